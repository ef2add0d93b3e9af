"""GPU parity of the INT8 group-64 and FP8 row-scale cache formats beyond the
shared small cases: tokens whose magnitudes differ by powers of two inside a
page (per-token scales are the point of both formats), pages whose rows past
the lane's tokens hold a previous lane's much larger rows, per-lane window
row counts, and the host-side limits of the two formats."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import ALL_KV, KV_NAMES, SM_SCALE, assert_close, assert_close_row_scaled, bf16_dev, i32_dev

pytestmark = pytest.mark.gpu
PAGE = 64


def _sdva():
    import speculative_decode_verify_append_gb300 as sdva
    return sdva


def _scaled(rng, shape, lo, hi):
    """Normal bf16 rows, each (token, head) row multiplied by 2^u with an
    integer u drawn from [lo, hi] (exact in bf16)."""
    x = synth.bf16_to_f32(synth.normal_bf16(rng, shape))
    u = rng.integers(lo, hi + 1, size=shape[:-1] + (1,)).astype(np.float32)
    return synth.to_bf16_bits(x * np.exp2(u))


def _append_both(gcache, ocache, k, v, table, L, status):
    sdva = _sdva()
    sdva.kv_append_quant(gcache, bf16_dev(k), bf16_dev(v), i32_dev(table), i32_dev(L), status)
    assert oracle.append(ocache, k, v, table, np.asarray(L, np.int32)) == 0


def _verify(gcache, q, table, L, Hkv, max_context):
    sdva = _sdva()
    B, W, Hq = q.shape[:3]
    out = torch.full((B, W, Hq, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(sdva.verify_attn_workspace_size(B, W, Hq, Hkv, max_context), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    sdva.verify_attn(gcache, bf16_dev(q), i32_dev(table), i32_dev(L), max_context, float(SM_SCALE), out, ws, st)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), int(st.item())


@pytest.mark.parametrize("dtype", ALL_KV, ids=lambda d: KV_NAMES[d])
def test_token_magnitudes_spread_inside_pages(dtype):
    """K rows scaled by 2^[-2, 1] and V rows by 2^[-6, 6], token by token: the
    V row scales of a page then span up to 2^12, inside the 2^14 that the
    FP8-row path widens to fp16 at full precision.  (The K spread stays
    small: the FP8 formats carry Q as two E4M3 terms, about bf16 precision,
    and larger keys sharpen the softmax's sensitivity to that.)  The bound's
    absolute term follows each output row's scale (assert_close_row_scaled):
    with V rows up to 2^6 times larger than the unit-scale data of the other
    tests, every format -- FP8 page scales included -- leaves errors of a
    few 1e-4 of the row's largest element on elements that cancel."""
    sdva = _sdva()
    rng = np.random.default_rng(2024 + dtype)
    lens, W, Hq, Hkv = np.array([300, 1000, 64], np.int32), 8, 24, 4
    B = len(lens)
    need = (int(lens.max()) + W + PAGE - 1) // PAGE
    table = rng.permutation(need * B).astype(np.int32).reshape(B, need)
    gcache = sdva.KVCache(dtype, need * B, Hkv)
    ocache = oracle.Cache(dtype, need * B, Hkv)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    for b in range(B):
        n = int(lens[b])
        k, v = _scaled(rng, (1, n, Hkv, 128), -2, 1), _scaled(rng, (1, n, Hkv, 128), -6, 6)
        _append_both(gcache, ocache, k, v, table[b:b + 1], [0], st)
    kw, vw = _scaled(rng, (B, W, Hkv, 128), -2, 1), _scaled(rng, (B, W, Hkv, 128), -6, 6)
    _append_both(gcache, ocache, kw, vw, table, lens, st)
    q = synth.normal_bf16(rng, (B, W, Hq, 128))
    got, status = _verify(gcache, q, table, lens, Hkv, int(lens.max()))
    assert status == 0 and int(st.item()) == 0
    want, ost = oracle.verify_attn(ocache, q, table, lens, SM_SCALE, threads=8)
    assert ost == 0
    worst = assert_close_row_scaled(got, want, f"spread {KV_NAMES[dtype]}")
    print(f"spread {KV_NAMES[dtype]}: max error / row scale {worst:.3g}")


@pytest.mark.parametrize("dtype", ALL_KV, ids=lambda d: KV_NAMES[d])
def test_rows_past_the_lane_hold_larger_stale_rows(dtype):
    """A lane reuses pages that an earlier lane filled with rows 2^10 times
    larger; the rows past its own tokens keep those codes and scales.  They
    are invisible, and must not change (or overflow) the visible result: for
    FP8 row scales the page's largest V row scale is taken over the lane's
    written rows only, and the other rows are widened to zero."""
    sdva = _sdva()
    rng = np.random.default_rng(77 + dtype)
    Hq, Hkv, W = 8, 2, 8
    table = np.array([[3, 1, 4]], np.int32)
    gcache = sdva.KVCache(dtype, 5, Hkv)
    ocache = oracle.Cache(dtype, 5, Hkv)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    big = 3 * PAGE
    _append_both(gcache, ocache, _scaled(rng, (1, big, Hkv, 128), 10, 10), _scaled(rng, (1, big, Hkv, 128), 10, 10),
                 table, [0], st)
    for L in (60, 64 + 57, 5):  # the window ends inside page 1, inside page 2 (57 + 8 > 64), inside page 0
        k, v = synth.normal_bf16(rng, (1, L, Hkv, 128)), synth.normal_bf16(rng, (1, L, Hkv, 128))
        _append_both(gcache, ocache, k, v, table, [0], st)
        kw, vw = synth.normal_bf16(rng, (1, W, Hkv, 128)), synth.normal_bf16(rng, (1, W, Hkv, 128))
        _append_both(gcache, ocache, kw, vw, table, [L], st)
        q = synth.normal_bf16(rng, (1, W, Hq, 128))
        got, status = _verify(gcache, q, table, np.array([L], np.int32), Hkv, L)
        assert status == 0 and int(st.item()) == 0
        assert np.isfinite(got).all()
        want, _ = oracle.verify_attn(ocache, q, table, np.array([L], np.int32), SM_SCALE, threads=4)
        assert_close(got, want, f"stale rows L={L} {KV_NAMES[dtype]}")


@pytest.mark.parametrize("dtype", [synth.KV_INT8, synth.KV_FP8_ROW], ids=lambda d: KV_NAMES[d])
def test_ragged_rows_new_formats(dtype):
    """verify_attn_ragged: rows past each lane's count are zero, the others
    match the oracle (a zero count, a full lane, a count in between)."""
    sdva = _sdva()
    rng = np.random.default_rng(31 + dtype)
    lens, W, Hq, Hkv = np.array([900, 64, 5, 2000], np.int32), 16, 8, 1
    B = len(lens)
    spec = synth.Spec("rf", 12, B, 0, 0, Hq, Hkv, W, dtype, None, 0.7, True)
    step = synth.make_step(spec, seq_lens=lens, with_accept=False)
    from gpu_util import fill_both
    g, o, _ = fill_both(spec, step, chunk=512)
    n = np.array([3, 16, 0, 9], np.int32)
    out = torch.full((B, W, Hq, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(sdva.verify_attn_workspace_size(B, W, Hq, Hkv, int(lens.max())), dtype=torch.uint8,
                     device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    sdva.verify_attn_ragged(g, bf16_dev(step.q), i32_dev(n), i32_dev(step.page_table), i32_dev(lens),
                            int(lens.max()), float(SM_SCALE), out, ws, st)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy()
    assert int(st.item()) == 0
    want, _ = oracle.verify_attn_ragged(o, step.q, step.page_table, lens, n, SM_SCALE, threads=8)
    for b in range(B):
        assert not got[b, n[b]:].any()
        assert_close(got[b, :n[b]], want[b, :n[b]], f"lane {b}")


@pytest.mark.parametrize("dtype", [synth.KV_INT8, synth.KV_FP8_ROW], ids=lambda d: KV_NAMES[d])
def test_more_than_128_rows_per_kv_head_is_unsupported(dtype):
    sdva = _sdva()
    g = sdva.KVCache(dtype, 2, 1)
    q = torch.zeros((1, 16, 16, 128), dtype=torch.bfloat16, device="cuda")  # 256 rows on one kv head
    t = torch.zeros((1, 2), dtype=torch.int32, device="cuda")
    L = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(1 << 22, dtype=torch.uint8, device="cuda")
    with pytest.raises(sdva.SdvaError) as e:
        sdva.verify_attn(g, q, t, L, 64, 0.088, q.clone(), ws)
    assert e.value.code == sdva.ERR_UNSUPPORTED
