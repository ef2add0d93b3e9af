"""GPU parity of kv_append_quant against the oracle: cache bytes and scales
must be bit-exact (FP8 codes, fp32 page scales, INT4 nibbles, INT8 codes,
fp16 group scales, fp32 row scales), over exhaustive bf16 exponent bands,
multi-step verify histories with scale growth, and the error paths."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import bf16_dev, cache_to_host, i32_dev

pytestmark = pytest.mark.gpu
PAGE = 64
ALL_KV = [synth.KV_FP8, synth.KV_INT4, synth.KV_INT8, synth.KV_FP8_ROW]


def _sdva():
    import speculative_decode_verify_append_gb300 as sdva
    return sdva


def _assert_cache_equal(gcache, ocache, what=""):
    g = cache_to_host(gcache)
    for n in ("k_codes", "v_codes", "k_scales", "v_scales"):
        want = getattr(ocache, n)
        got = g[n]
        if got.dtype == np.float16:
            got = got.view(np.uint16)
        if got.dtype == np.float32:
            got, want = got.view(np.uint32), want.view(np.uint32)
        diff = np.argwhere(got != want)
        assert diff.size == 0, f"{what} {n}: {len(diff)} differing entries, first {diff[:5].tolist()}"


def _band_block(rng, e_top, shape):
    """bf16 patterns whose exponent lies in [e_top-8, e_top]: every such
    pattern (both signs, all mantissas) once, the rest random in the band."""
    n = int(np.prod(shape))
    exps = np.arange(e_top - 8, e_top + 1)
    exps = exps[(exps >= 1) & (exps <= 254)]  # biased bf16 exponents, finite and normal
    allp = (exps[:, None] << 7) | np.arange(128)[None, :]
    allp = np.concatenate([allp.reshape(-1), (allp | 0x8000).reshape(-1)]).astype(np.uint16)
    if e_top - 8 < 1:  # include subnormals and zeros of both signs
        sub = np.arange(128, dtype=np.uint16)
        allp = np.concatenate([allp, sub, sub | 0x8000])
    rest = rng.choice(allp, size=max(0, n - allp.size))
    out = np.concatenate([allp, rest])[:n]
    return rng.permutation(out).reshape(shape).astype(np.uint16)


@pytest.mark.parametrize("dtype", ALL_KV)
def test_exhaustive_bf16_bands(dtype):
    sdva = _sdva()
    Hkv = 4
    rng = np.random.default_rng(1234)
    bands = list(range(1, 255))  # every biased exponent as the top of a band
    blocks_per_page = Hkv * 2
    NP = (len(bands) + blocks_per_page - 1) // blocks_per_page
    k = np.zeros((1, NP * PAGE, Hkv, 128), np.uint16)
    v = np.zeros_like(k)
    for idx, e_top in enumerate(bands):
        p, rem = divmod(idx, blocks_per_page)
        h, kv = divmod(rem, 2)
        blk = _band_block(rng, e_top, (PAGE, 128))
        (v if kv else k)[0, p * PAGE:(p + 1) * PAGE, h] = blk
    table = np.arange(NP, dtype=np.int32)[None]
    gcache = sdva.KVCache(dtype, NP, Hkv)
    ocache = oracle.Cache(dtype, NP, Hkv)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sdva.kv_append_quant(gcache, bf16_dev(k), bf16_dev(v), i32_dev(table), i32_dev(np.zeros(1)), status)
    assert oracle.append(ocache, k, v, table, np.zeros(1, np.int32)) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    _assert_cache_equal(gcache, ocache, "bands")


@pytest.mark.parametrize("dtype", ALL_KV)
def test_growth_reencode_bands(dtype):
    """Half a page at a small scale, then the other half at scales up to 2^40
    larger: every earlier code is re-encoded (FP8)."""
    sdva = _sdva()
    Hkv = 2
    rng = np.random.default_rng(99)
    NP = 16
    table = rng.permutation(NP).astype(np.int32)[None]
    gcache = sdva.KVCache(dtype, NP, Hkv)
    ocache = oracle.Cache(dtype, NP, Hkv)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    L = 0
    for step in range(NP * 2):
        e_top = 60 + (step * 37) % 130
        k = _band_block(rng, e_top, (1, 32, Hkv, 128))
        v = _band_block(rng, e_top + 3, (1, 32, Hkv, 128))
        sdva.kv_append_quant(gcache, bf16_dev(k), bf16_dev(v), i32_dev(table), i32_dev(np.array([L])), status)
        assert oracle.append(ocache, k, v, table, np.array([L], np.int32)) == 0
        L += 32
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    _assert_cache_equal(gcache, ocache, "growth")


@pytest.mark.parametrize("dtype", ALL_KV)
@pytest.mark.parametrize("W", [1, 5, 16])
def test_verify_history_bit_exact(dtype, W):
    """Many verify steps with random accept lengths (rejected slots are
    overwritten next step), lanes crossing page boundaries, permuted table."""
    sdva = _sdva()
    B, Hkv, steps = 5, 3, 12
    rng = np.random.default_rng(W * 10 + dtype)
    L = np.array([0, 63, 64, 130, 1000][:B], np.int32)
    need = int((L.max() + steps * W + W + 63) // 64)
    table = rng.permutation(need * B).astype(np.int32).reshape(B, need)
    gcache = sdva.KVCache(dtype, need * B, Hkv)
    ocache = oracle.Cache(dtype, need * B, Hkv)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    spec = synth.Spec("h", 7, B, 0, 0, Hkv, Hkv, W, dtype, 64, 0.7, True)
    for b in range(B):
        if L[b]:
            k, v = synth.context_chunk(spec, b, 0, int(L[b]))
            sdva.kv_append_quant(gcache, bf16_dev(k[None]), bf16_dev(v[None]), i32_dev(table[b:b + 1]),
                                 i32_dev(np.zeros(1)), status)
            oracle.append(ocache, k[None], v[None], table[b:b + 1], np.zeros(1, np.int32))
    for s in range(steps):
        k = synth.normal_bf16(rng, (B, W, Hkv, 128))
        v = synth.normal_bf16(rng, (B, W, Hkv, 128))
        if s % 4 == 2:
            k[:, :, :, 3] = synth.to_bf16_bits(np.float32(30.0 + s) * np.ones((B, W, Hkv), np.float32))
        sdva.kv_append_quant(gcache, bf16_dev(k), bf16_dev(v), i32_dev(table), i32_dev(L), status)
        oracle.append(ocache, k, v, table, L)
        L = L + 1 + rng.integers(0, W, size=B).astype(np.int32)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    _assert_cache_equal(gcache, ocache, f"history W={W}")


def test_error_lanes_flagged_and_untouched():
    sdva = _sdva()
    Hkv = 1
    gcache = sdva.KVCache(synth.KV_FP8, 4, Hkv)
    k = synth.normal_bf16(np.random.default_rng(0), (3, 4, Hkv, 128))
    table = np.array([[0, 1], [2, 9], [3, 3]], np.int32)  # lane 1 maps a page past num_pages
    L = np.array([10, 62, 126], np.int32)  # lane 2 overflows its 2-page row
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sdva.kv_append_quant(gcache, bf16_dev(k), bf16_dev(k), i32_dev(table), i32_dev(L), status)
    torch.cuda.synchronize()
    assert int(status.item()) == 3
    codes = gcache.k_codes.cpu().numpy()
    assert codes[0, 0, 10:14].any()          # lane 0 written
    assert not codes[2:].any()               # lanes 1, 2 untouched
    status.zero_()
    sdva.kv_append_quant(gcache, bf16_dev(k[:1]), bf16_dev(k[:1]), i32_dev(table[:1]), i32_dev(np.array([-5])),
                         status)
    torch.cuda.synchronize()
    assert int(status.item()) == 2


def test_host_argument_errors():
    sdva = _sdva()
    gcache = sdva.KVCache(synth.KV_FP8, 2, 1)
    k = bf16_dev(np.zeros((1, 1, 1, 128), np.uint16))
    t = i32_dev(np.zeros((1, 2)))
    with pytest.raises(sdva.SdvaError) as e:
        sdva.kv_append_quant(gcache, k[:, :0], k[:, :0], t, i32_dev(np.zeros(1)))
    assert e.value.code == sdva.ERR_INVALID


# ---- per-lane token counts -------------------------------------------------

@pytest.mark.parametrize("dtype", ALL_KV)
def test_ragged_append_history_parity(dtype):
    sdva = _sdva()
    rng = np.random.default_rng(77 + dtype)
    B, W, H, steps = 5, 16, 4, 8
    L = np.array([0, 5, 63, 64, 130], np.int32)
    need = (int(L.max()) + steps * W + W + PAGE - 1) // PAGE
    table = rng.permutation(need * B).astype(np.int32).reshape(B, need)
    gcache = sdva.KVCache(dtype, need * B, H)
    ocache = oracle.Cache(dtype, need * B, H)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    tdev = i32_dev(table)
    for b in range(B):  # starting context, one plain append per lane
        if L[b]:
            k = synth.normal_bf16(rng, (1, int(L[b]), H, 128))
            sdva.kv_append_quant(gcache, bf16_dev(k), bf16_dev(k), tdev[b:b + 1], i32_dev(np.zeros(1)), st)
            assert oracle.append(ocache, k, k, table[b:b + 1], np.zeros(1, np.int32)) == 0
    for s in range(steps):
        k = synth.normal_bf16(rng, (B, W, H, 128))
        v = synth.normal_bf16(rng, (B, W, H, 128))
        if s == 3:  # padding past lane 1's count is huge: it must not reach the page scale
            k[1, 2:, :, :] = synth.to_bf16_bits(np.array([3.0e4], np.float32))[0]
        if s == 5:  # a large token inside lane 2's count forces a growth re-encode
            v[2, 0, 3, 11] = synth.to_bf16_bits(np.array([-500.0], np.float32))[0]
        n = rng.integers(0, W + 1, size=B).astype(np.int32)
        n[s % B] = 0
        n[(s + 1) % B] = W
        if s == 3:
            n[1] = 2
        sdva.kv_append_quant_ragged(gcache, bf16_dev(k), bf16_dev(v), i32_dev(n), tdev, i32_dev(L), st)
        assert oracle.append_ragged(ocache, k, v, table, L, n) == 0
        L = L + rng.integers(0, n + 1).astype(np.int32)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    _assert_cache_equal(gcache, ocache, "ragged history")


def test_ragged_invalid_and_empty_counts():
    sdva = _sdva()
    rng = np.random.default_rng(78)
    B, W, H = 3, 4, 1
    table = np.array([[0, 1], [2, 3], [-5, 4]], np.int32)  # lane 2 has a bad page id
    L = np.array([0, 10, 0], np.int32)
    k = synth.normal_bf16(rng, (B, W, H, 128))
    gcache = sdva.KVCache(synth.KV_FP8, 5, H)
    ocache = oracle.Cache(synth.KV_FP8, 5, H)
    for n in (np.array([W + 1, -1, 0], np.int32), np.array([2, 0, 1], np.int32)):
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        sdva.kv_append_quant_ragged(gcache, bf16_dev(k), bf16_dev(k), i32_dev(n), i32_dev(table), i32_dev(L), st)
        torch.cuda.synchronize()
        assert int(st.item()) == oracle.append_ragged(ocache, k, k, table, L, n)
        _assert_cache_equal(gcache, ocache, f"counts {n.tolist()}")
