"""The three calls together, as a serving loop issues them: several verify
steps with commits (append -> verify_attn -> spec_accept), checked against
the oracle replaying the same steps; CUDA-graph replay of a step; and
checkpoint / restore of the caller-owned state."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import SM_SCALE, assert_close, bf16_dev, fill_both, i32_dev

pytestmark = pytest.mark.gpu


def _sdva():
    import speculative_decode_verify_append_gb300 as sdva
    from speculative_decode_verify_append_gb300.step import VerifyStep
    return sdva, VerifyStep


@pytest.mark.parametrize("dtype", [synth.KV_FP8, synth.KV_INT4, synth.KV_INT8, synth.KV_FP8_ROW])
def test_multi_step_loop_matches_oracle(dtype):
    sdva, VerifyStep = _sdva()
    W, Hq, Hkv, V = 6, 12, 2, 3000
    lens = np.array([100, 640, 1333], np.int32)
    steps = 5
    spec = synth.Spec("loop", 11, 3, 0, 0, Hq, Hkv, W, dtype, V, 0.7, True)
    # capacity for all steps
    table, total = synth.page_table_for(spec, lens + steps * W, W)
    step0 = synth.make_step(spec, seq_lens=lens, with_accept=False)
    step0.page_table, step0.num_pages = table, total
    gcache, ocache, st = fill_both(spec, step0, chunk=256)  # includes step 0's window append
    vs = VerifyStep(3, W, Hq, Hkv, int(lens.max()) + steps * W, V)
    L_host = lens.copy()
    L_dev = i32_dev(lens)
    tdev = i32_dev(table)
    for s in range(steps):
        stp = synth.make_step(spec, seq_lens=L_host, tag=f"s{s}")
        if s > 0:  # step 0's window is already appended by fill_both
            vs.append(gcache, bf16_dev(stp.k_win), bf16_dev(stp.v_win), tdev, L_dev)
            assert oracle.append(ocache, stp.k_win, stp.v_win, table, L_host) == 0
        vs.attend(gcache, bf16_dev(stp.q), tdev, L_dev)
        vs.accept(torch.from_numpy(stp.logits).cuda(), i32_dev(stp.drafts), L_dev)
        torch.cuda.synchronize()
        want, _ = oracle.verify_attn(ocache, stp.q, table, L_host, SM_SCALE, threads=8)
        assert_close(vs.out.float().cpu().numpy(), want, f"step {s}")
        acc, tok, newL, _ = oracle.spec_accept(stp.logits, stp.drafts, L_host)
        assert np.array_equal(vs.accept_len.cpu().numpy(), acc)
        assert np.array_equal(vs.out_tokens.cpu().numpy(), tok)
        assert np.array_equal(L_dev.cpu().numpy(), newL)
        L_host = newL
    assert int(vs.status.item()) == 0
    g = {n: getattr(gcache, n).cpu().numpy() for n in ("k_codes", "v_codes")}
    assert np.array_equal(g["k_codes"], ocache.k_codes) and np.array_equal(g["v_codes"], ocache.v_codes)


@pytest.mark.parametrize("dtype", [synth.KV_FP8, synth.KV_INT4, synth.KV_INT8, synth.KV_FP8_ROW])
def test_ragged_step_loop_matches_oracle(dtype):
    """Lanes with their own draft counts d_b in one padded window: the ragged
    append writes 1 + d_b tokens per lane, verify rows 0 .. d_b are compared,
    verify_attn_ragged gives the same rows bit for bit and zeros past each
    count (every row against the oracle), and the lazy acceptance uses the
    same counts."""
    sdva, VerifyStep = _sdva()
    W, Hq, Hkv, V = 8, 12, 2, 3000
    lens = np.array([70, 640, 1333, 5], np.int32)
    B, steps = len(lens), 5
    spec = synth.Spec("ragged", 12, B, 0, 0, Hq, Hkv, W, dtype, V, 0.8, True)
    table, total = synth.page_table_for(spec, lens + steps * W, W)
    step0 = synth.make_step(spec, seq_lens=lens, with_accept=False)
    step0.page_table, step0.num_pages = table, total
    # the starting contexts (every window, step 0's included, goes through the ragged append)
    gcache = sdva.KVCache(dtype, total, Hkv)
    ocache = oracle.Cache(dtype, total, Hkv)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    tdev = i32_dev(table)
    for b, L in enumerate(lens):
        for start, n in synth.fill_chunks(int(L), 256):
            k, v = synth.context_chunk(spec, b, start, n)
            sdva.kv_append_quant(gcache, bf16_dev(k[None]), bf16_dev(v[None]), tdev[b:b + 1],
                                 i32_dev(np.array([start])), st)
            assert oracle.append(ocache, k[None], v[None], table[b:b + 1], np.array([start], np.int32)) == 0
    vs = VerifyStep(B, W, Hq, Hkv, int(lens.max()) + steps * W, V)
    rng = np.random.default_rng(13)
    L_host, L_dev = lens.copy(), i32_dev(lens)
    for s in range(steps):
        stp = synth.make_step(spec, seq_lens=L_host, tag=f"r{s}")
        d = rng.integers(0, W, size=B).astype(np.int32)
        d[s % B] = W - 1
        d[(s + 2) % B] = 0
        vs.append_ragged(gcache, bf16_dev(stp.k_win), bf16_dev(stp.v_win), i32_dev(d + 1), tdev, L_dev)
        assert oracle.append_ragged(ocache, stp.k_win, stp.v_win, table, L_host, d + 1) == 0
        vs.attend(gcache, bf16_dev(stp.q), tdev, L_dev)
        q_dev = bf16_dev(stp.q)
        out_r = torch.full_like(vs.out, float("nan"))
        sdva.verify_attn_ragged(gcache, q_dev, i32_dev(d + 1), tdev, L_dev, vs.max_context, vs.sm_scale, out_r,
                                vs.workspace, vs.status)
        vs.accept_lazy(torch.from_numpy(stp.logits).cuda(), i32_dev(stp.drafts), i32_dev(d), L_dev)
        torch.cuda.synchronize()
        want, _ = oracle.verify_attn(ocache, stp.q, table, L_host, SM_SCALE, threads=8)
        got = vs.out.float().cpu().numpy()
        for b in range(B):  # rows past a lane's count attend to padding: not compared
            assert_close(got[b, :d[b] + 1], want[b, :d[b] + 1], f"step {s} lane {b}")
        # the ragged verify: every row, the ones past a lane's count zero
        want_r, st_r = oracle.verify_attn_ragged(ocache, stp.q, table, L_host, d + 1, SM_SCALE, threads=8)
        assert st_r == 0
        got_r = out_r.float().cpu().numpy()
        assert_close(got_r, want_r, f"ragged verify step {s}")
        for b in range(B):
            assert not got_r[b, d[b] + 1:].any()
            assert np.array_equal(got_r[b, :d[b] + 1], got[b, :d[b] + 1])
        acc, tok, newL, _ = oracle.spec_accept_lazy(stp.logits, stp.drafts, d, L_host)
        assert np.array_equal(vs.accept_len.cpu().numpy(), acc)
        assert np.array_equal(vs.out_tokens.cpu().numpy(), tok)
        assert np.array_equal(L_dev.cpu().numpy(), newL)
        L_host = newL
    assert int(vs.status.item()) == 0
    for n in ("k_codes", "v_codes", "k_scales", "v_scales"):
        g = getattr(gcache, n).cpu().numpy()
        w = getattr(ocache, n)
        assert np.array_equal(g.view(np.uint8), w.view(np.uint8)), n


def test_cuda_graph_replay_matches_eager():
    sdva, VerifyStep = _sdva()
    spec = synth.WORKLOADS["multi_lane"]
    lens = np.array([4096, 700, 9000, 64], np.int32)
    spec = synth.Spec("g", 3, 4, 0, 0, 24, 4, 16, synth.KV_FP8, 151936, 0.7, True)
    stp = synth.make_step(spec, seq_lens=lens)
    gcache, _, _ = fill_both(spec, stp, with_oracle=False)
    vs = VerifyStep(4, 16, 24, 4, 9000, 151936)
    q, t, L = bf16_dev(stp.q), i32_dev(stp.page_table), i32_dev(lens)
    lg, dr = torch.from_numpy(stp.logits).cuda(), i32_dev(stp.drafts)
    kw, vw = bf16_dev(stp.k_win), bf16_dev(stp.v_win)
    vs.run(gcache, q, kw, vw, t, L, lg, dr, commit=False)
    torch.cuda.synchronize()
    eager = (vs.out.clone(), vs.accept_len.clone(), vs.out_tokens.clone())
    vs.out.zero_()
    vs.accept_len.zero_()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            vs.run(gcache, q, kw, vw, t, L, lg, dr, commit=False, stream=s)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(vs.out, eager[0])
    assert torch.equal(vs.accept_len, eager[1]) and torch.equal(vs.out_tokens, eager[2])


def test_checkpoint_restore_continues_identically():
    sdva, VerifyStep = _sdva()
    W = 4
    lens = np.array([500, 90], np.int32)
    spec = synth.Spec("ck", 21, 2, 0, 0, 8, 2, W, synth.KV_FP8, 500, 0.7, True)
    table, total = synth.page_table_for(spec, lens + 3 * W, W)
    s0 = synth.make_step(spec, seq_lens=lens, with_accept=False)
    s0.page_table, s0.num_pages = table, total
    gcache, _, _ = fill_both(spec, s0, with_oracle=False)
    vs = VerifyStep(2, W, 8, 2, 600, 500)
    tdev = i32_dev(table)
    L = i32_dev(lens)

    def one_step(tag):
        L_host = L.cpu().numpy()
        stp = synth.make_step(spec, seq_lens=L_host, tag=tag)
        vs.run(gcache, bf16_dev(stp.q), bf16_dev(stp.k_win), bf16_dev(stp.v_win), tdev, L,
               torch.from_numpy(stp.logits).cuda(), i32_dev(stp.drafts))
        torch.cuda.synchronize()
        return vs.out.clone(), vs.accept_len.clone()

    one_step("a")
    saved = [x.clone() for x in (gcache.k_codes, gcache.v_codes, gcache.k_scales, gcache.v_scales, L)]
    first = [one_step("b"), one_step("c")]
    for dst, src in zip((gcache.k_codes, gcache.v_codes, gcache.k_scales, gcache.v_scales, L), saved):
        dst.copy_(src)
    second = [one_step("b"), one_step("c")]
    for (o1, a1), (o2, a2) in zip(first, second):
        assert torch.equal(o1, o2) and torch.equal(a1, a2)


@pytest.mark.parametrize("dtype", [synth.KV_FP8, synth.KV_INT4, synth.KV_INT8, synth.KV_FP8_ROW])
def test_verify_step_equals_the_three_calls(dtype):
    """verify_step (the chained launch) leaves the same cache bytes, attention
    rows, accept lengths, tokens, committed lengths and status as
    kv_append_quant, verify_attn and spec_accept called in order -- bit for
    bit -- over three steps, with and without the commit."""
    sdva, VerifyStep = _sdva()
    W, Hq, Hkv, V = 16 if dtype == synth.KV_FP8 else 8, 24, 4, 151936
    lens = np.array([4096, 700, 9000, 64, 33000, 5], np.int32)
    B = len(lens)
    spec = synth.Spec("chain", 14 + dtype, B, 0, 0, Hq, Hkv, W, dtype, V, 0.7, True)
    table, total = synth.page_table_for(spec, lens + 3 * W, W)
    caches = []
    for _ in range(2):
        g = sdva.KVCache(dtype, total, Hkv)
        tdev = i32_dev(table)
        for b, L in enumerate(lens):
            for start, n in synth.fill_chunks(int(L), 4096):
                k, v = synth.context_chunk(spec, b, start, n)
                sdva.kv_append_quant(g, bf16_dev(k[None]), bf16_dev(v[None]), tdev[b:b + 1],
                                     i32_dev(np.array([start])))
        caches.append(g)
    va, vb = (VerifyStep(B, W, Hq, Hkv, int(lens.max()) + 3 * W, V) for _ in range(2))
    La, Lb = i32_dev(lens), i32_dev(lens)
    tdev = i32_dev(table)
    L_host = lens.copy()
    for s in range(3):
        stp = synth.make_step(spec, seq_lens=L_host, tag=f"c{s}")
        q, kw, vw = bf16_dev(stp.q), bf16_dev(stp.k_win), bf16_dev(stp.v_win)
        lg, dr = torch.from_numpy(stp.logits).cuda(), i32_dev(stp.drafts)
        commit = s != 1
        va.run(caches[0], q, kw, vw, tdev, La, lg, dr, commit=commit)
        vb.step(caches[1], q, kw, vw, tdev, Lb, lg, dr, commit=commit)
        torch.cuda.synchronize()
        for x, y, name in ((va.out, vb.out, "out"), (va.accept_len, vb.accept_len, "accept_len"),
                           (va.out_tokens, vb.out_tokens, "out_tokens"), (La, Lb, "seq_lens"),
                           (va.status, vb.status, "status")):
            assert torch.equal(x, y), (s, name)
        L_host = La.cpu().numpy()
    assert int(va.status.item()) == 0
    for n in ("k_codes", "v_codes", "k_scales", "v_scales"):
        assert torch.equal(getattr(caches[0], n), getattr(caches[1], n)), n


def test_verify_step_in_a_cuda_graph():
    """verify_step captures and replays in a CUDA graph with the eager results."""
    sdva, VerifyStep = _sdva()
    lens = np.array([4096, 700, 9000, 64], np.int32)
    spec = synth.Spec("g2", 3, 4, 0, 0, 24, 4, 16, synth.KV_FP8, 151936, 0.7, True)
    stp = synth.make_step(spec, seq_lens=lens)
    gcache, _, _ = fill_both(spec, stp, with_oracle=False)
    vs = VerifyStep(4, 16, 24, 4, 9000, 151936)
    q, t, L = bf16_dev(stp.q), i32_dev(stp.page_table), i32_dev(lens)
    lg, dr = torch.from_numpy(stp.logits).cuda(), i32_dev(stp.drafts)
    kw, vw = bf16_dev(stp.k_win), bf16_dev(stp.v_win)
    vs.step(gcache, q, kw, vw, t, L, lg, dr, commit=False)
    torch.cuda.synchronize()
    eager = (vs.out.clone(), vs.accept_len.clone(), vs.out_tokens.clone())
    vs.out.zero_()
    vs.accept_len.zero_()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            vs.step(gcache, q, kw, vw, t, L, lg, dr, commit=False, stream=s)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(vs.out, eager[0]) and torch.equal(vs.accept_len, eager[1])
    assert torch.equal(vs.out_tokens, eager[2])
    assert int(vs.status.item()) == 0


@pytest.mark.parametrize("V,W,Hq,Hkv,offset", [
    (151936, 16, 24, 4, 0),   # 96 rows per kv head, vector loads of the logits
    (32003, 8, 8, 1, 0),      # odd vocab: scalar loads
    (4096, 8, 16, 2, 1),      # rows not 16-byte aligned: scalar loads
    (4, 4, 8, 8, 0),          # one float4 per row
    (151937, 16, 32, 4, 0),   # 128 rows per kv head
], ids=["vec", "odd", "unaligned", "v4", "r128"])
def test_verify_step_argmax_on_hostile_logits(V, W, Hq, Hkv, offset):
    """verify_step's acceptance on logits with heavy ties, NaN rows and
    half-NaN rows, signed zeros and -inf rows, on lanes so short that most
    CTAs of the split kernel have no pages: tokens, accept lengths and
    committed lengths equal the oracle's exactly, and the attention rows
    equal the three calls' bit for bit."""
    sdva, VerifyStep = _sdva()
    lens = np.array([5, 64, 130, 1], np.int32)
    B = len(lens)
    rng = np.random.default_rng(V + W)
    spec = synth.Spec("hostile", 5, B, 0, 0, Hq, Hkv, W, synth.KV_FP8, V, 0.7, True)
    table, total = synth.page_table_for(spec, lens + W, W)
    stp = synth.make_step(spec, seq_lens=lens, with_accept=False)
    stp.page_table, stp.num_pages = table, total
    caches = [fill_both(spec, stp, with_oracle=False)[0] for _ in range(2)]
    logits = rng.integers(-2, 3, size=(B, W, V)).astype(np.float32)
    logits[0, 0, :] = np.nan
    logits[1, 1, : V // 2] = np.nan
    logits[2, 2, :] = -0.0
    logits[2, 2, V - 1] = 0.0
    logits[3, 3, :] = -np.inf
    drafts = np.argmax(np.nan_to_num(logits, nan=-9.0), axis=2)[:, :W - 1].astype(np.int32)
    drafts[1, 2] = (drafts[1, 2] + 1) % V  # one lane rejects in the middle
    flat = torch.from_numpy(logits.reshape(-1))
    buf = torch.empty(flat.numel() + offset, dtype=torch.float32, device="cuda")
    lg = buf[offset:].view(logits.shape)
    lg.copy_(flat.view(logits.shape))
    dr = i32_dev(drafts)
    tdev = i32_dev(table)
    q, kw, vw = bf16_dev(stp.q), bf16_dev(stp.k_win), bf16_dev(stp.v_win)
    va, vb = (VerifyStep(B, W, Hq, Hkv, int(lens.max()) + W, V) for _ in range(2))
    La, Lb = i32_dev(lens), i32_dev(lens)
    # both caches hold the window already (fill_both); both sides append it again
    va.run(caches[0], q, kw, vw, tdev, La, lg, dr, commit=True)
    vb.step(caches[1], q, kw, vw, tdev, Lb, lg, dr, commit=True)
    torch.cuda.synchronize()
    acc, tok, newL, st = oracle.spec_accept(logits, drafts, lens)
    assert np.array_equal(vb.out_tokens.cpu().numpy(), tok)
    assert np.array_equal(vb.accept_len.cpu().numpy(), acc)
    assert np.array_equal(Lb.cpu().numpy(), newL)
    assert int(vb.status.item()) == st == 0
    assert torch.equal(va.out, vb.out)
    assert torch.equal(va.out_tokens, vb.out_tokens) and torch.equal(va.accept_len, vb.accept_len)
    assert torch.equal(La, Lb)
