"""Pins for the oracle's verify attention (no GPU).

Checked against: the brute-force pure-Python statement (its own cache,
its own attention with math.fsum); PyTorch's fp64 softmax on caches
dequantised through PyTorch's float8_e4m3fn table; the oracle's separately
written single-pass decode routine (window of 1); and closed forms and
invariants (page-table permutation, causality inside the window, Q = 0, an
empty context, one dominant key)."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from oracle import brute

PAGE = 64
SM = np.float32(1.0 / math.sqrt(128.0))
_E4M3 = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()


def build(dtype, lens, W, Hq, Hkv, seed=5, permuted=True, scale_k=None):
    spec = synth.Spec("t", seed, len(lens), 0, 0, Hq, Hkv, W, dtype, 64, 0.7, permuted)
    step = synth.make_step(spec, seq_lens=np.array(lens, np.int32), with_accept=False)
    cache = oracle.Cache(dtype, step.num_pages, Hkv)
    for b, L in enumerate(lens):
        for start, n in synth.fill_chunks(L, 100):
            k, v = synth.context_chunk(spec, b, start, n)
            if scale_k is not None:
                k = synth.to_bf16_bits(synth.bf16_to_f32(k) * scale_k)
            assert oracle.append(cache, k[None], v[None], step.page_table[b:b + 1],
                                 np.array([start], np.int32)) == 0
    assert oracle.append(cache, step.k_win, step.v_win, step.page_table, step.seq_lens) == 0
    return spec, step, cache


def dense(cache, table_row, n, kv):
    """Dequantised [Hkv][n][128] fp64 through the library E4M3 table / numpy fp16."""
    H = cache.num_kv_heads
    out = np.zeros((H, n, 128))
    for t in range(n):
        pid, off = table_row[t // PAGE], t % PAGE
        for h in range(H):
            if cache.dtype == oracle.KV_FP8:
                codes = (cache.v_codes if kv else cache.k_codes)[pid, h, off]
                s = float((cache.v_scales if kv else cache.k_scales)[pid, h])
                out[h, t] = _E4M3[codes] * s
            else:
                packed = (cache.v_codes if kv else cache.k_codes)[pid, h, off]
                lo = ((packed & 0xF).astype(np.int8) ^ 8) - 8
                hi = ((packed >> 4).astype(np.int8) ^ 8) - 8
                q = np.stack([lo, hi], 1).reshape(-1).astype(np.float64)
                sc = (cache.v_scales if kv else cache.k_scales)[pid, h, off].view(np.float16).astype(np.float64)
                out[h, t] = q * np.repeat(sc, 32)
    return out


def torch_reference(step, cache):
    B, W, Hq = step.q.shape[:3]
    G = Hq // cache.num_kv_heads
    out = np.zeros((B, W, Hq, 128))
    for b in range(B):
        L = int(step.seq_lens[b])
        K = torch.from_numpy(dense(cache, step.page_table[b], L + W, 0))
        V = torch.from_numpy(dense(cache, step.page_table[b], L + W, 1))
        q = torch.from_numpy(synth.bf16_to_f32(step.q[b]).astype(np.float64))
        for i in range(W):
            for h in range(Hq):
                s = (K[h // G, :L + i + 1] @ q[i, h]) * float(SM)
                out[b, i, h] = (torch.softmax(s, 0) @ V[h // G, :L + i + 1]).numpy()
    return out


@pytest.mark.parametrize("dtype", [oracle.KV_FP8, oracle.KV_INT4])
def test_verify_matches_torch_softmax(dtype):
    spec, step, cache = build(dtype, [70, 5, 130], 4, 6, 2)
    got, st = oracle.verify_attn(cache, step.q, step.page_table, step.seq_lens, SM)
    assert st == 0
    want = torch_reference(step, cache)
    assert np.abs(got - want).max() < 1e-12


@pytest.mark.parametrize("dtype", [oracle.KV_FP8, oracle.KV_INT4])
def test_verify_matches_brute(dtype):
    lens, W, Hq, Hkv = [66, 3], 3, 4, 2
    spec, step, cache = build(dtype, lens, W, Hq, Hkv, seed=9)
    got, st = oracle.verify_attn(cache, step.q, step.page_table, step.seq_lens, SM)
    # the brute statement builds its own cache from the same inputs
    bc = brute.Cache(dtype)
    for b, L in enumerate(lens):
        for start, n in synth.fill_chunks(L, 100):
            k, v = synth.context_chunk(spec, b, start, n)
            rows = [[[list(map(int, k[t, h])) for h in range(Hkv)] for t in range(n)],
                    [[list(map(int, v[t, h])) for h in range(Hkv)] for t in range(n)]]
            brute.append(bc, rows, list(step.page_table[b]), start)
        rows = [[[list(map(int, step.k_win[b, t, h])) for h in range(Hkv)] for t in range(W)],
                [[list(map(int, step.v_win[b, t, h])) for h in range(Hkv)] for t in range(W)]]
        brute.append(bc, rows, list(step.page_table[b]), L)
    G = Hq // Hkv
    for b, L in enumerate(lens):
        for i in range(W):
            for h in range(Hq):
                want = brute.attention_row(bc, list(map(int, step.q[b, i, h])), list(step.page_table[b]),
                                           h // G, L + i + 1, float(SM))
                assert np.abs(got[b, i, h] - np.array(want)).max() < 1e-12, (b, i, h)


def test_window_of_one_equals_plain_decode():
    spec, step, cache = build(oracle.KV_FP8, [1000, 64, 0], 1, 6, 2, seed=4)
    got, st = oracle.verify_attn(cache, step.q, step.page_table, step.seq_lens, SM)
    for b, L in enumerate(step.seq_lens):
        for h in range(6):
            want = oracle.decode_row(cache, step.q[b, 0, h], h // 3, step.page_table[b], int(L) + 1, SM)
            assert np.abs(got[b, 0, h] - want).max() < 1e-12


def test_page_table_permutation_invariance():
    lens, W = [300, 77], 5
    s1, step1, c1 = build(oracle.KV_FP8, lens, W, 4, 1, seed=2, permuted=False)
    s2, step2, c2 = build(oracle.KV_FP8, lens, W, 4, 1, seed=2, permuted=True)
    assert not np.array_equal(step1.page_table, step2.page_table)
    o1, _ = oracle.verify_attn(c1, step1.q, step1.page_table, step1.seq_lens, SM)
    o2, _ = oracle.verify_attn(c2, step2.q, step2.page_table, step2.seq_lens, SM)
    assert np.array_equal(o1, o2)


def test_causality_inside_window():
    lens, W = [100], 6
    spec, step, cache = build(oracle.KV_FP8, lens, W, 4, 2, seed=3)
    o1, _ = oracle.verify_attn(cache, step.q, step.page_table, step.seq_lens, SM)
    j = 3
    step.k_win[0, j] = synth.normal_bf16(np.random.default_rng(99), step.k_win[0, j].shape)
    step.v_win[0, j] = synth.normal_bf16(np.random.default_rng(98), step.v_win[0, j].shape)
    cache2 = oracle.Cache(oracle.KV_FP8, step.num_pages, 2)
    for start, n in synth.fill_chunks(100, 100):
        k, v = synth.context_chunk(spec, 0, start, n)
        oracle.append(cache2, k[None], v[None], step.page_table, np.array([start], np.int32))
    oracle.append(cache2, step.k_win, step.v_win, step.page_table, step.seq_lens)
    o2, _ = oracle.verify_attn(cache2, step.q, step.page_table, step.seq_lens, SM)
    assert np.array_equal(o1[:, :j], o2[:, :j])
    assert not np.array_equal(o1[:, j:], o2[:, j:])


def test_zero_query_gives_mean_of_values():
    lens, W = [90, 10], 3
    spec, step, cache = build(oracle.KV_INT4, lens, W, 4, 2, seed=8)
    step.q[:] = 0
    got, _ = oracle.verify_attn(cache, step.q, step.page_table, step.seq_lens, SM)
    for b, L in enumerate(lens):
        V = dense(cache, step.page_table[b], L + W, 1)
        for i in range(W):
            for h in range(4):
                assert np.abs(got[b, i, h] - V[h // 2, :L + i + 1].mean(0)).max() < 1e-12


def test_empty_context_returns_the_single_value():
    spec, step, cache = build(oracle.KV_FP8, [0], 1, 4, 1, seed=6)
    got, _ = oracle.verify_attn(cache, step.q, step.page_table, step.seq_lens, SM)
    V = dense(cache, step.page_table[0], 1, 1)
    for h in range(4):
        assert np.array_equal(got[0, 0, h], V[0, 0])


def test_dominant_key_takes_all_weight():
    spec, step, cache = build(oracle.KV_FP8, [200], 1, 4, 1, seed=7)
    # make q parallel to key 37 and large: its logit dominates by > 40
    K = dense(cache, step.page_table[0], 201, 0)
    V = dense(cache, step.page_table[0], 201, 1)
    q = K[0, 37] / np.linalg.norm(K[0, 37]) * 400.0
    step.q[0, 0, 0] = synth.to_bf16_bits(q.astype(np.float32))
    got, _ = oracle.verify_attn(cache, step.q, step.page_table, step.seq_lens, SM)
    qf = synth.bf16_to_f32(step.q[0, 0, 0]).astype(np.float64)
    logits = K[0] @ qf * float(SM)
    assert np.sort(logits)[-1] - np.sort(logits)[-2] > 40
    assert np.abs(got[0, 0, 0] - V[0, 37]).max() < 1e-12


def test_invalid_lane_is_zero_and_flagged():
    spec, step, cache = build(oracle.KV_FP8, [70, 70], 2, 4, 1, seed=1)
    table = step.page_table.copy()
    table[1, 1] = step.num_pages + 5
    got, st = oracle.verify_attn(cache, step.q, table, step.seq_lens, SM)
    assert st == 1
    assert not got[1].any() and got[0].any()
    got, st = oracle.verify_attn(cache, step.q, step.page_table, np.array([70, 10 ** 6], np.int32), SM)
    assert st == 2 and not got[1].any()


def test_row_subset_matches_full():
    spec, step, cache = build(oracle.KV_FP8, [150, 20], 4, 6, 2, seed=12)
    full, _ = oracle.verify_attn(cache, step.q, step.page_table, step.seq_lens, SM, threads=3)
    rows = [(1, 3, 5), (0, 0, 0), (0, 2, 4)]
    part, _ = oracle.verify_attn(cache, step.q, step.page_table, step.seq_lens, SM, rows=rows)
    for k, (b, i, h) in enumerate(rows):
        assert np.array_equal(part[k], full[b, i, h])


@pytest.mark.parametrize("dtype", [oracle.KV_FP8, oracle.KV_INT4])
def test_ragged_window_rows(dtype):
    """Per-lane window row counts: rows i < n_b equal the attention of a
    window truncated to n_b rows (a separate oracle call with a shorter
    window) and the torch fp64 softmax; rows past the count are zero; a
    count outside [0, W] zeroes the lane and sets bit 16."""
    lens, W, Hq, Hkv = [70, 5, 130], 6, 6, 2
    spec, step, cache = build(dtype, lens, W, Hq, Hkv, seed=21)
    n = np.array([0, 4, 6], np.int32)
    got, st = oracle.verify_attn_ragged(cache, step.q, step.page_table, step.seq_lens, n, SM)
    assert st == 0
    want = torch_reference(step, cache)
    for b in range(len(lens)):
        assert not got[b, n[b]:].any()
        assert np.abs(got[b, :n[b]] - want[b, :n[b]]).max(initial=0.0) < 1e-12
        if n[b]:
            short, _ = oracle.verify_attn(cache, np.ascontiguousarray(step.q[b:b + 1, :n[b]]),
                                          step.page_table[b:b + 1], step.seq_lens[b:b + 1], SM)
            assert np.abs(got[b, :n[b]] - short[0]).max() < 1e-12
    got2, st2 = oracle.verify_attn_ragged(cache, step.q, step.page_table, step.seq_lens,
                                          np.array([7, 4, -1], np.int32), SM)
    assert st2 == 16
    assert not got2[0].any() and not got2[2].any()
    assert np.abs(got2[1] - got[1]).max() == 0.0
