"""Pins for the oracle's cache append (no GPU): the C oracle against the
independent brute-force statement on tiny multi-step histories, plus
invariants of the scale semantics (fresh page resets, growth re-encodes,
the dequantised error bound)."""
import numpy as np
import pytest

import oracle
import synth
from oracle import brute

PAGE = 64


def _rows(k, v, b):
    """brute layout: new_rows[kv][t][h] = list of 128 bf16 ints"""
    return [[[list(map(int, k[b, t, h])) for h in range(k.shape[2])] for t in range(k.shape[1])],
            [[list(map(int, v[b, t, h])) for h in range(v.shape[2])] for t in range(v.shape[1])]]


def _compare(cache, bc, dtype, table, lens_written):
    H = cache.num_kv_heads
    for kv, (codes, scales) in enumerate(((cache.k_codes, cache.k_scales), (cache.v_codes, cache.v_scales))):
        for b, n in enumerate(lens_written):
            for pos in range(n):
                pid, off = int(table[b, pos // PAGE]), pos % PAGE
                for h in range(H):
                    want = bc.codes[kv][(pid, h, off)]
                    if dtype == oracle.KV_FP8:
                        assert list(codes[pid, h, off]) == want, (kv, b, pos, h)
                        assert scales[pid, h] == np.float32(bc.scales[kv][(pid, h)])
                    else:
                        packed = codes[pid, h, off]
                        lo = ((packed & 0xF).astype(np.int8) ^ 8) - 8
                        hi = ((packed >> 4).astype(np.int8) ^ 8) - 8
                        got = np.stack([lo, hi], 1).reshape(-1)
                        assert list(got) == want, (kv, b, pos, h)
                        assert list(scales[pid, h, off]) == bc.scales[kv][(pid, h, off)]


def _history(dtype, seed, steps=6, W=5, lanes=2, H=2, big_at=None):
    spec = synth.Spec("t", seed, lanes, 0, 0, 2 * H, H, W, dtype, 64, 0.7, True)
    rng = np.random.default_rng(seed)
    L0 = np.array([3, 60][:lanes] + [0] * max(0, lanes - 2), np.int32)
    max_tokens = int(L0.max()) + steps * W + W
    need = (max_tokens + PAGE - 1) // PAGE
    perm = rng.permutation(need * lanes).astype(np.int32)
    table = perm.reshape(lanes, need)
    cache = oracle.Cache(dtype, need * lanes, H)
    bc = brute.Cache(dtype)
    # prefill: one chunk per lane of L0 tokens
    for b in range(lanes):
        if L0[b] == 0:
            continue
        k, v = synth.context_chunk(spec, b, 0, int(L0[b]))
        st = oracle.append(cache, k[None], v[None], table[b:b + 1], np.zeros(1, np.int32))
        assert st == 0
        brute.append(bc, _rows(k[None], v[None], 0), list(table[b]), 0)
    L = L0.copy()
    written = L0.copy()
    for s in range(steps):
        k = synth.normal_bf16(rng, (lanes, W, H, 128))
        v = synth.normal_bf16(rng, (lanes, W, H, 128))
        if big_at is not None and s == big_at:
            # a large-magnitude token forces the page scale to grow
            k[0, 1, 0, 5] = synth.to_bf16_bits(np.array([40.0], np.float32))[0]
            v[1, 0, 1, 7] = synth.to_bf16_bits(np.array([-90.0], np.float32))[0]
        st = oracle.append(cache, k, v, table, L)
        assert st == 0
        for b in range(lanes):
            brute.append(bc, _rows(k, v, b), list(table[b]), int(L[b]))
        written = np.maximum(written, L + W)
        L = L + 1 + rng.integers(0, W, size=lanes).astype(np.int32)
    return cache, bc, table, written


@pytest.mark.parametrize("dtype", [oracle.KV_FP8, oracle.KV_INT4])
@pytest.mark.parametrize("big_at", [None, 2])
def test_append_matches_brute(dtype, big_at):
    cache, bc, table, written = _history(dtype, 21 + (big_at or 0), big_at=big_at)
    _compare(cache, bc, dtype, table, written)


def test_fp8_fresh_page_resets_scale_and_growth_reencodes():
    H = 1
    cache = oracle.Cache(oracle.KV_FP8, 2, H)
    table = np.array([[0, 1]], np.int32)
    one = synth.to_bf16_bits(np.full((1, 3, H, 128), 1.0, np.float32))
    st = oracle.append(cache, one, one, table, np.array([0], np.int32))
    assert st == 0
    s1 = cache.k_scales[0, 0]
    assert s1 == np.float32(1.0) / np.float32(448.0)
    assert (cache.k_codes[0, 0, :3] == oracle.e4m3_encode(np.float32(1.0) / s1)).all()
    # a token twice as large grows the scale; earlier tokens are re-encoded
    two = synth.to_bf16_bits(np.full((1, 1, H, 128), 2.0, np.float32))
    oracle.append(cache, two, two, table, np.array([3], np.int32))
    s2 = cache.k_scales[0, 0]
    assert s2 == np.float32(2.0) / np.float32(448.0)
    deq = np.array([oracle.e4m3_decode(c) * float(s2) for c in cache.k_codes[0, 0, :4, 0]])
    # 1.0 at scale 2/448 is code 224 exactly: E4M3 holds 224 (0x76); 2.0 is 448
    assert list(cache.k_codes[0, 0, :4, 0]) == [0x76, 0x76, 0x76, 0x7E]
    assert np.allclose(deq, [1.0, 1.0, 1.0, 2.0], rtol=1e-6, atol=0)
    # a smaller token does not shrink the scale
    half = synth.to_bf16_bits(np.full((1, 1, H, 128), 0.5, np.float32))
    oracle.append(cache, half, half, table, np.array([4], np.int32))
    assert cache.k_scales[0, 0] == s2
    # an append starting at page offset 0 resets the scale of that page
    oracle.append(cache, half, half, table, np.array([64], np.int32))
    assert cache.k_scales[1, 0] == np.float32(0.5) / np.float32(448.0)


def test_fp8_dequant_error_bound():
    spec = synth.WORKLOADS["plain_decode"]
    k, v = synth.context_chunk(spec, 0, 0, 128)
    cache = oracle.Cache(oracle.KV_FP8, 2, 4)
    table = np.array([[0, 1]], np.int32)
    assert oracle.append(cache, k[None], v[None], table, np.zeros(1, np.int32)) == 0
    x = synth.bf16_to_f32(k).astype(np.float64)
    for t in range(128):
        pid, off = t // 64, t % 64
        for h in range(4):
            s = float(cache.k_scales[pid, h])
            deq = np.array([oracle.e4m3_decode(c) for c in cache.k_codes[pid, h, off]]) * s
            # E4M3 has 3 mantissa bits: relative error <= 2^-4 above the
            # subnormal range, absolute <= 2^-10 * s below it
            tol = np.maximum(np.abs(x[t, h]) * 2.0 ** -4, 2.0 ** -10 * s) * (1 + 1e-6)
            assert (np.abs(deq - x[t, h]) <= tol).all()


def test_overflow_and_bad_page_are_flagged_and_skipped():
    cache = oracle.Cache(oracle.KV_FP8, 2, 1)
    k = synth.normal_bf16(np.random.default_rng(0), (1, 4, 1, 128))
    table = np.array([[0, 1]], np.int32)
    before = cache.k_codes.copy()
    assert oracle.append(cache, k, k, table, np.array([125], np.int32)) == 2
    assert (cache.k_codes == before).all()
    bad = np.array([[0, 7]], np.int32)
    assert oracle.append(cache, k, k, bad, np.array([62], np.int32)) == 1
    assert (cache.k_codes == before).all()
    assert oracle.append(cache, k, k, table, np.array([-1], np.int32)) == 2


# ---- per-lane token counts (a padded window whose lanes drafted different numbers of tokens) ----

def _ragged_history(dtype, seed, steps=6, W=6, lanes=3, H=2):
    rng = np.random.default_rng(seed)
    L = np.array([5, 62, 0][:lanes], np.int32)
    need = (int(L.max()) + steps * W + W + PAGE - 1) // PAGE
    table = rng.permutation(need * lanes).astype(np.int32).reshape(lanes, need)
    cache = oracle.Cache(dtype, need * lanes, H)
    bc = brute.Cache(dtype)
    for b in range(lanes):  # the lanes' starting context
        if L[b]:
            k = synth.normal_bf16(rng, (1, int(L[b]), H, 128))
            assert oracle.append(cache, k, k, table[b:b + 1], np.zeros(1, np.int32)) == 0
            brute.append(bc, _rows(k, k, 0), list(table[b]), 0)
    written = L.copy()
    for s in range(steps):
        k = synth.normal_bf16(rng, (lanes, W, H, 128))
        v = synth.normal_bf16(rng, (lanes, W, H, 128))
        if s == 2:
            k[1, 0, 1, 9] = synth.to_bf16_bits(np.array([70.0], np.float32))[0]  # forces a scale growth
        n = rng.integers(0, W + 1, size=lanes).astype(np.int32)
        assert oracle.append_ragged(cache, k, v, table, L, n) == 0
        for b in range(lanes):
            if n[b]:
                brute.append(bc, _rows(k[:, :n[b]], v[:, :n[b]], b), list(table[b]), int(L[b]))
        written = np.maximum(written, L + n)
        L = L + rng.integers(0, n + 1).astype(np.int32)
    return cache, bc, table, written


@pytest.mark.parametrize("dtype", [oracle.KV_FP8, oracle.KV_INT4])
def test_ragged_append_matches_brute(dtype):
    cache, bc, table, written = _ragged_history(dtype, 31)
    _compare(cache, bc, dtype, table, written)


@pytest.mark.parametrize("dtype", [oracle.KV_FP8, oracle.KV_INT4])
def test_ragged_with_full_counts_is_the_plain_append(dtype):
    rng = np.random.default_rng(32)
    B, W, H = 3, 7, 2
    table = rng.permutation(4 * B).astype(np.int32).reshape(B, 4)
    L = np.array([10, 63, 120], np.int32)
    k = synth.normal_bf16(rng, (B, W, H, 128))
    v = synth.normal_bf16(rng, (B, W, H, 128))
    a, b = oracle.Cache(dtype, 4 * B, H), oracle.Cache(dtype, 4 * B, H)
    assert oracle.append(a, k, v, table, L) == 0
    assert oracle.append_ragged(b, k, v, table, L, np.full(B, W, np.int32)) == 0
    for n in ("k_codes", "v_codes", "k_scales", "v_scales"):
        assert np.array_equal(getattr(a, n), getattr(b, n)), n


def test_ragged_int4_in_two_parts_equals_one_append():
    # INT4 scales belong to single tokens, so writing a window in two parts changes nothing
    rng = np.random.default_rng(33)
    B, W, H = 2, 9, 3
    table = rng.permutation(3 * B).astype(np.int32).reshape(B, 3)
    L = np.array([60, 3], np.int32)
    k = synth.normal_bf16(rng, (B, W, H, 128))
    v = synth.normal_bf16(rng, (B, W, H, 128))
    whole, parts = oracle.Cache(oracle.KV_INT4, 3 * B, H), oracle.Cache(oracle.KV_INT4, 3 * B, H)
    assert oracle.append(whole, k, v, table, L) == 0
    n1 = np.array([4, 0], np.int32)
    assert oracle.append_ragged(parts, k, v, table, L, n1) == 0
    rest_k = np.stack([np.roll(k[b], -n1[b], axis=0) for b in range(B)])
    rest_v = np.stack([np.roll(v[b], -n1[b], axis=0) for b in range(B)])
    assert oracle.append_ragged(parts, rest_k, rest_v, table, L + n1, W - n1) == 0
    for n in ("k_codes", "v_codes", "k_scales", "v_scales"):
        assert np.array_equal(getattr(whole, n), getattr(parts, n)), n


def test_ragged_invalid_and_empty_counts():
    rng = np.random.default_rng(34)
    B, W, H = 3, 4, 1
    table = np.array([[0, 1], [2, 3], [-5, 4]], np.int32)  # lane 2 has a bad page id
    L = np.array([0, 10, 0], np.int32)
    k = synth.normal_bf16(rng, (B, W, H, 128))
    c = oracle.Cache(oracle.KV_FP8, 5, H)
    st = oracle.append_ragged(c, k, k, table, L, np.array([W + 1, -1, 0], np.int32))
    assert st == 16  # lane 2 writes nothing, so its bad page is never examined
    assert not c.k_codes.any() and not c.k_scales.any()
    assert oracle.append_ragged(c, k, k, table, L, np.array([2, 0, 1], np.int32)) == 1
    assert c.k_codes[0, 0, :2].any() and not c.k_codes[0, 0, 2:].any()
