"""Pins for the oracle's other KV formats (no GPU): INT8 group-64 with fp16
scales and FP8 E4M3 with one fp32 scale per (token, head) row.  Codecs against
the brute-force statements and hand-worked cases (ties to even, the clamp a
subnormal scale needs, zero groups), dequantisation error bounds, multi-step
append histories against brute force, and attention over each format
against the brute-force attention row."""
import math

import numpy as np
import pytest

import oracle
import synth
from oracle import brute

PAGE = 64


def test_int8_group_matches_brute_and_hand_cases():
    rng = np.random.default_rng(120)
    for trial in range(200):
        x = (rng.standard_normal(64) * 10.0 ** rng.uniform(-6, 4)).astype(np.float32)
        if trial % 7 == 0:
            x[rng.integers(0, 64, 5)] = 0.0
        s, q = oracle.int8_group(x)
        sb, qb = brute.int_group([float(v) for v in x], 127)
        assert s == sb and list(q) == qb, trial
    # amax 127 gives scale 1: halves go to even, the extremes stay in range
    x = np.array([127.0, 2.5, 3.5, -2.5, 126.5, -127.0] + [0.0] * 58, np.float32)
    s, q = oracle.int8_group(x)
    assert s == 0x3C00 and list(q[:6]) == [127, 2, 4, -2, 126, -127]
    # a subnormal fp16 scale is coarse: 1e-5 / 127 rounds to 2^-24, and the codes clamp at 127
    x = np.zeros(64, np.float32)
    x[0], x[1] = 1e-5, -1e-5
    s, q = oracle.int8_group(x)
    assert s == 0x0001 and q[0] == 127 and q[1] == -127
    # a zero group
    s, q = oracle.int8_group(np.zeros(64, np.float32))
    assert s == 0 and not q.any()


def test_fp8_row_matches_brute_and_bounds():
    rng = np.random.default_rng(121)
    for trial in range(200):
        x = (rng.standard_normal(128) * 10.0 ** rng.uniform(-5, 4)).astype(np.float32)
        s, c = oracle.fp8_row(x)
        sb, cb = brute.fp8_row([float(v) for v in x])
        assert s == sb and list(c) == cb, trial
        deq = np.array([brute.e4m3_value(int(k)) for k in c]) * s
        # E4M3 keeps 3 mantissa bits: half an ulp relative, or half the subnormal step
        assert (np.abs(deq - x) <= np.maximum(np.abs(x) * 2.0 ** -4, s * 2.0 ** -10)).all()
        assert int(np.argmax(np.abs(x))) in np.flatnonzero(np.isin(c, (0x7E, 0xFE)))
    s, c = oracle.fp8_row(np.zeros(128, np.float32))
    assert s == 0.0 and not c.any()


def test_int8_dequant_error_bound():
    rng = np.random.default_rng(122)
    for _ in range(100):
        x = (rng.standard_normal(64) * 3.0).astype(np.float32)
        s, q = oracle.int8_group(x)
        sv = float(np.frombuffer(np.uint16(s).tobytes(), np.float16)[0])
        assert (np.abs(q.astype(np.float64) * sv - x) <= 0.5 * sv * (1 + 1e-6) + 1e-30).all()


def _rows(k, v, b):
    return [[[list(map(int, k[b, t, h])) for h in range(k.shape[2])] for t in range(k.shape[1])],
            [[list(map(int, v[b, t, h])) for h in range(v.shape[2])] for t in range(v.shape[1])]]


def _history(dtype, seed, steps=4, W=5, lanes=2, H=2):
    rng = np.random.default_rng(seed)
    L = np.array([3, 61], np.int32)[:lanes]
    need = (int(L.max()) + steps * W + W + PAGE - 1) // PAGE
    table = rng.permutation(need * lanes).astype(np.int32).reshape(lanes, need)
    cache = oracle.Cache(dtype, need * lanes, H)
    bc = brute.Cache(dtype)
    written = L.copy()
    for b in range(lanes):
        k = synth.normal_bf16(rng, (1, int(L[b]), H, 128))
        assert oracle.append(cache, k, k, table[b:b + 1], np.zeros(1, np.int32)) == 0
        brute.append(bc, _rows(k, k, 0), list(table[b]), 0)
    for s in range(steps):
        k = synth.normal_bf16(rng, (lanes, W, H, 128))
        v = synth.normal_bf16(rng, (lanes, W, H, 128))
        assert oracle.append(cache, k, v, table, L) == 0
        for b in range(lanes):
            brute.append(bc, _rows(k, v, b), list(table[b]), int(L[b]))
        written = np.maximum(written, L + W)
        L = L + 1 + rng.integers(0, W, size=lanes).astype(np.int32)
    return cache, bc, table, written


@pytest.mark.parametrize("dtype", [oracle.KV_INT8, oracle.KV_FP8_ROW])
def test_append_history_matches_brute(dtype):
    cache, bc, table, written = _history(dtype, 123 + dtype)
    for kv, (codes, scales) in enumerate(((cache.k_codes, cache.k_scales), (cache.v_codes, cache.v_scales))):
        for b, n in enumerate(written):
            for pos in range(n):
                pid, off = int(table[b, pos // PAGE]), pos % PAGE
                for h in range(cache.num_kv_heads):
                    want = bc.codes[kv][(pid, h, off)]
                    if dtype == oracle.KV_INT8:
                        assert list(codes[pid, h, off].view(np.int8)) == want, (kv, b, pos, h)
                        assert list(scales[pid, h, off]) == bc.scales[kv][(pid, h, off)]
                    else:
                        assert list(codes[pid, h, off]) == want, (kv, b, pos, h)
                        assert scales[pid, h, off] == np.float32(bc.scales[kv][(pid, h, off)])


@pytest.mark.parametrize("dtype", [oracle.KV_INT8, oracle.KV_FP8_ROW])
def test_attention_over_the_format_matches_brute(dtype):
    cache, bc, table, written = _history(dtype, 124 + dtype, steps=2, W=4, lanes=1, H=1)
    L = np.array([int(written[0]) - 4], np.int32)  # the last window: rows see keys 0 .. L + i
    rng = np.random.default_rng(125)
    q = synth.normal_bf16(rng, (1, 4, 2, 128))
    sm = float(np.float32(1.0 / math.sqrt(128.0)))
    out, st = oracle.verify_attn(cache, q, table, L, sm)
    assert st == 0
    for i in range(4):
        for h in range(2):
            want = brute.attention_row(bc, [int(x) for x in q[0, i, h]], list(table[0]), 0, int(L[0]) + i + 1, sm)
            assert np.allclose(out[0, i, h], want, rtol=1e-12, atol=1e-12), (i, h)
