"""Pins for the oracle's codecs (no GPU).

The oracle's FP8/fp16/INT4 codecs are checked against things other than
themselves: PyTorch's float8_e4m3fn and numpy's float16 (independent library
implementations of the same IEEE/OCP formats), hand-worked cases in
tests/golden/, and the brute-force nearest-value search in oracle/brute.py.
"""
import os
import struct

import numpy as np
import pytest
import torch

import oracle
from oracle import brute

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _f32(x):
    return struct.unpack("<f", struct.pack("<f", x))[0]


def test_e4m3_decode_all_codes_match_library():
    lib = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    for c in range(256):
        v = oracle.e4m3_decode(c)
        if np.isnan(lib[c]):
            assert np.isnan(v), c
            assert c in (0x7F, 0xFF)
        else:
            assert v == float(lib[c]), (c, v, lib[c])
            assert np.signbit(v) == bool(c & 0x80)


def test_e4m3_encode_golden_cases():
    with open(os.path.join(GOLDEN, "e4m3_encode_cases.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            x, code, *_ = line.split()
            assert oracle.e4m3_encode(float(x)) == int(code, 16), line


def test_e4m3_encode_matches_library_in_range():
    # every finite bf16 pattern below the saturation threshold: library RNE cast
    bits = np.arange(65536, dtype=np.uint32)
    x = (bits << 16).view(np.float32)
    x = x[np.isfinite(x) & (np.abs(x) < 464.0)]
    lib = torch.from_numpy(x.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(float(v)) for v in x], np.uint8)
    bad = np.nonzero(got != lib)[0]
    assert bad.size == 0, [(float(x[i]), got[i], lib[i]) for i in bad[:10]]


def test_e4m3_encode_saturates():
    for x in (448.0, 449.0, 464.0, 480.0, 1e6, 3.0e38):
        assert oracle.e4m3_encode(x) == 0x7E
        assert oracle.e4m3_encode(-x) == 0xFE
    assert oracle.e4m3_encode(float("nan")) == 0x7F


def test_e4m3_encode_matches_brute_search():
    rng = np.random.default_rng(7)
    xs = np.concatenate([
        rng.standard_normal(600).astype(np.float32) * 50,
        (rng.random(300).astype(np.float32) * 0.03),
        np.array([0.0, -0.0, 447.9, 448.1, 2.0 ** -10, 2.0 ** -9 * 1.5], np.float32),
    ])
    for x in xs:
        x = float(x)
        assert oracle.e4m3_encode(x) == brute.e4m3_encode(x), x


def test_e4m3_roundtrip_is_identity_on_grid():
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        assert oracle.e4m3_encode(oracle.e4m3_decode(c)) == c


def test_f16_encode_matches_numpy():
    rng = np.random.default_rng(3)
    xs = np.concatenate([
        rng.standard_normal(4000).astype(np.float32) * np.float32(1e3),
        rng.random(4000).astype(np.float32) * np.float32(1e-4),  # subnormal region
        rng.random(1000).astype(np.float32) * np.float32(1e-7),
        np.array([65504.0, 65519.0, 65520.0, 6.1e-5, 5.96e-8, 2.98e-8, 0.0, -0.0], np.float32),
    ])
    with np.errstate(over="ignore"):
        lib = xs.astype(np.float16)
    for x, want in zip(xs, lib):
        got = oracle.f16_encode(float(x))
        assert got == int(want.view(np.uint16)), (float(x), hex(got), hex(int(want.view(np.uint16))))
        if not np.isinf(want):
            assert oracle.f16_decode(got) == float(want)


def test_int4_golden_cases():
    with open(os.path.join(GOLDEN, "int4_cases.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            head, want = line.split("->")
            amax, x = head.split("|")
            group = np.zeros(32, np.float32)
            group[0] = float(amax)
            group[1] = float(x)
            s, codes = oracle.int4_group(group)
            assert codes[1] == int(want), line
            assert codes[0] == 7


def test_int4_matches_brute_and_bounds():
    rng = np.random.default_rng(11)
    for trial in range(300):
        scale = [1.0, 1e-3, 1e3, 1e-6, 1e5][trial % 5]
        x = (rng.standard_normal(32) * scale).astype(np.float32)
        s, codes = oracle.int4_group(x)
        bs, bcodes = brute.int4_group([float(v) for v in x])
        assert s == bs, trial
        assert list(codes) == bcodes, trial
        assert codes.min() >= -7 and codes.max() <= 7
    s, codes = oracle.int4_group(np.zeros(32, np.float32))
    assert s == 0 and not codes.any()
    # amax / 7 above fp16 range: the scale clamps to 65504 and codes saturate
    x = np.full(32, 1e6, np.float32)
    s, codes = oracle.int4_group(x)
    assert s == 0x7BFF and (codes == 7).all()


def test_int4_error_within_half_step():
    rng = np.random.default_rng(12)
    for _ in range(200):
        x = rng.standard_normal(32).astype(np.float32)
        s, codes = oracle.int4_group(x)
        sv = oracle.f16_decode(s)
        err = np.abs(codes * sv - x.astype(np.float64))
        # half a quantisation step, plus the fp16 rounding of the scale at the ends
        assert (err <= 0.5 * sv + 7 * abs(sv - np.abs(x).max() / 7) + 1e-12).all()
