"""Helpers shared by the GPU parity tests: move seeded synthetic inputs to the
device and build the same cache twice -- with the library's kernels on the GPU
and with the oracle on the CPU -- from the same calls."""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
import synth

SM_SCALE = np.float32(1.0 / math.sqrt(128.0))
KV_NAMES = {synth.KV_FP8: "fp8", synth.KV_INT4: "int4", synth.KV_INT8: "int8", synth.KV_FP8_ROW: "fp8row"}
ALL_KV = list(KV_NAMES)


def bf16_dev(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def i32_dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(device)


def cache_to_host(c) -> dict:
    return {n: getattr(c, n).cpu().numpy() for n in ("k_codes", "v_codes", "k_scales", "v_scales")}


def fill_both(spec: synth.Spec, step: synth.Step, lanes=None, chunk: int = 4096, with_oracle: bool = True):
    """Fill the lanes' contexts on the GPU (all lanes) and in the oracle
    (`lanes`, default all) with the same page-aligned chunk sequence, then
    append the window on both.  Returns (gpu_cache, oracle_cache, gpu_status)."""
    import speculative_decode_verify_append_gb300 as sdva

    Hkv = spec.num_kv_heads
    gcache = sdva.KVCache(spec.kv_dtype, step.num_pages, Hkv)
    ocache = oracle.Cache(spec.kv_dtype, step.num_pages, Hkv) if with_oracle else None
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    table_dev = i32_dev(step.page_table)
    lanes = range(len(step.seq_lens)) if lanes is None else lanes
    for b, L in enumerate(step.seq_lens):
        for start, n in synth.fill_chunks(int(L), chunk):
            k, v = synth.context_chunk(spec, b, start, n)
            sdva.kv_append_quant(gcache, bf16_dev(k[None]), bf16_dev(v[None]), table_dev[b:b + 1],
                                 i32_dev(np.array([start])), status)
            if with_oracle and b in lanes:
                st = oracle.append(ocache, k[None], v[None], step.page_table[b:b + 1], np.array([start], np.int32))
                assert st == 0
    sdva.kv_append_quant(gcache, bf16_dev(step.k_win), bf16_dev(step.v_win), table_dev, i32_dev(step.seq_lens),
                         status)
    if with_oracle:
        sel = np.array(sorted(lanes))
        st = oracle.append(ocache, step.k_win[sel], step.v_win[sel], step.page_table[sel], step.seq_lens[sel])
        assert st == 0
    return gcache, ocache, status


def lane_pages(step: synth.Step, b: int) -> np.ndarray:
    n = (int(step.seq_lens[b]) + step.q.shape[1] + 63) // 64
    return step.page_table[b, :n]


def assert_close(got: np.ndarray, want: np.ndarray, what: str = "") -> tuple[float, float]:
    """|g - r| <= 2e-3 + 1e-2 |r| elementwise; returns (max abs, max rel)."""
    got = got.astype(np.float64)
    err = np.abs(got - want)
    bound = 2e-3 + 1e-2 * np.abs(want)
    bad = np.argwhere(err > bound)
    assert bad.size == 0, (f"{what}: {len(bad)} elements out of tolerance, first at {bad[:5].tolist()}, "
                           f"max abs {err.max():.3g}")
    if err.size == 0:
        return 0.0, 0.0
    rel = err / np.maximum(np.abs(want), 1e-30)
    return float(err.max()), float(rel.max())


def assert_close_row_scaled(got: np.ndarray, want: np.ndarray, what: str = "") -> float:
    """|g - r| <= 2e-3 s + 1e-2 |r| elementwise, s = max(1, max |r| over the
    output row): assert_close's absolute term taken relative to the row's
    own scale.  An output element is a softmax-weighted sum of V rows; when
    those rows are much larger than the element (inputs scaled by up to 2^6
    with partial cancellation), the fp16 rounding of P and V leaves an error
    that follows their magnitude, not the element's.  Returns the largest
    error relative to s."""
    got = got.astype(np.float64)
    err = np.abs(got - want)
    s = np.maximum(1.0, np.abs(want).max(axis=-1, keepdims=True))
    bad = np.argwhere(err > 2e-3 * s + 1e-2 * np.abs(want))
    assert bad.size == 0, (f"{what}: {len(bad)} elements out of tolerance, first at {bad[:5].tolist()}, "
                           f"max abs {err.max():.3g}")
    return float((err / s).max()) if err.size else 0.0


def both_fraction(got: np.ndarray, want: np.ndarray) -> float:
    """Fraction of elements within the stricter reading of the tolerance:
    |g - r| <= 2e-3 and |g - r| <= 1e-2 |r| at once."""
    err = np.abs(got.astype(np.float64) - want)
    ok = (err <= 2e-3) & (err <= 1e-2 * np.abs(want))
    return float(ok.mean())
