"""Seeded synthetic inputs for the speculative-decoding verify step.

Shared by the tests and the benchmark for both the GPU library and the CPU
oracle.  It holds none of the method's arithmetic (no quantisation, no
attention, no argmax): only random numbers, shapes and page tables.

Every array is drawn from numpy's PCG64 generator seeded by a tuple
(workload seed, stream name, lane, chunk), so any piece regenerates on its own
without drawing the rest first.

Workloads (names say what they are):

=================  =====================================================================
tiny               1 lane, context 512, 4 q / 1 kv heads, window 1+3, FP8, vocab 4096, p=0.7
plain_decode       1 lane, context 32,768, 24 q / 4 kv heads, window 1, FP8,
                   4 outlier K channels per kv head scaled x8
multi_lane         8 lanes, contexts U[4096, 65536], 24/4 heads, window 1+15, FP8,
                   permuted page table, vocab 151,936, p=0.7
long_context       1 lane, context 240,000, 24/4 heads, window 1+5, FP8, vocab 151,936, p=0.7
int4_12slot        12 lanes, contexts U[8192, 131072], 24/4 heads, window 1+7, INT4 g32,
                   permuted page table, vocab 151,936, p=0.5
=================  =====================================================================

All values: Q/K/V ~ N(0, 1) rounded to bf16 (nearest even); logits ~ N(0, 1)
fp32 with the target token of each row planted as the unique maximum; each
draft equals its row's target with probability p, else a uniform other id.
"""
from __future__ import annotations

import dataclasses
import zlib

import numpy as np

PAGE = 64
HEAD_DIM = 128
KV_FP8 = 0
KV_INT4 = 1
KV_INT8 = 2
KV_FP8_ROW = 3


@dataclasses.dataclass(frozen=True)
class Spec:
    name: str
    seed: int
    num_lanes: int
    ctx_lo: int
    ctx_hi: int
    num_q_heads: int
    num_kv_heads: int
    window: int
    kv_dtype: int
    vocab: int | None
    match_p: float
    permuted: bool
    outlier_k_channels: int = 0
    outlier_scale: float = 8.0


WORKLOADS = {
    "tiny": Spec("tiny", 1, 1, 512, 512, 4, 1, 4, KV_FP8, 4096, 0.7, False),
    "plain_decode": Spec("plain_decode", 2, 1, 32768, 32768, 24, 4, 1, KV_FP8, None, 0.7, False, 4),
    "multi_lane": Spec("multi_lane", 3, 8, 4096, 65536, 24, 4, 16, KV_FP8, 151936, 0.7, True),
    "long_context": Spec("long_context", 4, 1, 240000, 240000, 24, 4, 6, KV_FP8, 151936, 0.7, False),
    "int4_12slot": Spec("int4_12slot", 5, 12, 8192, 131072, 24, 4, 8, KV_INT4, 151936, 0.5, True),
}


def _rng(seed: int, *key) -> np.random.Generator:
    words = [int(seed) & 0xFFFFFFFF]
    for k in key:
        if isinstance(k, str):
            words.append(zlib.crc32(k.encode()))
        else:
            words.append(int(k) & 0xFFFFFFFF)
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(words)))


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (round to nearest even); inputs are finite."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(bits, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16(rng: np.random.Generator, shape, scale_channels=None) -> np.ndarray:
    x = rng.standard_normal(shape, dtype=np.float32)
    if scale_channels is not None:
        x = x * scale_channels
    return to_bf16_bits(x)


@dataclasses.dataclass
class Step:
    """One verify step's inputs (host arrays)."""
    spec: Spec
    seq_lens: np.ndarray  # int32 [B], cached length before the step
    page_table: np.ndarray  # int32 [B][max_pages]
    num_pages: int
    q: np.ndarray  # uint16 bf16 [B][W][Hq][128]
    k_win: np.ndarray  # uint16 bf16 [B][W][Hkv][128]
    v_win: np.ndarray  # uint16 bf16 [B][W][Hkv][128]
    logits: np.ndarray | None  # float32 [B][W][V]
    drafts: np.ndarray | None  # int32 [B][W-1]
    targets: np.ndarray | None  # int32 [B][W] planted argmax of each row

    @property
    def max_pages(self) -> int:
        return self.page_table.shape[1]


def context_lengths(spec: Spec) -> np.ndarray:
    rng = _rng(spec.seed, "ctx")
    if spec.ctx_lo == spec.ctx_hi:
        return np.full(spec.num_lanes, spec.ctx_lo, np.int32)
    return rng.integers(spec.ctx_lo, spec.ctx_hi + 1, size=spec.num_lanes).astype(np.int32)


def page_table_for(spec: Spec, seq_lens: np.ndarray, window: int, extra_pages: int = 0):
    """Each lane owns exactly the pages holding tokens [0, L_b + window);
    identity order or one seeded random permutation of all pages."""
    need = [(int(L) + window + PAGE - 1) // PAGE for L in seq_lens]
    total = sum(need) + extra_pages
    ids = np.arange(total, dtype=np.int32)
    if spec.permuted:
        ids = _rng(spec.seed, "perm").permutation(total).astype(np.int32)
    max_pages = max(need)
    table = np.full((len(need), max_pages), -1, np.int32)
    o = 0
    for b, n in enumerate(need):
        table[b, :n] = ids[o:o + n]
        o += n
    return table, total


def outlier_channels(spec: Spec) -> np.ndarray | None:
    """Per-kv-head multiplier over head dims: 4 seeded distinct channels x scale."""
    if not spec.outlier_k_channels:
        return None
    rng = _rng(spec.seed, "outliers")
    m = np.ones((spec.num_kv_heads, HEAD_DIM), np.float32)
    for h in range(spec.num_kv_heads):
        ch = rng.choice(HEAD_DIM, size=spec.outlier_k_channels, replace=False)
        m[h, ch] = spec.outlier_scale
    return m


def context_chunk(spec: Spec, lane: int, start: int, count: int):
    """K and V (bf16 bits [count][Hkv][128]) for cached tokens [start, start+count)
    of one lane.  Drawn per 64-token block so any block regenerates alone."""
    mult = outlier_channels(spec)
    ks, vs = [], []
    t = start
    while t < start + count:
        blk = t // PAGE
        b0 = blk * PAGE
        rk = _rng(spec.seed, "k", lane, blk)
        rv = _rng(spec.seed, "v", lane, blk)
        kb = normal_bf16(rk, (PAGE, spec.num_kv_heads, HEAD_DIM), mult)
        vb = normal_bf16(rv, (PAGE, spec.num_kv_heads, HEAD_DIM))
        lo = t - b0
        hi = min(PAGE, start + count - b0)
        ks.append(kb[lo:hi])
        vs.append(vb[lo:hi])
        t = b0 + hi
    if not ks:
        z = np.zeros((0, spec.num_kv_heads, HEAD_DIM), np.uint16)
        return z, z.copy()
    return np.concatenate(ks), np.concatenate(vs)


def acceptance_inputs(spec: Spec, num_lanes: int, window: int, vocab: int, p: float, tag: str = "accept"):
    """Logits with a planted unique maximum per row, and drafts that match the
    planted token with probability p."""
    rng = _rng(spec.seed, tag)
    logits = rng.standard_normal((num_lanes, window, vocab), dtype=np.float32)
    targets = rng.integers(0, vocab, size=(num_lanes, window)).astype(np.int32)
    bump = (8.0 + np.abs(rng.standard_normal((num_lanes, window)))).astype(np.float32)
    for b in range(num_lanes):
        for i in range(window):
            logits[b, i, targets[b, i]] = bump[b, i]
    d = window - 1
    match = rng.random((num_lanes, d)) < p
    other = rng.integers(0, vocab - 1, size=(num_lanes, d)).astype(np.int32)
    other = np.where(other >= targets[:, :d], other + 1, other).astype(np.int32)
    drafts = np.where(match, targets[:, :d], other).astype(np.int32)
    return logits, drafts, targets


def make_step(spec: Spec, seq_lens: np.ndarray | None = None, window: int | None = None,
              num_q_heads: int | None = None, num_kv_heads: int | None = None, with_accept: bool = True,
              tag: str = "step") -> Step:
    """Inputs for one verify step of `spec` (optionally overriding sizes, for
    small parity cases that keep the workload's structure)."""
    if num_q_heads is not None or num_kv_heads is not None:
        spec = dataclasses.replace(spec, num_q_heads=num_q_heads or spec.num_q_heads,
                                   num_kv_heads=num_kv_heads or spec.num_kv_heads)
    W = window or spec.window
    if seq_lens is None:
        seq_lens = context_lengths(spec)
    seq_lens = np.asarray(seq_lens, np.int32)
    if W != spec.window or len(seq_lens) != spec.num_lanes:
        spec = dataclasses.replace(spec, window=W, num_lanes=len(seq_lens))
    B = len(seq_lens)
    table, total = page_table_for(spec, seq_lens, W)
    rng = _rng(spec.seed, tag, "q")
    q = normal_bf16(rng, (B, W, spec.num_q_heads, HEAD_DIM))
    k_win = np.zeros((B, W, spec.num_kv_heads, HEAD_DIM), np.uint16)
    v_win = np.zeros_like(k_win)
    for b in range(B):
        k, v = context_chunk(spec, b, int(seq_lens[b]), W)
        k_win[b], v_win[b] = k, v
    logits = drafts = targets = None
    if with_accept and spec.vocab:
        logits, drafts, targets = acceptance_inputs(spec, B, W, spec.vocab, spec.match_p, tag + "/accept")
    return Step(spec, seq_lens, table, total, q, k_win, v_win, logits, drafts, targets)


def fill_chunks(seq_len: int, chunk: int = 4096):
    """(start, count) pieces used to fill a lane's context before the step:
    page-aligned chunks of `chunk` tokens, the last one ragged."""
    out = []
    t = 0
    while t < seq_len:
        n = min(chunk, seq_len - t)
        out.append((t, n))
        t += n
    return out
