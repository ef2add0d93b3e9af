"""Brute-force restatement of the verify step, pure Python, tiny inputs only.

TEST INFRASTRUCTURE ONLY.  It shares no code with ``oracle.c``: the FP8
value table comes from PyTorch's float8_e4m3fn type (an independent library
implementation of OCP E4M3), encoding is a nearest-value search over that
table, fp16 rounding is Python's ``struct`` half-float packing, fp32 results
are produced by rounding exact (or correctly rounded fp64) Python floats with
``struct`` single packing, and attention uses ``math.fsum``.

fp32 division through fp64: for fp32 operands the fp64 quotient rounded once
more to fp32 equals the correctly rounded fp32 quotient (53 >= 2*24 + 2), and
an fp32 product is exact in fp64, so every fp32 step here is IEEE-exact.
"""
from __future__ import annotations

import math
import struct

PAGE = 64
HEAD_DIM = 128

_E4M3 = None


def _table():
    global _E4M3
    if _E4M3 is None:
        import torch
        codes = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().tolist()
        _E4M3 = codes
    return _E4M3


def f32(x: float) -> float:
    return struct.unpack("<f", struct.pack("<f", x))[0]


def bf16(bits: int) -> float:
    return struct.unpack("<f", struct.pack("<I", (bits & 0xFFFF) << 16))[0]


def e4m3_value(code: int) -> float:
    return _table()[code]


def e4m3_encode(x: float) -> int:
    """Nearest finite E4M3 value; ties to the code with an even last bit;
    magnitudes above 448 saturate; the sign of zero is kept."""
    if x != x:
        return 0x7F
    sign = 0x80 if math.copysign(1.0, x) < 0 else 0
    a = abs(x)
    tab = _table()
    best, best_err = 0, None
    for c in range(0x7F):  # 0x00 .. 0x7E: all finite non-negative codes
        err = abs(tab[c] - a)
        if best_err is None or err < best_err or (err == best_err and c % 2 == 0):
            best, best_err = c, err
    return sign | best


def f16_bits(x: float) -> int:
    return struct.unpack("<H", struct.pack("<e", x))[0]


def f16_value(bits: int) -> float:
    return struct.unpack("<e", struct.pack("<H", bits))[0]


def int_group(xs, qmax):
    """Symmetric group codec to [-qmax, qmax]: the fp16 scale of amax / qmax,
    codes = x / s rounded half to even and clamped.  Returns (scale bits, codes)."""
    amax = max(abs(x) for x in xs)
    t = min(f32(amax / qmax), 65504.0)
    s_bits = f16_bits(t)
    s = f16_value(s_bits)
    if s == 0.0:
        return s_bits, [0] * len(xs)
    return s_bits, [max(-qmax, min(qmax, round(f32(x / s)))) for x in xs]


def fp8_row(xs):
    """Row codec: one fp32 scale amax / 448, codes E4M3 of x / s.  Returns (scale, codes)."""
    s = f32(max(abs(x) for x in xs) / 448.0)
    if s == 0.0:
        return s, [0] * len(xs)
    return s, [e4m3_encode(f32(x / s)) for x in xs]


def int4_group(xs):
    amax = max(abs(x) for x in xs)
    t = f32(amax / 7.0)
    t = min(t, 65504.0)
    s = f16_bits(t)
    sv = f16_value(s)
    codes = []
    for x in xs:
        if sv == 0.0:
            codes.append(0)
        else:
            r = f32(x / sv)
            k = round(r)  # Python rounds halves to even
            codes.append(max(-7, min(7, k)))
    return s, codes


class Cache:
    """Dict-of-pages cache: fp8 -> codes[(pid, h, off)] = list of 128 ints,
    scales[(pid, h)]; int4 -> codes[(pid, h, off)] = list of 128 ints in
    [-7, 7], scales[(pid, h, off)] = list of 4 fp16 bit patterns."""

    def __init__(self, dtype: int):
        self.dtype = dtype
        self.codes = {0: {}, 1: {}}
        self.scales = {0: {}, 1: {}}

    def value(self, kv: int, pid: int, h: int, off: int, d: int) -> float:
        if self.dtype == 0:
            return e4m3_value(self.codes[kv][(pid, h, off)][d]) * self.scales[kv][(pid, h)]
        if self.dtype == 2:
            return self.codes[kv][(pid, h, off)][d] * f16_value(self.scales[kv][(pid, h, off)][d // 64])
        if self.dtype == 3:
            return e4m3_value(self.codes[kv][(pid, h, off)][d]) * self.scales[kv][(pid, h, off)]
        return self.codes[kv][(pid, h, off)][d] * f16_value(self.scales[kv][(pid, h, off)][d // 32])


def append(cache: Cache, new_rows, page_row, L: int):
    """new_rows[kv][t][h] = list of 128 bf16 bit patterns for token L + t."""
    n = len(new_rows[0])
    H = len(new_rows[0][0]) if n else 0
    for kv in (0, 1):
        for h in range(H):
            if cache.dtype in (2, 3):
                for t in range(n):
                    pos = L + t
                    pid, off = page_row[pos // PAGE], pos % PAGE
                    xs = [bf16(b) for b in new_rows[kv][t][h]]
                    if cache.dtype == 2:
                        scales, codes = [], []
                        for g in range(2):
                            sc, c = int_group(xs[64 * g:64 * g + 64], 127)
                            scales.append(sc)
                            codes.extend(c)
                    else:
                        scales, codes = fp8_row(xs)
                    cache.codes[kv][(pid, h, off)] = codes
                    cache.scales[kv][(pid, h, off)] = scales
                continue
            if cache.dtype == 1:
                for t in range(n):
                    pos = L + t
                    pid, off = page_row[pos // PAGE], pos % PAGE
                    xs = [bf16(b) for b in new_rows[kv][t][h]]
                    scales, codes = [], []
                    for g in range(4):
                        s, c = int4_group(xs[32 * g:32 * g + 32])
                        scales.append(s)
                        codes.extend(c)
                    cache.codes[kv][(pid, h, off)] = codes
                    cache.scales[kv][(pid, h, off)] = scales
                continue
            # FP8: group the new tokens by page
            by_page = {}
            for t in range(n):
                by_page.setdefault((L + t) // PAGE, []).append(t)
            for lp, ts in sorted(by_page.items()):
                pid = page_row[lp]
                start = (L + ts[0]) % PAGE
                xs = {t: [bf16(b) for b in new_rows[kv][t][h]] for t in ts}
                amax = max(abs(x) for t in ts for x in xs[t])
                s_c = f32(amax / 448.0)
                if start == 0:
                    s_new = s_c
                else:
                    s_old = cache.scales[kv][(pid, h)]
                    s_new = max(s_c, s_old)
                    if s_new > s_old:
                        for off in range(start):
                            old = cache.codes[kv][(pid, h, off)]
                            cache.codes[kv][(pid, h, off)] = [
                                e4m3_encode(f32(f32(e4m3_value(c) * s_old) / s_new)) for c in old]
                for t in ts:
                    off = (L + t) % PAGE
                    if s_new == 0.0:
                        cache.codes[kv][(pid, h, off)] = [0] * HEAD_DIM
                    else:
                        cache.codes[kv][(pid, h, off)] = [e4m3_encode(f32(x / s_new)) for x in xs[t]]
                cache.scales[kv][(pid, h)] = s_new


def attention_row(cache: Cache, q_bits, page_row, hk: int, n_keys: int, sm_scale: float):
    q = [bf16(b) for b in q_bits]
    logits = []
    for j in range(n_keys):
        pid, off = page_row[j // PAGE], j % PAGE
        logits.append(sm_scale * math.fsum(q[d] * cache.value(0, pid, hk, off, d) for d in range(HEAD_DIM)))
    m = max(logits)
    w = [math.exp(x - m) for x in logits]
    z = math.fsum(w)
    out = []
    for d in range(HEAD_DIM):
        out.append(math.fsum(w[j] * cache.value(1, page_row[j // PAGE], hk, j % PAGE, d) for j in range(n_keys)) / z)
    return out


def argmax(row) -> int:
    best = None
    for i, x in enumerate(row):
        if x != x:
            continue
        if best is None or x > row[best]:
            best = i
    return 0 if best is None else best


def accept(logits_rows, drafts):
    """logits_rows: W rows; drafts: W-1 ids.  Returns (a, targets)."""
    t = [argmax(r) for r in logits_rows]
    a = 0
    while a < len(drafts) and drafts[a] == t[a]:
        a += 1
    return a, t


def accept_lazy(logits_rows, drafts, d):
    """Per-lane draft count d (0 <= d <= len(drafts)).  a is the largest k <= d
    such that the first k drafts equal the first k argmaxes; the argmaxes of
    rows 0 .. a are reported and -1 after them.  Returns (a, tokens)."""
    t = [argmax(r) for r in logits_rows]
    a = max(k for k in range(d + 1) if all(drafts[i] == t[i] for i in range(k)))
    return a, t[:a + 1] + [-1] * (len(logits_rows) - a - 1)


def accept_sampled(logits_rows, q_rows, drafts, u_accept, u_sample):
    """Lossless stochastic acceptance restated with exact sums: the ratio test
    u < p(x) / q(x) (a zero q accepts), the residual max(0, p - q), and the
    inverse CDF through exactly rounded prefix sums.  Returns (a, tokens)."""
    import math

    def softmax(row):
        m = max(row)
        e = [math.exp(v - m) for v in row]
        s = math.fsum(e)
        return [v / s for v in e]

    d = len(drafts)
    n = len(logits_rows[0])
    a = d
    for i in range(d):
        x = drafts[i]
        if not 0 <= x < n:
            a = i
            break
        p = softmax(logits_rows[i])
        q = q_rows[i][x]
        if not (q == 0.0 or u_accept[i] < p[x] / q):
            a = i
            break
    p = softmax(logits_rows[a])
    w = [max(0.0, p[x] - q_rows[a][x]) for x in range(n)] if a < d else p
    if math.fsum(w) <= 0.0:
        w = p
    z = math.fsum(w)
    target = u_sample * z
    k = next((x for x in range(n) if math.fsum(w[:x + 1]) > target), None)
    if k is None:
        k = max(x for x in range(n) if w[x] > 0.0)
    return a, list(drafts[:a]) + [k] + [-1] * (len(logits_rows) - a - 1)


def attention_keys(cache: Cache, q_bits, page_row, hk: int, positions, sm_scale: float):
    """Attention of one query row over an explicit list of cached positions."""
    import math
    q = [bf16(b) for b in q_bits]
    logits = []
    for pos in positions:
        pid, off = page_row[pos // PAGE], pos % PAGE
        logits.append(sm_scale * math.fsum(q[d] * cache.value(0, pid, hk, off, d) for d in range(HEAD_DIM)))
    m = max(logits)
    w = [math.exp(x - m) for x in logits]
    z = math.fsum(w)
    out = []
    for d in range(HEAD_DIM):
        out.append(math.fsum(w[k] * cache.value(1, page_row[pos // PAGE], hk, pos % PAGE, d)
                             for k, pos in enumerate(positions)) / z)
    return out


def tree_accept(logits_rows, tokens, parent):
    """Draft-tree acceptance stated over root-to-node paths: a node is accepted
    when every node on its path from the root carries the argmax of its
    parent's row; among accepted nodes the deepest wins, ties to the path
    that is smaller slot by slot.  Returns (a, path, out_tokens)."""
    W = len(tokens)
    t = [argmax(r) for r in logits_rows]

    def chain(i):
        out = [i]
        while out[-1] != 0:
            out.append(parent[out[-1]])
        return out[::-1]

    best = [0]
    for i in range(1, W):
        p = chain(i)
        if all(tokens[p[k + 1]] == t[p[k]] for k in range(len(p) - 1)):
            if len(p) > len(best) or (len(p) == len(best) and p < best):
                best = p
    a = len(best) - 1
    out = [tokens[s] for s in best[1:]] + [t[best[-1]]]
    return a, best + [-1] * (W - len(best)), out + [-1] * (W - len(out))
