"""Plain CPU oracle for the speculative-decoding verify step.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg are the only callers.  The GPU library never imports this
package and this package never imports the GPU library.

The arithmetic lives in ``oracle.c`` (fp32 codecs written from their IEEE /
OCP definitions, fp64 attention, plain loops); this module compiles it with
gcc and marshals numpy arrays into it.  ``brute.py`` next to it is a second,
independent pure-Python statement of the same definitions used to pin the C
code on tiny inputs.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()

KV_FP8 = 0
KV_INT4 = 1
KV_INT8 = 2      # INT8 group-64 (fp16 scales), oracle only
KV_FP8_ROW = 3   # FP8 E4M3 with one fp32 scale per (token, head) row, oracle only
PAGE = 64
HEAD_DIM = 128


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (IEEE semantics: no contraction)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call([
            "gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
            "-o", tmp, _SRC, "-lm", "-lpthread",
        ])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            I = ctypes.c_int
            lib.oracle_e4m3_decode.restype = ctypes.c_double
            lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_encode.restype = ctypes.c_uint8
            lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
            lib.oracle_f16_decode.restype = ctypes.c_double
            lib.oracle_f16_decode.argtypes = [ctypes.c_uint16]
            lib.oracle_f16_encode.restype = ctypes.c_uint16
            lib.oracle_f16_encode.argtypes = [ctypes.c_float]
            lib.oracle_int4_group.restype = ctypes.c_uint16
            lib.oracle_int4_group.argtypes = [P, I, P]
            lib.oracle_int8_group.restype = ctypes.c_uint16
            lib.oracle_int8_group.argtypes = [P, I, P]
            lib.oracle_fp8_row.restype = ctypes.c_float
            lib.oracle_fp8_row.argtypes = [P, I, P]
            lib.oracle_append.restype = I
            lib.oracle_append.argtypes = [I, I, I, P, P, P, P, P, P, I, I, P, I, P, P]
            lib.oracle_verify_attn.restype = I
            lib.oracle_verify_attn.argtypes = [I, I, I, P, P, P, P, P, I, I, I, P, I, P, ctypes.c_float,
                                               P, P, I, I, P]
            lib.oracle_tree_attn.restype = I
            lib.oracle_tree_attn.argtypes = [I, I, I, P, P, P, P, P, I, I, I, P, I, P, P, ctypes.c_float, P, I, P]
            lib.oracle_tree_accept.restype = I
            lib.oracle_tree_accept.argtypes = [P, I, I, I, P, P, P, P, P, P, P]
            lib.oracle_decode_row.restype = I
            lib.oracle_decode_row.argtypes = [I, I, I, P, P, P, P, P, I, P, I, ctypes.c_float, P]
            lib.oracle_argmax.restype = I
            lib.oracle_argmax.argtypes = [P, I]
            lib.oracle_spec_accept.restype = I
            lib.oracle_spec_accept.argtypes = [P, I, I, I, P, P, P, P, P]
            lib.oracle_spec_accept_lazy.restype = I
            lib.oracle_spec_accept_lazy.argtypes = [P, I, I, I, P, P, P, P, P, P]
            lib.oracle_spec_accept_sampled.restype = I
            lib.oracle_spec_accept_sampled.argtypes = [P, P, I, I, I, P, P, P, P, P, P, P]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _as(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------------------
# codecs
# --------------------------------------------------------------------------
def e4m3_decode(code: int) -> float:
    return _load().oracle_e4m3_decode(int(code))


def e4m3_encode(x: float) -> int:
    return _load().oracle_e4m3_encode(float(x))


def f16_encode(x: float) -> int:
    return _load().oracle_f16_encode(float(x))


def f16_decode(bits: int) -> float:
    return _load().oracle_f16_decode(int(bits))


def int4_group(x) -> tuple[int, np.ndarray]:
    x = _as(x, np.float32)
    codes = np.zeros(x.size, np.int8)
    s = _load().oracle_int4_group(_ptr(x), x.size, _ptr(codes))
    return s, codes


def int8_group(x) -> tuple[int, np.ndarray]:
    """INT8 group codec: (fp16 scale bits, codes in [-127, 127])."""
    x = _as(x, np.float32)
    codes = np.zeros(x.size, np.int8)
    s = _load().oracle_int8_group(_ptr(x), x.size, _ptr(codes))
    return s, codes


def fp8_row(x) -> tuple[float, np.ndarray]:
    """FP8 row codec: (fp32 scale, E4M3 codes)."""
    x = _as(x, np.float32)
    codes = np.zeros(x.size, np.uint8)
    s = _load().oracle_fp8_row(_ptr(x), x.size, _ptr(codes))
    return float(np.float32(s)), codes


# --------------------------------------------------------------------------
# the cache
# --------------------------------------------------------------------------
class Cache:
    """Host copy of a paged KV cache in the library's byte layout.

    FP8:  codes uint8 [pages][Hkv][64][128], scales float32 [pages][Hkv]
    INT4: codes uint8 [pages][Hkv][64][64],  scales uint16 (fp16 bits) [pages][Hkv][64][4]
    INT8: codes uint8 (int8 bits) [pages][Hkv][64][128], scales uint16 (fp16 bits) [pages][Hkv][64][2]
    FP8_ROW: codes uint8 [pages][Hkv][64][128], scales float32 [pages][Hkv][64]
    """

    def __init__(self, dtype: int, num_pages: int, num_kv_heads: int):
        self.dtype = dtype
        self.num_pages = num_pages
        self.num_kv_heads = num_kv_heads
        if dtype == KV_FP8:
            shape = (num_pages, num_kv_heads, PAGE, HEAD_DIM)
            sshape, sdt = (num_pages, num_kv_heads), np.float32
        elif dtype == KV_INT8:
            shape = (num_pages, num_kv_heads, PAGE, HEAD_DIM)
            sshape, sdt = (num_pages, num_kv_heads, PAGE, HEAD_DIM // 64), np.uint16
        elif dtype == KV_FP8_ROW:
            shape = (num_pages, num_kv_heads, PAGE, HEAD_DIM)
            sshape, sdt = (num_pages, num_kv_heads, PAGE), np.float32
        else:
            shape = (num_pages, num_kv_heads, PAGE, HEAD_DIM // 2)
            sshape, sdt = (num_pages, num_kv_heads, PAGE, HEAD_DIM // 32), np.uint16
        self.k_codes = np.zeros(shape, np.uint8)
        self.v_codes = np.zeros(shape, np.uint8)
        self.k_scales = np.zeros(sshape, sdt)
        self.v_scales = np.zeros(sshape, sdt)

    def copy(self) -> "Cache":
        c = Cache.__new__(Cache)
        c.dtype, c.num_pages, c.num_kv_heads = self.dtype, self.num_pages, self.num_kv_heads
        for n in ("k_codes", "v_codes", "k_scales", "v_scales"):
            setattr(c, n, getattr(self, n).copy())
        return c

    def _args(self):
        return (self.dtype, self.num_pages, self.num_kv_heads, _ptr(self.k_codes), _ptr(self.v_codes),
                _ptr(self.k_scales), _ptr(self.v_scales))


def append(cache: Cache, k_new_bf16: np.ndarray, v_new_bf16: np.ndarray, page_table: np.ndarray,
           seq_lens: np.ndarray) -> int:
    """Write tokens [L_b, L_b + n_new) of every lane into the cache in place.

    k_new_bf16 / v_new_bf16: uint16 bf16 bits [B][n_new][Hkv][128].
    Returns the status bits (1 bad page id, 2 lane range overflow)."""
    k = _as(k_new_bf16, np.uint16)
    v = _as(v_new_bf16, np.uint16)
    pt = _as(page_table, np.int32)
    sl = _as(seq_lens, np.int32)
    B, n_new = k.shape[0], k.shape[1]
    st = np.zeros(1, np.int32)
    _load().oracle_append(*cache._args(), _ptr(k), _ptr(v), B, n_new, _ptr(pt), pt.shape[1], _ptr(sl), _ptr(st))
    return int(st[0])


def append_ragged(cache: Cache, k_new_bf16: np.ndarray, v_new_bf16: np.ndarray, page_table: np.ndarray,
                  seq_lens: np.ndarray, n_lane: np.ndarray) -> int:
    """Per-lane token counts: lane b writes only its first n_lane[b] tokens
    (0 <= n_lane[b] <= n_new), i.e. exactly what appending that lane's
    truncated window on its own writes; a lane with no token is not examined.
    A count outside [0, n_new] sets status bit 16 and leaves the lane alone.
    Returns the OR of the status bits."""
    k = _as(k_new_bf16, np.uint16)
    v = _as(v_new_bf16, np.uint16)
    pt = _as(page_table, np.int32)
    sl = _as(seq_lens, np.int32)
    n_new = k.shape[1]
    st = 0
    for b in range(k.shape[0]):
        n = int(n_lane[b])
        if n < 0 or n > n_new:
            st |= 16
        elif n > 0:
            st |= append(cache, k[b:b + 1, :n], v[b:b + 1, :n], pt[b:b + 1], sl[b:b + 1])
    return st


def verify_attn(cache: Cache, q_bf16: np.ndarray, page_table: np.ndarray, seq_lens: np.ndarray,
                sm_scale: float, rows=None, threads: int = 1) -> tuple[np.ndarray, int]:
    """fp64 attention of every window row over its visible keys.

    q_bf16: uint16 [B][W][Hq][128].  Returns (out, status) with out fp64
    [B][W][Hq][128], or [len(rows)][128] for an explicit list of (b, i, h)."""
    q = _as(q_bf16, np.uint16)
    pt = _as(page_table, np.int32)
    sl = _as(seq_lens, np.int32)
    B, W, Hq = q.shape[0], q.shape[1], q.shape[2]
    st = np.zeros(1, np.int32)
    if rows is None:
        out = np.zeros((B, W, Hq, HEAD_DIM), np.float64)
        rows_a, nrows = None, 0
    else:
        rows_a = _as(np.asarray(rows).reshape(-1, 3), np.int32)
        nrows = rows_a.shape[0]
        out = np.zeros((nrows, HEAD_DIM), np.float64)
    rc = _load().oracle_verify_attn(*cache._args(), _ptr(q), Hq, B, W, _ptr(pt), pt.shape[1], _ptr(sl),
                                    float(sm_scale), _ptr(out), _ptr(rows_a), nrows, int(threads), _ptr(st))
    if rc != 0:
        raise ValueError("oracle_verify_attn: invalid arguments")
    return out, int(st[0])


def verify_attn_ragged(cache: Cache, q_bf16: np.ndarray, page_table: np.ndarray, seq_lens: np.ndarray,
                       n_lane: np.ndarray, sm_scale: float, threads: int = 1) -> tuple[np.ndarray, int]:
    """Attention of a padded window with a row count per lane: lane b's rows
    i < n_lane[b] are verify_attn's rows (keys 0 .. L_b + i), its rows
    i >= n_lane[b] are zero; a count outside [0, W] zeroes the lane and sets
    status bit 16 (the per-workload draft count, as in append_ragged)."""
    q = _as(q_bf16, np.uint16)
    B, W = q.shape[0], q.shape[1]
    out, st = verify_attn(cache, q, page_table, seq_lens, sm_scale, threads=threads)
    for b in range(B):
        n = int(n_lane[b])
        if n < 0 or n > W:
            st |= 16
            out[b] = 0.0
        else:
            out[b, n:] = 0.0
    return out, st


def tree_attn(cache: Cache, q_bf16: np.ndarray, page_table: np.ndarray, seq_lens: np.ndarray,
              parent: np.ndarray, sm_scale: float, threads: int = 1) -> tuple[np.ndarray, int]:
    """fp64 attention of a draft tree's window: row i sees the context and the
    window keys of its ancestors and itself.  parent int32 [B][W] (entry 0
    unused, 0 <= parent[i] < i).  Returns (out fp64 [B][W][Hq][128], status)."""
    q = _as(q_bf16, np.uint16)
    pt = _as(page_table, np.int32)
    sl = _as(seq_lens, np.int32)
    par = _as(parent, np.int32)
    B, W, Hq = q.shape[0], q.shape[1], q.shape[2]
    st = np.zeros(1, np.int32)
    out = np.zeros((B, W, Hq, HEAD_DIM), np.float64)
    rc = _load().oracle_tree_attn(*cache._args(), _ptr(q), Hq, B, W, _ptr(pt), pt.shape[1], _ptr(sl), _ptr(par),
                                  float(sm_scale), _ptr(out), int(threads), _ptr(st))
    if rc != 0:
        raise ValueError("oracle_tree_attn: invalid arguments")
    return out, int(st[0])


def tree_accept(logits: np.ndarray, tokens: np.ndarray, parent: np.ndarray, seq_lens: np.ndarray | None = None):
    """Greedy acceptance of a draft tree.  logits [B][W][V]; tokens, parent int32
    [B][W].  Returns (accept_len [B], path [B][W] of accepted slots (root first,
    -1 after), out_tokens [B][W] (accepted tokens, the bonus, -1 after),
    new seq_lens or None, status)."""
    lg = _as(logits, np.float32)
    B, W, V = lg.shape
    tk = _as(tokens, np.int32).reshape(B, W)
    par = _as(parent, np.int32).reshape(B, W)
    acc = np.zeros(B, np.int32)
    path = np.zeros((B, W), np.int32)
    tok = np.zeros((B, W), np.int32)
    sl = None if seq_lens is None else _as(seq_lens, np.int32).copy()
    st = np.zeros(1, np.int32)
    _load().oracle_tree_accept(_ptr(lg), B, W, V, _ptr(tk), _ptr(par), _ptr(acc), _ptr(path), _ptr(tok), _ptr(sl),
                               _ptr(st))
    return acc, path, tok, sl, int(st[0])


def decode_row(cache: Cache, q_row_bf16: np.ndarray, kv_head: int, page_row: np.ndarray, n_keys: int,
               sm_scale: float) -> np.ndarray:
    """Independent single-pass plain decode of one query row over n_keys keys."""
    q = _as(q_row_bf16, np.uint16)
    pr = _as(page_row, np.int32)
    out = np.zeros(HEAD_DIM, np.float64)
    _load().oracle_decode_row(*cache._args(), _ptr(q), int(kv_head), _ptr(pr), int(n_keys), float(sm_scale),
                              _ptr(out))
    return out


def argmax(x: np.ndarray) -> int:
    x = _as(x, np.float32)
    return _load().oracle_argmax(_ptr(x), x.size)


def spec_accept(logits: np.ndarray, drafts: np.ndarray, seq_lens: np.ndarray | None = None):
    """Returns (accept_len [B], out_tokens [B][W], new seq_lens or None, status)."""
    lg = _as(logits, np.float32)
    B, W, V = lg.shape
    dr = _as(drafts, np.int32).reshape(B, W - 1) if W > 1 else np.zeros((B, 0), np.int32)
    acc = np.zeros(B, np.int32)
    tok = np.zeros((B, W), np.int32)
    sl = None if seq_lens is None else _as(seq_lens, np.int32).copy()
    st = np.zeros(1, np.int32)
    _load().oracle_spec_accept(_ptr(lg), B, W, V, _ptr(dr) if dr.size else None, _ptr(acc), _ptr(tok), _ptr(sl),
                               _ptr(st))
    return acc, tok, sl, int(st[0])


def spec_accept_lazy(logits: np.ndarray, drafts: np.ndarray, num_drafts: np.ndarray | None = None,
                     seq_lens: np.ndarray | None = None):
    """Lazy acceptance with per-lane draft counts (None: window - 1 each).
    Returns (accept_len [B], out_tokens [B][W] with -1 after row a, new seq_lens or None, status)."""
    lg = _as(logits, np.float32)
    B, W, V = lg.shape
    dr = _as(drafts, np.int32).reshape(B, W - 1) if W > 1 else np.zeros((B, 0), np.int32)
    nd = None if num_drafts is None else _as(num_drafts, np.int32).reshape(B)
    acc = np.zeros(B, np.int32)
    tok = np.zeros((B, W), np.int32)
    sl = None if seq_lens is None else _as(seq_lens, np.int32).copy()
    st = np.zeros(1, np.int32)
    _load().oracle_spec_accept_lazy(_ptr(lg), B, W, V, _ptr(dr) if dr.size else None, _ptr(nd), _ptr(acc),
                                    _ptr(tok), _ptr(sl), _ptr(st))
    return acc, tok, sl, int(st[0])


def spec_accept_sampled(logits: np.ndarray, draft_probs: np.ndarray, drafts: np.ndarray, u_accept: np.ndarray,
                        u_sample: np.ndarray, seq_lens: np.ndarray | None = None):
    """Lossless stochastic acceptance.  logits [B][W][V], draft_probs [B][W-1][V],
    drafts [B][W-1], u_accept [B][W-1], u_sample [B] (uniforms in [0, 1)).
    Returns (accept_len [B], out_tokens [B][W]: drafts, the drawn token, -1 after;
    new seq_lens or None, status)."""
    lg = _as(logits, np.float32)
    B, W, V = lg.shape
    q = _as(draft_probs, np.float32).reshape(B, W - 1, V) if W > 1 else np.zeros((B, 0, V), np.float32)
    dr = _as(drafts, np.int32).reshape(B, W - 1) if W > 1 else np.zeros((B, 0), np.int32)
    ua = _as(u_accept, np.float32).reshape(B, W - 1) if W > 1 else np.zeros((B, 0), np.float32)
    us = _as(u_sample, np.float32).reshape(B)
    acc = np.zeros(B, np.int32)
    tok = np.zeros((B, W), np.int32)
    sl = None if seq_lens is None else _as(seq_lens, np.int32).copy()
    st = np.zeros(1, np.int32)
    rc = _load().oracle_spec_accept_sampled(_ptr(lg), _ptr(q) if q.size else None, B, W, V,
                                            _ptr(dr) if dr.size else None, _ptr(ua) if ua.size else None, _ptr(us),
                                            _ptr(acc), _ptr(tok), _ptr(sl), _ptr(st))
    assert rc == 0
    return acc, tok, sl, int(st[0])
