"""Python binding of libsdva, the GB300 verify-step library.

Argument marshalling only: every step of the verify path runs in the CUDA
kernels of ``libsdva.so`` (built in-tree by ``build.py``).  There is no
Python or CPU fallback; importing this package without the built library
raises.  PyTorch supplies device memory and streams.

The calls mirror ``include/sdva.h``:

    kv_append_quant(cache, k_new, v_new, page_table, seq_lens, status=None, stream=None)
    kv_append_quant_ragged(cache, k_new, v_new, n_lane, page_table, seq_lens, status=None, stream=None)
    verify_attn_workspace_size(num_lanes, window, num_q_heads, num_kv_heads, max_context, num_sms=0)
    verify_attn(cache, q, page_table, seq_lens, max_context, sm_scale, out, workspace, status=None, stream=None)
    verify_attn_tree(cache, q, parent, page_table, seq_lens, max_context, sm_scale, out, workspace, status=None,
                     stream=None)
    verify_attn_ragged(cache, q, n_lane, page_table, seq_lens, max_context, sm_scale, out, workspace, status=None,
                       stream=None)
    verify_step(cache, k_new, v_new, q, page_table, seq_lens, max_context, sm_scale, out, workspace, logits, drafts,
                accept_len, out_tokens, commit=True, status=None, stream=None)
    spec_accept(logits, drafts, accept_len, out_tokens, seq_lens_inout=None, status=None, stream=None)
    spec_accept_lazy(logits, drafts, accept_len, out_tokens, num_drafts=None, seq_lens_inout=None, status=None,
                     stream=None)
    spec_accept_tree(logits, tokens, parent, accept_len, path, out_tokens, seq_lens_inout=None, status=None,
                     stream=None)
    spec_accept_sampled_workspace_size(num_lanes, window)
    spec_accept_sampled(logits, draft_probs, drafts, u_accept, u_sample, accept_len, out_tokens, workspace,
                        seq_lens_inout=None, status=None, stream=None)
    sdva_status_string(code)
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libsdva.so")

KV_FP8_E4M3 = 0
KV_INT4_G32 = 1
KV_INT8_G64 = 2
KV_FP8_ROW = 3
PAGE = 64
HEAD_DIM = 128
MAX_WINDOW = 16

OK = 0
ERR_INVALID = -1
ERR_UNSUPPORTED = -2
ERR_WORKSPACE = -3
ERR_CUDA = -4
STATUS_BAD_PAGE = 1
STATUS_OVERFLOW = 2
STATUS_BAD_DRAFT = 4
STATUS_TIMEOUT = 8
STATUS_BAD_COUNT = 16
STATUS_BAD_TREE = 32
LAZY_WALK_MIN_LANES = 48  # SDVA_LAZY_WALK_MIN_LANES: spec_accept_lazy walks rows from this many lanes on

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()' "
        "or python speculative_decode_verify_append_gb300/build.py)")

_lib = ctypes.CDLL(LIB_PATH)


class _KVCacheStruct(ctypes.Structure):
    _fields_ = [
        ("dtype", ctypes.c_int32),
        ("num_pages", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("k_codes", ctypes.c_void_p),
        ("v_codes", ctypes.c_void_p),
        ("k_scales", ctypes.c_void_p),
        ("v_scales", ctypes.c_void_p),
    ]


_P = ctypes.c_void_p
_I = ctypes.c_int
_lib.kv_append_quant.restype = _I
_lib.kv_append_quant.argtypes = [ctypes.POINTER(_KVCacheStruct), _P, _P, _I, _I, _P, _I, _P, _P, _P]
_lib.kv_append_quant_ragged.restype = _I
_lib.kv_append_quant_ragged.argtypes = [ctypes.POINTER(_KVCacheStruct), _P, _P, _I, _I, _P, _P, _I, _P, _P, _P]
_lib.verify_attn_workspace_size.restype = ctypes.c_size_t
_lib.verify_attn_workspace_size.argtypes = [_I, _I, _I, _I, _I, _I]
_lib.verify_attn.restype = _I
_lib.verify_attn.argtypes = [ctypes.POINTER(_KVCacheStruct), _P, _I, _I, _I, _P, _I, _P, _I, ctypes.c_float, _P,
                             _P, ctypes.c_size_t, _P, _P]
_lib.verify_attn_tree.restype = _I
_lib.verify_attn_tree.argtypes = [ctypes.POINTER(_KVCacheStruct), _P, _I, _I, _I, _P, _P, _I, _P, _I, ctypes.c_float,
                                  _P, _P, ctypes.c_size_t, _P, _P]
_lib.verify_attn_ragged.restype = _I
_lib.verify_attn_ragged.argtypes = [ctypes.POINTER(_KVCacheStruct), _P, _I, _I, _I, _P, _P, _I, _P, _I, ctypes.c_float,
                                    _P, _P, ctypes.c_size_t, _P, _P]
_lib.verify_step.restype = _I
_lib.verify_step.argtypes = [ctypes.POINTER(_KVCacheStruct), _P, _P, _P, _I, _I, _I, _P, _I, _P, _I, ctypes.c_float,
                             _P, _P, ctypes.c_size_t, _P, _I, _P, _P, _P, _I, _P, _P]
_lib.verify_attn_noalloc.restype = _I
_lib.verify_attn_noalloc.argtypes = [ctypes.POINTER(_KVCacheStruct), _P, _I, _I, _I, _P, _I, _P, _I, ctypes.c_float,
                                     _P, _P, _P]
_lib.spec_accept.restype = _I
_lib.spec_accept.argtypes = [_P, _I, _I, _I, _P, _P, _P, _P, _P, _P]
_lib.spec_accept_lazy.restype = _I
_lib.spec_accept_lazy.argtypes = [_P, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P]
_lib.spec_accept_tree.restype = _I
_lib.spec_accept_tree.argtypes = [_P, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P]
_lib.spec_accept_sampled_workspace_size.restype = ctypes.c_size_t
_lib.spec_accept_sampled_workspace_size.argtypes = [_I, _I]
_lib.spec_accept_sampled.restype = _I
_lib.spec_accept_sampled.argtypes = [_P, _P, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P, _P]
_lib.sdva_debug_set_wait_limit.restype = ctypes.c_longlong
_lib.sdva_debug_set_wait_limit.argtypes = [ctypes.c_longlong]
_lib.sdva_status_string.restype = ctypes.c_char_p
_lib.sdva_status_string.argtypes = [_I]

EXPORTED = ("kv_append_quant", "kv_append_quant_ragged", "verify_attn_workspace_size", "verify_attn",
            "verify_attn_tree", "verify_attn_ragged", "verify_step", "verify_attn_noalloc", "spec_accept", "spec_accept_lazy", "spec_accept_tree",
            "spec_accept_sampled_workspace_size", "spec_accept_sampled", "sdva_debug_set_wait_limit",
            "sdva_status_string")
NOALLOC_SCRATCH_BYTES = 32 << 20


class SdvaError(RuntimeError):
    def __init__(self, call: str, code: int):
        super().__init__(f"{call}: {sdva_status_string(code)} (code {code})")
        self.code = code


def sdva_debug_set_wait_limit(cycles: int) -> int:
    """Bound every device wait of verify_attn's tensor-core kernels at `cycles`
    clock cycles (negative: the default, about two seconds); returns the
    previous bound.  A wait that runs out raises STATUS_TIMEOUT."""
    return int(_lib.sdva_debug_set_wait_limit(int(cycles)))


def sdva_status_string(code: int) -> str:
    return _lib.sdva_status_string(int(code)).decode()


def _check(call: str, rc: int) -> None:
    if rc != OK:
        raise SdvaError(call, rc)


def _dptr(t: torch.Tensor | None, dtype: torch.dtype | None = None, name: str = "tensor"):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


class KVCache:
    """Caller-owned paged KV cache (device tensors in the library's layout).

    FP8:  k_codes/v_codes uint8 [pages][Hkv][64][128]; k_scales/v_scales float32 [pages][Hkv]
    INT4: k_codes/v_codes uint8 [pages][Hkv][64][64];  k_scales/v_scales float16 [pages][Hkv][64][4]
    INT8: k_codes/v_codes uint8 (int8 bits) [pages][Hkv][64][128]; k_scales/v_scales float16 [pages][Hkv][64][2]
    FP8_ROW: k_codes/v_codes uint8 [pages][Hkv][64][128]; k_scales/v_scales float32 [pages][Hkv][64]
    """

    def __init__(self, dtype: int, num_pages: int, num_kv_heads: int, device="cuda", tensors=None):
        self.dtype = int(dtype)
        self.num_pages = int(num_pages)
        self.num_kv_heads = int(num_kv_heads)
        if tensors is not None:
            self.k_codes, self.v_codes, self.k_scales, self.v_scales = tensors
        elif self.dtype == KV_FP8_E4M3:
            shape = (num_pages, num_kv_heads, PAGE, HEAD_DIM)
            self.k_codes = torch.zeros(shape, dtype=torch.uint8, device=device)
            self.v_codes = torch.zeros(shape, dtype=torch.uint8, device=device)
            self.k_scales = torch.zeros((num_pages, num_kv_heads), dtype=torch.float32, device=device)
            self.v_scales = torch.zeros((num_pages, num_kv_heads), dtype=torch.float32, device=device)
        elif self.dtype in (KV_INT4_G32, KV_INT8_G64, KV_FP8_ROW):
            if self.dtype == KV_INT4_G32:
                shape = (num_pages, num_kv_heads, PAGE, HEAD_DIM // 2)
                sshape, sdt = (num_pages, num_kv_heads, PAGE, HEAD_DIM // 32), torch.float16
            elif self.dtype == KV_INT8_G64:
                shape = (num_pages, num_kv_heads, PAGE, HEAD_DIM)
                sshape, sdt = (num_pages, num_kv_heads, PAGE, HEAD_DIM // 64), torch.float16
            else:
                shape = (num_pages, num_kv_heads, PAGE, HEAD_DIM)
                sshape, sdt = (num_pages, num_kv_heads, PAGE), torch.float32
            self.k_codes = torch.zeros(shape, dtype=torch.uint8, device=device)
            self.v_codes = torch.zeros(shape, dtype=torch.uint8, device=device)
            self.k_scales = torch.zeros(sshape, dtype=sdt, device=device)
            self.v_scales = torch.zeros(sshape, dtype=sdt, device=device)
        else:
            raise ValueError(f"unknown kv dtype {dtype}")

    @property
    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in (self.k_codes, self.v_codes, self.k_scales, self.v_scales))

    def struct(self) -> _KVCacheStruct:
        return _KVCacheStruct(self.dtype, self.num_pages, PAGE, self.num_kv_heads, HEAD_DIM,
                              _dptr(self.k_codes, name="k_codes"), _dptr(self.v_codes, name="v_codes"),
                              _dptr(self.k_scales, name="k_scales"), _dptr(self.v_scales, name="v_scales"))


def kv_append_quant(cache: KVCache, k_new: torch.Tensor, v_new: torch.Tensor, page_table: torch.Tensor,
                    seq_lens: torch.Tensor, status: torch.Tensor | None = None, stream=None) -> None:
    """k_new, v_new: bf16 [B][n_new][Hkv][128]; page_table int32 [B][max_pages]; seq_lens int32 [B]."""
    B, n_new = k_new.shape[0], k_new.shape[1]
    s = cache.struct()
    rc = _lib.kv_append_quant(ctypes.byref(s), _dptr(k_new, torch.bfloat16, "k_new"),
                              _dptr(v_new, torch.bfloat16, "v_new"), B, n_new,
                              _dptr(page_table, torch.int32, "page_table"), page_table.shape[1],
                              _dptr(seq_lens, torch.int32, "seq_lens"), _dptr(status, torch.int32, "status"),
                              _stream(stream))
    _check("kv_append_quant", rc)


def kv_append_quant_ragged(cache: KVCache, k_new: torch.Tensor, v_new: torch.Tensor, n_lane: torch.Tensor,
                           page_table: torch.Tensor, seq_lens: torch.Tensor, status: torch.Tensor | None = None,
                           stream=None) -> None:
    """As kv_append_quant; lane b writes only its first n_lane[b] tokens (int32 [B] on the device)."""
    B, n_new = k_new.shape[0], k_new.shape[1]
    if n_lane is None:
        raise ValueError("n_lane is required")
    s = cache.struct()
    rc = _lib.kv_append_quant_ragged(ctypes.byref(s), _dptr(k_new, torch.bfloat16, "k_new"),
                                     _dptr(v_new, torch.bfloat16, "v_new"), B, n_new,
                                     _dptr(n_lane, torch.int32, "n_lane"),
                                     _dptr(page_table, torch.int32, "page_table"), page_table.shape[1],
                                     _dptr(seq_lens, torch.int32, "seq_lens"), _dptr(status, torch.int32, "status"),
                                     _stream(stream))
    _check("kv_append_quant_ragged", rc)


def verify_attn_workspace_size(num_lanes: int, window: int, num_q_heads: int, num_kv_heads: int, max_context: int,
                               num_sms: int = 0) -> int:
    return int(_lib.verify_attn_workspace_size(num_lanes, window, num_q_heads, num_kv_heads, max_context, num_sms))


def verify_attn(cache: KVCache, q: torch.Tensor, page_table: torch.Tensor, seq_lens: torch.Tensor,
                max_context: int, sm_scale: float, out: torch.Tensor, workspace: torch.Tensor,
                status: torch.Tensor | None = None, stream=None) -> None:
    """q, out: bf16 [B][W][Hq][128]; workspace: uint8 device tensor of at least
    verify_attn_workspace_size(...) bytes (its contents do not matter)."""
    B, W, Hq = q.shape[0], q.shape[1], q.shape[2]
    s = cache.struct()
    rc = _lib.verify_attn(ctypes.byref(s), _dptr(q, torch.bfloat16, "q"), Hq, B, W,
                          _dptr(page_table, torch.int32, "page_table"), page_table.shape[1],
                          _dptr(seq_lens, torch.int32, "seq_lens"), int(max_context), float(sm_scale),
                          _dptr(out, torch.bfloat16, "out"), _dptr(workspace, None, "workspace"),
                          workspace.numel() * workspace.element_size(), _dptr(status, torch.int32, "status"),
                          _stream(stream))
    _check("verify_attn", rc)


def verify_attn_tree(cache: KVCache, q: torch.Tensor, parent: torch.Tensor | None, page_table: torch.Tensor,
                     seq_lens: torch.Tensor, max_context: int, sm_scale: float, out: torch.Tensor,
                     workspace: torch.Tensor, status: torch.Tensor | None = None, stream=None) -> None:
    """verify_attn over a draft-tree window: parent int32 [B][W] (slot 0 unused);
    row i sees the context and the window keys of its ancestors and itself."""
    B, W, Hq = q.shape[0], q.shape[1], q.shape[2]
    s = cache.struct()
    rc = _lib.verify_attn_tree(ctypes.byref(s), _dptr(q, torch.bfloat16, "q"), Hq, B, W,
                               _dptr(parent, torch.int32, "parent"), _dptr(page_table, torch.int32, "page_table"),
                               page_table.shape[1], _dptr(seq_lens, torch.int32, "seq_lens"), int(max_context),
                               float(sm_scale), _dptr(out, torch.bfloat16, "out"), _dptr(workspace, None, "workspace"),
                               workspace.numel() * workspace.element_size(), _dptr(status, torch.int32, "status"),
                               _stream(stream))
    _check("verify_attn_tree", rc)


def verify_attn_ragged(cache: KVCache, q: torch.Tensor, n_lane: torch.Tensor, page_table: torch.Tensor,
                       seq_lens: torch.Tensor, max_context: int, sm_scale: float, out: torch.Tensor,
                       workspace: torch.Tensor, status: torch.Tensor | None = None, stream=None) -> None:
    """verify_attn with a window row count per lane: n_lane int32 [B]; rows
    past a lane's count are written as zeros."""
    B, W, Hq = q.shape[0], q.shape[1], q.shape[2]
    s = cache.struct()
    rc = _lib.verify_attn_ragged(ctypes.byref(s), _dptr(q, torch.bfloat16, "q"), Hq, B, W,
                                 _dptr(n_lane, torch.int32, "n_lane"), _dptr(page_table, torch.int32, "page_table"),
                                 page_table.shape[1], _dptr(seq_lens, torch.int32, "seq_lens"), int(max_context),
                                 float(sm_scale), _dptr(out, torch.bfloat16, "out"),
                                 _dptr(workspace, None, "workspace"), workspace.numel() * workspace.element_size(),
                                 _dptr(status, torch.int32, "status"), _stream(stream))
    _check("verify_attn_ragged", rc)


def verify_step(cache: KVCache, k_new: torch.Tensor, v_new: torch.Tensor, q: torch.Tensor, page_table: torch.Tensor,
                seq_lens: torch.Tensor, max_context: int, sm_scale: float, out: torch.Tensor, workspace: torch.Tensor,
                logits: torch.Tensor, drafts: torch.Tensor | None, accept_len: torch.Tensor, out_tokens: torch.Tensor,
                commit: bool = True, status: torch.Tensor | None = None, stream=None) -> None:
    """kv_append_quant + verify_attn + spec_accept as one chain of programmatic
    dependent launches (same results as the three calls in order); with commit,
    seq_lens is advanced by 1 + accept_len."""
    B, W, Hq = q.shape[0], q.shape[1], q.shape[2]
    if logits.dim() != 3 or logits.shape[0] != B or logits.shape[1] != W:
        raise ValueError("logits must be [B][W][V]")
    s = cache.struct()
    rc = _lib.verify_step(ctypes.byref(s), _dptr(k_new, torch.bfloat16, "k_new"), _dptr(v_new, torch.bfloat16, "v_new"),
                          _dptr(q, torch.bfloat16, "q"), Hq, B, W, _dptr(page_table, torch.int32, "page_table"),
                          page_table.shape[1], _dptr(seq_lens, torch.int32, "seq_lens"), int(max_context),
                          float(sm_scale), _dptr(out, torch.bfloat16, "out"), _dptr(workspace, None, "workspace"),
                          workspace.numel() * workspace.element_size(), _dptr(logits, torch.float32, "logits"),
                          logits.shape[2], _dptr(drafts, torch.int32, "drafts"),
                          _dptr(accept_len, torch.int32, "accept_len"), _dptr(out_tokens, torch.int32, "out_tokens"),
                          1 if commit else 0, _dptr(status, torch.int32, "status"), _stream(stream))
    _check("verify_step", rc)


def verify_attn_noalloc(cache: KVCache, q: torch.Tensor, page_table: torch.Tensor, seq_lens: torch.Tensor,
                        max_context: int, sm_scale: float, out: torch.Tensor, status: torch.Tensor | None = None,
                        stream=None) -> None:
    """verify_attn with the library's fixed device scratch instead of a
    caller workspace (for callers that cannot allocate device memory)."""
    B, W, Hq = q.shape[0], q.shape[1], q.shape[2]
    s = cache.struct()
    rc = _lib.verify_attn_noalloc(ctypes.byref(s), _dptr(q, torch.bfloat16, "q"), Hq, B, W,
                                  _dptr(page_table, torch.int32, "page_table"), page_table.shape[1],
                                  _dptr(seq_lens, torch.int32, "seq_lens"), int(max_context), float(sm_scale),
                                  _dptr(out, torch.bfloat16, "out"), _dptr(status, torch.int32, "status"),
                                  _stream(stream))
    _check("verify_attn_noalloc", rc)


def spec_accept(logits: torch.Tensor, drafts: torch.Tensor | None, accept_len: torch.Tensor,
                out_tokens: torch.Tensor, seq_lens_inout: torch.Tensor | None = None,
                status: torch.Tensor | None = None, stream=None) -> None:
    """logits fp32 [B][W][V]; drafts int32 [B][W-1]; accept_len int32 [B]; out_tokens int32 [B][W]."""
    B, W, V = logits.shape
    rc = _lib.spec_accept(_dptr(logits, torch.float32, "logits"), B, W, V,
                          _dptr(drafts, torch.int32, "drafts") if W > 1 else None,
                          _dptr(accept_len, torch.int32, "accept_len"), _dptr(out_tokens, torch.int32, "out_tokens"),
                          _dptr(seq_lens_inout, torch.int32, "seq_lens_inout"), _dptr(status, torch.int32, "status"),
                          _stream(stream))
    _check("spec_accept", rc)


def spec_accept_lazy(logits: torch.Tensor, drafts: torch.Tensor | None, accept_len: torch.Tensor,
                     out_tokens: torch.Tensor, num_drafts: torch.Tensor | None = None,
                     seq_lens_inout: torch.Tensor | None = None, status: torch.Tensor | None = None,
                     stream=None) -> None:
    """As spec_accept, reading each lane's rows only up to its first disagreement;
    num_drafts int32 [B] (None: W-1 each); out_tokens is -1 after row accept_len."""
    B, W, V = logits.shape
    rc = _lib.spec_accept_lazy(_dptr(logits, torch.float32, "logits"), B, W, V,
                               _dptr(drafts, torch.int32, "drafts") if W > 1 else None,
                               _dptr(num_drafts, torch.int32, "num_drafts"),
                               _dptr(accept_len, torch.int32, "accept_len"),
                               _dptr(out_tokens, torch.int32, "out_tokens"),
                               _dptr(seq_lens_inout, torch.int32, "seq_lens_inout"),
                               _dptr(status, torch.int32, "status"), _stream(stream))
    _check("spec_accept_lazy", rc)


def spec_accept_tree(logits: torch.Tensor, tokens: torch.Tensor | None, parent: torch.Tensor | None,
                     accept_len: torch.Tensor, path: torch.Tensor, out_tokens: torch.Tensor,
                     seq_lens_inout: torch.Tensor | None = None, status: torch.Tensor | None = None,
                     stream=None) -> None:
    """logits fp32 [B][W][V]; tokens, parent int32 [B][W]; accept_len int32 [B];
    path, out_tokens int32 [B][W]."""
    B, W, V = logits.shape
    rc = _lib.spec_accept_tree(_dptr(logits, torch.float32, "logits"), B, W, V,
                               _dptr(tokens, torch.int32, "tokens") if W > 1 else None,
                               _dptr(parent, torch.int32, "parent") if W > 1 else None,
                               _dptr(accept_len, torch.int32, "accept_len"), _dptr(path, torch.int32, "path"),
                               _dptr(out_tokens, torch.int32, "out_tokens"),
                               _dptr(seq_lens_inout, torch.int32, "seq_lens_inout"),
                               _dptr(status, torch.int32, "status"), _stream(stream))
    _check("spec_accept_tree", rc)


def spec_accept_sampled_workspace_size(num_lanes: int, window: int) -> int:
    return int(_lib.spec_accept_sampled_workspace_size(num_lanes, window))


def spec_accept_sampled(logits: torch.Tensor, draft_probs: torch.Tensor | None, drafts: torch.Tensor | None,
                        u_accept: torch.Tensor | None, u_sample: torch.Tensor, accept_len: torch.Tensor,
                        out_tokens: torch.Tensor, workspace: torch.Tensor, seq_lens_inout: torch.Tensor | None = None,
                        status: torch.Tensor | None = None, stream=None) -> None:
    """logits fp32 [B][W][V]; draft_probs fp32 [B][W-1][V]; drafts int32 [B][W-1];
    u_accept fp32 [B][W-1]; u_sample fp32 [B]; workspace: uint8 device tensor of at
    least spec_accept_sampled_workspace_size(B, W) bytes."""
    B, W, V = logits.shape
    rc = _lib.spec_accept_sampled(_dptr(logits, torch.float32, "logits"),
                                  _dptr(draft_probs, torch.float32, "draft_probs") if W > 1 else None, B, W, V,
                                  _dptr(drafts, torch.int32, "drafts") if W > 1 else None,
                                  _dptr(u_accept, torch.float32, "u_accept") if W > 1 else None,
                                  _dptr(u_sample, torch.float32, "u_sample"),
                                  _dptr(accept_len, torch.int32, "accept_len"),
                                  _dptr(out_tokens, torch.int32, "out_tokens"),
                                  _dptr(seq_lens_inout, torch.int32, "seq_lens_inout"),
                                  _dptr(workspace, None, "workspace"), workspace.numel() * workspace.element_size(),
                                  _dptr(status, torch.int32, "status"), _stream(stream))
    _check("spec_accept_sampled", rc)


def raw_library() -> ctypes.CDLL:
    """The loaded C library (for callers that pass raw pointers themselves)."""
    return _lib
