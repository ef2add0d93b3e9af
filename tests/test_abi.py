"""The C ABI (no GPU): libsdva.so builds for sm_103a, loads, exports every
function include/sdva.h declares, and its pure-host logic (workspace sizing,
status strings, argument validation that returns before any CUDA call)
behaves as the header documents."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    path = __graft_entry__._load_builder().build()
    return ctypes.CDLL(path)


def _declared_functions():
    names = []
    for hdr in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not hdr.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", hdr)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M):
            name = m.group(1)
            if name not in ("if", "while", "sizeof", "defined"):
                names.append(name)
    return sorted(set(names))


def test_header_declares_the_three_calls():
    names = _declared_functions()
    for n in ("kv_append_quant", "verify_attn", "spec_accept", "verify_attn_workspace_size", "sdva_status_string"):
        assert n in names, names


def test_every_declared_symbol_is_exported(lib):
    path = lib._name
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for n in _declared_functions():
        assert n in exported, n
        assert getattr(lib, n) is not None


def test_library_targets_sm103a(lib):
    out = subprocess.run(["cuobjdump", "--list-elf", lib._name], capture_output=True, text=True)
    if out.returncode != 0:
        pytest.skip("cuobjdump unavailable")
    assert "sm_103a" in out.stdout


def test_workspace_size_host_logic(lib):
    f = lib.verify_attn_workspace_size
    f.restype = ctypes.c_size_t
    f.argtypes = [ctypes.c_int] * 6
    a = f(8, 16, 24, 4, 65536, 152)
    b = f(8, 16, 24, 4, 131072, 152)
    assert a > 0 and b >= a
    assert f(1, 1, 24, 4, 32768, 152) > 0
    assert f(1, 17, 24, 4, 1000, 152) == 0     # window > 16
    assert f(1, 4, 25, 4, 1000, 152) == 0      # Hq % Hkv != 0
    assert f(0, 4, 24, 4, 1000, 152) == 0
    # partials: (m, l) + 128 fp32 per row per split, 256-byte aligned sections
    assert a % 4 == 0


def test_status_strings(lib):
    f = lib.sdva_status_string
    f.restype = ctypes.c_char_p
    f.argtypes = [ctypes.c_int]
    for code in (0, -1, -2, -3, -4, 1, 2, 4, 8, 16, 32, 3, -99):
        s = f(code)
        assert s and len(s) >= 2


class _Cache(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int32), ("num_pages", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("k_codes", ctypes.c_void_p),
                ("v_codes", ctypes.c_void_p), ("k_scales", ctypes.c_void_p), ("v_scales", ctypes.c_void_p)]


def test_argument_validation_returns_before_cuda(lib):
    P = ctypes.c_void_p
    fake = P(0x1000)  # never dereferenced: every call below fails validation first
    c = _Cache(0, 4, 64, 1, 128, fake, fake, fake, fake)
    rag = lib.kv_append_quant_ragged
    rag.restype = ctypes.c_int
    assert rag(ctypes.byref(c), fake, fake, 1, 1, None, fake, 1, fake, None, None) == -1  # counts required
    assert rag(ctypes.byref(c), fake, fake, 1, 0, fake, fake, 1, fake, None, None) == -1
    app = lib.kv_append_quant
    app.restype = ctypes.c_int
    assert app(ctypes.byref(c), None, fake, 1, 1, fake, 1, fake, None, None) == -1
    assert app(ctypes.byref(c), fake, fake, 1, 0, fake, 1, fake, None, None) == -1
    c.head_dim = 64
    assert app(ctypes.byref(c), fake, fake, 1, 1, fake, 1, fake, None, None) == -2
    c.head_dim, c.page_size = 128, 32
    assert app(ctypes.byref(c), fake, fake, 1, 1, fake, 1, fake, None, None) == -2
    c.page_size, c.dtype = 64, 7
    assert app(ctypes.byref(c), fake, fake, 1, 1, fake, 1, fake, None, None) == -2
    c.dtype = -1
    assert app(ctypes.byref(c), fake, fake, 1, 1, fake, 1, fake, None, None) == -2
    # every format's four cache arrays must be 16-byte aligned
    for dt in range(4):
        for field in ("k_codes", "v_codes", "k_scales", "v_scales"):
            c.dtype = dt
            setattr(c, field, P(0x1004))
            assert app(ctypes.byref(c), fake, fake, 1, 1, fake, 1, fake, None, None) == -1, (dt, field)
            setattr(c, field, fake)
    c.dtype = 0
    va = lib.verify_attn
    va.restype = ctypes.c_int
    va.argtypes = [P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, ctypes.c_int, P, ctypes.c_int, ctypes.c_float,
                   P, P, ctypes.c_size_t, P, P]
    assert va(ctypes.byref(c), fake, 4, 1, 17, fake, 1, fake, 10, 0.088, fake, fake, 1 << 20, None, None) == -2
    c.num_kv_heads = 2
    assert va(ctypes.byref(c), fake, 3, 1, 4, fake, 1, fake, 10, 0.088, fake, fake, 1 << 20, None, None) == -1
    c.num_kv_heads = 1
    assert va(ctypes.byref(c), fake, 4, 1, 4, fake, 1, fake, 10, -1.0, fake, fake, 1 << 20, None, None) == -1
    assert va(ctypes.byref(c), None, 4, 1, 4, fake, 1, fake, 10, 0.088, fake, fake, 1 << 20, None, None) == -1
    # q and out are read and written in 16-byte vectors: both must be 16-byte aligned
    odd = P(0x1008)
    assert va(ctypes.byref(c), odd, 4, 1, 4, fake, 1, fake, 10, 0.088, fake, fake, 1 << 20, None, None) == -1
    assert va(ctypes.byref(c), fake, 4, 1, 4, fake, 1, fake, 10, 0.088, odd, fake, 1 << 20, None, None) == -1
    for dt in range(4):
        c.dtype, c.v_scales = dt, P(0x1004)
        assert va(ctypes.byref(c), fake, 4, 1, 4, fake, 1, fake, 10, 0.088, fake, fake, 1 << 20, None, None) == -1
    c.dtype, c.v_scales = 4, fake
    assert va(ctypes.byref(c), fake, 4, 1, 4, fake, 1, fake, 10, 0.088, fake, fake, 1 << 20, None, None) == -2
    c.dtype = 0
    sa = lib.spec_accept
    sa.restype = ctypes.c_int
    assert sa(fake, 1, 4, 100, None, fake, fake, None, None, None) == -1   # drafts needed when window > 1
    assert sa(fake, 0, 4, 100, fake, fake, fake, None, None, None) == -1
    assert sa(fake, 1, 17, 100, fake, fake, fake, None, None, None) == -2
    ws = lib.spec_accept_sampled_workspace_size
    ws.restype = ctypes.c_size_t
    ws.argtypes = [ctypes.c_int, ctypes.c_int]
    assert ws(8, 16) >= 8 * 16 * 8 and ws(8, 16) % 256 == 0 and ws(0, 4) == 0
    sm = lib.spec_accept_sampled
    sm.restype = ctypes.c_int
    sm.argtypes = [P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, P, P, P, P, P, ctypes.c_size_t, P, P]
    assert sm(fake, None, 2, 4, 100, fake, fake, fake, fake, fake, None, fake, 4096, None, None) == -1  # q needed
    assert sm(fake, fake, 2, 4, 100, fake, fake, None, fake, fake, None, fake, 4096, None, None) == -1  # u_sample
    assert sm(fake, fake, 2, 17, 100, fake, fake, fake, fake, fake, None, fake, 4096, None, None) == -2
    assert sm(fake, fake, 2, 4, 100, fake, fake, fake, fake, fake, None, fake, 8, None, None) == -3  # too small
    assert sm(fake, fake, 2, 4, 100, fake, fake, fake, fake, fake, None, None, 4096, None, None) == -3
    assert sm(fake, fake, 2, 4, 100, fake, fake, fake, fake, fake, None, P(0x1004), 4096, None, None) == -3
    tr = lib.spec_accept_tree
    tr.restype = ctypes.c_int
    assert tr(fake, 2, 4, 100, None, fake, fake, fake, fake, None, None, None) == -1  # tokens needed
    assert tr(fake, 2, 4, 100, fake, fake, fake, None, fake, None, None, None) == -1  # path needed
    assert tr(fake, 2, 17, 100, fake, fake, fake, fake, fake, None, None, None) == -2
    lz = lib.spec_accept_lazy
    lz.restype = ctypes.c_int
    assert lz(fake, 1, 4, 100, None, None, fake, fake, None, None, None) == -1   # drafts needed when window > 1
    assert lz(fake, 1, 4, 0, fake, None, fake, fake, None, None, None) == -1
    assert lz(fake, 1, 4, 100, fake, None, None, fake, None, None, None) == -1
    assert lz(fake, 1, 17, 100, fake, fake, fake, fake, None, None, None) == -2
    assert lz(fake, 5000, 16, 100, fake, fake, fake, fake, None, None, None) == -2  # more than 65535 rows


def test_header_constants_match_the_binding(lib):
    text = open(os.path.join(ROOT, "include", "sdva.h")).read()
    defs = dict(re.findall(r"#define (SDVA_\w+) \(?(-?\d+)\)?", text))
    import speculative_decode_verify_append_gb300 as sdva
    assert int(defs["SDVA_LAZY_WALK_MIN_LANES"]) == sdva.LAZY_WALK_MIN_LANES
    assert int(defs["SDVA_STATUS_BAD_COUNT"]) == sdva.STATUS_BAD_COUNT
    assert int(defs["SDVA_STATUS_BAD_TREE"]) == sdva.STATUS_BAD_TREE
    assert int(defs["SDVA_STATUS_BAD_DRAFT"]) == sdva.STATUS_BAD_DRAFT
    assert int(defs["SDVA_ERR_WORKSPACE"]) == sdva.ERR_WORKSPACE
    kinds = dict(re.findall(r"SDVA_KV_(\w+) = (\d+)", text))
    assert {k: int(v) for k, v in kinds.items()} == {"FP8_E4M3": 0, "INT4_G32": 1, "INT8_G64": 2, "FP8_ROW": 3}
    assert (sdva.KV_FP8_E4M3, sdva.KV_INT4_G32, sdva.KV_INT8_G64, sdva.KV_FP8_ROW) == (0, 1, 2, 3)
    import oracle
    import synth
    assert (oracle.KV_FP8, oracle.KV_INT4, oracle.KV_INT8, oracle.KV_FP8_ROW) == (0, 1, 2, 3)
    assert (synth.KV_FP8, synth.KV_INT4, synth.KV_INT8, synth.KV_FP8_ROW) == (0, 1, 2, 3)
    m = re.search(r"#define SDVA_NOALLOC_SCRATCH_BYTES \(\(size_t\)(\d+) << (\d+)\)", text)
    assert m, "SDVA_NOALLOC_SCRATCH_BYTES not found"
    assert int(m.group(1)) << int(m.group(2)) == sdva.NOALLOC_SCRATCH_BYTES


def test_tree_verify_rejects_a_missing_parent_array(lib):
    """verify_attn_tree validates its arguments on the host: a window of more
    than one slot needs the parent array."""
    f = lib.verify_attn_tree
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p]
    fake = ctypes.c_void_p(256)
    assert f(fake, fake, 24, 2, 4, None, fake, 8, fake, 1000, 0.088, fake, fake, 1 << 20, None, None) == -1
    g = lib.verify_attn_ragged  # the per-lane row counts are required
    g.restype, g.argtypes = ctypes.c_int, f.argtypes
    assert g(fake, fake, 24, 2, 4, None, fake, 8, fake, 1000, 0.088, fake, fake, 1 << 20, None, None) == -1


def test_header_is_plain_c(tmp_path):
    """sdva.h compiles as C99 with warnings as errors, and every prototype
    has the type a C caller expects."""
    src = tmp_path / "use_sdva.c"
    src.write_text(r'''
#include "sdva.h"
typedef int (*append_fn)(const sdva_kv_cache*, const void*, const void*, int, int, const int32_t*, int,
                         const int32_t*, int32_t*, sdva_stream_t);
typedef int (*ragged_fn)(const sdva_kv_cache*, const void*, const void*, int, int, const int32_t*,
                         const int32_t*, int, const int32_t*, int32_t*, sdva_stream_t);
typedef size_t (*ws_fn)(int, int, int, int, int, int);
typedef int (*verify_fn)(const sdva_kv_cache*, const void*, int, int, int, const int32_t*, int, const int32_t*,
                         int, float, void*, void*, size_t, int32_t*, sdva_stream_t);
typedef int (*accept_fn)(const float*, int, int, int, const int32_t*, int32_t*, int32_t*, int32_t*, int32_t*,
                         sdva_stream_t);
typedef int (*lazy_fn)(const float*, int, int, int, const int32_t*, const int32_t*, int32_t*, int32_t*, int32_t*,
                       int32_t*, sdva_stream_t);
typedef int (*tree_fn)(const float*, int, int, int, const int32_t*, const int32_t*, int32_t*, int32_t*, int32_t*,
                       int32_t*, int32_t*, sdva_stream_t);
typedef int (*noalloc_fn)(const sdva_kv_cache*, const void*, int, int, int, const int32_t*, int, const int32_t*,
                          int, float, void*, int32_t*, sdva_stream_t);
typedef int (*step_fn)(const sdva_kv_cache*, const void*, const void*, const void*, int, int, int, const int32_t*, int,
                       int32_t*, int, float, void*, void*, size_t, const float*, int, const int32_t*, int32_t*,
                       int32_t*, int, int32_t*, sdva_stream_t);
typedef int (*tree_verify_fn)(const sdva_kv_cache*, const void*, int, int, int, const int32_t*, const int32_t*, int,
                              const int32_t*, int, float, void*, void*, size_t, int32_t*, sdva_stream_t);
typedef size_t (*sws_fn)(int, int);
typedef int (*sampled_fn)(const float*, const float*, int, int, int, const int32_t*, const float*, const float*,
                          int32_t*, int32_t*, int32_t*, void*, size_t, int32_t*, sdva_stream_t);
typedef const char* (*str_fn)(int);
typedef long long (*limit_fn)(long long);
int check(void) {
    append_fn a = kv_append_quant;
    ragged_fn r = kv_append_quant_ragged;
    ws_fn w = verify_attn_workspace_size;
    verify_fn v = verify_attn;
    accept_fn s = spec_accept;
    lazy_fn l = spec_accept_lazy;
    tree_fn t = spec_accept_tree;
    noalloc_fn n = verify_attn_noalloc;
    tree_verify_fn tv = verify_attn_tree;
    tree_verify_fn rv = verify_attn_ragged;
    step_fn vs = verify_step;
    sws_fn sw = spec_accept_sampled_workspace_size;
    sampled_fn sm = spec_accept_sampled;
    str_fn st = sdva_status_string;
    limit_fn lim = sdva_debug_set_wait_limit;
    return (a != 0) + (r != 0) + (w != 0) + (v != 0) + (n != 0) + (tv != 0) + (rv != 0) + (vs != 0) + (s != 0) + (l != 0) +
           (t != 0) +
           (sw != 0) +
           (sm != 0) +
           (st != 0) + (lim != 0) + SDVA_OK + SDVA_KV_FP8_E4M3 + SDVA_LAZY_WALK_MIN_LANES;
}
''')
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I",
                        os.path.join(ROOT, "include"), "-c", str(src), "-o", str(tmp_path / "use_sdva.o")],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
