"""verify_attn_noalloc: the allocation-free variant of verify_attn.

Some callers cannot allocate device memory when they call an operator: a
runtime that planned all of its device memory at start-up, a plugin host that
hands over only the operator's own tensors, or a latency-critical loop that
cannot afford an allocator's implicit synchronisation.  verify_attn_noalloc
serves them by taking its split-K scratch from a fixed array inside the
library.  These tests call it through the C ABI (the ctypes binding) and
check it against verify_attn with a fresh caller workspace, bit for bit (the
same kernels run on the same inputs), on two calls in a row of different
sizes -- a large one, then a smaller one that would expose anything the first
left behind in the shared array; and check that sizes whose scratch would
not fit the fixed array are refused before anything runs.

This file is named so that pytest collects it last."""
import numpy as np
import pytest
import torch

import synth
from gpu_util import SM_SCALE, bf16_dev, fill_both, i32_dev

pytestmark = pytest.mark.gpu


def _case(dtype, lens, W, seed):
    spec = synth.Spec("noalloc", seed, len(lens), 0, 0, 24, 4, W, dtype, None, 0.7, True)
    step = synth.make_step(spec, seq_lens=np.array(lens, np.int32), with_accept=False)
    gcache, _, _ = fill_both(spec, step, with_oracle=False)
    return spec, step, gcache


def _reference(sdva, gcache, step, q, table, seq, max_context):
    """verify_attn with a freshly allocated workspace filled with NaN bytes."""
    B, W, Hq = step.q.shape[:3]
    n = sdva.verify_attn_workspace_size(B, W, Hq, 4, max_context)
    ws = torch.full((n,), 0xFF, dtype=torch.uint8, device="cuda")
    ref = torch.empty((B, W, Hq, 128), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    sdva.verify_attn(gcache, q, table, seq, max_context, float(SM_SCALE), ref, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return ref


@pytest.mark.parametrize("dtype", [synth.KV_FP8, synth.KV_INT4, synth.KV_INT8, synth.KV_FP8_ROW])
def test_noalloc_matches_workspace_call_large_then_small(dtype):
    """Two calls in a row through the C ABI: first a large case (8 lanes up to
    60,000 tokens, the scratch filled with its split-K partials), then a
    smaller, different one (3 short lanes, other splits), so that a partial
    left over from the first call would show in the second.  Each equals
    verify_attn with a fresh NaN-filled workspace bit for bit: the two run
    the same kernels on the same inputs."""
    import speculative_decode_verify_append_gb300 as sdva

    cases = [([3000, 700, 12000, 60000, 64, 9000, 31000, 150], 16, 31), ([500, 64, 1300], 8, 32)]
    for lens, W, seed in cases:
        spec, step, gcache = _case(dtype, lens, W if dtype in (synth.KV_FP8, synth.KV_FP8_ROW) else min(W, 8), seed)
        B, Wn, Hq = step.q.shape[:3]
        max_context = max(lens)
        q, table, seq = bf16_dev(step.q), i32_dev(step.page_table), i32_dev(step.seq_lens)
        out = torch.full((B, Wn, Hq, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        sdva.verify_attn_noalloc(gcache, q, table, seq, max_context, float(SM_SCALE), out, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        ref = _reference(sdva, gcache, step, q, table, seq, max_context)
        assert torch.isfinite(ref.float()).all()
        assert torch.equal(out, ref), (lens, float((out.float() - ref.float()).abs().max()))


def test_noalloc_refuses_sizes_beyond_its_scratch():
    import speculative_decode_verify_append_gb300 as sdva

    g = sdva.KVCache(synth.KV_FP8, 4, 4)
    B, W, Hq = 64, 16, 24
    max_context = 1 << 20
    assert sdva.verify_attn_workspace_size(B, W, Hq, 4, max_context) > sdva.NOALLOC_SCRATCH_BYTES
    q = torch.zeros((B, W, Hq, 128), dtype=torch.bfloat16, device="cuda")
    table = torch.zeros((B, 4), dtype=torch.int32, device="cuda")
    seq = torch.zeros(B, dtype=torch.int32, device="cuda")
    out = torch.zeros_like(q)
    with pytest.raises(sdva.SdvaError) as e:
        sdva.verify_attn_noalloc(g, q, table, seq, max_context, float(SM_SCALE), out)
    assert e.value.code == sdva.ERR_WORKSPACE
