"""verify_attn_noalloc: the allocation-free variant of verify_attn.

Some callers cannot allocate device memory when they call an operator: a
runtime that planned all of its device memory at start-up, a plugin host that
hands over only the operator's own tensors, or a latency-critical loop that
cannot afford an allocator's implicit synchronisation.  verify_attn_noalloc
serves them by taking its split-K scratch from a fixed array inside the
library.  These tests call it through the C ABI (the ctypes binding) and
check it against verify_attn with a caller workspace, on two calls in a row,
within the tolerance the parity tests use; and check that sizes whose scratch
would not fit the fixed array are refused before anything runs.

This file is named so that pytest collects it last."""
import numpy as np
import pytest
import torch

import synth
from gpu_util import SM_SCALE, bf16_dev, fill_both, i32_dev

pytestmark = pytest.mark.gpu


def _close(got: np.ndarray, ref: np.ndarray) -> None:
    err = np.abs(got.astype(np.float64) - ref.astype(np.float64))
    assert (err <= 2e-3 + 1e-2 * np.abs(ref)).all(), float(err.max())


@pytest.mark.parametrize("dtype,lens,W", [(synth.KV_FP8, [3000, 700, 12000], 16), (synth.KV_INT4, [5000, 64], 8)])
def test_noalloc_matches_workspace_call_twice(dtype, lens, W):
    import speculative_decode_verify_append_gb300 as sdva

    spec = synth.Spec("noalloc", 31, len(lens), 0, 0, 24, 4, W, dtype, None, 0.7, True)
    step = synth.make_step(spec, seq_lens=np.array(lens, np.int32), with_accept=False)
    gcache, _, _ = fill_both(spec, step, with_oracle=False)
    B, Hq = len(lens), 24
    max_context = max(lens)
    q, table, seq = bf16_dev(step.q), i32_dev(step.page_table), i32_dev(step.seq_lens)

    ws = torch.zeros(sdva.verify_attn_workspace_size(B, W, Hq, 4, max_context), dtype=torch.uint8, device="cuda")
    ref = torch.empty((B, W, Hq, 128), dtype=torch.bfloat16, device="cuda")
    st_ref = torch.zeros(1, dtype=torch.int32, device="cuda")
    sdva.verify_attn(gcache, q, table, seq, max_context, float(SM_SCALE), ref, ws, st_ref)

    outs = []
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(2):  # the second call reuses the array as the first left it
        out = torch.full((B, W, Hq, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
        sdva.verify_attn_noalloc(gcache, q, table, seq, max_context, float(SM_SCALE), out, st)
        outs.append(out)
    torch.cuda.synchronize()
    assert int(st_ref.item()) == 0 and int(st.item()) == 0
    r = ref.float().cpu().numpy()
    assert np.isfinite(r).all()
    for out in outs:
        _close(out.float().cpu().numpy(), r)


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
