"""A bounded device wait that runs out, on the GPU, without a fault.

The diagnostic hook sdva_debug_set_wait_limit makes every wait of
verify_attn's tensor-core kernels give up at once (a limit of zero cycles),
so that the first wait that is not already satisfied runs out -- the "flag
that nothing sets" of a real hang.  The call must raise SDVA_STATUS_TIMEOUT
and return; its kernels must drain their own copies and MMAs and free their
tensor memory, so that the next normal call (whose kernels allocate tensor
memory again) runs and is correct."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import SM_SCALE, assert_close, bf16_dev, fill_both, i32_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", [synth.KV_FP8, synth.KV_INT4, synth.KV_INT8, synth.KV_FP8_ROW])
def test_wait_that_runs_out_is_reported_and_recovered(dtype):
    import speculative_decode_verify_append_gb300 as sdva
    lens, W = [3000, 700, 12000, 64], 8
    spec = synth.Spec("timeout", 71, len(lens), 0, 0, 24, 4, W, dtype, None, 0.7, True)
    step = synth.make_step(spec, seq_lens=np.array(lens, np.int32), with_accept=False)
    g, o, _ = fill_both(spec, step)
    B, Hq = len(lens), 24
    q, t, L = bf16_dev(step.q), i32_dev(step.page_table), i32_dev(step.seq_lens)
    ws = torch.empty(sdva.verify_attn_workspace_size(B, W, Hq, 4, max(lens)), dtype=torch.uint8, device="cuda")
    out = torch.zeros((B, W, Hq, 128), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    prev = sdva.sdva_debug_set_wait_limit(0)
    try:
        sdva.verify_attn(g, q, t, L, max(lens), float(SM_SCALE), out, ws, st)
        torch.cuda.synchronize()  # the call returned: no hang, no fault
    finally:
        sdva.sdva_debug_set_wait_limit(prev)
    assert int(st.item()) & sdva.STATUS_TIMEOUT
    # the next calls, with the default limit, run and are right
    want, _ = oracle.verify_attn(o, step.q, step.page_table, step.seq_lens, SM_SCALE, threads=16)
    for _ in range(2):
        st.zero_()
        out.fill_(float("nan"))
        sdva.verify_attn(g, q, t, L, max(lens), float(SM_SCALE), out, ws, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert_close(out.float().cpu().numpy(), want, "after the timeout")
