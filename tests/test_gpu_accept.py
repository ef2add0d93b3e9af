"""GPU parity of spec_accept against the oracle: accept lengths, argmax
tokens and committed lengths bit-exact, on the workloads' vocabularies and on
hand-built ties, NaNs, signed zeros and odd vocabulary sizes."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import i32_dev

pytestmark = pytest.mark.gpu


def _run(logits, drafts, seq_lens=None):
    import speculative_decode_verify_append_gb300 as sdva
    B, W, V = logits.shape
    lg = torch.from_numpy(np.ascontiguousarray(logits)).cuda()
    dr = i32_dev(drafts.reshape(B, max(W - 1, 0))) if W > 1 else None
    acc = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    tok = torch.full((B, W), -1, dtype=torch.int32, device="cuda")
    sl = i32_dev(seq_lens) if seq_lens is not None else None
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    sdva.spec_accept(lg, dr, acc, tok, sl, st)
    torch.cuda.synchronize()
    return (acc.cpu().numpy(), tok.cpu().numpy(), None if sl is None else sl.cpu().numpy(), int(st.item()))


@pytest.mark.parametrize("name", ["tiny", "multi_lane", "long_context", "int4_12slot"])
def test_workload_parity(name):
    spec = synth.WORKLOADS[name]
    B, W = spec.num_lanes, spec.window
    logits, drafts, targets = synth.acceptance_inputs(spec, B, W, spec.vocab, spec.match_p)
    L = synth.context_lengths(spec)
    got = _run(logits, drafts, L)
    want = oracle.spec_accept(logits, drafts, L)
    assert np.array_equal(got[0], want[0]) and np.array_equal(got[1], want[1]) and np.array_equal(got[2], want[2])
    assert got[3] == want[3] == 0
    assert np.array_equal(got[1], targets)


def test_ties_nan_signed_zero_and_odd_vocab():
    rng = np.random.default_rng(3)
    for V in (1, 3, 7, 1000, 4097, 151937):
        B, W = 3, 5
        logits = rng.integers(-2, 3, size=(B, W, V)).astype(np.float32)  # heavy ties
        logits[0, 0, :] = np.nan
        logits[1, 1, : V // 2] = np.nan
        logits[2, 2, :] = -0.0
        logits[2, 2, V - 1] = 0.0
        logits[2, 3, :] = -np.inf
        drafts = rng.integers(0, 3, size=(B, W - 1)).astype(np.int32)
        got = _run(logits, drafts)
        want = oracle.spec_accept(logits, drafts)
        assert np.array_equal(got[1], want[1]), V
        assert np.array_equal(got[0], want[0]), V


def test_no_drafts_and_bad_drafts():
    logits = np.random.default_rng(0).standard_normal((4, 1, 999)).astype(np.float32)
    got = _run(logits, np.zeros((4, 0), np.int32), np.array([1, 2, 3, 4], np.int32))
    assert (got[0] == 0).all() and list(got[2]) == [2, 3, 4, 5]
    logits = np.zeros((2, 3, 50), np.float32)
    logits[:, :, 7] = 1.0
    got = _run(logits, np.array([[7, 50], [-1, 7]], np.int32))
    assert list(got[0]) == [1, 0] and got[3] == 4
