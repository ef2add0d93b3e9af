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


def _logits_dev(logits, offset=0):
    """Device copy of the logits; offset > 0 shifts the base by that many
    floats, so the rows are not 16-byte aligned."""
    flat = torch.from_numpy(np.ascontiguousarray(logits).reshape(-1))
    buf = torch.empty(flat.numel() + offset, dtype=torch.float32, device="cuda")
    lg = buf[offset:].view(logits.shape)
    lg.copy_(flat.view(logits.shape))
    return lg


def _run(logits, drafts, seq_lens=None, offset=0):
    import speculative_decode_verify_append_gb300 as sdva
    B, W, V = logits.shape
    lg = _logits_dev(logits, offset)
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


def test_unaligned_logits_take_the_scalar_path():
    rng = np.random.default_rng(8)
    logits = rng.integers(-3, 4, size=(3, 4, 4096)).astype(np.float32)
    drafts = logits.argmax(axis=2)[:, :3].astype(np.int32)
    got = _run(logits, drafts, offset=1)
    want = oracle.spec_accept(logits, drafts)
    assert np.array_equal(got[0], want[0]) and np.array_equal(got[1], want[1])


# ---- lazy acceptance with per-lane draft counts --------------------------

def _run_lazy(logits, drafts, num_drafts=None, seq_lens=None, offset=0):
    import speculative_decode_verify_append_gb300 as sdva
    B, W, V = logits.shape
    lg = _logits_dev(logits, offset)
    dr = i32_dev(drafts.reshape(B, max(W - 1, 0))) if W > 1 else None
    nd = i32_dev(num_drafts) if num_drafts is not None else None
    acc = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    tok = torch.full((B, W), -7, dtype=torch.int32, device="cuda")
    sl = i32_dev(seq_lens) if seq_lens is not None else None
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    sdva.spec_accept_lazy(lg, dr, acc, tok, nd, sl, st)
    torch.cuda.synchronize()
    return (acc.cpu().numpy(), tok.cpu().numpy(), None if sl is None else sl.cpu().numpy(), int(st.item()))


def _same(got, want):
    assert np.array_equal(got[0], want[0]), (got[0], want[0])
    assert np.array_equal(got[1], want[1])
    assert (got[2] is None and want[2] is None) or np.array_equal(got[2], want[2])
    assert got[3] == want[3]


@pytest.mark.parametrize("name", ["tiny", "multi_lane", "long_context", "int4_12slot"])
def test_lazy_workload_parity(name):
    spec = synth.WORKLOADS[name]
    B, W = spec.num_lanes, spec.window
    logits, drafts, _ = synth.acceptance_inputs(spec, B, W, spec.vocab, spec.match_p)
    L = synth.context_lengths(spec)
    want = oracle.spec_accept_lazy(logits, drafts, None, L)
    _same(_run_lazy(logits, drafts, None, L), want)
    # the eager call agrees on the accept length and on rows 0 .. a
    eager = oracle.spec_accept(logits, drafts)
    assert np.array_equal(want[0], eager[0])
    nd = np.random.default_rng(spec.seed).integers(0, W, size=B).astype(np.int32)
    _same(_run_lazy(logits, drafts, nd, L), oracle.spec_accept_lazy(logits, drafts, nd, L))


@pytest.mark.parametrize("offset", [0, 1])
def test_lazy_ties_nan_odd_vocab_and_deep_walks(offset):
    rng = np.random.default_rng(30 + offset)
    for V in (1, 3, 7, 1000, 4096, 4097, 32768, 151936, 151937):
        B, W = 5, 16
        logits = rng.integers(-2, 3, size=(B, W, V)).astype(np.float32)  # heavy ties
        logits[0, 1, :] = np.nan
        logits[1, 2, : V // 2] = np.nan
        logits[2, 3, :] = -0.0
        logits[2, 3, V - 1] = 0.0
        logits[3, 0, :] = -np.inf
        targets = np.array([[oracle.argmax(logits[b, i]) for i in range(W)] for b in range(B)], np.int32)
        # drafts agree with probability 0.9, so most lanes walk deep into the window
        drafts = np.where(rng.random((B, W - 1)) < 0.9, targets[:, :W - 1], (targets[:, :W - 1] + 1) % V)
        drafts = drafts.astype(np.int32)
        nd = np.array([15, 0, 7, 15, 3], np.int32)
        for counts in (None, nd):
            _same(_run_lazy(logits, drafts, counts, offset=offset), oracle.spec_accept_lazy(logits, drafts, counts))


def test_lazy_bad_counts_and_bad_drafts():
    rng = np.random.default_rng(9)
    B, W, V = 6, 8, 5000
    logits = rng.standard_normal((B, W, V)).astype(np.float32)
    targets = logits.argmax(axis=2).astype(np.int32)
    drafts = targets[:, :W - 1].copy()
    drafts[4, 5] = V + 3   # inside lane 4's count: flagged
    drafts[5, 6] = -1      # past lane 5's count: not read
    nd = np.array([7, -1, 8, 0, 7, 4], np.int32)
    L = np.arange(B, dtype=np.int32) * 100
    got = _run_lazy(logits, drafts, nd, L)
    want = oracle.spec_accept_lazy(logits, drafts, nd, L)
    _same(got, want)
    assert got[3] == 16 | 4 and list(got[0]) == [7, 0, 0, 0, 5, 4]
    assert (got[1][1] == -1).all() and (got[1][2] == -1).all() and list(got[2][1:3]) == [100, 200]


def test_lazy_window_of_one():
    logits = np.random.default_rng(1).standard_normal((3, 1, 151936)).astype(np.float32)
    got = _run_lazy(logits, np.zeros((3, 0), np.int32), None, np.array([4, 5, 6], np.int32))
    _same(got, oracle.spec_accept_lazy(logits, np.zeros((3, 0), np.int32), None, np.array([4, 5, 6], np.int32)))


# With 48 lanes or more the lazy call walks each lane's rows in order; the
# cases below sit on that side of the switch (the ones above on the other).
@pytest.mark.parametrize("V,offset", [(151936, 0), (151936, 1), (4097, 0), (1000, 0)])
def test_lazy_walk_parity(V, offset):
    rng = np.random.default_rng(40 + offset + V % 7)
    B, W = 48, 16
    logits = rng.standard_normal((B, W, V)).astype(np.float32)
    logits[3, 2, :] = np.nan
    logits[4, :, 5] = logits[4, :, 9] = 50.0  # a tie on every row of lane 4
    targets = np.array([[oracle.argmax(logits[b, i]) for i in range(W)] for b in range(B)], np.int32)
    drafts = np.where(rng.random((B, W - 1)) < 0.85, targets[:, :W - 1], (targets[:, :W - 1] + 1) % V)
    drafts = drafts.astype(np.int32)
    drafts[7, 0] = V  # out of vocabulary
    nd = rng.integers(0, W, size=B).astype(np.int32)
    nd[1], nd[2] = -1, W  # invalid counts
    L = rng.integers(0, 1000, size=B).astype(np.int32)
    for counts in (None, nd):
        _same(_run_lazy(logits, drafts, counts, L, offset=offset), oracle.spec_accept_lazy(logits, drafts, counts, L))


def test_lazy_walk_window_of_one_and_full_agreement():
    rng = np.random.default_rng(41)
    logits = rng.standard_normal((49, 1, 5000)).astype(np.float32)
    _same(_run_lazy(logits, np.zeros((49, 0), np.int32)), oracle.spec_accept_lazy(logits, np.zeros((49, 0), np.int32)))
    logits = rng.standard_normal((64, 16, 8192)).astype(np.float32)
    drafts = logits.argmax(axis=2)[:, :15].astype(np.int32)
    got = _run_lazy(logits, drafts)
    _same(got, oracle.spec_accept_lazy(logits, drafts))
    assert (got[0] == 15).all()
