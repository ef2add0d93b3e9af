"""Pins for the oracle's acceptance rule (no GPU): brute force, hand-built
edge cases (ties, NaN, +-0, all-match, first mismatch) and the closed form
of the mean accept length when each draft matches independently with
probability p: E[a] = sum_{k=1..d} p^k."""
import numpy as np
import pytest

import oracle
import synth
from oracle import brute


def test_matches_brute_on_random_rows():
    rng = np.random.default_rng(4)
    for trial in range(40):
        B, W, V = 3, 1 + trial % 6, 50
        logits = rng.integers(-3, 4, size=(B, W, V)).astype(np.float32)  # many ties
        drafts = rng.integers(0, 4, size=(B, W - 1)).astype(np.int32)
        acc, tok, sl, st = oracle.spec_accept(logits, drafts, np.array([10, 20, 30], np.int32))
        for b in range(B):
            a, t = brute.accept(logits[b].tolist(), [int(x) for x in drafts[b]])
            assert acc[b] == a and list(tok[b]) == t
            assert sl[b] == [10, 20, 30][b] + 1 + a


def test_ties_nan_and_signed_zero():
    assert oracle.argmax(np.array([1.0, 3.0, 3.0, 2.0], np.float32)) == 1
    assert oracle.argmax(np.array([np.nan, -1.0, -1.0], np.float32)) == 1
    assert oracle.argmax(np.array([np.nan, np.nan], np.float32)) == 0
    assert oracle.argmax(np.array([-0.0, 0.0], np.float32)) == 0
    assert oracle.argmax(np.array([-np.inf, -np.inf], np.float32)) == 0
    assert oracle.argmax(np.array([-np.inf, np.nan, 5.0, np.inf], np.float32)) == 3


def test_all_match_and_first_mismatch():
    spec = synth.WORKLOADS["tiny"]
    logits, drafts, targets = synth.acceptance_inputs(spec, 4, 6, 300, 1.0)
    acc, tok, _, st = oracle.spec_accept(logits, drafts)
    assert (acc == 5).all() and (tok == targets).all() and st == 0
    drafts[:, 0] = (targets[:, 0] + 1) % 300
    acc, tok, _, _ = oracle.spec_accept(logits, drafts)
    assert (acc == 0).all()
    # bonus token = target at position a
    drafts[:, 0] = targets[:, 0]
    drafts[:, 2] = (targets[:, 2] + 1) % 300
    acc, tok, _, _ = oracle.spec_accept(logits, drafts)
    assert (acc == 2).all() and (tok[:, 2] == targets[:, 2]).all()


def test_window_of_one_has_no_drafts():
    logits = np.random.default_rng(0).standard_normal((2, 1, 40)).astype(np.float32)
    acc, tok, sl, _ = oracle.spec_accept(logits, np.zeros((2, 0), np.int32), np.array([5, 6], np.int32))
    assert (acc == 0).all() and list(sl) == [6, 7]
    assert list(tok[:, 0]) == [int(np.argmax(logits[0, 0])), int(np.argmax(logits[1, 0]))]


def test_out_of_vocab_draft_is_flagged_and_never_matches():
    logits = np.zeros((1, 3, 8), np.float32)
    logits[0, :, 2] = 1.0
    acc, tok, _, st = oracle.spec_accept(logits, np.array([[2, 99]], np.int32))
    assert st == 4 and acc[0] == 1


@pytest.mark.parametrize("d,p", [(3, 0.7), (15, 0.7), (5, 0.7), (7, 0.5)])
def test_mean_accept_length_closed_form(d, p):
    spec = synth.WORKLOADS["tiny"]
    lanes = 4000
    logits, drafts, _ = synth.acceptance_inputs(spec, lanes, d + 1, 64, p, tag=f"mean{d}")
    acc, _, _, _ = oracle.spec_accept(logits, drafts)
    want = sum(p ** k for k in range(1, d + 1))
    # standard error of the mean is below 0.05 at these sizes; allow 4 sigma
    var = np.var(acc)
    assert abs(acc.mean() - want) < 4 * np.sqrt(var / lanes) + 1e-9


# ---- lazy acceptance with per-lane draft counts --------------------------

def test_lazy_matches_brute_with_per_lane_counts():
    rng = np.random.default_rng(14)
    for trial in range(40):
        B, W, V = 4, 1 + trial % 7, 30
        logits = rng.integers(-3, 4, size=(B, W, V)).astype(np.float32)  # many ties
        logits[0, rng.integers(0, W), rng.integers(0, V, size=5)] = np.nan
        targets = logits.argmax(axis=2)
        drafts = np.where(rng.random((B, W - 1)) < 0.6, targets[:, :W - 1],
                          rng.integers(0, V, size=(B, W - 1))).astype(np.int32)
        nd = rng.integers(0, W, size=B).astype(np.int32)
        L = np.array([3, 1, 4, 1], np.int32)
        acc, tok, sl, st = oracle.spec_accept_lazy(logits, drafts, nd, L)
        assert st == 0
        for b in range(B):
            a, t = brute.accept_lazy(logits[b].tolist(), [int(x) for x in drafts[b]], int(nd[b]))
            assert acc[b] == a and list(tok[b]) == t, (trial, b)
            assert sl[b] == L[b] + 1 + a


def test_lazy_rows_after_the_first_disagreement_decide_nothing():
    rng = np.random.default_rng(15)
    B, W, V = 6, 9, 200
    logits = rng.standard_normal((B, W, V)).astype(np.float32)
    targets = logits.argmax(axis=2)
    drafts = np.where(rng.random((B, W - 1)) < 0.7, targets[:, :W - 1], (targets[:, :W - 1] + 1) % V)
    drafts = drafts.astype(np.int32)
    acc, tok, _, _ = oracle.spec_accept_lazy(logits, drafts)
    poisoned = logits.copy()
    for b in range(B):
        poisoned[b, acc[b] + 1:, :] = np.nan
        poisoned[b, acc[b] + 1:, 7] = np.inf
    acc2, tok2, _, _ = oracle.spec_accept_lazy(poisoned, drafts)
    assert np.array_equal(acc, acc2) and np.array_equal(tok, tok2)
    # the eager rule agrees on the accept length and on rows 0 .. a
    acc3, tok3, _, _ = oracle.spec_accept(logits, drafts)
    assert np.array_equal(acc, acc3)
    for b in range(B):
        assert list(tok[b, :acc[b] + 1]) == list(tok3[b, :acc[b] + 1])
        assert (tok[b, acc[b] + 1:] == -1).all()


def test_lazy_counts_zero_full_and_invalid():
    spec = synth.WORKLOADS["tiny"]
    logits, drafts, targets = synth.acceptance_inputs(spec, 5, 6, 300, 1.0)
    # every draft agrees: a = d_b, bonus = the target at row d_b
    nd = np.array([0, 1, 5, 3, 2], np.int32)
    acc, tok, sl, st = oracle.spec_accept_lazy(logits, drafts, nd, np.zeros(5, np.int32))
    assert list(acc) == list(nd) and st == 0 and list(sl) == list(1 + nd)
    for b in range(5):
        assert list(tok[b, :nd[b] + 1]) == list(targets[b, :nd[b] + 1]) and (tok[b, nd[b] + 1:] == -1).all()
    # no count array means window - 1 drafts everywhere
    acc, tok, _, _ = oracle.spec_accept_lazy(logits, drafts)
    assert (acc == 5).all() and np.array_equal(tok, targets)
    # a count outside [0, window - 1]: flagged, lane skipped, no commit
    nd = np.array([-1, 6, 2, 0, 5], np.int32)
    acc, tok, sl, st = oracle.spec_accept_lazy(logits, drafts, nd, np.full(5, 10, np.int32))
    assert st == 16 and list(acc) == [0, 0, 2, 0, 5]
    assert (tok[:2] == -1).all() and list(sl) == [10, 10, 13, 11, 16]


def test_lazy_bad_drafts_only_within_the_lane_count():
    logits = np.zeros((2, 4, 8), np.float32)
    logits[:, :, 2] = 1.0
    drafts = np.array([[2, 2, 99], [2, -5, 2]], np.int32)
    _, _, _, st = oracle.spec_accept_lazy(logits, drafts, np.array([2, 1], np.int32))
    assert st == 0  # the bad ids lie past each lane's count
    acc, _, _, st = oracle.spec_accept_lazy(logits, drafts, np.array([3, 2], np.int32))
    assert st == 4 and list(acc) == [2, 1]


@pytest.mark.parametrize("p", [0.7, 0.5])
def test_lazy_mean_accept_length_closed_form_per_lane_count(p):
    spec = synth.WORKLOADS["tiny"]
    lanes, W = 4000, 10
    logits, drafts, _ = synth.acceptance_inputs(spec, lanes, W, 64, p, tag=f"lazy{p}")
    nd = (np.arange(lanes) % W).astype(np.int32)
    acc, _, _, _ = oracle.spec_accept_lazy(logits, drafts, nd)
    want = np.mean([sum(p ** k for k in range(1, int(d) + 1)) for d in nd])
    assert abs(acc.mean() - want) < 4 * np.sqrt(np.var(acc) / lanes) + 1e-9
