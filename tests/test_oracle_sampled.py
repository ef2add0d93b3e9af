"""Pins for the oracle's lossless stochastic acceptance (no GPU): the exact
restatement in brute.py, hand-worked cases (ratio test, residual, inverse CDF,
zero draft probability, q = p), and the property that defines the method:
with the draft drawn from q and the uniforms uniform, the emitted token at
the first position is distributed as the target p (chi-square on seeded
trials), and so is the bonus token after a fully accepted window."""
import math

import numpy as np
import pytest

import oracle
from oracle import brute


def _probs(rng, shape, sharp=1.0):
    z = np.exp(sharp * rng.standard_normal(shape))
    return (z / z.sum(axis=-1, keepdims=True)).astype(np.float32)


def test_matches_brute_on_random_windows():
    rng = np.random.default_rng(50)
    for trial in range(60):
        B, W, V = 3, 1 + trial % 5, 40
        logits = (2.0 * rng.standard_normal((B, W, V))).astype(np.float32)
        q = _probs(rng, (B, W - 1, V), 1.5)
        drafts = np.array([[rng.choice(V, p=q[b, i] / q[b, i].sum()) for i in range(W - 1)] for b in range(B)],
                          np.int32).reshape(B, W - 1)
        ua = rng.random((B, W - 1)).astype(np.float32)
        us = rng.random(B).astype(np.float32)
        acc, tok, sl, st = oracle.spec_accept_sampled(logits, q, drafts, ua, us, np.array([1, 2, 3], np.int32))
        assert st == 0
        for b in range(B):
            a, t = brute.accept_sampled(logits[b].astype(np.float64).tolist(), q[b].astype(np.float64).tolist(),
                                        [int(x) for x in drafts[b]], [float(u) for u in ua[b]], float(us[b]))
            assert acc[b] == a and list(tok[b]) == t, (trial, b)
            assert sl[b] == [1, 2, 3][b] + 1 + a


def test_hand_worked_ratio_residual_and_inverse_cdf():
    # p = (0.5, 0.25, 0.25); q = (0.1, 0.8, 0.1); draft 1 has ratio 0.3125
    logits = np.log(np.array([[[2.0, 1.0, 1.0], [1.0, 1.0, 1.0]]], np.float64)).astype(np.float32)
    q = np.array([[[0.1, 0.8, 0.1]]], np.float32)
    drafts = np.array([[1]], np.int32)
    # accepted (u = 0.3 < 0.3125): the bonus comes from p_1 = uniform thirds
    acc, tok, _, _ = oracle.spec_accept_sampled(logits, q, drafts, np.array([[0.3]], np.float32),
                                                np.array([0.7], np.float32))
    assert acc[0] == 1 and list(tok[0]) == [1, 2]
    # rejected (u = 0.5): residual (0.4, 0, 0.15) / 0.55; targets 0.275 -> 0 and 0.44 -> 2
    for us, k in ((0.5, 0), (0.8, 2), (0.7, 0), (0.73, 2)):
        acc, tok, _, _ = oracle.spec_accept_sampled(logits, q, drafts, np.array([[0.5]], np.float32),
                                                    np.array([us], np.float32))
        assert acc[0] == 0 and list(tok[0]) == [k, -1], us
    # window of one: inverse CDF of p = (0.5, 0.25, 0.25)
    for us, k in ((0.2, 0), (0.6, 1), (0.8, 2), (0.0, 0)):
        _, tok, _, _ = oracle.spec_accept_sampled(logits[:, :1], np.zeros((1, 0, 3), np.float32),
                                                  np.zeros((1, 0), np.int32), np.zeros((1, 0), np.float32),
                                                  np.array([us], np.float32))
        assert tok[0, 0] == k, us


def test_q_equal_p_always_accepts_and_zero_q_accepts():
    rng = np.random.default_rng(51)
    B, W, V = 50, 6, 30
    logits = (1.5 * rng.standard_normal((B, W, V))).astype(np.float32)
    p = np.exp(logits - logits.max(axis=2, keepdims=True))
    p = (p / p.sum(axis=2, keepdims=True)).astype(np.float32)
    q = (p[:, :W - 1] * (1 - 1e-6)).astype(np.float32)  # a hair below p: every ratio exceeds 1
    drafts = rng.integers(0, V, size=(B, W - 1)).astype(np.int32)
    acc, _, _, _ = oracle.spec_accept_sampled(logits, q, drafts, rng.random((B, W - 1)).astype(np.float32),
                                              rng.random(B).astype(np.float32))
    assert (acc == W - 1).all()
    q0 = q.copy()
    for b in range(B):
        q0[b, 0, drafts[b, 0]] = 0.0
    acc, _, _, _ = oracle.spec_accept_sampled(logits, q0, drafts, np.full((B, W - 1), 0.999, np.float32),
                                              rng.random(B).astype(np.float32))
    assert (acc >= 1).all()


def test_bad_draft_is_a_flagged_rejection():
    logits = np.zeros((2, 3, 5), np.float32)
    q = np.full((2, 2, 5), 0.2, np.float32)
    acc, tok, _, st = oracle.spec_accept_sampled(logits, q, np.array([[1, 9], [-1, 2]], np.int32),
                                                 np.zeros((2, 2), np.float32), np.array([0.5, 0.5], np.float32))
    assert st == 4 and list(acc) == [1, 0]
    assert tok[0, 0] == 1 and tok[0, 2] == -1 and tok[1, 1] == -1


def _chi2_ok(counts, probs, n):
    exp = probs * n
    chi2 = float(((counts - exp) ** 2 / exp).sum())
    dof = len(probs) - 1
    # Wilson-Hilferty: upper 1e-4 tail of chi-square with dof degrees of freedom
    z = 3.719
    bound = dof * (1 - 2 / (9 * dof) + z * math.sqrt(2 / (9 * dof))) ** 3
    return chi2 < bound, chi2, bound


@pytest.mark.parametrize("seed", [52, 53])
def test_first_token_is_distributed_as_the_target(seed):
    rng = np.random.default_rng(seed)
    V, N = 8, 40000
    l0 = (1.2 * rng.standard_normal(V)).astype(np.float32)
    p0 = np.exp(l0.astype(np.float64) - l0.max())
    p0 /= p0.sum()
    q0 = _probs(rng, (V,), 1.0).astype(np.float64)
    q0 /= q0.sum()
    logits = np.broadcast_to(np.stack([l0, l0]), (N, 2, V)).astype(np.float32)
    q = np.broadcast_to(q0.astype(np.float32), (N, 1, V)).copy()
    drafts = rng.choice(V, size=(N, 1), p=q0).astype(np.int32)
    acc, tok, _, _ = oracle.spec_accept_sampled(logits, q, drafts, rng.random((N, 1)).astype(np.float32),
                                                rng.random(N).astype(np.float32))
    counts = np.bincount(tok[:, 0], minlength=V)
    ok, chi2, bound = _chi2_ok(counts, p0, N)
    assert ok, (chi2, bound)
    # and the rejection rate is the total variation distance between p and q
    tv = 0.5 * np.abs(p0 - q0).sum()
    assert abs((acc == 0).mean() - tv) < 4 * math.sqrt(tv * (1 - tv) / N)


def test_bonus_token_is_distributed_as_the_last_row():
    rng = np.random.default_rng(54)
    V, N = 6, 30000
    l = (1.0 * rng.standard_normal((2, V))).astype(np.float32)
    p = np.exp(l.astype(np.float64) - l.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    q = np.broadcast_to((p[0] * (1 - 1e-6)).astype(np.float32), (N, 1, V)).copy()  # always accepted
    drafts = rng.choice(V, size=(N, 1), p=p[0]).astype(np.int32)
    logits = np.broadcast_to(l, (N, 2, V)).astype(np.float32)
    acc, tok, _, _ = oracle.spec_accept_sampled(logits, q, drafts, rng.random((N, 1)).astype(np.float32),
                                                rng.random(N).astype(np.float32))
    assert (acc == 1).all()
    ok, chi2, bound = _chi2_ok(np.bincount(tok[:, 1], minlength=V), p[1], N)
    assert ok, (chi2, bound)


def test_zero_residual_falls_back_to_the_target():
    # q = 3 p (not normalised): every draft is rejected at u = 0.5 and max(0, p - q)
    # has no mass, so the token is drawn from p itself
    rng = np.random.default_rng(55)
    B, W, V = 6, 3, 25
    logits = rng.standard_normal((B, W, V)).astype(np.float32)
    p = np.exp(logits.astype(np.float64) - logits.max(axis=2, keepdims=True))
    p /= p.sum(axis=2, keepdims=True)
    q = (3.0 * p[:, :W - 1]).astype(np.float32)
    drafts = rng.integers(0, V, size=(B, W - 1)).astype(np.int32)
    ua = np.full((B, W - 1), 0.5, np.float32)
    us = rng.random(B).astype(np.float32)
    acc, tok, _, _ = oracle.spec_accept_sampled(logits, q, drafts, ua, us)
    assert (acc == 0).all()
    for b in range(B):
        a, t = brute.accept_sampled(logits[b].astype(np.float64).tolist(), q[b].astype(np.float64).tolist(),
                                    [int(x) for x in drafts[b]], [0.5] * (W - 1), float(us[b]))
        assert (a, t) == (0, list(tok[b]))
        cdf = np.cumsum(p[b, 0])
        assert tok[b, 0] == int(np.searchsorted(cdf, us[b] * cdf[-1], side="right"))
