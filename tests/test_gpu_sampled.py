"""GPU parity of spec_accept_sampled (lossless stochastic acceptance) against
the oracle.  The kernel decides in fp32 with hardware exp2, the oracle in
fp64, so a decision whose uniform lies within rounding of its boundary may
go either way: every lane is run through the oracle three times, with both
uniforms as given and scaled by (1 - 1e-4) and (1 + 1e-4).  Accept lengths
and accepted drafts must match exactly where the three runs agree; the drawn
token must lie between the draws at the two scaled uniforms (a window of
1e-4 of the probability mass), which is exact where they agree.  The
distribution of the GPU's own draws is also checked against the target
(chi-square), independently of the oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_util import i32_dev

pytestmark = pytest.mark.gpu
DELTA = 1e-4


def _inputs(seed, B, W, V, sharp=2.0):
    rng = np.random.default_rng(seed)
    logits = (sharp * rng.standard_normal((B, W, V))).astype(np.float32)
    # a draft distribution correlated with the target
    z = 0.8 * logits[:, :W - 1].astype(np.float64) + 0.6 * rng.standard_normal((B, W - 1, V))
    q = np.exp(z - z.max(axis=2, keepdims=True))
    q = (q / q.sum(axis=2, keepdims=True)).astype(np.float32)
    cdf = np.cumsum(q.astype(np.float64), axis=2)
    u = rng.random((B, W - 1)) * cdf[:, :, -1]
    drafts = np.array([[min(V - 1, int(np.searchsorted(cdf[b, i], u[b, i], side="right"))) for i in range(W - 1)]
                       for b in range(B)], np.int32).reshape(B, W - 1)
    ua = rng.random((B, W - 1)).astype(np.float32)
    us = rng.random(B).astype(np.float32)
    return logits, q, drafts, ua, us


def _dev_f32(a, offset=0):
    flat = torch.from_numpy(np.ascontiguousarray(a, np.float32).reshape(-1))
    buf = torch.empty(flat.numel() + offset, dtype=torch.float32, device="cuda")
    buf[offset:].copy_(flat)
    return buf[offset:].view(a.shape)


def _run(logits, q, drafts, ua, us, seq_lens=None, offset=0):
    import speculative_decode_verify_append_gb300 as sdva
    B, W, V = logits.shape
    ws = torch.empty(sdva.spec_accept_sampled_workspace_size(B, W), dtype=torch.uint8, device="cuda")
    acc = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    tok = torch.full((B, W), -7, dtype=torch.int32, device="cuda")
    sl = i32_dev(seq_lens) if seq_lens is not None else None
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    sdva.spec_accept_sampled(_dev_f32(logits, offset), _dev_f32(q, offset) if W > 1 else None,
                             i32_dev(drafts) if W > 1 else None, _dev_f32(ua) if W > 1 else None, _dev_f32(us),
                             acc, tok, ws, sl, st)
    torch.cuda.synchronize()
    return acc.cpu().numpy(), tok.cpu().numpy(), None if sl is None else sl.cpu().numpy(), int(st.item())


def _check(logits, q, drafts, ua, us, got, seq_lens=None):
    """The accept length must be the oracle's wherever that is robust to the
    uniforms' rounding (else one of the nearby lengths).  Given it, the
    accepted drafts and the -1 tail are exact, and the drawn token lies
    between the oracle's draws at u_sample * (1 - 1e-4) and * (1 + 1e-4)
    (the inverse CDF is monotone in the uniform): exact where they agree.
    Returns the number of lanes checked exactly."""
    one = np.float32(np.nextafter(np.float32(1), np.float32(0)))
    runs = [oracle.spec_accept_sampled(logits, q, drafts, np.minimum(ua * f, one).astype(np.float32),
                                       np.minimum(us * f, one).astype(np.float32), seq_lens)
            for f in (1.0, 1.0 - DELTA, 1.0 + DELTA)]
    assert got[3] == runs[0][3]
    W = logits.shape[1]
    exact = 0
    for b in range(logits.shape[0]):
        a = int(got[0][b])
        lens = {int(r[0][b]) for r in runs}
        assert a in lens, (b, a, lens)
        if len(lens) > 1:
            continue  # the accept decision itself sits on its boundary
        tok = got[1][b]
        assert list(tok[:a]) == list(drafts[b, :a]) and (tok[a + 1:] == -1).all(), (b, tok)
        ks = [int(r[1][b][a]) for r in runs]
        lo, hi = min(ks), max(ks)
        assert lo <= tok[a] <= hi, (b, int(tok[a]), ks)
        exact += lo == hi
        if seq_lens is not None:
            assert got[2][b] == seq_lens[b] + 1 + a
    return exact


@pytest.mark.parametrize("B,W,V,offset", [(8, 16, 151936, 0), (12, 8, 151936, 0), (8, 16, 151936, 1),
                                          (5, 4, 4097, 0), (3, 6, 1000, 0), (6, 2, 7, 0)])
def test_sampled_parity(B, W, V, offset):
    logits, q, drafts, ua, us = _inputs(60 + B + W, B, W, V)
    L = np.arange(B, dtype=np.int32) * 10
    got = _run(logits, q, drafts, ua, us, L, offset)
    exact = _check(logits, q, drafts, ua, us, got, L)
    if V <= 5000:  # wide bins: nearly every draw is pinned exactly
        assert exact >= B - 1, exact
    assert (got[0] >= 0).all() and (got[0] <= W - 1).all()


def test_sampled_window_of_one_and_peaked_rows():
    rng = np.random.default_rng(70)
    B, V = 40, 151936
    logits = rng.standard_normal((B, 1, V)).astype(np.float32)
    logits[:, 0, 17] = 14.0  # most of the mass (about 0.83) on one token
    us = rng.random(B).astype(np.float32)
    got = _run(logits, None, np.zeros((B, 0), np.int32), np.zeros((B, 0), np.float32), us)
    exact = _check(logits, np.zeros((B, 0, V), np.float32), np.zeros((B, 0), np.int32),
                   np.zeros((B, 0), np.float32), us, got)
    assert (got[0] == 0).all() and exact >= B // 2  # token 17 holds most of the mass: its draws are exact


def test_sampled_bad_drafts_and_zero_draft_probability():
    logits, q, drafts, ua, us = _inputs(71, 4, 5, 3000)
    drafts[0, 2] = 3000   # out of vocabulary: a flagged rejection
    drafts[1, 0] = -1
    q[2, 0, drafts[2, 0]] = 0.0  # the draft model could not have drawn it: accepted
    ua[2, 0] = 0.999
    got = _run(logits, q, drafts, ua, us)
    _check(logits, q, drafts, ua, us, got)
    assert got[3] == 4 and got[0][0] <= 2 and got[0][1] == 0 and got[0][2] >= 1


def test_gpu_first_token_is_distributed_as_the_target():
    rng = np.random.default_rng(72)
    V, N = 8, 20000
    l0 = (1.2 * rng.standard_normal(V)).astype(np.float32)
    p0 = np.exp(l0.astype(np.float64) - l0.max())
    p0 /= p0.sum()
    q0 = rng.random(V) + 0.2
    q0 /= q0.sum()
    logits = np.broadcast_to(np.stack([l0, l0]), (N, 2, V)).astype(np.float32)
    q = np.broadcast_to(q0.astype(np.float32), (N, 1, V)).copy()
    drafts = rng.choice(V, size=(N, 1), p=q0).astype(np.int32)
    got = _run(logits, q, drafts, rng.random((N, 1)).astype(np.float32), rng.random(N).astype(np.float32))
    counts = np.bincount(got[1][:, 0], minlength=V)
    chi2 = float(((counts - p0 * N) ** 2 / (p0 * N)).sum())
    dof = V - 1
    bound = dof * (1 - 2 / (9 * dof) + 3.719 * math.sqrt(2 / (9 * dof))) ** 3  # upper 1e-4 tail
    assert chi2 < bound, (chi2, bound)


def test_workspace_too_small_is_refused():
    import speculative_decode_verify_append_gb300 as sdva
    logits, q, drafts, ua, us = _inputs(73, 2, 3, 100)
    ws = torch.empty(8, dtype=torch.uint8, device="cuda")
    acc = torch.zeros(2, dtype=torch.int32, device="cuda")
    tok = torch.zeros((2, 3), dtype=torch.int32, device="cuda")
    with pytest.raises(sdva.SdvaError) as e:
        sdva.spec_accept_sampled(_dev_f32(logits), _dev_f32(q), i32_dev(drafts), _dev_f32(ua), _dev_f32(us), acc,
                                 tok, ws)
    assert e.value.code == sdva.ERR_WORKSPACE
