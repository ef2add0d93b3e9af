"""GPU parity of spec_accept_sampled (lossless stochastic acceptance) against
the oracle.  The kernel decides in fp32 with the hardware exp2, the oracle in
fp64.  The test bounds the kernel's fp32 error from its arithmetic (see
_eps_row) and checks each decision against the fp64 value with that bound:
- a ratio test u q < p whose fp64 margin exceeds the bound must come out as
  in fp64; the lanes where one sits inside it ("straddle" lanes) are counted
  and reported, and their accept length must be one the bound allows;
- the drawn token's cumulative-mass interval must hold the fp64 target
  u_sample Z to within the bound; the token must equal the fp64 draw on at
  least a stated share of the lanes.
The fp64 reference values (softmax, cumulative residual mass) are checked
against the oracle's own decisions at the exact uniforms.  The distribution
of the GPU's draws is also checked against the target (chi-square),
independently of the oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_util import i32_dev

pytestmark = pytest.mark.gpu
U = 2.0 ** -24  # fp32 unit roundoff
# bound assumed for the relative error of the hardware exp2 (ex2.approx.ftz.f32)
E = 2.0 ** -21
LN2 = math.log(2.0)
LOG2E = 1.0 / LN2


def _stats_parts(rows):
    """CTAs per logits row of the statistics kernel, chosen as the host does:
    enough to cover every SM about four times, at most one 8-CTA cluster."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    parts = 1
    while parts < 8 and rows * parts < 4 * sms:
        parts *= 2
    return parts


def _eps_row(lrow, parts):
    """Relative error bound of the kernel's p(x) = exp2((l_x - M) log2e) / S
    over one fp32 logits row.  S is summed per thread in groups of four
    (each group: one rescale of the partial by exp2 and four additions), then
    combined over 5 warp levels, 7 sequential warp partials and parts - 1
    cluster partials (each a rescale and an addition).  Along any path to S:
    at most 1 + levels exp2 evaluations (E each), 3 + 2 levels roundings (U
    each), and an exp2 argument error of 3U |arg| per evaluation, where the
    arguments of one path's rescales add up to at most the row's range R (the
    running max only grows) and the element's own argument is bounded in the
    weighted mean.  p adds its own exp2 (E + 3U |arg|) and the division (U).
    Returns (eps for the element with argument a, as a function; the bound
    at the row's largest argument)."""
    V = lrow.size
    x = lrow.astype(np.float64)
    M = x.max()
    arg = (M - x) * LOG2E
    w = np.exp2(-arg)
    abar = float((w * arg).sum() / w.sum())
    R = float(arg.max())
    chunk = (((V + parts - 1) // parts) + 3) & ~3
    g = -(-chunk // 1024)
    levels = g + 5 + 7 + (parts - 1)
    eps_s = E * (1 + levels) + U * (3 + 2 * levels) + 3 * U * LN2 * (abar + R)

    def eps(a):
        return eps_s + E + 3 * U * LN2 * a + U
    return eps, eps(R)


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


def _softmax64(l):
    x = l.astype(np.float64)
    e = np.exp(x - x.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


def _check(logits, q, drafts, ua, us, got, seq_lens=None):
    """Checks one GPU run (see the module docstring).  Returns (lanes whose
    token equals the fp64 draw, straddle lanes, largest cumulative-mass miss
    of a draw, the largest bound allowed for it)."""
    B, W, V = logits.shape
    d = W - 1
    parts = _stats_parts(B * W)
    orc = oracle.spec_accept_sampled(logits, q, drafts, ua, us, seq_lens)
    assert got[3] == orc[3]
    n_tiles = -(-V // 1024)
    slices = min(64, max(1, -(-V // 4096)))
    exact = straddle = 0
    worst_miss = worst_eta = 0.0
    for b in range(B):
        P = _softmax64(logits[b])
        possible = []
        for i in range(d):
            x = int(drafts[b, i])
            if x < 0 or x >= V:
                possible.append(i)
                break
            eps, _ = _eps_row(logits[b, i], parts)
            px = P[i, x]
            margin = (px - float(ua[b, i]) * float(q[b, i, x])) / px
            tol = eps((logits[b, i].astype(np.float64).max() - float(logits[b, i, x])) * LOG2E) + 2 * U
            if margin > tol:
                continue
            possible.append(i)
            if margin < -tol:
                break  # a clear rejection
            # inside the bound: either outcome is allowed; continue as accepted
        else:
            possible.append(d)
        a = int(got[0][b])
        assert a in possible, (b, a, possible)
        straddle += len(possible) > 1
        assert int(orc[0][b]) in possible, (b, int(orc[0][b]), possible)
        tok = got[1][b]
        assert list(tok[:a]) == list(drafts[b, :a]) and (tok[a + 1:] == -1).all(), (b, tok)
        # the draw from row a: the residual max(0, p - q), or p after a full acceptance
        w = np.maximum(0.0, P[a] - q[b, a].astype(np.float64)) if a < d else P[a]
        if not w.sum() > 0.0:
            w = P[a]
        C = np.cumsum(w)
        Z = C[-1]
        T = float(us[b]) * Z
        k_ref = min(int(np.searchsorted(C, T, side="right")), int(np.nonzero(w > 0)[0][-1]))
        if int(orc[0][b]) == a:  # the fp64 reference agrees with the oracle's own draw
            assert int(orc[1][b][a]) == k_ref, (b, int(orc[1][b][a]), k_ref)
        k = int(tok[a])
        lo_c = C[k - 1] if k > 0 else 0.0
        hi_c = C[k]
        miss = 0.0 if lo_c <= T < hi_c else (lo_c - T if T < lo_c else T - hi_c)
        _, eps_p = _eps_row(logits[b, a], parts)
        # cumulative and total mass: the weights' error (eps_p of a mass <= 1),
        # the sums (4-term, 1024-logit block scan, tiles of a slice, slices),
        # and the target's product
        eta = 2.0 * (eps_p + U * (2 + 13 + n_tiles + slices)) + U
        assert miss <= eta, (b, k, k_ref, miss, eta)
        worst_miss, worst_eta = max(worst_miss, miss), max(worst_eta, eta)
        exact += k == k_ref
        if seq_lens is not None:
            assert got[2][b] == seq_lens[b] + 1 + a
    return exact, straddle, worst_miss, worst_eta


@pytest.mark.parametrize("B,W,V,offset", [(8, 16, 151936, 0), (12, 8, 151936, 0), (8, 16, 151936, 1),
                                          (5, 4, 4097, 0), (3, 6, 1000, 0), (6, 2, 7, 0)])
def test_sampled_parity(B, W, V, offset):
    logits, q, drafts, ua, us = _inputs(60 + B + W, B, W, V)
    L = np.arange(B, dtype=np.int32) * 10
    got = _run(logits, q, drafts, ua, us, L, offset)
    exact, straddle, miss, eta = _check(logits, q, drafts, ua, us, got, L)
    print(f"B={B} W={W} V={V}: {exact}/{B} draws equal the fp64 draw, {straddle} straddle lanes, "
          f"largest mass miss {miss:.3g} (bound {eta:.3g})")
    assert straddle <= 1, straddle
    # the fp32 error (measured far below the bound) moves a draw only when the
    # target sits that close to a token boundary
    assert exact >= B - (1 if V <= 5000 else 2), exact
    assert (got[0] >= 0).all() and (got[0] <= W - 1).all()


def test_sampled_window_of_one_and_peaked_rows():
    rng = np.random.default_rng(70)
    B, V = 40, 151936
    logits = rng.standard_normal((B, 1, V)).astype(np.float32)
    logits[:, 0, 17] = 14.0  # most of the mass (about 0.83) on one token
    us = rng.random(B).astype(np.float32)
    got = _run(logits, None, np.zeros((B, 0), np.int32), np.zeros((B, 0), np.float32), us)
    exact, straddle, _, _ = _check(logits, np.zeros((B, 0, V), np.float32), np.zeros((B, 0), np.int32),
                                   np.zeros((B, 0), np.float32), us, got)
    assert (got[0] == 0).all() and straddle == 0 and exact >= B - 2


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
