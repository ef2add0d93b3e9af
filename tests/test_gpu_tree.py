"""GPU parity of the draft-tree calls against the oracle.

spec_accept_tree: accept lengths, accepted paths, tokens, commits and status
bits bit-exact, on random trees (distinct and duplicate sibling tokens),
chain trees (which must equal spec_accept), invalid trees and
out-of-vocabulary tokens, up to a 151,936-token vocabulary.

verify_attn_tree: every element within the attention tolerance of the
oracle's fp64 ancestor-masked attention on random trees (FP8 and INT4, small
cases and one full multi-lane lane), chain trees bit-identical to verify_attn,
and invalid lanes zeroed and flagged."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import i32_dev
from test_oracle_tree import _random_tree, _tokens_for

pytestmark = pytest.mark.gpu


def _run(logits, tokens, parent, seq_lens=None):
    import speculative_decode_verify_append_gb300 as sdva
    B, W, V = logits.shape
    acc = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    path = torch.full((B, W), -7, dtype=torch.int32, device="cuda")
    tok = torch.full((B, W), -7, dtype=torch.int32, device="cuda")
    sl = i32_dev(seq_lens) if seq_lens is not None else None
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    sdva.spec_accept_tree(torch.from_numpy(np.ascontiguousarray(logits)).cuda(), i32_dev(tokens), i32_dev(parent),
                          acc, path, tok, sl, st)
    torch.cuda.synchronize()
    return (acc.cpu().numpy(), path.cpu().numpy(), tok.cpu().numpy(), None if sl is None else sl.cpu().numpy(),
            int(st.item()))


def _same(got, want):
    for g, w, name in zip(got, want, ("accept_len", "path", "out_tokens", "seq_lens", "status")):
        if w is None:
            assert g is None
        else:
            assert np.array_equal(np.asarray(g), np.asarray(w)), name


@pytest.mark.parametrize("B,W,V", [(8, 16, 151936), (12, 8, 151936), (5, 7, 4097), (30, 16, 1000), (4, 2, 50)])
def test_random_trees(B, W, V):
    rng = np.random.default_rng(100 + W)
    logits = rng.standard_normal((B, W, V)).astype(np.float32)
    targets = logits.argmax(axis=2)
    parent = np.stack([_random_tree(rng, W) for _ in range(B)])
    tokens = np.stack([_tokens_for(rng, parent[b], targets[b], V, 0.8) for b in range(B)])
    if W > 3:  # a duplicate sibling token on one lane: the first slot wins
        kids = [i for i in range(1, W) if parent[0, i] == 0]
        if len(kids) >= 2:
            tokens[0, kids[1]] = tokens[0, kids[0]]
    L = np.arange(B, dtype=np.int32) * 3
    _same(_run(logits, tokens, parent, L), oracle.tree_accept(logits, tokens, parent, L))


def test_chain_tree_equals_spec_accept():
    import speculative_decode_verify_append_gb300 as sdva
    rng = np.random.default_rng(110)
    B, W, V = 8, 16, 151936
    logits = rng.standard_normal((B, W, V)).astype(np.float32)
    t = logits.argmax(axis=2).astype(np.int32)
    drafts = np.where(rng.random((B, W - 1)) < 0.8, t[:, :W - 1], (t[:, :W - 1] + 1) % V).astype(np.int32)
    parent = np.tile(np.maximum(np.arange(-1, W - 1, dtype=np.int32), 0), (B, 1))
    tokens = np.concatenate([np.zeros((B, 1), np.int32), drafts], axis=1)
    got = _run(logits, tokens, parent)
    acc = torch.zeros(B, dtype=torch.int32, device="cuda")
    tok = torch.zeros((B, W), dtype=torch.int32, device="cuda")
    sdva.spec_accept(torch.from_numpy(logits).cuda(), i32_dev(drafts), acc, tok)
    torch.cuda.synchronize()
    a_e, t_e = acc.cpu().numpy(), tok.cpu().numpy()
    assert np.array_equal(got[0], a_e)
    for b in range(B):
        assert list(got[2][b, :a_e[b] + 1]) == list(t_e[b, :a_e[b] + 1])
        assert list(got[1][b, :a_e[b] + 1]) == list(range(a_e[b] + 1))


def test_invalid_trees_bad_tokens_and_window_of_one():
    rng = np.random.default_rng(111)
    B, W, V = 4, 6, 300
    logits = rng.standard_normal((B, W, V)).astype(np.float32)
    targets = logits.argmax(axis=2)
    parent = np.stack([_random_tree(rng, W) for _ in range(B)])
    tokens = np.stack([_tokens_for(rng, parent[b], targets[b], V, 0.9) for b in range(B)])
    parent[1, 3] = 3       # not an earlier slot
    parent[2, 5] = -1
    tokens[3, 4] = V + 5   # out of vocabulary
    L = np.full(B, 40, np.int32)
    got = _run(logits, tokens, parent, L)
    _same(got, oracle.tree_accept(logits, tokens, parent, L))
    assert got[4] == 32 | 4
    one = rng.standard_normal((3, 1, 999)).astype(np.float32)
    z = np.zeros((3, 1), np.int32)
    _same(_run(one, z, z), oracle.tree_accept(one, z, z))


# ---------------------------------------------------------------------------
# verify_attn_tree: the ancestor-masked attention of a draft-tree window
# ---------------------------------------------------------------------------
def _tree_verify(spec, step, gcache, parent, max_context=None):
    import speculative_decode_verify_append_gb300 as sdva
    from gpu_util import SM_SCALE, bf16_dev
    B, W, Hq = step.q.shape[:3]
    max_context = int(step.seq_lens.max()) if max_context is None else max_context
    out = torch.full((B, W, Hq, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(sdva.verify_attn_workspace_size(B, W, Hq, spec.num_kv_heads, max_context), dtype=torch.uint8,
                     device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    sdva.verify_attn_tree(gcache, bf16_dev(step.q), i32_dev(parent), i32_dev(step.page_table),
                          i32_dev(step.seq_lens), max_context, float(SM_SCALE), out, ws, st)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), int(st.item())


TREE_CASES = [
    # (kv dtype, lens, W, Hq, Hkv)
    (0, [5, 200, 1500, 63], 16, 24, 4),
    (0, [0, 64, 4097], 7, 8, 1),
    (1, [0, 129, 900], 8, 24, 4),
    (1, [700, 31], 16, 8, 1),
    (2, [0, 129, 900], 8, 24, 4),
    (3, [5, 200, 1500, 63], 16, 24, 4),
]
KV_NAMES = {0: "fp8", 1: "int4", 2: "int8", 3: "fp8row"}


@pytest.mark.parametrize("case", TREE_CASES, ids=lambda c: f"{KV_NAMES[c[0]]}-W{c[2]}-{c[3]}q{c[4]}kv")
def test_tree_attention_random_trees(case):
    """Every element of every row within |g - r| <= 2e-3 + 1e-2 |r| of the
    oracle's fp64 ancestor-masked attention, on random trees."""
    import synth
    from gpu_util import SM_SCALE, assert_close, fill_both
    dtype, lens, W, Hq, Hkv = case
    spec = synth.Spec("tree", 40 + W, len(lens), 0, 0, Hq, Hkv, W, dtype, None, 0.7, True)
    step = synth.make_step(spec, seq_lens=np.array(lens, np.int32), with_accept=False)
    gcache, ocache, _ = fill_both(spec, step, chunk=512)
    rng = np.random.default_rng(7 + W)
    parent = np.stack([_random_tree(rng, W) for _ in range(len(lens))]).astype(np.int32)
    got, status = _tree_verify(spec, step, gcache, parent)
    assert status == 0
    want, ost = oracle.tree_attn(ocache, step.q, step.page_table, step.seq_lens, parent, SM_SCALE, threads=8)
    assert ost == 0
    assert_close(got, want, f"tree {case}")


@pytest.mark.parametrize("dtype", [0, 1, 2, 3])
def test_chain_tree_equals_causal_verify(dtype):
    """A chain tree (parent i - 1) is the causal window: bit-identical to verify_attn."""
    import synth
    from gpu_util import fill_both
    import speculative_decode_verify_append_gb300 as sdva
    from gpu_util import SM_SCALE, bf16_dev
    lens, W = [300, 4000, 64], 16
    spec = synth.Spec("chain", 51, len(lens), 0, 0, 24, 4, W, dtype, None, 0.7, True)
    step = synth.make_step(spec, seq_lens=np.array(lens, np.int32), with_accept=False)
    gcache, _, _ = fill_both(spec, step, with_oracle=False)
    parent = np.tile(np.maximum(np.arange(-1, W - 1, dtype=np.int32), 0), (len(lens), 1))
    got, st = _tree_verify(spec, step, gcache, parent)
    B, Hq = len(lens), 24
    out = torch.zeros((B, W, Hq, 128), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(sdva.verify_attn_workspace_size(B, W, Hq, 4, max(lens)), dtype=torch.uint8, device="cuda")
    sdva.verify_attn(gcache, bf16_dev(step.q), i32_dev(step.page_table), i32_dev(step.seq_lens), max(lens),
                     float(SM_SCALE), out, ws)
    torch.cuda.synchronize()
    assert st == 0
    assert np.array_equal(got, out.float().cpu().numpy())


def test_tree_attention_invalid_lane_is_zero_and_flagged():
    """A lane whose parent array is not a tree gets zero rows and
    SDVA_STATUS_BAD_TREE; the other lanes equal the oracle."""
    import synth
    from gpu_util import SM_SCALE, assert_close, fill_both
    import speculative_decode_verify_append_gb300 as sdva
    lens, W = [500, 2000, 90], 8
    spec = synth.Spec("badtree", 61, len(lens), 0, 0, 24, 4, W, 0, None, 0.7, True)
    step = synth.make_step(spec, seq_lens=np.array(lens, np.int32), with_accept=False)
    gcache, ocache, _ = fill_both(spec, step)
    rng = np.random.default_rng(62)
    parent = np.stack([_random_tree(rng, W) for _ in range(len(lens))]).astype(np.int32)
    bad = parent.copy()
    bad[1, 5] = 6  # not an earlier slot
    got, status = _tree_verify(spec, step, gcache, bad)
    assert status == sdva.STATUS_BAD_TREE
    assert not got[1].any()
    want, _ = oracle.tree_attn(ocache, step.q, step.page_table, step.seq_lens, parent, SM_SCALE, threads=8)
    assert_close(got[[0, 2]], want[[0, 2]], "valid lanes")


def test_tree_attention_full_workload_rows():
    """The multi-lane workload (8 lanes up to 65,536 tokens, 16-slot trees):
    every row of one lane, in the benchmark's launch configuration."""
    import synth
    from gpu_util import SM_SCALE, assert_close, fill_both
    spec = synth.WORKLOADS["multi_lane"]
    step = synth.make_step(spec, with_accept=False)
    B, W, Hq = step.q.shape[:3]
    lane = 3
    gcache, ocache, _ = fill_both(spec, step, lanes=[lane])
    rng = np.random.default_rng(63)
    parent = np.stack([_random_tree(rng, W) for _ in range(B)]).astype(np.int32)
    got, status = _tree_verify(spec, step, gcache, parent, max_context=spec.ctx_hi)
    assert status == 0
    sel = np.array([lane])
    want, _ = oracle.tree_attn(ocache, step.q[sel], step.page_table[sel], step.seq_lens[sel], parent[sel], SM_SCALE,
                               threads=16)
    assert_close(got[lane], want[0], "multi-lane tree lane")
