"""GPU parity of spec_accept_tree against the oracle: accept lengths, accepted
paths, tokens, commits and status bits bit-exact, on random trees (distinct
and duplicate sibling tokens), chain trees (which must equal spec_accept),
invalid trees and out-of-vocabulary tokens, up to a 151,936-token vocabulary."""
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
