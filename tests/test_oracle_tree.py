"""Pins for the oracle's draft-tree verification (no GPU).  Acceptance: the
greedy walk against the path formulation in brute.py (deepest accepted node)
on random trees with distinct sibling tokens, a chain tree against the
ordinary acceptance, the tie rule for duplicate siblings, invalid trees.
Attention: the ancestor mask against brute-force attention over explicit key
positions, a chain tree against the causal verify attention, and, with INT4
(per-token scales), a star tree's row i against a causal two-token window
holding only the root and token i."""
import math

import numpy as np
import pytest

import oracle
import synth
from oracle import brute

PAGE = 64


def _random_tree(rng, W):
    return np.array([0] + [int(rng.integers(0, i)) for i in range(1, W)], np.int32)


def _tokens_for(rng, parent, targets, V, p_follow=0.7):
    """Window tokens with distinct siblings; a child carries its parent's
    argmax with probability p_follow (at most one child per parent does)."""
    W = len(parent)
    tok = np.zeros(W, np.int32)
    used = {}
    for i in range(1, W):
        n = int(parent[i])
        taken = used.setdefault(n, set())
        t = int(targets[n])
        if not (rng.random() < p_follow and t not in taken):
            t = int(rng.integers(0, V))
            while t in taken or t == int(targets[n]):
                t = int(rng.integers(0, V))
        taken.add(t)
        tok[i] = t
    tok[0] = int(rng.integers(0, V))
    return tok


def test_tree_accept_matches_the_path_formulation():
    rng = np.random.default_rng(90)
    for trial in range(80):
        B, W, V = 3, 2 + trial % 15, 40
        logits = rng.standard_normal((B, W, V)).astype(np.float32)
        targets = logits.argmax(axis=2)
        parent = np.stack([_random_tree(rng, W) for _ in range(B)])
        tokens = np.stack([_tokens_for(rng, parent[b], targets[b], V) for b in range(B)])
        acc, path, tok, sl, st = oracle.tree_accept(logits, tokens, parent, np.array([5, 6, 7], np.int32))
        assert st == 0
        for b in range(B):
            a, p, t = brute.tree_accept(logits[b].tolist(), [int(x) for x in tokens[b]], [int(x) for x in parent[b]])
            assert (acc[b], list(path[b]), list(tok[b])) == (a, p, t), (trial, b)
            assert sl[b] == [5, 6, 7][b] + 1 + a


def test_chain_tree_is_the_ordinary_acceptance():
    spec = synth.WORKLOADS["tiny"]
    logits, drafts, _ = synth.acceptance_inputs(spec, 6, 9, 500, 0.7, tag="chain")
    B, W = 6, 9
    parent = np.tile(np.arange(-1, W - 1, dtype=np.int32), (B, 1))
    parent[:, 0] = 0
    tokens = np.concatenate([np.zeros((B, 1), np.int32), drafts], axis=1)
    acc, path, tok, _, st = oracle.tree_accept(logits, tokens, parent)
    acc_e, tok_e, _, _ = oracle.spec_accept(logits, drafts)
    assert st == 0 and np.array_equal(acc, acc_e)
    for b in range(B):
        assert list(path[b, :acc[b] + 1]) == list(range(acc[b] + 1))
        assert list(tok[b, :acc[b] + 1]) == list(tok_e[b, :acc[b] + 1]) and (tok[b, acc[b] + 1:] == -1).all()


def test_duplicate_siblings_take_the_first_slot_and_invalid_trees_are_flagged():
    V = 10
    logits = np.zeros((2, 5, V), np.float32)
    logits[:, :, 3] = 1.0  # every row's argmax is 3
    parent = np.array([[0, 0, 0, 2, 1], [0, 0, 2, 1, 1]], np.int32)  # lane 1: parent[2] = 2 is invalid
    tokens = np.array([[9, 3, 3, 3, 4], [9, 3, 3, 3, 3]], np.int32)
    acc, path, tok, sl, st = oracle.tree_accept(logits, tokens, parent, np.array([0, 0], np.int32))
    # lane 0: slots 1 and 2 both carry 3: slot 1 is taken (its child 4 carries 4, so the walk ends there)
    assert acc[0] == 1 and list(path[0]) == [0, 1, -1, -1, -1] and list(tok[0]) == [3, 3, -1, -1, -1]
    assert st == 32 and acc[1] == 0 and (path[1] == -1).all() and (tok[1] == -1).all()
    assert list(sl) == [2, 0]


def _ancestors(parent, i):
    out = [i]
    while out[-1] != 0:
        out.append(int(parent[out[-1]]))
    return sorted(out)


def _cache_with_window(dtype, seed, L, W, H, Hq):
    spec = synth.Spec("tree", seed, 1, 0, 0, Hq, H, W, dtype, 64, 0.7, True)
    step = synth.make_step(spec, seq_lens=np.array([L], np.int32), with_accept=False)
    cache = oracle.Cache(dtype, step.num_pages, H)
    for start, n in synth.fill_chunks(L, 64):
        k, v = synth.context_chunk(spec, 0, start, n)
        assert oracle.append(cache, k[None], v[None], step.page_table, np.array([start], np.int32)) == 0
    assert oracle.append(cache, step.k_win, step.v_win, step.page_table, step.seq_lens) == 0
    return spec, step, cache


@pytest.mark.parametrize("dtype", [oracle.KV_FP8, oracle.KV_INT4])
def test_tree_attention_matches_brute_force(dtype):
    L, W, H, Hq = 70, 7, 1, 2
    spec, step, cache = _cache_with_window(dtype, 91, L, W, H, Hq)
    parent = np.array([[0, 0, 1, 0, 3, 3, 1]], np.int32)
    sm = float(np.float32(1.0 / math.sqrt(128.0)))  # the oracle takes the scale as fp32
    out, st = oracle.tree_attn(cache, step.q, step.page_table, step.seq_lens, parent, sm)
    assert st == 0
    bc = brute.Cache(dtype)
    # the brute cache holds the same bytes: read them back through its value()
    for pid in range(step.num_pages):
        for h in range(H):
            if dtype == oracle.KV_FP8:
                for kv, (codes, scales) in enumerate(((cache.k_codes, cache.k_scales),
                                                      (cache.v_codes, cache.v_scales))):
                    bc.scales[kv][(pid, h)] = float(scales[pid, h])
                    for off in range(PAGE):
                        bc.codes[kv][(pid, h, off)] = [int(c) for c in codes[pid, h, off]]
            else:
                for kv, (codes, scales) in enumerate(((cache.k_codes, cache.k_scales),
                                                      (cache.v_codes, cache.v_scales))):
                    for off in range(PAGE):
                        packed = codes[pid, h, off]
                        lo = ((packed & 0xF).astype(np.int8) ^ 8) - 8
                        hi = ((packed >> 4).astype(np.int8) ^ 8) - 8
                        bc.codes[kv][(pid, h, off)] = [int(x) for x in np.stack([lo, hi], 1).reshape(-1)]
                        bc.scales[kv][(pid, h, off)] = [int(x) for x in scales[pid, h, off].view(np.uint16)]
    row = list(step.page_table[0])
    for i in range(W):
        pos = list(range(L)) + [L + j for j in _ancestors(parent[0], i)]
        for h in range(Hq):
            want = brute.attention_keys(bc, [int(x) for x in step.q[0, i, h]], row, h // (Hq // H), pos, sm)
            assert np.allclose(out[0, i, h], want, rtol=1e-12, atol=1e-12), (i, h)


def test_chain_tree_attention_is_the_causal_window():
    L, W, H, Hq = 130, 6, 2, 4
    spec, step, cache = _cache_with_window(oracle.KV_FP8, 92, L, W, H, Hq)
    chain = np.array([[0, 0, 1, 2, 3, 4]], np.int32)
    sm = float(np.float32(1.0 / math.sqrt(128.0)))  # the oracle takes the scale as fp32
    got, _ = oracle.tree_attn(cache, step.q, step.page_table, step.seq_lens, chain, sm)
    want, _ = oracle.verify_attn(cache, step.q, step.page_table, step.seq_lens, sm)
    assert np.array_equal(got, want)


def test_star_tree_row_equals_a_two_token_causal_window_int4():
    # INT4 scales belong to single tokens, so a token's cached values do not
    # depend on its neighbours: row i of a star tree (every parent the root)
    # must equal row 1 of a causal window holding only the root and token i
    L, W, H, Hq = 90, 5, 1, 3
    spec, step, cache = _cache_with_window(oracle.KV_INT4, 93, L, W, H, Hq)
    star = np.zeros((1, W), np.int32)
    sm = float(np.float32(1.0 / math.sqrt(128.0)))  # the oracle takes the scale as fp32
    got, _ = oracle.tree_attn(cache, step.q, step.page_table, step.seq_lens, star, sm)
    for i in range(1, W):
        other = oracle.Cache(oracle.KV_INT4, step.num_pages, H)
        for start, n in synth.fill_chunks(L, 64):
            k, v = synth.context_chunk(spec, 0, start, n)
            oracle.append(other, k[None], v[None], step.page_table, np.array([start], np.int32))
        kw = step.k_win[:, [0, i]]
        vw = step.v_win[:, [0, i]]
        assert oracle.append(other, kw, vw, step.page_table, step.seq_lens) == 0
        want, _ = oracle.verify_attn(other, step.q[:, [0, i]], step.page_table, step.seq_lens, sm)
        assert np.array_equal(got[0, i], want[0, 1]), i


def test_invalid_tree_is_refused():
    L, W, H, Hq = 10, 4, 1, 1
    spec, step, cache = _cache_with_window(oracle.KV_FP8, 94, L, W, H, Hq)
    with pytest.raises(ValueError):
        oracle.tree_attn(cache, step.q, step.page_table, step.seq_lens, np.array([[0, 0, 2, 1]], np.int32), 0.1)


def test_compaction_by_ragged_reappend_int4():
    # after acceptance the path's K/V must sit at L + 1 .. L + a: re-appending the
    # accepted slots' rows there (a ragged append of a tokens) leaves, with INT4's
    # per-token scales, exactly what appending the accepted chain directly leaves
    rng = np.random.default_rng(95)
    L, W, H = 100, 8, 2
    spec = synth.Spec("tree", 95, 1, 0, 0, 2 * H, H, W, oracle.KV_INT4, 64, 0.7, True)
    step = synth.make_step(spec, seq_lens=np.array([L], np.int32), with_accept=False)
    parent = np.array([[0, 0, 1, 0, 2, 4, 3, 5]], np.int32)
    path = [0, 1, 2, 4, 5]  # an accepted path of the tree, a = 4
    a = len(path) - 1

    def fresh():
        c = oracle.Cache(oracle.KV_INT4, step.num_pages, H)
        for start, n in synth.fill_chunks(L, 64):
            k, v = synth.context_chunk(spec, 0, start, n)
            oracle.append(c, k[None], v[None], step.page_table, np.array([start], np.int32))
        return c

    tree = fresh()
    assert oracle.append(tree, step.k_win, step.v_win, step.page_table, step.seq_lens) == 0
    kg = np.ascontiguousarray(step.k_win[:, path[1:]])
    vg = np.ascontiguousarray(step.v_win[:, path[1:]])
    pad = np.zeros((1, W - 1 - a) + kg.shape[2:], kg.dtype)
    assert oracle.append_ragged(tree, np.concatenate([kg, pad], 1), np.concatenate([vg, pad], 1), step.page_table,
                                step.seq_lens + 1, np.array([a], np.int32)) == 0
    chain = fresh()
    assert oracle.append(chain, step.k_win[:, path], step.v_win[:, path], step.page_table, step.seq_lens) == 0
    row = step.page_table[0]
    for pos in range(L + a + 1):
        pid, off = row[pos // PAGE], pos % PAGE
        for n in ("k_codes", "v_codes", "k_scales", "v_scales"):
            assert np.array_equal(getattr(tree, n)[pid, :, off], getattr(chain, n)[pid, :, off]), (pos, n)
