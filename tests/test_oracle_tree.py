"""Pins for the oracle's draft-tree construction.

The pages give the idea (EAGLE-2: keep the most confident candidates, EAGLE-3
visual reading "EAGLE-2"; top-k children per node with k = 4 at the root, EAGLE
review appendix A.1) and not the steps; the oracle's reading is written out in
eagle_oracle.c.  Pinned here by: a hand-worked example (tests/golden), numpy's
lexsort for the per-row top-k, searchsorted for sampled children, and structural
invariants that any correct reading must satisfy (ancestor-closed, parents
first, cumulative path log-probabilities, kept >= dropped, masks = ancestors).
"""
import json
import os

import numpy as np
import pytest
from scipy.special import log_softmax

import oracle
from eagle_speculative_decoding_tree_gb300 import synth
from spec_helpers import OracleDynamicBuilder, OracleStaticBuilder, drive_tree_build

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _ancestors(parent, i):
    out = []
    while i >= 0:
        out.append(i)
        i = parent[i]
    return out


def _mask_of(parent, i, W):
    m = np.zeros(W, np.uint64)
    for a in _ancestors(parent, i):
        m[a // 64] |= np.uint64(1) << np.uint64(a % 64)
    return m


def test_hand_worked_dynamic_tree():
    g = json.load(open(os.path.join(GOLDEN, "dynamic_tree_hand_v4.json")))
    V, k, D = g["vocab"], g["top_k"], g["depth"]
    root_rows = np.log(np.array([[g["root_q"]]], np.float32))
    lvl2_rows = np.log(np.array([g["level2_q"]], np.float32))
    for case in g["cases"]:
        N = case["total_tokens"]
        t = oracle.DynamicTree(1, V, D, k, N)
        fr1 = t.expand(root_rows)
        assert t.frontier_tokens()[0].tolist() == [0, 1]
        fr2 = t.expand(lvl2_rows)
        assert t.frontier_tokens()[0].tolist() == g["level2_frontier_tokens"]
        assert t.frontier_parent_slot(fr1)[0].tolist() == g["level2_frontier_parent_slot"]
        out = t.finalize(np.array([g["root_token"]], np.int32), np.array([g["seq_len"]], np.int32))
        assert out["tokens"][0].tolist() == case["tokens"]
        assert out["parent"][0].tolist() == case["parent"]
        assert out["depth"][0].tolist() == case["depth"]
        assert out["pos_id"][0].tolist() == [g["seq_len"] + d for d in case["depth"]]
        np.testing.assert_allclose(np.exp(out["score"][0]), case["prob"], rtol=1e-6)
        for i in range(N + 1):
            assert np.array_equal(out["anc_mask"][0, i], _mask_of(case["parent"], i, 1))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_row_topk_matches_lexsort(dtype):
    g = synth.rng(0, 9100)
    V, k = 5000, 16
    rows = synth.normal_row(g, (3, V), 2.0)
    rows[2, :] = np.round(rows[2, :])  # many exact ties
    st = oracle.StaticTree(3, V, np.array([-1] + [0] * k, np.int32), False, 1.0)
    st.expand(synth.as_dtype_bytes(rows[:, None, :], dtype))
    vals = synth.bf16_value(synth.bf16_bits(rows)) if dtype == "bf16" else rows
    for b in range(3):
        order = np.lexsort((np.arange(V), -vals[b].astype(np.float64)))
        assert st.tokens[b, 1:].tolist() == order[:k].tolist()


def test_sampled_children_match_searchsorted():
    g = synth.rng(0, 9200)
    B, V, T = 300, 700, 0.8
    par = synth.static_parents(synth.TINY_STATIC_CHOICES)
    st = oracle.StaticTree(B, V, par, True, T)
    rows = synth.normal_row(g, (B, 1, V), 2.0)
    ud = synth.uniforms(g, (B, len(par)))
    st.expand(rows, ud)
    p = np.exp((rows[:, 0].astype(np.float64) - rows[:, 0].max(axis=1, keepdims=True)) / T)
    c = np.cumsum(p, axis=1)
    ok = st.near_tie == 0
    assert ok.mean() > 0.95
    for b in np.nonzero(ok)[0]:
        for child in (1, 2, 3, 4):
            expect = np.searchsorted(c[b], ud[b, child] * c[b, -1], side="right")
            assert st.tokens[b, child] == expect


@pytest.mark.parametrize("V,k,D,N,dtype", [(200, 6, 5, 25, "bf16"), (64, 4, 4, 16, "f32"), (300, 8, 3, 40, "bf16")])
def test_dynamic_tree_invariants(V, k, D, N, dtype):
    B = 6
    lm = synth.HashLM(V, "normal", 2.0, 0.6, dtype)
    roots = synth.rng(0, 9300).integers(0, V, B).astype(np.int32)
    hroot = [synth.root_hash(0, b, V) for b in range(B)]
    seq_len = np.arange(B, dtype=np.int32) * 10 + 50
    bld = OracleDynamicBuilder(B, V, D, k, N)
    rec = []
    tree = drive_tree_build(bld, lm, D, roots, hroot, seq_len, record=rec)
    t = bld.t
    R = N + 1
    W = max(1, -(-R // 64))
    for b in range(B):
        par, tok, dep = tree["parent"][b], tree["tokens"][b], tree["depth"][b]
        assert par[0] == -1 and dep[0] == 0 and tok[0] == roots[b]
        hs = [hroot[b]]
        for i in range(1, R):
            assert 0 <= par[i] < i
            assert dep[i] == dep[par[i]] + 1
            hs.append(synth.child_hash(hs[par[i]], int(tok[i])))
            # the token is among the parent's top-k draft tokens
            row = lm.draft_row(hs[par[i]]).astype(np.float64)
            order = np.lexsort((np.arange(V), -row))
            assert tok[i] in order[:k].tolist()
            # siblings come in rank order
            sib = [j for j in range(1, i) if par[j] == par[i]]
            if sib:
                assert order.tolist().index(tok[sib[-1]]) < order.tolist().index(tok[i])
            # score = cumulative ln q along the path (draft confidence at temperature 1)
            path_score = sum(log_softmax(lm.draft_row(hs[par[a]]).astype(np.float64))[tok[a]]
                             for a in _ancestors(par, i) if a > 0)
            assert abs(tree["score"][b, i] - path_score) < 1e-9
            assert np.array_equal(tree["anc_mask"][b, i], _mask_of(par, i, W))
            assert tree["pos_id"][b, i] == seq_len[b] + dep[i]
        # kept >= dropped, over the whole pool
        kept = set()
        sc = t.pool_score[b, : t.n_pool[b]]
        kept_scores = np.sort(tree["score"][b, 1:])
        dropped = np.sort(sc)[::-1][N:]
        if len(dropped):
            assert kept_scores.min() >= dropped.max() - 1e-12
    # each level's frontier is the best k of that level's new candidates
    for b in range(B):
        base = 0
        for level in range(1, D + 1):
            F = 1 if level == 1 else k
            new = np.arange(base, base + F * k)
            best = new[np.lexsort((new, -t.pool_score[b, new]))][:k]
            base += F * k
            if level == D:
                assert sorted(best.tolist()) == t.frontier[b].tolist()


def test_dynamic_tree_keeps_whole_pool_when_n_equals_pool():
    V, k, D = 30, 3, 3
    N = k + (D - 1) * k * k
    lm = synth.HashLM(V, "normal", 2.0, 0.5, "f32")
    bld = OracleDynamicBuilder(2, V, D, k, N)
    tree = drive_tree_build(bld, lm, D, np.array([1, 2], np.int32), [11, 12], np.zeros(2, np.int32))
    assert (np.bincount(tree["depth"][0], minlength=D + 1) == [1, k, k * k, k * k]).all()


def test_equal_logits_pick_lowest_ids():
    V, k = 50, 5
    t = oracle.DynamicTree(1, V, 1, k, k)
    t.expand(np.zeros((1, 1, V), np.float32))
    out = t.finalize(np.array([3], np.int32), np.array([0], np.int32))
    assert out["tokens"][0, 1:].tolist() == [0, 1, 2, 3, 4]
    np.testing.assert_allclose(out["score"][0, 1:], -np.log(V), rtol=1e-12)


def test_static_topk_tree_children_are_ranked_tokens():
    V = 120
    par = synth.static_parents(synth.TINY_STATIC_CHOICES)
    lm = synth.HashLM(V, "normal", 2.0, 0.5, "bf16")
    bld = OracleStaticBuilder(2, V, par, False, 0.0)
    hroot = [5, 6]
    tree = drive_tree_build(bld, lm, 3, np.array([7, 8], np.int32), hroot, np.array([10, 20], np.int32))
    choices = ((),) + synth.TINY_STATIC_CHOICES
    for b in range(2):
        hs = [hroot[b]]
        for i in range(1, len(par)):
            hs.append(synth.child_hash(hs[par[i]], int(tree["tokens"][b, i])))
            row = lm.draft_row(hs[par[i]]).astype(np.float64)
            order = np.lexsort((np.arange(V), -row))
            assert tree["tokens"][b, i] == order[choices[i][-1]]


@pytest.mark.parametrize("choices", [synth.TINY_STATIC_CHOICES,
                                     tuple((0,) * d for d in range(1, 8)),
                                     tuple((i,) for i in range(70)) + ((0, 0), (69, 3))])
def test_static_finalize_from_the_choice_paths(choices):
    """StaticTree.finalize against the static tree written as child-rank paths (EAGLE
    review appendix A.1, a fixed tree shape): node j is an ancestor of node i exactly
    when j's path is a prefix of i's (the root's empty path is a prefix of every path),
    a node's depth is its path length and its position is seq_len + depth.  Covers the
    tiny tree, the 8-row chain and a 73-row tree that needs two mask words."""
    paths = ((),) + tuple(tuple(c) for c in choices)
    R = len(paths)
    W = -(-R // 64)
    par = synth.static_parents(choices)
    t = oracle.StaticTree(2, 50, par, False, 0.0)
    seq_len = np.array([5, 1234], np.int32)
    out = t.finalize(np.array([11, 22], np.int32), seq_len)
    for i, pi in enumerate(paths):
        want = np.zeros(W, np.uint64)
        for j, pj in enumerate(paths):
            if pi[:len(pj)] == pj:
                want[j // 64] |= np.uint64(1) << np.uint64(j % 64)
        for b in range(2):
            assert np.array_equal(out["anc_mask"][b, i], want), (i, pi)
            assert out["depth"][b, i] == len(pi)
            assert out["pos_id"][b, i] == seq_len[b] + len(pi)
            assert out["parent"][b, i] == (-1 if i == 0 else paths.index(pi[:-1]))
    assert out["tokens"][:, 0].tolist() == [11, 22]
