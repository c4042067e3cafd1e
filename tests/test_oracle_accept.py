"""Pins for the oracle's acceptance (multi-round speculative sampling).

What the pages fix, and how each is checked here:
  * losslessness: the emitted tokens follow the target distribution, greedy and
    non-greedy (EAGLE review sections 3.3 and 4; lesson "Leviathan rule") --
    chi-square over 10^6 trials on a 16-token vocabulary, for the dynamic top-k
    tree, the static sampled tree and the sampled chain, on the first emitted
    token and on the first two jointly (lesson step 5 runs the same check);
  * the planted non-lossless reading (draft softmax as the proposal of a
    deterministically chosen candidate) must fail the same test;
  * E[tokens per verify] = (1 - a^(N+1)) / (1 - a) for a chain with per-token
    acceptance a (lesson "what sets the speedup");
  * the Fig. 3 toy distribution p(am) = 0.6, p(always) = 0.4 (EAGLE review /
    EAGLE-3 visual reading, Figure 3), reproduced exactly on a uniform grid;
  * the lesson's accept snippet: a draft probability <= 0 accepts;
  * special cases: p == q accepts everything, a one-hot target is greedy, a leaf
    draws from the untouched target (checked against numpy's searchsorted).
"""
import numpy as np
import pytest
from scipy.special import softmax

import oracle
from eagle_speculative_decoding_tree_gb300 import synth
from spec_helpers import chisquare_pvalue, first_two_tokens

V16 = 16
TRIALS = 1_000_000


def _lm():
    return synth.BigramLM(V16, sigma=1.5, draft_sigma=0.7, seed_key=1)


def _joint_expected(lm, root, T=1.0):
    p1 = softmax(lm.target[root].astype(np.float64) / T)
    p2 = softmax(lm.target.astype(np.float64) / T, axis=1)
    return p1, p1[:, None] * p2


def _check_lossless(t1, t2, lm, root):
    p1, joint = _joint_expected(lm, root)
    c1 = np.bincount(t1, minlength=V16)
    c12 = np.bincount(t1 * V16 + t2, minlength=V16 * V16)
    return chisquare_pvalue(c1, p1), chisquare_pvalue(c12, joint)


@pytest.mark.parametrize("mode,proposal,seed,kw", [
    ("dynamic", oracle.DELTA, 1, dict(depth=3, top_k=4, total_tokens=10)),
    ("static_sampled", oracle.SAMPLED, 2, dict(static_parent=synth.static_parents(synth.TINY_STATIC_CHOICES))),
    ("static_sampled", oracle.SAMPLED, 3, dict(static_parent=synth.static_parents(synth.CHAIN7))),
], ids=["dynamic-delta", "static10-sampled", "chain7-sampled"])
def test_chisquare_lossless(mode, proposal, seed, kw):
    lm = _lm()
    root = 3
    t1, t2 = first_two_tokens(lm, root, mode, proposal, 1.0, TRIALS, seed=seed, **kw)
    p_first, p_joint = _check_lossless(t1, t2, lm, root)
    print(f"chi-square p-values: first token {p_first:.4f}, first two tokens {p_joint:.4f}")
    assert p_first > 1e-3, p_first
    assert p_joint > 1e-3, p_joint


def test_chisquare_detects_planted_non_lossless_rule():
    """Top-k candidates judged with the draft softmax as their proposal (the literal
    reading of p/q for a deterministic candidate) is not lossless; the test must see it."""
    lm = _lm()
    t1, t2 = first_two_tokens(lm, 3, "dynamic", oracle.SAMPLED, 1.0, 200_000, seed=11,
                              depth=3, top_k=4, total_tokens=10)
    p_first, p_joint = _check_lossless(t1, t2, lm, 3)
    assert p_first < 1e-6 and p_joint < 1e-6, (p_first, p_joint)


@pytest.mark.parametrize("alpha,expected", [(0.5, 1.992), (0.6, 2.458), (0.8, 4.161), (0.9, 5.695)])
def test_expected_tokens_per_verify_closed_form(alpha, expected):
    N, V, trials = 7, 4, TRIALS
    e_closed = (1 - alpha ** (N + 1)) / (1 - alpha)
    assert abs(e_closed - expected) < 5e-4  # the printed values of the closed form
    R = N + 1
    parent = np.arange(-1, N, dtype=np.int32)
    tokens = np.zeros(R, np.int32)
    # draft: point mass on token 0; target: p(0) = alpha, the rest shares 1 - alpha
    draft = np.full((R, V), -np.inf, np.float32)
    draft[:, 0] = 0.0
    target = np.full((R, V), np.log((1 - alpha) / (V - 1)), np.float32)
    target[:, 0] = np.log(alpha)
    # exact law of X = n_acc + 1: P(X = j+1) = a^j (1-a) for j < N, P(X = N+1) = a^N
    js = np.arange(N + 1)
    px = np.where(js < N, alpha ** js * (1 - alpha), alpha ** N)
    mean_x = (px * (js + 1)).sum()
    sd_x = np.sqrt((px * (js + 1) ** 2).sum() - mean_x ** 2)
    assert abs(mean_x - e_closed) < 1e-12
    total = 0
    chunk = 100_000
    for c in range(trials // chunk):
        g = synth.rng(0, 8100, int(alpha * 100), c)
        ua = synth.uniforms(g, (chunk, R))
        uf = synth.uniforms(g, (chunk,))
        res = oracle.accept(np.broadcast_to(target, (chunk, R, V)), np.broadcast_to(tokens, (chunk, R)), parent,
                            ua, uf, 1.0, oracle.SAMPLED, R, draft=np.broadcast_to(draft, (chunk, R, V)))
        total += int(res["n_acc"].sum()) + chunk
    mean = total / trials
    assert abs(mean - e_closed) < 4 * sd_x / np.sqrt(trials), (mean, e_closed)


def test_fig3_toy_distribution_exact_on_grid():
    """After "I": p(am) = 0.6, p(always) = 0.4.  A single top-1 draft "am" is accepted
    iff u < 0.6; otherwise the residual puts all mass on "always"."""
    M = 10000
    u = ((np.arange(M) + 0.5) / M).astype(np.float32)
    target = np.log(np.array([[[0.6, 0.4], [0.5, 0.5]]], np.float32))  # rows: root, node "am"
    tokens = np.array([[7, 0]], np.int32)  # root token, child token 0 = "am"
    parent = np.array([[-1, 0]], np.int32)
    B = M
    tgt = np.broadcast_to(target, (B, 2, 2))
    ua = np.stack([np.zeros(M, np.float32), u], axis=1)
    res = oracle.accept(tgt, np.broadcast_to(tokens, (B, 2)), parent, ua, np.full(B, 0.5, np.float32), 1.0,
                        oracle.DELTA, 2)
    first = res["out_tok"][:, 0]
    assert (first == 0).sum() == 6000 and (first == 1).sum() == 4000
    # the literal reading (draft softmax q = (0.9, 0.1) as the proposal) gives 2/3 instead
    draft = np.log(np.array([[[0.9, 0.1], [0.5, 0.5]]], np.float32))
    res2 = oracle.accept(tgt, np.broadcast_to(tokens, (B, 2)), parent, ua, np.full(B, 0.5, np.float32), 1.0,
                         oracle.SAMPLED, 2, draft=np.broadcast_to(draft, (B, 2, 2)))
    assert (res2["out_tok"][:, 0] == 0).sum() == 6667


def test_zero_draft_probability_accepts():
    """Lesson step 1: a draft probability <= 0 accepts."""
    target = np.log(np.array([[[0.5, 0.5, 0.0 + 1e-30], [0.3, 0.3, 0.4]]], np.float32))
    draft = np.array([[[0.0, 0.0, -np.inf], [0.0, 0.0, 0.0]]], np.float32)
    res = oracle.accept(target, np.array([[0, 2]], np.int32), np.array([[-1, 0]], np.int32),
                        np.array([[0.0, 0.999]], np.float32), np.array([0.1], np.float32), 1.0, oracle.SAMPLED, 2,
                        draft=draft)
    assert res["n_acc"][0] == 1 and res["out_tok"][0, 0] == 2


def test_equal_draft_and_target_accept_everything():
    lm = synth.BigramLM(32, 2.0, 0.0, seed_key=2)
    parent = synth.static_parents(synth.TINY_STATIC_CHOICES)
    from spec_helpers import build_tree_bigram
    B = 2000
    g = synth.rng(0, 8200)
    roots = g.integers(0, 32, B).astype(np.int32)
    tree = build_tree_bigram(lm, roots, "static_sampled", static_parent=parent, u_draft=synth.uniforms(g, (B, 11)))
    tgt = lm.target[tree["tokens"]]
    res = oracle.accept(tgt, tree["tokens"], tree["parent"], synth.uniforms(g, (B, 11)), synth.uniforms(g, (B,)),
                        1.0, oracle.SAMPLED, 4, draft=tgt)
    # the first child is always accepted, so the walk follows the first-child chain 0-1-5-9
    assert (res["n_acc"] == 3).all()
    assert (res["path"] == np.array([0, 1, 5, 9])).all()


def test_one_hot_target_behaves_like_greedy():
    g = synth.rng(0, 8300)
    B, R, V = 500, 11, 50
    parent = synth.static_parents(synth.TINY_STATIC_CHOICES)
    target = synth.normal_row(g, (B, R, V), 3.0)
    tokens = g.integers(0, V, (B, R)).astype(np.int32)
    # make a child token the argmax in some rows
    tokens[:, 1] = np.argmax(target[:, 0], axis=1)
    onehot = np.where(target == target.max(axis=2, keepdims=True), np.float32(0.0), np.float32(-1e4))
    ua, uf = synth.uniforms(g, (B, R)), synth.uniforms(g, (B,))
    r_soft = oracle.accept(onehot, tokens, parent, ua, uf, 1.0, oracle.DELTA, 4)
    r_greedy = oracle.accept(target, tokens, parent, ua, uf, 0.0, oracle.DELTA, 4)
    for key in ("n_acc", "path", "out_tok"):
        assert np.array_equal(r_soft[key], r_greedy[key]), key
    assert (r_greedy["n_acc"] >= 1).all()


def test_leaf_draws_from_untouched_target():
    g = synth.rng(0, 8400)
    B, V = 4000, 300
    for T in (1.0, 0.7):
        target = synth.normal_row(g, (B, 1, V), 2.0)
        uf = synth.uniforms(g, (B,))
        res = oracle.accept(target, np.zeros((B, 1), np.int32), np.full((B, 1), -1, np.int32),
                            np.zeros((B, 1), np.float32), uf, T, oracle.DELTA, 1)
        assert (res["n_acc"] == 0).all()
        p = softmax(target[:, 0].astype(np.float64) / T, axis=1)
        c = np.cumsum(p, axis=1)
        expect = np.array([np.searchsorted(c[b], uf[b] * c[b, -1], side="right") for b in range(B)])
        ok = res["near_tie"] == 0
        assert ok.mean() > 0.99
        assert np.array_equal(res["out_tok"][ok, 0], expect[ok])


def test_temperature_is_logit_scaling():
    g = synth.rng(0, 8500)
    B, R, V = 1000, 11, 64
    parent = synth.static_parents(synth.TINY_STATIC_CHOICES)
    target = synth.normal_row(g, (B, R, V), 1.0)
    draft = synth.normal_row(g, (B, R, V), 1.0)
    tokens = g.integers(0, V, (B, R)).astype(np.int32)
    ua, uf = synth.uniforms(g, (B, R)), synth.uniforms(g, (B,))
    a = oracle.accept(target, tokens, parent, ua, uf, 0.5, oracle.SAMPLED, 4, draft=draft)
    b = oracle.accept(2 * target, tokens, parent, ua, uf, 1.0, oracle.SAMPLED, 4, draft=2 * draft)
    for key in ("n_acc", "out_tok"):
        assert np.array_equal(a[key], b[key])


def test_near_tie_is_reported():
    target = np.log(np.array([[[0.25, 0.75], [0.5, 0.5]]], np.float32))
    p0 = softmax(target[0, 0].astype(np.float64))[0]
    for du, near in ((0.0, 1), (3e-6, 1), (5e-5, 0)):  # accept test: |u - p/q| < 1e-5
        res = oracle.accept(target, np.array([[1, 0]], np.int32), np.array([[-1, 0]], np.int32),
                            np.array([[0.0, p0 + du]], np.float32), np.array([0.9], np.float32), 1.0, oracle.DELTA, 2)
        assert res["near_tie"][0] == near, du
