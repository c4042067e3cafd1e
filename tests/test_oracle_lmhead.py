"""Pins for the oracle's LM-head statistics (what acceptance needs from each node's
distribution: max, argmax and sum exp((x - max) / T) per vocabulary tile, and each
node's token logit under its parent's row), checked against things other than the
oracle itself: exact integer dot products, scipy's logsumexp, numpy's argmax over
whole rows, and the acceptance walk on materialised logits."""
import numpy as np
import pytest
from scipy.special import logsumexp

import oracle
from eagle_speculative_decoding_tree_gb300 import synth


def _bf16(x):
    return synth.bf16_bits(np.asarray(x, np.float32))


def test_integer_inputs_give_exact_logits_and_children():
    """Small integers are exact in bf16 and their dot products exact in any precision:
    the oracle's logits and child logits equal Python integer arithmetic."""
    g = np.random.default_rng(1)
    B, R, h, V = 2, 5, 24, 300
    H = g.integers(-3, 4, (B * R, h))
    W = g.integers(-3, 4, (V, h))
    par = np.array([[-1, 0, 0, 1, 2], [-1, 0, 1, 1, 3]])
    tok = g.integers(0, V, (B, R))
    st = oracle.lmhead_stats(_bf16(H), _bf16(W), 1.0, 64, tok, par)
    for r in range(B * R):
        for v in range(0, V, 37):
            assert st["logits"][r, v] == sum(int(a) * int(b) for a, b in zip(H[r], W[v]))
    for b in range(B):
        assert np.isnan(st["child"][b, 0])
        for i in range(1, R):
            want = sum(int(a) * int(c) for a, c in zip(H[b * R + par[b, i]], W[tok[b, i]]))
            assert st["child"][b, i] == want


@pytest.mark.parametrize("T,tile,V", [(1.0, 128, 1000), (0.7, 128, 1000), (1.0, 64, 777), (0.0, 256, 513)])
def test_tile_records_rebuild_the_row_log_normaliser_and_argmax(T, tile, V):
    g = np.random.default_rng(2)
    M, h = 7, 64
    H = _bf16(g.normal(0, 1, (M, h)))
    W = _bf16(g.normal(0, 1 / np.sqrt(h), (V, h)))
    st = oracle.lmhead_stats(H, W, T, tile)
    x = st["logits"]
    Tn = T if T > 0 else 1.0
    for r in range(M):
        Mx = st["max"][r].max()
        lse = Mx / Tn + np.log(np.sum(st["sum"][r] * np.exp((st["max"][r] - Mx) / Tn)))
        assert abs(lse - logsumexp(x[r] / Tn)) < 1e-12 * max(1.0, abs(lse))
        best = int(np.argmax(st["max"][r]))  # first tile holding the row max
        assert st["argmax"][r, best] == int(np.argmax(x[r]))
    assert st["max"].shape[1] == -(-V // tile)


def test_ties_in_a_tile_take_the_lowest_index():
    H = _bf16(np.ones((1, 8)))
    W = np.zeros((200, 8), np.float32)
    W[[30, 10, 150], :] = 1.0  # equal top logits at 10, 30 (tile 0) and 150 (tile 1)
    st = oracle.lmhead_stats(H, _bf16(W), 1.0, 128)
    assert st["argmax"][0, 0] == 10 and st["argmax"][0, 1] == 150


def test_acceptance_from_hidden_states_equals_acceptance_on_materialised_logits():
    g = np.random.default_rng(3)
    B, R, h, V = 3, 6, 32, 400
    H = _bf16(g.normal(0, 1, (B * R, h)))
    W = _bf16(g.normal(0, 1, (V, h)))
    par = np.array([[-1, 0, 0, 1, 1, 2]] * B, np.int32)
    tok = g.integers(0, V, (B, R)).astype(np.int32)
    ua = synth.uniforms(g, (B, R))
    uf = synth.uniforms(g, (B,))
    x = np.asarray(oracle.lmhead_logits(H, W), np.float32).reshape(B, R, V)
    ref = oracle.accept(x, tok, par, ua, uf, 1.0, oracle.DELTA, 4)
    got = oracle.lmhead_accept(H, W, tok, par, ua, uf, 1.0, oracle.DELTA, 4)
    for k in ("n_acc", "path", "out_tok"):
        assert np.array_equal(ref[k], got[k])
