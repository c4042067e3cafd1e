"""Pins for the oracle's tree attention.

Tree attention is defined on the pages as "each candidate attends only to its
ancestors" (EAGLE review, terms "tree attention"; lesson glossary "Tree
attention").  The pins below check the oracle against things that do not share its
formulation: per-path causal attention over an explicitly built token sequence,
closed forms, and GQA head replication.
"""
import numpy as np
import pytest
from scipy.special import logsumexp, softmax

import oracle
from eagle_speculative_decoding_tree_gb300 import synth


def _causal_attention(q, k, v, scale):
    """Plain causal attention over one sequence: q,k,v [T][D] -> out [T][D], lse [T]."""
    T = q.shape[0]
    x = (q @ k.T) * scale
    x = np.where(np.tril(np.ones((T, T), bool)), x, -np.inf)
    return softmax(x, axis=1) @ v, logsumexp(x, axis=1)


def _inputs(dtype, B=2, R=11, Hq=4, Hkv=2, D=16, P=40, seed=0):
    g = synth.rng(0, 1000 + seed)
    f = lambda *s: synth.as_dtype_bytes(synth.normal_row(g, s, 1.0), dtype)
    q, kc, vc = f(B, R, Hq, D), f(B, Hkv, P, D), f(B, Hkv, P, D)
    tk, tv = f(B, Hkv, R, D), f(B, Hkv, R, D)
    val = (lambda a: synth.bf16_value(a)) if dtype == "bf16" else (lambda a: a)
    return (q, kc, vc, tk, tv), [val(a).astype(np.float64) for a in (q, kc, vc, tk, tv)]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_tree_attention_equals_per_path_causal_attention(dtype):
    B, R, Hq, Hkv, D, P = 2, 11, 4, 2, 16, 40
    G = Hq // Hkv
    raw, (q, kc, vc, tk, tv) = _inputs(dtype, B, R, Hq, Hkv, D, P)
    parent = synth.static_parents(synth.TINY_STATIC_CHOICES)
    seq_len = np.array([17, 33], np.int32)
    scale = 1.0 / np.sqrt(D)
    out, lse = oracle.tree_attn(*raw, seq_len, np.broadcast_to(parent, (B, R)), scale)

    leaves = [i for i in range(R) if i not in set(parent.tolist())]
    checked = set()
    for b in range(B):
        L = int(seq_len[b])
        for leaf in leaves:
            path = []
            a = leaf
            while a >= 0:
                path.append(a)
                a = parent[a]
            path = path[::-1]  # root .. leaf
            for hq in range(Hq):
                h = hq // G  # query head hq reads KV head hq // G
                seq_k = np.concatenate([kc[b, h, :L], tk[b, h, path]])
                seq_v = np.concatenate([vc[b, h, :L], tv[b, h, path]])
                seq_q = np.concatenate([np.zeros((L, D)), q[b, path, hq]])
                o, l = _causal_attention(seq_q, seq_k, seq_v, scale)
                for t, node in enumerate(path):
                    np.testing.assert_allclose(out[b, node, hq], o[L + t], rtol=0, atol=1e-12)
                    assert abs(lse[b, node, hq] - l[L + t]) < 1e-12
                    checked.add((b, node, hq))
    assert len(checked) == B * R * Hq


def test_single_key_returns_its_value():
    # empty prefix, root only: softmax over one key is 1
    raw, vals = _inputs("f32", B=1, R=1, Hq=2, Hkv=1, D=8, P=4)
    out, lse = oracle.tree_attn(*raw, np.zeros(1, np.int32), np.array([[-1]], np.int32), 0.5)
    q, _, _, tk, tv = vals
    for hq in range(2):
        np.testing.assert_allclose(out[0, 0, hq], tv[0, 0, 0], atol=1e-15)
        assert abs(lse[0, 0, hq] - 0.5 * q[0, 0, hq] @ tk[0, 0, 0]) < 1e-12


def test_equal_keys_give_mean_of_visible_values():
    B, R, Hq, Hkv, D, P = 1, 11, 2, 2, 8, 16
    raw, vals = _inputs("f32", B, R, Hq, Hkv, D, P)
    q, kc, vc, tk, tv = raw
    kc[:] = 0.25
    tk[:] = 0.25
    parent = synth.static_parents(synth.TINY_STATIC_CHOICES)
    L = 9
    out, lse = oracle.tree_attn(q, kc, vc, tk, tv, np.array([L], np.int32), parent[None], 1.0)
    vcv, tvv = vc.astype(np.float64), tv.astype(np.float64)
    for i in range(R):
        anc = []
        a = i
        while a >= 0:
            anc.append(a)
            a = parent[a]
        for h in range(Hq):
            vis = np.concatenate([vcv[0, h, :L], tvv[0, h, anc]])
            np.testing.assert_allclose(out[0, i, h], vis.mean(axis=0), atol=1e-14)
            x = 0.25 * q[0, i, h].astype(np.float64).sum()
            assert abs(lse[0, i, h] - (x + np.log(L + len(anc)))) < 1e-12


def test_siblings_do_not_see_each_other():
    # changing a node's K/V must not change the output of any node that is not its descendant
    B, R, Hq, Hkv, D, P = 1, 11, 2, 1, 8, 8
    raw, _ = _inputs("f32", B, R, Hq, Hkv, D, P, seed=3)
    parent = synth.static_parents(synth.TINY_STATIC_CHOICES)
    sl = np.array([5], np.int32)
    base, _ = oracle.tree_attn(*raw, sl, parent[None], 0.3)
    q, kc, vc, tk, tv = [a.copy() for a in raw]
    tk[0, 0, 5] += 1.0
    tv[0, 0, 5] -= 2.0
    moved, _ = oracle.tree_attn(q, kc, vc, tk, tv, sl, parent[None], 0.3)
    descendants_of_5 = {5, 9, 10}
    for i in range(R):
        changed = not np.allclose(base[0, i], moved[0, i], atol=0, rtol=0)
        assert changed == (i in descendants_of_5), i


def test_rejects_bad_parent():
    raw, _ = _inputs("f32", B=1, R=3, Hq=1, Hkv=1, D=4, P=4)
    with pytest.raises(ValueError):
        oracle.tree_attn(*raw, np.array([2], np.int32), np.array([[-1, 2, 0]], np.int32), 1.0)
