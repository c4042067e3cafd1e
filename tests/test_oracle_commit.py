"""Pins for the oracle's KV commit (KV rollback bookkeeping).

Commit keeps the accepted path and drops the rest: path node m's K/V goes to cache
slot seq_len + m (m = 0 is the root, the pending token whose K/V the verify pass
computed), and the logical length becomes seq_len + n_acc + 1 (EAGLE review,
section 3.3 and data path step 7; lesson "KV cache rollback" and step 4).  The
emitted correction/bonus token is the next step's root; its K/V comes from the
next verify pass.
"""
import numpy as np

import oracle
from eagle_speculative_decoding_tree_gb300 import synth


def test_commit_is_an_exact_byte_copy():
    g = synth.rng(0, 9500)
    L, B, H, P, R, D, Fw = 3, 2, 2, 40, 11, 8, 6
    kc = synth.bf16_bits(synth.normal_row(g, (L, B, H, P, D), 1.0))
    vc = synth.bf16_bits(synth.normal_row(g, (L, B, H, P, D), 1.0))
    tk = synth.bf16_bits(synth.normal_row(g, (L, B, H, R, D), 1.0))
    tv = synth.bf16_bits(synth.normal_row(g, (L, B, H, R, D), 1.0))
    fc = synth.normal_row(g, (B, P, Fw), 1.0)
    tf = synth.normal_row(g, (B, R, Fw), 1.0)
    seq_len = np.array([20, 7], np.int32)
    n_acc = np.array([3, 0], np.int32)
    path = np.array([[0, 1, 5, 9], [0, -1, -1, -1]], np.int32)
    kc0, vc0, fc0 = kc.copy(), vc.copy(), fc.copy()
    new_len, pos = oracle.kv_commit(kc, vc, tk, tv, n_acc, path, seq_len, fc, tf)
    assert new_len.tolist() == [24, 8]
    assert pos.tolist() == [[20, 21, 22, 23], [7, -1, -1, -1]]
    for b in range(B):
        touched = set()
        for m in range(n_acc[b] + 1):
            s = seq_len[b] + m
            touched.add(s)
            assert kc[:, b, :, s].tobytes() == tk[:, b, :, path[b, m]].tobytes()
            assert vc[:, b, :, s].tobytes() == tv[:, b, :, path[b, m]].tobytes()
            assert fc[b, s].tobytes() == tf[b, path[b, m]].tobytes()
        for s in range(P):
            if s not in touched:
                assert kc[:, b, :, s].tobytes() == kc0[:, b, :, s].tobytes()
                assert vc[:, b, :, s].tobytes() == vc0[:, b, :, s].tobytes()
                assert fc[b, s].tobytes() == fc0[b, s].tobytes()


def test_two_sequence_rollback_exercise():
    """Lesson exercise: sequence A accepts every draft, sequence B rejects the
    draft at position 2.  Both logical lengths must come out right and nothing
    past them may be committed."""
    N, V = 4, 8
    R = N + 1
    parent = np.arange(-1, N, dtype=np.int32)
    tokens = np.array([[7, 1, 2, 3, 4], [7, 1, 2, 3, 4]], np.int32)
    target = np.full((2, R, V), -5.0, np.float32)
    for i in range(R):
        target[0, i, (tokens[0, i + 1] if i + 1 < R else 6)] = 5.0   # A: argmax follows the chain
        target[1, i, (tokens[1, i + 1] if i + 1 < R else 6)] = 5.0
    target[1, 1, :] = -5.0
    target[1, 1, 5] = 5.0                                            # B: draft 2 (token 2) loses to token 5
    res = oracle.accept(target, tokens, parent, np.zeros((2, R), np.float32), np.zeros(2, np.float32), 0.0,
                        oracle.DELTA, R)
    assert res["n_acc"].tolist() == [4, 1]
    assert res["out_tok"][0].tolist() == [1, 2, 3, 4, 6]
    assert res["out_tok"][1].tolist() == [1, 5, -1, -1, -1]
    L, H, P, D = 1, 1, 32, 4
    kc = np.zeros((L, 2, H, P, D), np.float32)
    vc = np.zeros((L, 2, H, P, D), np.float32)
    tk = np.arange(L * 2 * H * R * D, dtype=np.float32).reshape(L, 2, H, R, D) + 1
    tv = -tk
    seq_len = np.array([10, 10], np.int32)
    new_len, _ = oracle.kv_commit(kc, vc, tk, tv, res["n_acc"], res["path"], seq_len)
    assert new_len.tolist() == [15, 12]
    assert (kc[0, 0, 0, 10:15] == tk[0, 0, 0, 0:5]).all() and (kc[0, 0, 0, 15:] == 0).all()
    assert (kc[0, 1, 0, 10:12] == tk[0, 1, 0, 0:2]).all() and (kc[0, 1, 0, 12:] == 0).all()
