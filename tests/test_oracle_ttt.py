"""Pins for the oracle's training-time-test attention (EAGLE-3: causal on the original
sequence, diagonal on the earlier TTT steps' predictions, one softmax over both),
against torch's scaled_dot_product_attention in float64: with is_causal for step 0,
and over the explicitly concatenated key set (trunk then branch) with the mask the
pages describe for later steps."""
import numpy as np
import pytest
import torch

import oracle


def _case(K, S, Hq, Hkv, D, seed):
    g = np.random.default_rng(seed)
    q = g.normal(0, 1, (K, S, Hq, D)).astype(np.float32)
    kt = g.normal(0, 1, (Hkv, S, D)).astype(np.float32)
    vt = g.normal(0, 1, (Hkv, S, D)).astype(np.float32)
    kb = g.normal(0, 1, (K, Hkv, S, D)).astype(np.float32)
    vb = g.normal(0, 1, (K, Hkv, S, D)).astype(np.float32)
    return q, kt, vt, kb, vb


def test_step0_is_causal_attention():
    q, kt, vt, kb, vb = _case(2, 37, 4, 2, 16, 1)
    out, lse = oracle.ttt_attn(q, kt, vt, kb, vb, 0.25)
    for hq in range(4):
        h = hq // 2
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q[0, :, hq]).double()[None], torch.from_numpy(kt[h]).double()[None],
            torch.from_numpy(vt[h]).double()[None], is_causal=True, scale=0.25)[0].numpy()
        assert np.abs(out[0, :, hq] - ref).max() < 1e-12


@pytest.mark.parametrize("K", [3, 7])
def test_later_steps_attend_to_trunk_prefix_and_own_predecessors(K):
    S, Hq, Hkv, D, scale = 29, 2, 1, 8, 0.3
    q, kt, vt, kb, vb = _case(K, S, Hq, Hkv, D, K)
    out, lse = oracle.ttt_attn(q, kt, vt, kb, vb, scale)
    # keys: trunk positions 0..S-1, then branch (i, t) for i = 1..K-1, t = 0..S-1
    keys = np.concatenate([kt[0]] + [kb[i, 0] for i in range(1, K)], axis=0)
    vals = np.concatenate([vt[0]] + [vb[i, 0] for i in range(1, K)], axis=0)
    for j in range(K):
        mask = np.zeros((S, keys.shape[0]), bool)
        for t in range(S):
            mask[t, :t + 1] = True                      # causal on the original sequence
            for i in range(1, j + 1):
                mask[t, S * i + t] = True               # diagonal: its own predecessor only
        for hq in range(Hq):
            ref = torch.nn.functional.scaled_dot_product_attention(
                torch.from_numpy(q[j, :, hq]).double()[None], torch.from_numpy(keys).double()[None],
                torch.from_numpy(vals).double()[None], attn_mask=torch.from_numpy(mask)[None], scale=scale)[0].numpy()
            assert np.abs(out[j, :, hq] - ref).max() < 1e-12
            s = (q[j, :, hq].astype(np.float64) @ keys.T.astype(np.float64)) * scale
            s[~mask] = -np.inf
            m = s.max(axis=1)
            assert np.abs(lse[j, :, hq] - (m + np.log(np.exp(s - m[:, None]).sum(axis=1)))).max() < 1e-12
