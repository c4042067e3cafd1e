"""GPU parity: eagle_ttt_attn (EAGLE-3 training-time-test attention: causal trunk on the
tensor cores, each prediction's own predecessors in earlier TTT steps folded into the
same softmax) against the oracle.  bf16 inputs N(0, 1), fp32 accumulation: max abs
error 2e-3 plus the one rounding of a bf16 output (2^-8 |O|); lse within 2e-3."""
import math

import numpy as np
import pytest
import torch

import oracle
from eagle_speculative_decoding_tree_gb300 import binding as B
from eagle_speculative_decoding_tree_gb300 import synth

pytestmark = pytest.mark.gpu


def _case(K, S, Hq, Hkv, seed, q_scale=1.0):
    g = np.random.default_rng(seed)
    bits = lambda shape, sc=1.0: synth.bf16_bits((g.normal(0, 1, shape) * sc).astype(np.float32))
    return (bits((K, S, Hq, 128), q_scale), bits((Hkv, S, 128)), bits((Hkv, S, 128)), bits((K, Hkv, S, 128)),
            bits((K, Hkv, S, 128)))


def _run(ins, Hq, Hkv, out_f32=False):
    q, kt, vt, kb, vb = ins
    K, S = q.shape[:2]
    dv = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)
    desc = B.TttDesc(K, S, Hq, Hkv, 128, 1.0 / math.sqrt(128), B.EAGLE_F32 if out_f32 else B.EAGLE_BF16)
    ws = torch.zeros(B.workspace_size(B.EAGLE_WS_TTT_ATTN, desc), dtype=torch.uint8, device="cuda")
    out = torch.full((K, S, Hq, 128), float("nan"), dtype=torch.float32 if out_f32 else torch.bfloat16, device="cuda")
    lse = torch.empty(K, S, Hq, dtype=torch.float32, device="cuda")
    B.eagle_ttt_attn(desc, dv(q), dv(kt), dv(vt), dv(kb), dv(vb), out, lse, ws)
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32).item()) == 0, "a bounded wait gave up"
    return out.float().cpu().numpy(), lse.cpu().numpy()


@pytest.mark.parametrize("K,S,Hq,Hkv,q_scale", [(4, 333, 8, 2, 1.0), (7, 200, 4, 4, 1.0), (1, 129, 4, 1, 1.0),
                                                (3, 260, 8, 2, 4.0)])
def test_ttt_attention(K, S, Hq, Hkv, q_scale):
    ins = _case(K, S, Hq, Hkv, seed=K * 100 + S, q_scale=q_scale)
    ref, ref_lse = oracle.ttt_attn(*ins, 1.0 / math.sqrt(128))
    for out_f32 in (False, True):
        out, lse = _run(ins, Hq, Hkv, out_f32)
        err = np.abs(out - ref)
        bound = 2e-3 + (0.0 if out_f32 else 2.0 ** -8 * np.abs(ref))
        assert (err <= bound).all(), f"max error {err.max():.3e} (out_f32={out_f32})"
        assert np.abs(lse - ref_lse).max() < 2e-3


def test_ttt_attention_training_shape():
    """An 8B-shaped draft layer in training: 32 q / 8 kv heads x 128, sequence 2048,
    7 TTT steps; heads 0 and 31 of steps 0, 3 and 6 against the oracle."""
    K, S, Hq, Hkv = 7, 2048, 32, 8
    ins = _case(K, S, Hq, Hkv, seed=99)
    out, lse = _run(ins, Hq, Hkv)
    q, kt, vt, kb, vb = ins
    for hq in (0, 31):
        h = hq // (Hq // Hkv)
        sub = (np.ascontiguousarray(q[:, :, hq:hq + 1]), np.ascontiguousarray(kt[h:h + 1]),
               np.ascontiguousarray(vt[h:h + 1]), np.ascontiguousarray(kb[:, h:h + 1]),
               np.ascontiguousarray(vb[:, h:h + 1]))
        ref, ref_lse = oracle.ttt_attn(*sub, 1.0 / math.sqrt(128))
        for j in (0, 3, 6):
            err = np.abs(out[j, :, hq] - ref[j, :, 0])
            assert (err <= 2e-3 + 2.0 ** -8 * np.abs(ref[j, :, 0])).all(), (hq, j, err.max())
            assert np.abs(lse[j, :, hq] - ref_lse[j, :, 0]).max() < 2e-3
