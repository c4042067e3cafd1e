"""GPU parity: eagle_lmhead_stats (vocabulary statistics at every tree node from the
hidden states and the LM head, logits never written) against the oracle's float64
statistics of the materialised logits.  Hidden ~ N(0, 1), head ~ N(0, 1/h), both
bf16, so logits ~ N(0, 1); fp32 accumulation over h = 4096 products.  Tolerances:
max and child logits within 1e-4 absolute; a tile sum of exp((x - max) / T) then
moves by at most a factor exp(2e-4 / T), so tile sums within 2e-4 / T relative;
argmax exact except where the tile's two largest logits are within 1e-4 (counted)."""
import numpy as np
import pytest
import torch

import oracle
from conftest import record_near_ties
from eagle_speculative_decoding_tree_gb300 import binding as B
from eagle_speculative_decoding_tree_gb300 import synth
from gpu_helpers import random_tree

pytestmark = pytest.mark.gpu


def _inputs(M, h, V, seed):
    g = np.random.default_rng(seed)
    H = synth.bf16_bits(g.normal(0, 1, (M, h)).astype(np.float32))
    W = synth.bf16_bits(g.normal(0, 1 / np.sqrt(h), (V, h)).astype(np.float32))
    return H, W


def _run(H, W, R, T, tokens=None, parent=None):
    M, h = H.shape
    V = W.shape[0]
    desc = B.LmHeadDesc(M, R, h, V, T)
    C = -(-V // B.EAGLE_LMHEAD_TILE)
    rec = torch.zeros(M, C, 4, dtype=torch.int32, device="cuda")
    child = torch.full((M,), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dv = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)
    i32 = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()
    B.eagle_lmhead_stats(desc, dv(H), dv(W), i32(tokens), i32(parent), rec, child if tokens is not None else None,
                         status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    r = rec.cpu().numpy()
    return dict(max=r[..., 0].view(np.float32), argmax=r[..., 1], sum=r[..., 2].view(np.float32).astype(np.float64)
                + r[..., 3].view(np.float32).astype(np.float64), child=child.cpu().numpy())


def _compare(got, ref, rows, label, T=1.0):
    tile = B.EAGLE_LMHEAD_TILE
    x = ref["logits"]
    assert np.abs(got["max"][rows] - ref["max"]).max() < 1e-4
    rel = np.abs(got["sum"][rows] - ref["sum"]) / ref["sum"]
    assert rel.max() < np.expm1(2e-4 / (T if T > 0 else 1.0)), rel.max()
    near = 0
    for i, r in enumerate(rows):
        for c in range(ref["max"].shape[1]):
            blk = np.sort(x[i, c * tile:(c + 1) * tile])
            if blk.size > 1 and blk[-1] - blk[-2] < 1e-4:
                near += 1
                continue
            assert got["argmax"][r, c] == ref["argmax"][i, c], (r, c)
    record_near_ties(label, near, len(rows) * ref["max"].shape[1])
    assert near <= max(1, len(rows) * ref["max"].shape[1] // 1000)


@pytest.mark.parametrize("M,R,V,T", [(61, 61, 8192 + 77, 1.0), (128, 64, 1000, 0.7), (8, 8, 130, 0.0)])
def test_lmhead_stats_small(M, R, V, T):
    h = 4096 if M > 8 else 64
    H, W = _inputs(M, h, V, seed=M + V)
    Bn = M // R
    par = np.stack([random_tree(R, seed=31 + b)[0] for b in range(Bn)])
    g = np.random.default_rng(5)
    tok = g.integers(0, V, (Bn, R)).astype(np.int32)
    got = _run(H, W, R, T, tok, par)
    ref = oracle.lmhead_stats(H, W, T, B.EAGLE_LMHEAD_TILE, tok, par)
    _compare(got, ref, np.arange(M), f"lmhead M={M} V={V}", T)
    want = ref["child"].reshape(-1)
    ok = ~np.isnan(want)
    assert np.abs(got["child"][ok] - want[ok]).max() < 1e-4
    assert np.isnan(got["child"][~ok]).all()  # roots untouched


def test_lmhead_stats_full_vocabulary():
    """The LLaMA-3.1-8B shape: hidden 4096, vocabulary 128256, 61 tree rows and a second
    request's 61; sampled rows against the oracle."""
    M, R, h, V = 122, 61, 4096, 128256
    H, W = _inputs(M, h, V, seed=7)
    par = np.stack([random_tree(R, seed=41 + b)[0] for b in range(2)])
    tok = np.random.default_rng(6).integers(0, V, (2, R)).astype(np.int32)
    got = _run(H, W, R, 1.0, tok, par)
    rows = np.array([0, 1, 17, 60, 61, 90, 121])
    ref = oracle.lmhead_stats(H[rows], W, 1.0, B.EAGLE_LMHEAD_TILE)
    _compare(got, ref, rows, "lmhead full vocabulary")
    # children whose parent is a sampled row
    x = ref["logits"]
    where = {int(r): i for i, r in enumerate(rows)}
    checked = 0
    for b in range(2):
        for i in range(1, R):
            pr = b * R + int(par[b, i])
            if pr in where:
                assert abs(got["child"][b * R + i] - x[where[pr], tok[b, i]]) < 1e-4
                checked += 1
    assert checked > 0
