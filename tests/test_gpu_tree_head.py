"""GPU parity: eagle_tree_build_head (the draft LM head fused with tree expansion)
against the oracle's tree construction on the oracle's logits.

At every level both sides receive the same frontier hidden states (bf16) and the same
head (bf16): the oracle forms the logits in float64 (lmhead_logits, rounded to fp32) and
builds the level from them; the GPU reduces its tensor-core logits (fp32 accumulation)
to the rows' statistics and top lists without writing them.  Frontier tokens and parent
slots, then the final tree (tokens, parents, depths, position ids, ancestor masks), must
agree bit for bit; scores within 1e-4.  Besides the selection near-ties both sides flag
(scores within 1e-5), a request is excluded from the level on when one of its rows has
its last kept and first dropped logits within 1e-4: the two sides' logits differ by the
accumulation order (about 1e-6 here), so such a row's top list is not determined.
"""
import numpy as np
import pytest
import torch

import oracle
from conftest import near_tie_cap, record_near_ties
from eagle_speculative_decoding_tree_gb300 import synth
from eagle_speculative_decoding_tree_gb300.step import GpuTreeBuilder
from spec_helpers import OracleDynamicBuilder, OracleStaticBuilder

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS


def _bits(a):
    return synth.bf16_bits(np.asarray(a, np.float32))


def _kept_per_row(w, level, F):
    """Tokens each frontier row contributes at this level: k (dynamic) or the node's
    children (static top-k)."""
    if w.tree_mode == "dynamic":
        return np.full(F, w.top_k)
    par = synth.static_parents(w.static_choices)
    dep = np.zeros(len(par), np.int32)
    for i in range(1, len(par)):
        dep[i] = dep[par[i]] + 1
    nodes = np.nonzero(dep == level - 1)[0]
    return np.array([(par == n).sum() for n in nodes])


def build_head_both(w, batch, h, seed, label, logits_levels=()):
    g = np.random.default_rng(seed)
    V = w.vocab
    Wb = _bits(g.normal(0, 1 / np.sqrt(h), (V, h)))
    Wd = torch.from_numpy(Wb.view(np.int16)).cuda().view(torch.bfloat16)
    root_tok = g.integers(0, V, batch).astype(np.int32)
    seq_len = synth.prefix_lengths(w, batch)
    gpu = GpuTreeBuilder(w, batch)
    gpu.set_context(root_tok, seq_len)
    if w.tree_mode == "dynamic":
        ora = OracleDynamicBuilder(batch, V, w.depth, w.top_k, w.total_tokens)
    else:
        ora = OracleStaticBuilder(batch, V, synth.static_parents(w.static_choices), False, 1.0)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    excluded = np.zeros(batch, bool)
    gap = np.zeros(batch, bool)  # undetermined top lists (from the oracle's logits alone)
    F = 1
    for level in range(1, gpu.depth + 1):
        H = _bits(g.normal(0, 1, (batch, F, h)))
        lo = oracle.lmhead_logits(H.reshape(-1, h), Wb).reshape(batch, F, V)
        kept = _kept_per_row(w, level, F)
        srt = -np.sort(-lo, axis=2)
        for f in range(F):
            kf = int(kept[f])
            if 0 < kf < V:
                gap |= (srt[:, f, kf - 1] - srt[:, f, kf]) < 1e-4
        excluded |= gap
        if level in logits_levels:  # this level from the logits themselves (fp32 rows)
            lg = lo.astype(np.float32)
            gt, gs = gpu.expand(level, lg)
            ot, os_ = ora.expand(level, lg)
        else:
            gt, gs = gpu.expand_head(level, H, Wd, status)
            ot, os_ = ora.expand(level, lo.astype(np.float32))
        excluded |= ora.t.near_tie > 0
        for b in np.nonzero(~excluded)[0]:
            assert np.array_equal(gt[b], ot[b]), (level, b, gt[b], ot[b])
            assert np.array_equal(gs[b], os_[b]), (level, b, gs[b], os_[b])
        F = ot.shape[1]
    torch.cuda.synchronize()
    assert int(status.item()) == 0, "a bounded wait of the head kernel gave up"
    tg = gpu.finalize(root_tok, seq_len)
    to = ora.finalize(root_tok, seq_len)
    excluded |= (to["near_tie"] > 0) | (tg["near_tie"] > 0)
    for b in np.nonzero(~excluded)[0]:
        for key in ("tokens", "parent", "depth", "pos_id", "anc_mask"):
            assert np.array_equal(tg[key][b], to[key][b]), (key, b)
        np.testing.assert_allclose(tg["score"][b], to["score"][b], atol=1e-4, rtol=1e-5)
    record_near_ties(label, excluded.sum(), batch)
    # selection boundaries within 1e-5: about 1e-4 per level
    flagged = excluded & ~gap
    assert flagged.sum() <= near_tie_cap(batch, 2e-4 * gpu.depth), f"{flagged.sum()} of {batch} flagged"
    assert excluded.sum() < batch, "no request was compared"


def test_tree_head_small_dynamic():
    w = W["vicuna7b"].with_(vocab=5000, top_k=4, depth=3, total_tokens=12)
    build_head_both(w, 8, 128, seed=11, label="tree from head V=5000 h=128")


def test_tree_head_static_topk():
    w = W["tiny"].with_(tree_mode="static_topk", dtype="bf16", vocab=3000, temperature=0.0)
    build_head_both(w, 4, 64, seed=12, label="tree from head static top-k")


def test_tree_head_ragged_vocab_and_batch():
    # a vocabulary that is not a multiple of the 128-token tile, fewer tiles than records
    w = W["vicuna7b"].with_(vocab=9001, top_k=8, depth=4, total_tokens=30)
    build_head_both(w, 16, 192, seed=13, label="tree from head V=9001 B=16")


def test_tree_head_llama8b_draft_shape():
    """A LLaMA-3.1-8B-shaped draft head (vocab 128256, hidden 4096) over the llama8b
    workload's dynamic tree (depth 7, top-8, 60 drafts)."""
    build_head_both(W["llama8b"], 1, 4096, seed=14, label="tree from head llama8b")


def test_tree_levels_from_logits_and_from_the_head_mix():
    """Level 1 from the logits (eagle_tree_build), the later levels from hidden states
    (eagle_tree_build_head) in the same workspace."""
    w = W["vicuna7b"].with_(vocab=7000, top_k=6, depth=4, total_tokens=20, dtype="f32")
    build_head_both(w, 8, 128, seed=15, label="tree from logits then head", logits_levels=(1,))
