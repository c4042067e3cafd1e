"""GPU parity: eagle_tree_build against the oracle's tree construction.

Both builders receive the same draft rows at every level (rows of the synthetic
path-keyed LM at the oracle's frontier), and must agree bit for bit on each
level's frontier tokens and parent slots and on the final tree (tokens, parents,
depths, position ids, ancestor masks).  A request whose selection boundary or
draw landed near a tie (selection scores within 1e-5, a draw within 1e-7 of the
mass of a bin edge; reported by either side) is excluded from the
comparison from that level on and counted; the counts are reported in the test
summary and capped near their expected rates: a selection boundary within 1e-5 is
rare at these vocabulary sizes, while a draw's chance of landing within 1e-7 of the
mass of a bin edge is about the sum over tokens of min(p, 2e-7), up to a few percent
per draw at 128K tokens.  Cumulative scores agree within 1e-4.
"""
import numpy as np
import pytest

from conftest import draw_rate_of, near_tie_cap, record_near_ties
from eagle_speculative_decoding_tree_gb300 import synth
from eagle_speculative_decoding_tree_gb300.step import GpuTreeBuilder
from spec_helpers import OracleDynamicBuilder, OracleStaticBuilder

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS


class RoundedLM(synth.HashLM):
    """Rows rounded to integers: many exact ties inside a row."""

    def draft_row(self, h):
        return np.round(super().draft_row(h)).astype(np.float32)


def build_both(w, batch, seed, lm=None, max_excluded=None, label=None):
    lm = lm or synth.hash_lm(w)
    root_tok = synth.rng(w.config_id, 31, seed).integers(0, w.vocab, batch).astype(np.int32)
    root_h = [synth.root_hash(w.config_id, b, seed) for b in range(batch)]
    seq_len = synth.prefix_lengths(w, batch)
    gpu = GpuTreeBuilder(w, batch)
    gpu.set_context(root_tok, seq_len)
    if w.tree_mode == "dynamic":
        ora = OracleDynamicBuilder(batch, w.vocab, w.depth, w.top_k, w.total_tokens)
    else:
        ora = OracleStaticBuilder(batch, w.vocab, synth.static_parents(w.static_choices),
                                  w.tree_mode == "static_sampled", w.temperature)
    ud = synth.uniforms(synth.rng(w.config_id, 32, seed), (batch, w.rows)) \
        if w.tree_mode == "static_sampled" else None
    excluded = np.zeros(batch, bool)
    front = [[h] for h in root_h]
    draw_rows = None
    for level in range(1, gpu.depth + 1):
        rows = synth.as_dtype_bytes(np.stack([lm.rows(front[b], "draft") for b in range(batch)]), w.dtype)
        if draw_rows is None:
            draw_rows = synth.bf16_value(rows[:4, :1]) if w.dtype == "bf16" else np.asarray(rows[:4, :1], np.float32)
        gt, gs = gpu.expand(level, rows, ud)
        ot, os_ = ora.expand(level, rows, ud)
        excluded |= ora.t.near_tie > 0
        for b in np.nonzero(~excluded)[0]:
            assert np.array_equal(gt[b], ot[b]), (level, b, gt[b], ot[b])
            assert np.array_equal(gs[b], os_[b]), (level, b, gs[b], os_[b])
        front = [[synth.child_hash(front[b][int(os_[b, j])], int(ot[b, j])) for j in range(ot.shape[1])]
                 for b in range(batch)]
    tg = gpu.finalize(root_tok, seq_len)
    to = ora.finalize(root_tok, seq_len)
    excluded |= (to["near_tie"] > 0) | (tg["near_tie"] > 0)
    for b in np.nonzero(~excluded)[0]:
        for key in ("tokens", "parent", "depth", "pos_id", "anc_mask"):
            assert np.array_equal(tg[key][b], to[key][b]), (key, b)
        np.testing.assert_allclose(tg["score"][b], to["score"][b], atol=1e-4, rtol=1e-5)
    record_near_ties(label or f"tree build {w.name} B={batch}", excluded.sum(), batch)
    # selection boundaries: ~1e-4 per level; sampled trees: one draw per node, at the
    # rate of the draft rows' distributions
    draws = (w.rows - 1) if w.tree_mode == "static_sampled" else 0
    rate = draw_rate_of(draw_rows, w.temperature, draws) if draws else 0.0
    limit = max_excluded if max_excluded is not None else near_tie_cap(batch, rate + 1e-4 * max(1, gpu.depth))
    assert excluded.sum() <= limit, f"{excluded.sum()} of {batch} requests hit near-ties"
    assert excluded.sum() < batch, "no request was compared"
    return int(excluded.sum())


@pytest.mark.parametrize("name,batch", [("vicuna7b", 4), ("llama8b", 2), ("tiny", 16), ("long128k", 16)])
def test_tree_build_workloads(name, batch):
    build_both(W[name], batch, seed=1)


@pytest.mark.parametrize("batch", [8, 32])
def test_tree_build_concurrency(batch):
    """The concurrency workload's full shape (vocab 128256, dynamic trees of 60 drafts,
    depth 6, top-8) at batch 8 and 32."""
    build_both(W["concurrency"].with_(batch=batch), batch, seed=2)


def test_static_topk_tree():
    w = W["tiny"].with_(tree_mode="static_topk", dtype="bf16", vocab=5000, temperature=0.0)
    build_both(w, 4, seed=3)


def test_small_vocab_fewer_tokens_than_list_slots():
    w = W["vicuna7b"].with_(vocab=10, top_k=4, depth=3, total_tokens=12, dtype="f32")
    build_both(w, 8, seed=4)


def test_many_exact_ties():
    """Rows rounded to integers: many exact ties inside a row, broken by token id on
    both sides.  Ties across parents can put two scores within 1e-5 at the selection
    boundary (flagged), so at most half of the 16 requests may drop out."""
    w = W["vicuna7b"].with_(vocab=3000, top_k=6, depth=3, total_tokens=24)
    lm = RoundedLM(w.vocab, "normal", 3.0, 0.7, "bf16")
    build_both(w, 16, seed=5, lm=lm, max_excluded=8)


def test_dynamic_tree_whole_pool_and_max_rows():
    # N = pool size (every candidate kept), and the largest tree (127 drafts, two mask words)
    w = W["vicuna7b"].with_(vocab=2000, top_k=3, depth=4, total_tokens=3 + 3 * 9)
    build_both(w, 3, seed=6)
    w2 = W["vicuna7b"].with_(vocab=2000, top_k=8, depth=3, total_tokens=127)
    build_both(w2, 2, seed=7)
