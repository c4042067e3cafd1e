"""GPU parity: eagle_accept against the oracle's acceptance.

Trees come from the oracle's builder on the synthetic path-keyed LM; target (and
draft) rows are that LM's rows at the tree's nodes; uniforms are seeded.  The GPU
must reproduce the oracle's accepted lengths, paths and emitted tokens bit for
bit, except for requests where either side reports a near-tie (|u - p/q| < 1e-5,
or a draw within 1e-7 of the mass of a bin edge), which are counted, reported in
the test summary and capped near their expected rate (about 2e-5 per accept
decision, and up to a few percent per draw at 128K tokens).  A GPU-side chi-square
check repeats the losslessness test on the kernels themselves.
"""
import numpy as np
import pytest
import torch
from scipy.special import softmax

import oracle
from eagle_speculative_decoding_tree_gb300 import binding as B
from eagle_speculative_decoding_tree_gb300 import synth
from conftest import draw_rate, draw_rate_of, near_tie_cap, record_near_ties
from gpu_helpers import dev
from spec_helpers import OracleDynamicBuilder, OracleStaticBuilder, build_tree_bigram, chisquare_pvalue, \
    drive_tree_build, node_hashes

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS


def gpu_accept(w, tree, target, draft, ua, uf, proposal, T, max_depth):
    Bn, R = tree["tokens"].shape
    dt = B.EAGLE_F32 if w.dtype == "f32" else B.EAGLE_BF16
    desc = B.AcceptDesc(Bn, R, target.shape[-1], float(T), proposal, dt, max_depth)
    ws = torch.zeros(B.workspace_size(B.EAGLE_WS_ACCEPT, desc), dtype=torch.uint8, device="cuda")
    out = B.AcceptBuffers.allocate(Bn, max_depth)
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()
    B.eagle_accept(desc, dev(target, w.dtype), None if draft is None else dev(draft, w.dtype), i32(tree["tokens"]),
                   i32(tree["parent"]), torch.from_numpy(ua).cuda(), torch.from_numpy(uf).cuda(), out, ws)
    torch.cuda.synchronize()
    return {k: getattr(out, k).cpu().numpy() for k in ("n_acc", "path", "out_tok", "near_tie", "status")}


def accept_cap(n, V, target=None, dtype="bf16", T=1.0):
    """Near-tie cap for n requests over V tokens: one final draw each (its rate taken
    from the target rows when given, else the bound for V tokens) and up to eight
    accept decisions at 2e-5."""
    rate = draw_rate(V)
    if target is not None and T > 0:
        vals = synth.bf16_value(target[:16]) if dtype == "bf16" else np.asarray(target[:16], np.float32)
        rate = draw_rate_of(vals, T)
    return near_tie_cap(n, rate + 8 * 2e-5)


def compare(g, r, max_near, label="accept"):
    near = (g["near_tie"] > 0) | (r["near_tie"] > 0)
    record_near_ties(label, near.sum(), len(near))
    assert near.sum() < len(near), "no request was compared"
    ok = ~near
    for key in ("n_acc", "path", "out_tok"):
        bad = np.nonzero(ok & np.any(np.atleast_2d(g[key].reshape(len(near), -1) != r[key].reshape(len(near), -1)),
                                     axis=1))[0]
        assert len(bad) == 0, f"{key} differs for requests {bad[:8]}: gpu {g[key][bad[:2]]} oracle {r[key][bad[:2]]}"
    assert g["status"][0] == 0
    assert near.sum() <= max_near, near.sum()
    return int(near.sum())


def case(w, batch, seed, T=None, proposal=None):
    T = w.temperature if T is None else T
    proposal = proposal if proposal is not None else (oracle.SAMPLED if w.proposal == "sampled" else oracle.DELTA)
    lm = synth.hash_lm(w)
    root_tok = synth.rng(w.config_id, 41, seed).integers(0, w.vocab, batch).astype(np.int32)
    root_h = [synth.root_hash(w.config_id, b, 100 + seed) for b in range(batch)]
    seq_len = synth.prefix_lengths(w, batch)
    if w.tree_mode == "dynamic":
        bld = OracleDynamicBuilder(batch, w.vocab, w.depth, w.top_k, w.total_tokens)
        depth = w.depth
    else:
        par = synth.static_parents(w.static_choices)
        bld = OracleStaticBuilder(batch, w.vocab, par, w.tree_mode == "static_sampled", T if T > 0 else 1.0)
        depth = int(max(len(c) for c in w.static_choices))
    ud = synth.uniforms(synth.rng(w.config_id, 42, seed), (batch, w.rows))
    tree = drive_tree_build(bld, lm, depth, root_tok, root_h, seq_len, u_draft=ud)
    hs = node_hashes(tree, root_h)
    target = synth.as_dtype_bytes(np.stack([lm.rows(hs[b], "target") for b in range(batch)]), w.dtype)
    draft = synth.as_dtype_bytes(np.stack([lm.rows(hs[b], "draft") for b in range(batch)]), w.dtype) \
        if proposal == oracle.SAMPLED else None
    ua = synth.uniforms(synth.rng(w.config_id, 43, seed), (batch, tree["tokens"].shape[1]))
    uf = synth.uniforms(synth.rng(w.config_id, 44, seed), (batch,))
    max_depth = int(tree["depth"].max())
    r = oracle.accept(target, tree["tokens"], tree["parent"], ua, uf, T, proposal, max_depth + 1, draft=draft)
    g = gpu_accept(w, tree, target, draft, ua, uf, proposal, T, max_depth)
    g["_target"] = target
    return g, r


@pytest.mark.parametrize("name,batch,T", [
    ("vicuna7b", 8, 0.0), ("vicuna7b", 8, 1.0), ("llama8b", 8, 1.0), ("tiny", 64, 1.0), ("long128k", 8, 1.0),
])
def test_accept_workloads(name, batch, T):
    g, r = case(W[name], batch, seed=1, T=T)
    compare(g, r, max_near=accept_cap(batch, W[name].vocab, g["_target"], W[name].dtype, T),
            label=f"accept {name} T={T} B={batch}")


def test_accept_concurrency_batch32():
    """The concurrency workload's full shape: 32 requests, vocab 128256, 61-row trees."""
    w = W["concurrency"].with_(batch=32)
    g, r = case(w, 32, seed=2)
    compare(g, r, max_near=accept_cap(32, w.vocab, g["_target"], w.dtype, w.temperature), label="accept concurrency B=32")


def test_accept_temperature_07_delta():
    w = W["vicuna7b"].with_(vocab=5000, temperature=0.7)
    g, r = case(w, 32, seed=3)
    compare(g, r, max_near=accept_cap(32, w.vocab, g["_target"], w.dtype, 0.7), label="accept T=0.7 delta B=32")


def test_accept_sampled_static_multi_sibling_residuals():
    w = W["tiny"].with_(vocab=5000, dtype="bf16", temperature=0.8, draft_sigma=2.0)
    g, r = case(w, 64, seed=4)
    compare(g, r, max_near=accept_cap(64, w.vocab), label="accept sampled multi-sibling B=64")
    assert (r["n_acc"] < 3).sum() > 10  # rejections (and residual passes) happened


def test_accept_delta_with_duplicate_siblings():
    # children drawn with replacement, judged as point-mass proposals: a duplicate of a
    # rejected token has zero residual mass and must be rejected too
    w = W["tiny"].with_(vocab=40, dtype="f32", temperature=1.0, sigma=1.0)
    g, r = case(w, 128, seed=5, proposal=oracle.DELTA)
    compare(g, r, max_near=accept_cap(128, w.vocab), label="accept duplicate siblings B=128")


def test_accept_gpu_chisquare_first_token():
    """Losslessness on the GPU: 2e5 independent requests in one call, first emitted
    token against the target distribution (dynamic top-k tree, point-mass proposals)."""
    V, n = 16, 200_000
    lm = synth.BigramLM(V, sigma=1.5, draft_sigma=0.7, seed_key=1)
    root = 3
    tree = build_tree_bigram(lm, np.array([root], np.int32), "dynamic", depth=3, top_k=4, total_tokens=10)
    tree = {k: np.broadcast_to(v, (n,) + v.shape[1:]).copy() for k, v in tree.items()}
    target = lm.target[tree["tokens"]]
    g = synth.rng(0, 7777)
    ua, uf = synth.uniforms(g, (n, 11)), synth.uniforms(g, (n,))
    w = synth.WORKLOADS["tiny"]
    out = gpu_accept(w, tree, target, None, ua, uf, oracle.DELTA, 1.0, int(tree["depth"].max()))
    c1 = np.bincount(out["out_tok"][:, 0], minlength=V)
    p = softmax(lm.target[root].astype(np.float64))
    assert chisquare_pvalue(c1, p) > 1e-3


def test_accept_gpu_chisquare_sampled_static():
    V, n = 16, 100_000
    lm = synth.BigramLM(V, sigma=1.5, draft_sigma=0.7, seed_key=1)
    g = synth.rng(0, 7778)
    par = synth.static_parents(synth.TINY_STATIC_CHOICES)
    tree = build_tree_bigram(lm, np.full(n, 3, np.int32), "static_sampled", static_parent=par,
                             u_draft=synth.uniforms(g, (n, 11)))
    target, draft = lm.target[tree["tokens"]], lm.draft[tree["tokens"]]
    ua, uf = synth.uniforms(g, (n, 11)), synth.uniforms(g, (n,))
    out = gpu_accept(synth.WORKLOADS["tiny"], tree, target, draft, ua, uf, oracle.SAMPLED, 1.0, 3)
    c1 = np.bincount(out["out_tok"][:, 0], minlength=V)
    p = softmax(lm.target[3].astype(np.float64))
    assert chisquare_pvalue(c1, p) > 1e-3
    r = oracle.accept(target[:2000], tree["tokens"][:2000], tree["parent"][:2000], ua[:2000], uf[:2000], 1.0,
                      oracle.SAMPLED, 4, draft=draft[:2000])
    compare({k: v[:2000] if k != "status" else v for k, v in out.items()}, r, max_near=accept_cap(2000, V),
            label="accept sampled static (chi-square run) B=2000")


def test_accept_bad_token_is_flagged_and_rejected():
    w = W["tiny"].with_(vocab=50, dtype="f32")
    tree = {"tokens": np.array([[1, 60, 3]], np.int32), "parent": np.array([[-1, 0, 0]], np.int32)}
    target = np.zeros((1, 3, 50), np.float32)
    target[0, 0, 3] = 10.0
    g = gpu_accept(w, tree, target, None, np.zeros((1, 3), np.float32), np.zeros(1, np.float32), oracle.DELTA, 1.0, 1)
    assert g["status"][0] & B.EAGLE_STATUS_BAD_TOKEN
    assert g["n_acc"][0] == 1 and g["out_tok"][0, 0] == 3


@pytest.mark.parametrize("proposal", [oracle.DELTA, oracle.SAMPLED])
def test_accept_agreement_many_requests_128k(proposal):
    """Many requests over a 128K vocabulary: outside the requests either side reports as
    near-ties, the GPU and the oracle never disagree; near-ties stay rare."""
    from gpu_helpers import random_tree
    Bn, R, V, n_rows = 128, 12, 128256, 24
    g = synth.rng(0, 7900, proposal)
    pool_t = np.stack([synth.zipf_row(g, V) for _ in range(n_rows)])
    pool_d = (pool_t + synth.normal_row(g, pool_t.shape, 0.5)).astype(np.float32)
    which = g.integers(0, n_rows, (Bn, R))
    target = synth.bf16_bits(pool_t[which])
    draft = synth.bf16_bits(pool_d[which]) if proposal == oracle.SAMPLED else None
    tokens = np.zeros((Bn, R), np.int32)
    parent = np.zeros((Bn, R), np.int32)
    for b in range(Bn):
        par, _ = random_tree(R, seed=1000 + b)
        parent[b] = par
        for i in range(1, R):  # one of the parent row's three most likely tokens
            tokens[b, i] = np.argsort(-pool_d[which[b, par[i]]])[g.integers(0, 3)]
    ua, uf = synth.uniforms(g, (Bn, R)), synth.uniforms(g, (Bn,))
    max_depth = R - 1
    tree = {"tokens": tokens, "parent": parent}
    w = W["llama8b"]
    r = oracle.accept(target, tokens, parent, ua, uf, 1.0, proposal, max_depth + 1, draft=draft)
    out = gpu_accept(w, tree, target, draft, ua, uf, proposal, 1.0, max_depth)
    # each draw lands within 1e-7 of the mass of a bin edge with probability about
    # sum min(p, 2e-7) = 2.6% over a Zipf(1.1) row of 128256 tokens: ~3 of 128 expected
    near = compare(out, r, max_near=accept_cap(Bn, V, target, "bf16", 1.0),
                   label=f"accept 128K agreement proposal={proposal} B={Bn}")
    assert (r["n_acc"] > 0).sum() > Bn // 10
    print(f"near-ties: {near} of {Bn}")
