"""Test helpers: drive whole speculative steps through the oracle on synthetic LMs.

Used by the oracle pins (losslessness, greedy equivalence) and by the GPU parity
tests as the expected side.  Nothing here is method arithmetic beyond calling the
oracle's stages in the order of the pages' data path (draft levels, verify, accept,
commit: EAGLE review, "GPU / system data path" steps 4-7).
"""
import numpy as np
from scipy import stats

import oracle
from eagle_speculative_decoding_tree_gb300 import synth


def build_tree_bigram(lm: synth.BigramLM, roots: np.ndarray, mode: str, *, depth=3, top_k=4, total_tokens=10,
                      static_parent=None, temperature=1.0, u_draft=None):
    """Build one draft tree per request with the bigram LM's draft rows (row = draft[last token])."""
    B = len(roots)
    if mode == "dynamic":
        t = oracle.DynamicTree(B, lm.vocab, depth, top_k, total_tokens)
        toks = roots[:, None]
        for _ in range(depth):
            t.expand(lm.draft[toks])
            toks = t.frontier_tokens()
        return t.finalize(roots, np.zeros(B, np.int32))
    t = oracle.StaticTree(B, lm.vocab, static_parent, mode == "static_sampled", temperature)
    toks = np.zeros((B, t.R), np.int32)
    toks[:, 0] = roots
    for level in range(1, int(t.depths.max()) + 1):
        nodes = t.frontier_nodes(level)
        t.expand(lm.draft[toks[:, nodes]], u_draft)
        toks = t.tokens.copy()
        toks[:, 0] = roots
    return t.finalize(roots, np.zeros(B, np.int32))


def spec_step_bigram(lm, roots, mode, proposal, temperature, gen, **tree_kw):
    """One speculative step per request; returns (tree, accept result)."""
    B = len(roots)
    R_guess = None
    ud = None
    if mode == "static_sampled":
        R_guess = len(tree_kw["static_parent"])
        ud = synth.uniforms(gen, (B, R_guess))
    tree = build_tree_bigram(lm, roots, mode, temperature=temperature, u_draft=ud, **tree_kw)
    R = tree["tokens"].shape[1]
    ua = synth.uniforms(gen, (B, R))
    uf = synth.uniforms(gen, (B,))
    tgt = lm.target[tree["tokens"]]
    dft = lm.draft[tree["tokens"]] if proposal == oracle.SAMPLED else None
    max_path = int(tree["depth"].max()) + 1
    res = oracle.accept(tgt, tree["tokens"], tree["parent"], ua, uf, temperature, proposal, max_path, draft=dft)
    return tree, res


def first_two_tokens(lm, root, mode, proposal, temperature, trials, seed, chunk=50000, **tree_kw):
    """Emit the first two tokens after `root` for many independent trials.

    When a step emits only one token (n_acc == 0), a second step is run from it.
    """
    t1 = np.empty(trials, np.int64)
    t2 = np.empty(trials, np.int64)
    done = 0
    c = 0
    while done < trials:
        n = min(chunk, trials - done)
        gen = synth.rng(0, 7000 + seed, c)
        roots = np.full(n, root, np.int32)
        _, res = spec_step_bigram(lm, roots, mode, proposal, temperature, gen, **tree_kw)
        a = res["out_tok"][:, 0].astype(np.int64)
        b = res["out_tok"][:, 1].astype(np.int64)
        need = res["n_acc"] == 0
        if need.any():
            _, res2 = spec_step_bigram(lm, a[need].astype(np.int32), mode, proposal, temperature, gen, **tree_kw)
            b[need] = res2["out_tok"][:, 0]
        t1[done:done + n] = a
        t2[done:done + n] = b
        done += n
        c += 1
    return t1, t2


def chisquare_pvalue(counts: np.ndarray, probs: np.ndarray, min_expected: float = 5.0) -> float:
    """Pearson chi-square p-value, bins with expected count < min_expected merged into one."""
    counts = np.asarray(counts, np.float64).ravel()
    probs = np.asarray(probs, np.float64).ravel()
    n = counts.sum()
    exp = probs * n
    small = exp < min_expected
    obs_b = np.concatenate([counts[~small], [counts[small].sum()]]) if small.any() else counts
    exp_b = np.concatenate([exp[~small], [exp[small].sum()]]) if small.any() else exp
    keep = exp_b > 0
    assert obs_b[~keep].sum() == 0, "tokens emitted where the target has no mass"
    return float(stats.chisquare(obs_b[keep], exp_b[keep] * obs_b[keep].sum() / exp_b[keep].sum()).pvalue)


def softmax64(x, T=1.0):
    x = np.asarray(x, np.float64) / T
    e = np.exp(x - x.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


# ----------------------------------------------------------------------------- hash-LM drivers
class OracleDynamicBuilder:
    def __init__(self, B, V, depth, top_k, total_tokens):
        self.t = oracle.DynamicTree(B, V, depth, top_k, total_tokens)
        self.prev = None

    def expand(self, level, logits, u_draft=None):
        fr = self.t.expand(logits)
        slot = self.t.frontier_parent_slot(self.prev)
        self.prev = fr
        return self.t.frontier_tokens(), slot

    def finalize(self, root_tok, seq_len):
        return self.t.finalize(root_tok, seq_len)


class OracleStaticBuilder:
    def __init__(self, B, V, static_parent, sampled, temperature):
        self.t = oracle.StaticTree(B, V, static_parent, sampled, temperature)

    def expand(self, level, logits, u_draft=None):
        self.t.expand(logits, u_draft)
        nodes = self.t.frontier_nodes(level + 1)
        prev_nodes = list(self.t.frontier_nodes(level))
        slot = np.array([prev_nodes.index(self.t.parent[n]) for n in nodes], np.int32)
        B = self.t.B
        return self.t.tokens[:, nodes].copy(), np.broadcast_to(slot, (B, len(nodes))).copy()

    def finalize(self, root_tok, seq_len):
        return self.t.finalize(root_tok, seq_len)


def node_hashes(tree, root_hash):
    """Path hash of every tree node (row order), from the root hash and the tokens."""
    B, R = tree["tokens"].shape
    out = np.zeros((B, R), np.uint64)
    hs = [[0] * R for _ in range(B)]
    for b in range(B):
        hs[b][0] = int(root_hash[b])
        for i in range(1, R):
            hs[b][i] = synth.child_hash(hs[b][tree["parent"][b, i]], int(tree["tokens"][b, i]))
        out[b] = np.array(hs[b], dtype=np.uint64)
    return hs


def drive_tree_build(builder, lm: synth.HashLM, depth, root_tok, root_hash, seq_len, u_draft=None, record=None):
    """Run the level-by-level tree build, feeding each level the draft rows of the
    current frontier (keyed by path hash).  Returns the finalized tree."""
    B = len(root_tok)
    front = [[int(h)] for h in root_hash]
    for level in range(1, depth + 1):
        logits = np.stack([lm.rows(front[b], "draft") for b in range(B)])
        logits = synth.as_dtype_bytes(logits, lm.dtype)
        ftok, fslot = builder.expand(level, logits, u_draft)
        if record is not None:
            record.append((logits, ftok.copy(), fslot.copy()))
        front = [[synth.child_hash(front[b][int(fslot[b, j])], int(ftok[b, j])) for j in range(ftok.shape[1])]
                 for b in range(B)]
    return builder.finalize(root_tok, seq_len)
