"""CPU oracle for the EAGLE draft-tree verify step -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may
import this package.  The CUDA product path never calls it and shares no code with
it; the only thing both sides use is the seeded input generator module.

The heavy stages (tree attention, acceptance, tree construction) are plain float64
C loops in ``eagle_oracle.c``, built with gcc into ``_build/liboracle.so`` on first
use; this module marshals numpy arrays into them.  The KV commit is a plain numpy
copy here.  Page citations are at each function.

Parity pins: every function below is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_*.py`` against brute force, closed forms, library routines and
the pages' worked examples.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "eagle_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lib = None

F32, BF16 = 0, 1
DELTA, SAMPLED = 0, 1


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain -O2, no fast-math, no target flags)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
    return _lib


def _p(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    raise TypeError(f"oracle inputs are float32 or bf16 bits (uint16), got {a.dtype}")


def _c(a, dt):
    return np.ascontiguousarray(a, dtype=dt)


# ---------------------------------------------------------------------------- attention
def tree_attn(q, k_cache, v_cache, tree_k, tree_v, seq_len, parent, scale: float):
    """Tree attention: each node attends to the prefix and to its own ancestors.

    EAGLE review (zenmind), terms "tree attention"; lesson glossary "Tree attention".
    Shapes: q [B][R][Hq][D]; k/v cache [B][Hkv][P_max][D]; tree k/v [B][Hkv][R][D];
    seq_len [B]; parent [B][R] (root -1).  Returns (out [B][R][Hq][D], lse [B][R][Hq])
    in float64.
    """
    lib = _load()
    dt = _dtype_code(q)
    B, R, Hq, D = q.shape
    Hkv, P = k_cache.shape[1], k_cache.shape[2]
    args = [_c(x, q.dtype) for x in (q, k_cache, v_cache, tree_k, tree_v)]
    sl = _c(seq_len, np.int32)
    par = _c(np.broadcast_to(parent, (B, R)), np.int32)
    out = np.zeros((B, R, Hq, D), np.float64)
    lse = np.zeros((B, R, Hq), np.float64)
    fn = lib.oracle_tree_attn
    fn.restype = ctypes.c_int
    rc = fn(B, R, Hq, Hkv, D, P, ctypes.c_double(scale), dt, *[_p(a) for a in args], _p(sl), _p(par),
            _p(out), _p(lse))
    if rc:
        raise ValueError(f"oracle_tree_attn rc={rc}")
    return out, lse


# ---------------------------------------------------------------------------- accept
def accept(target, tokens, parent, u_accept, u_final, temperature: float, proposal: int,
           max_path: int, draft=None, want_ratio: bool = False):
    """Multi-round speculative sampling over a draft tree (greedy when T == 0).

    EAGLE review section 3.3 and appendix A.2 / Algorithm 1; lesson steps 1-2 and
    "bonus token".  target/draft [B][R][V]; tokens/parent [B][R]; u_accept [B][R];
    u_final [B].  Returns a dict with n_acc [B], path [B][max_path],
    out_tok [B][max_path], near_tie [B] and (optionally) ratio [B][R].
    """
    lib = _load()
    dt = _dtype_code(target)
    B, R, V = target.shape
    tgt = _c(target, target.dtype)
    dft = None if draft is None else _c(draft, target.dtype)
    tok = _c(tokens, np.int32)
    par = _c(np.broadcast_to(parent, (B, R)), np.int32)
    ua = _c(u_accept, np.float32)
    uf = _c(u_final, np.float32)
    n_acc = np.zeros(B, np.int32)
    path = np.zeros((B, max_path), np.int32)
    out_tok = np.zeros((B, max_path), np.int32)
    near = np.zeros(B, np.int32)
    ratio = np.zeros((B, R), np.float64) if want_ratio else None
    fn = lib.oracle_accept
    fn.restype = ctypes.c_int
    rc = fn(B, R, V, dt, ctypes.c_double(temperature), proposal, max_path, _p(tgt), _p(dft), _p(tok),
            _p(par), _p(ua), _p(uf), _p(n_acc), _p(path), _p(out_tok), _p(near), _p(ratio))
    if rc:
        raise ValueError(f"oracle_accept rc={rc}")
    res = dict(n_acc=n_acc, path=path, out_tok=out_tok, near_tie=near)
    if want_ratio:
        res["ratio"] = ratio
    return res


# ---------------------------------------------------------------------------- tree build
class DynamicTree:
    """EAGLE-2 dynamic draft tree, one level per call (see eagle_oracle.c for the reading).

    EAGLE-3 visual reading, "EAGLE-2" (confidence-driven dynamic tree); EAGLE review
    section 3.1 / appendix A.1 (top-k children per frontier node).
    """

    def __init__(self, batch: int, vocab: int, depth: int, top_k: int, total_tokens: int):
        self.B, self.V, self.depth, self.k, self.N = batch, vocab, depth, top_k, total_tokens
        self.cap = top_k + (depth - 1) * top_k * top_k
        self.pool_tok = np.zeros((batch, self.cap), np.int32)
        self.pool_parent = np.zeros((batch, self.cap), np.int32)
        self.pool_score = np.zeros((batch, self.cap), np.float64)
        self.pool_depth = np.zeros((batch, self.cap), np.int32)
        self.n_pool = np.zeros(batch, np.int32)
        self.frontier = np.zeros((batch, top_k), np.int32)
        self.near_tie = np.zeros(batch, np.int32)
        self.level = 0

    def expand(self, logits: np.ndarray) -> np.ndarray:
        """Add one level.  logits [B][F][V] are the draft rows of the current frontier
        (F = 1 at level 1, else k, in frontier order).  Returns the new frontier as
        pool indices [B][k] (pool-index order)."""
        lib = _load()
        self.level += 1
        F = 1 if self.level == 1 else self.k
        assert logits.shape == (self.B, F, self.V), logits.shape
        lg = _c(logits, logits.dtype)
        fn = lib.oracle_tree_level_dynamic
        fn.restype = ctypes.c_int
        rc = fn(self.B, self.V, _dtype_code(lg), self.k, self.level, _p(lg), self.cap, _p(self.pool_tok),
                _p(self.pool_parent), _p(self.pool_score), _p(self.pool_depth), _p(self.n_pool),
                _p(self.frontier), _p(self.near_tie))
        if rc:
            raise ValueError(f"oracle_tree_level_dynamic rc={rc}")
        return self.frontier.copy()

    def frontier_tokens(self) -> np.ndarray:
        return np.take_along_axis(self.pool_tok, self.frontier, axis=1)

    def frontier_parent_slot(self, prev_frontier: Optional[np.ndarray]) -> np.ndarray:
        """For each new frontier node, the slot of its parent in the previous frontier
        (0 at level 1, where the parent is the root)."""
        par = np.take_along_axis(self.pool_parent, self.frontier, axis=1)
        if prev_frontier is None:
            return np.zeros_like(par)
        out = np.zeros_like(par)
        for b in range(self.B):
            slot = {int(p): s for s, p in enumerate(prev_frontier[b])}
            out[b] = [slot[int(p)] for p in par[b]]
        return out

    def finalize(self, root_tok: np.ndarray, seq_len: np.ndarray):
        lib = _load()
        R = self.N + 1
        W = max(1, -(-R // 64))
        out = dict(tokens=np.zeros((self.B, R), np.int32), parent=np.zeros((self.B, R), np.int32),
                   depth=np.zeros((self.B, R), np.int32), pos_id=np.zeros((self.B, R), np.int32),
                   anc_mask=np.zeros((self.B, R, W), np.uint64), score=np.zeros((self.B, R), np.float64))
        fn = lib.oracle_tree_finalize_dynamic
        fn.restype = ctypes.c_int
        rc = fn(self.B, self.N, self.cap, _p(self.pool_tok), _p(self.pool_parent), _p(self.pool_score),
                _p(self.pool_depth), _p(self.n_pool), _p(_c(root_tok, np.int32)), _p(_c(seq_len, np.int32)), W,
                _p(out["tokens"]), _p(out["parent"]), _p(out["depth"]), _p(out["pos_id"]), _p(out["anc_mask"]),
                _p(out["score"]), _p(self.near_tie))
        if rc:
            raise ValueError(f"oracle_tree_finalize_dynamic rc={rc}")
        out["near_tie"] = self.near_tie.copy()
        return out


def static_depths(static_parent: np.ndarray) -> np.ndarray:
    dep = np.zeros(len(static_parent), np.int32)
    for i in range(1, len(static_parent)):
        dep[i] = dep[static_parent[i]] + 1
    return dep


class StaticTree:
    """Static draft tree (EAGLE review appendix A.1): greedy -> top-k children,
    non-greedy -> children drawn from the draft distribution."""

    def __init__(self, batch: int, vocab: int, static_parent: np.ndarray, sampled: bool, temperature: float):
        self.B, self.V = batch, vocab
        self.parent = np.asarray(static_parent, np.int32)
        self.R = len(self.parent)
        self.depths = static_depths(self.parent)
        self.sampled, self.T = sampled, temperature
        self.tokens = np.zeros((batch, self.R), np.int32)
        self.score = np.zeros((batch, self.R), np.float64)
        self.near_tie = np.zeros(batch, np.int32)
        self.level = 0

    def frontier_nodes(self, level: int) -> np.ndarray:
        """Node ids whose draft rows feed level `level` (the depth level-1 nodes)."""
        return np.nonzero(self.depths == level - 1)[0].astype(np.int32)

    def expand(self, logits: np.ndarray, u_draft: Optional[np.ndarray] = None):
        lib = _load()
        self.level += 1
        F = len(self.frontier_nodes(self.level))
        assert logits.shape == (self.B, F, self.V), (logits.shape, F)
        lg = _c(logits, logits.dtype)
        ud = _c(u_draft if u_draft is not None else np.zeros((self.B, self.R), np.float32), np.float32)
        fn = lib.oracle_tree_level_static
        fn.restype = ctypes.c_int
        rc = fn(self.B, self.V, _dtype_code(lg), self.R, _p(self.parent), self.level, int(self.sampled),
                ctypes.c_double(self.T), _p(lg), _p(ud), _p(self.tokens), _p(self.score), _p(self.near_tie))
        if rc:
            raise ValueError(f"oracle_tree_level_static rc={rc}")

    def finalize(self, root_tok: np.ndarray, seq_len: np.ndarray):
        R = self.R
        W = max(1, -(-R // 64))
        tokens = self.tokens.copy()
        tokens[:, 0] = root_tok
        mask = np.zeros((R, W), np.uint64)
        for i in range(R):
            if i > 0:
                mask[i] = mask[self.parent[i]]
            mask[i, i // 64] |= np.uint64(1) << np.uint64(i % 64)
        return dict(tokens=tokens, parent=np.broadcast_to(self.parent, (self.B, R)).copy(),
                    depth=np.broadcast_to(self.depths, (self.B, R)).copy(),
                    pos_id=(np.asarray(seq_len, np.int32)[:, None] + self.depths[None, :]).astype(np.int32),
                    anc_mask=np.broadcast_to(mask, (self.B, R, W)).copy(), score=self.score.copy(),
                    near_tie=self.near_tie.copy())


# ---------------------------------------------------------------------------- commit
def kv_commit(k_cache, v_cache, tree_k, tree_v, n_acc, path, seq_len, feat_cache=None, tree_feat=None):
    """Commit the accepted path: copy path node m's K/V (and feature row) to cache slot
    seq_len + m for m = 0..n_acc, then seq_len += n_acc + 1.

    EAGLE review section 3.3 ("accepted tokens and their features are recorded")
    and data path step 7; lesson "KV cache rollback" and step 4 (KV accounting).
    k/v cache [L][B][Hkv][P][D] (modified in place); tree k/v [L][B][Hkv][R][D];
    feat_cache [B][P][F]; tree_feat [B][R][F].  Returns (new seq_len, commit_pos [B][max_path]).
    """
    B = len(seq_len)
    max_path = path.shape[1]
    new_len = np.array(seq_len, np.int32)
    pos = np.full((B, max_path), -1, np.int32)
    for b in range(B):
        for m in range(int(n_acc[b]) + 1):
            node = int(path[b, m])
            slot = int(seq_len[b]) + m
            k_cache[:, b, :, slot, :] = tree_k[:, b, :, node, :]
            v_cache[:, b, :, slot, :] = tree_v[:, b, :, node, :]
            if feat_cache is not None:
                feat_cache[b, slot, :] = tree_feat[b, node, :]
            pos[b, m] = slot
        new_len[b] = int(seq_len[b]) + int(n_acc[b]) + 1
    return new_len, pos


# ---------------------------------------------------------------------------- LM-head statistics
def lmhead_logits(hidden, weight):
    """The target model's logits at the tree's nodes: hidden [M][h] times the LM head
    W [V][h] transposed, in float64 (inputs float32 or bf16 bits).  EAGLE review, data
    path steps 3 and 6 (the frozen LM head gives the distribution at every node)."""
    def f64(a):
        a = np.asarray(a)
        if a.dtype == np.uint16:
            return (a.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
        return a.astype(np.float64)
    return f64(hidden) @ f64(weight).T


def lmhead_stats(hidden, weight, temperature: float, tile: int, tokens=None, parent=None):
    """What acceptance needs from each node's distribution, from the logits
    x = hidden W^T (EAGLE review, section 3.3 / Algorithm 1: the accept test reads the
    target probability of each child's token, the bonus draw reads the distribution):
    per row and per tile of `tile` vocabulary entries, the max logit, its index (lowest
    on ties) and sum exp((x - max) / T) (T <= 0 counts as 1); and, given the tree
    (tokens, parent [B][R] with rows ordered b * R + node), each node's own token's
    logit under its parent's row (NaN at the roots).  Returns a dict of float64 /
    int64 arrays: max, argmax [M][C], sum [M][C], child [B][R]."""
    x = lmhead_logits(hidden, weight)
    M, V = x.shape
    T = temperature if temperature > 0 else 1.0
    C = -(-V // tile)
    mx = np.full((M, C), -np.inf)
    am = np.zeros((M, C), np.int64)
    sm = np.zeros((M, C))
    for c in range(C):
        blk = x[:, c * tile:(c + 1) * tile]
        mx[:, c] = blk.max(axis=1)
        am[:, c] = c * tile + np.argmax(blk, axis=1)  # first maximum: the lowest index
        sm[:, c] = np.exp((blk - mx[:, c:c + 1]) / T).sum(axis=1)
    out = dict(max=mx, argmax=am, sum=sm, logits=x)
    if tokens is not None:
        Bn, R = np.asarray(tokens).shape
        child = np.full((Bn, R), np.nan)
        for b in range(Bn):
            for i in range(1, R):
                child[b, i] = x[b * R + int(parent[b][i]), int(tokens[b][i])]
        out["child"] = child
    return out


def lmhead_accept(hidden, weight, tokens, parent, u_accept, u_final, temperature: float, proposal: int,
                  max_path: int):
    """Acceptance with the target rows given as hidden states and the LM head: the
    logits at every node (lmhead_logits), then the multi-round rule (accept)."""
    Bn, R = np.asarray(tokens).shape
    x = lmhead_logits(hidden, weight).astype(np.float32).reshape(Bn, R, -1)
    return accept(x, tokens, parent, u_accept, u_final, temperature, proposal, max_path)


# ---------------------------------------------------------------------------- TTT attention
def ttt_attn(q, k_trunk, v_trunk, k_branch, v_branch, scale: float):
    """Attention of EAGLE-3's training-time test (EAGLE-3 visual reading, "训练时的
    Attention Mask 设计"; Didi article sections 5.2-5.3).  TTT step j's prediction at
    position t attends causally to the original sequence (trunk keys t' <= t) and,
    through the diagonal mask, only to its own predecessors in the earlier TTT steps
    at the same position (branch keys (i, t), 1 <= i <= j); the two parts share one
    softmax (the streaming-softmax / LSE fusion of trunk and branch).
    Shapes: q [k][S][Hq][D]; k/v_trunk [Hkv][S][D]; k/v_branch [k][Hkv][S][D] (step 0
    unused); float32 or bf16 bits.  Returns (out [k][S][Hq][D], lse [k][S][Hq]) in
    float64, lse the natural log of the softmax normaliser of the scaled scores."""
    def f64(a):
        a = np.asarray(a)
        if a.dtype == np.uint16:
            return (a.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
        return a.astype(np.float64)
    q, kt, vt, kb, vb = (f64(x) for x in (q, k_trunk, v_trunk, k_branch, v_branch))
    K, S, Hq, D = q.shape
    Hkv = kt.shape[0]
    G = Hq // Hkv
    out = np.zeros((K, S, Hq, D))
    lse = np.zeros((K, S, Hq))
    causal = np.tril(np.ones((S, S), bool))
    for j in range(K):
        for hq in range(Hq):
            h = hq // G
            s_trunk = (q[j, :, hq] @ kt[h].T) * scale                       # [S][S]
            s_trunk = np.where(causal, s_trunk, -np.inf)
            s_br = np.stack([np.einsum("td,td->t", q[j, :, hq], kb[i, h]) * scale for i in range(1, j + 1)],
                            axis=1) if j > 0 else np.zeros((S, 0))          # [S][j]
            s = np.concatenate([s_trunk, s_br], axis=1)
            m = s.max(axis=1, keepdims=True)
            p = np.exp(s - m)
            l = p.sum(axis=1, keepdims=True)
            o = p[:, :S] @ vt[h]
            for i in range(1, j + 1):
                o += p[:, S + i - 1:S + i] * vb[i, h]
            out[j, :, hq] = o / l
            lse[j, :, hq] = (m + np.log(l))[:, 0]
    return out, lse
