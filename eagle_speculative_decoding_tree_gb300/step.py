"""One EAGLE verify step on the GPU: tree attention over L layers, acceptance, commit.

``VerifyStep`` owns the device buffers of a workload (caches, tree K/V, queries,
logits, uniforms, outputs) and enqueues the step's library calls on one stream:

    for each layer: eagle_tree_attn      (tree attention)
    eagle_accept                         (multi-round speculative sampling)
    eagle_kv_commit                      (accepted path -> contiguous cache)

This follows the verify half of the pages' data path (EAGLE review, "GPU / system
data path" steps 6-7).  Every step of it runs in libeagle's kernels; this module
only allocates memory with torch and passes pointers.  ``build_tree`` runs the
draft-tree build (eagle_tree_build, level by level) with draft rows from the
seeded synthetic LM, which stands in for the draft model.
"""
from __future__ import annotations

import math
from typing import Optional

import numpy as np
import torch

from . import binding as B
from . import synth


def _to_dev(x: np.ndarray, dtype: str, device) -> torch.Tensor:
    """Upload generator output (float32 values or bf16 bits) as a device tensor."""
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(device)


def tree_desc_for(w: synth.Workload, batch: int) -> B.TreeDesc:
    dt = B.EAGLE_F32 if w.dtype == "f32" else B.EAGLE_BF16
    if w.tree_mode == "dynamic":
        return B.tree_desc(batch, w.vocab, B.EAGLE_TREE_DYNAMIC, w.depth, w.top_k, w.total_tokens, dtype=dt)
    mode = B.EAGLE_TREE_STATIC_SAMPLED if w.tree_mode == "static_sampled" else B.EAGLE_TREE_STATIC_TOPK
    par = synth.static_parents(w.static_choices)
    return B.tree_desc(batch, w.vocab, mode, int(max(len(c) for c in w.static_choices)),
                       static_parent=par.tolist(), dtype=dt, temperature=w.temperature if w.temperature > 0 else 1.0)


class GpuTreeBuilder:
    """Level-by-level tree build through eagle_tree_build (the same driver interface
    as the tests' oracle builders: expand(level, logits, u_draft) -> (frontier tokens,
    frontier parent slots) on the host, finalize(root_tok, seq_len) -> tree dict)."""

    def __init__(self, w: synth.Workload, batch: int, device="cuda"):
        self.w, self.batch, self.device = w, batch, device
        self.desc = tree_desc_for(w, batch)
        self.ws = torch.zeros(B.workspace_size(B.EAGLE_WS_TREE_BUILD, self.desc), dtype=torch.uint8, device=device)
        self.out = B.TreeBuffers.allocate(self.desc, device)
        self.depth = w.depth if w.tree_mode == "dynamic" else self.desc.depth
        self.root_tok = None
        self.seq_len = None
        self.levels = []  # (level, device logits, device uniforms) of every expand call

    def set_context(self, root_tok: np.ndarray, seq_len: np.ndarray):
        self.root_tok = torch.from_numpy(np.asarray(root_tok, np.int32)).to(self.device)
        self.seq_len = torch.from_numpy(np.asarray(seq_len, np.int32)).to(self.device)

    def expand(self, level: int, logits: np.ndarray, u_draft: Optional[np.ndarray] = None):
        if self.root_tok is None:
            self.set_context(np.zeros(self.batch, np.int32), np.zeros(self.batch, np.int32))
        lg = _to_dev(logits, self.w.dtype, self.device)
        ud = None if u_draft is None else torch.from_numpy(np.asarray(u_draft, np.float32)).to(self.device)
        B.eagle_tree_build(self.desc, level, lg, ud, self.root_tok, self.seq_len, self.ws, self.out)
        self.levels = [lv for lv in self.levels if lv[0] < level] + [(level, lg, ud)]
        return self._frontier(level)

    def _frontier(self, level: int):
        if self.w.tree_mode == "dynamic":
            F = self.w.top_k
        else:  # the nodes created at this level (depth == level), in row order
            par = synth.static_parents(self.w.static_choices)
            dep = np.zeros(len(par), np.int32)
            for i in range(1, len(par)):
                dep[i] = dep[par[i]] + 1
            F = int((dep == level).sum())
        return self.out.frontier_tok[:, :F].cpu().numpy(), self.out.frontier_slot[:, :F].cpu().numpy()

    def expand_head(self, level: int, hidden: np.ndarray, head_weight: torch.Tensor, status: torch.Tensor):
        """One level from the frontier rows' hidden states (bf16 bits [B][F][h]) and the
        draft LM head (device bf16 [V][h]) through eagle_tree_build_head."""
        if self.root_tok is None:
            self.set_context(np.zeros(self.batch, np.int32), np.zeros(self.batch, np.int32))
        hd = torch.from_numpy(np.ascontiguousarray(hidden).view(np.int16)).to(self.device).view(torch.bfloat16)
        B.eagle_tree_build_head(self.desc, level, hd, head_weight, self.root_tok, self.seq_len, self.ws, self.out,
                                status)
        self.head_levels = [lv for lv in getattr(self, "head_levels", []) if lv[0] < level] + [(level, hd)]
        return self._frontier(level)

    def replay(self, stream=None):
        """Enqueue the whole build again (every level, inputs already on the device)."""
        for level, lg, ud in self.levels:
            B.eagle_tree_build(self.desc, level, lg, ud, self.root_tok, self.seq_len, self.ws, self.out, stream)

    def replay_head(self, head_weight: torch.Tensor, status: torch.Tensor, stream=None):
        """Enqueue the whole build from hidden states again (every level's hidden states
        already on the device)."""
        for level, hd in self.head_levels:
            B.eagle_tree_build_head(self.desc, level, hd, head_weight, self.root_tok, self.seq_len, self.ws,
                                    self.out, status, stream)

    def finalize(self, root_tok: np.ndarray, seq_len: np.ndarray):
        o = self.out
        return dict(tokens=o.tokens.cpu().numpy(), parent=o.parent.cpu().numpy(), depth=o.depth.cpu().numpy(),
                    pos_id=o.pos_id.cpu().numpy(), anc_mask=o.anc_mask.cpu().numpy().view(np.uint64),
                    score=o.score.cpu().numpy(), near_tie=o.near_tie.cpu().numpy())


def build_tree(w: synth.Workload, batch: int, root_tok: np.ndarray, root_hashes, seq_len: np.ndarray,
               u_draft: Optional[np.ndarray] = None, device="cuda"):
    """Draft-tree build on the GPU, fed level by level with the synthetic LM's draft rows."""
    lm = synth.hash_lm(w)
    bld = GpuTreeBuilder(w, batch, device)
    bld.set_context(root_tok, seq_len)
    front = [[int(h)] for h in root_hashes]
    for level in range(1, bld.depth + 1):
        rows = np.stack([lm.rows(front[b], "draft") for b in range(batch)])
        ftok, fslot = bld.expand(level, synth.as_dtype_bytes(rows, w.dtype), u_draft)
        front = [[synth.child_hash(front[b][int(fslot[b, j])], int(ftok[b, j])) for j in range(ftok.shape[1])]
                 for b in range(batch)]
    return bld.finalize(root_tok, seq_len), bld


def node_hashes(tokens: np.ndarray, parent: np.ndarray, root_hashes):
    Bn, R = tokens.shape
    hs = []
    for b in range(Bn):
        h = [int(root_hashes[b])]
        for i in range(1, R):
            h.append(synth.child_hash(h[int(parent[b, i])], int(tokens[b, i])))
        hs.append(h)
    return hs


class VerifyStep:
    """Device state and call sequence of one verify step for a workload.

    The tree (tokens, parents, ancestor masks) comes from ``build_tree`` on the GPU;
    target/draft logits are the synthetic LM's rows at the tree's nodes; Q, K/V and
    the uniforms are seeded normals / uniforms.  ``run`` enqueues the step;
    ``reset`` restores seq_len so that repeated runs process the same step.
    """

    def __init__(self, w: synth.Workload, batch: Optional[int] = None, layers: Optional[int] = None,
                 device="cuda", q_scale: float = 1.0, num_splits: int = 0, tree: Optional[dict] = None,
                 keep_host: bool = False, precision: int = B.EAGLE_ATTN_PRECISE):
        self.w = w
        self.B = batch if batch is not None else w.batch
        self.L = layers if layers is not None else w.layers
        self.device = device
        Bn, L = self.B, self.L
        self.seq_len0 = synth.prefix_lengths(w, Bn)
        self.root_tok = synth.root_tokens(w, Bn)
        self.root_hashes = [synth.root_hash(w.config_id, b) for b in range(Bn)]
        ua, uf, ud = synth.step_uniforms(w, Bn, w.rows)
        self.u_draft_host = ud
        self.builder = None
        if tree is None:
            tree, self.builder = build_tree(w, Bn, self.root_tok, self.root_hashes, self.seq_len0,
                                            ud if w.tree_mode == "static_sampled" else None, device)
        self.tree = tree
        R = tree["tokens"].shape[1]
        self.R = R
        # path arrays sized for the deepest tree the workload builds (step variants included)
        self.max_depth = max(int(tree["depth"].max()), w.depth if w.tree_mode == "dynamic" else 0)
        dev = torch.device(device)
        i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(dev)
        self.tokens, self.parent = i32(tree["tokens"]), i32(tree["parent"])
        self.anc_mask = torch.from_numpy(np.ascontiguousarray(tree["anc_mask"]).view(np.int64)).to(dev)
        self.seq_len = i32(self.seq_len0)
        self.seq_len_init = self.seq_len.clone()
        self.u_accept = torch.from_numpy(ua).to(dev)
        self.u_final = torch.from_numpy(uf).to(dev)

        # logits at the tree's nodes from the synthetic LM
        lm = synth.hash_lm(w)
        hs = node_hashes(tree["tokens"], tree["parent"], self.root_hashes)
        tgt = np.stack([lm.rows(hs[b], "target") for b in range(Bn)])
        self.target_host = synth.as_dtype_bytes(tgt, w.dtype)
        self.target = _to_dev(self.target_host, w.dtype, dev)
        self.draft = None
        self.draft_host = None
        if w.proposal == "sampled" and w.temperature > 0:
            dft = np.stack([lm.rows(hs[b], "draft") for b in range(Bn)])
            self.draft_host = synth.as_dtype_bytes(dft, w.dtype)
            self.draft = _to_dev(self.draft_host, w.dtype, dev)

        # per-layer attention tensors
        self.q, self.kc, self.vc, self.tk, self.tv, self.out = [], [], [], [], [], []
        self.host = [] if keep_host else None
        for l in range(L):
            q, kc, vc, tk, tv = synth.attn_tensors(w, l, Bn, self.seq_len0, R, q_scale)
            if keep_host:
                self.host.append((q, kc, vc, tk, tv))
            self.q.append(_to_dev(q, w.dtype, dev))
            self.kc.append(_to_dev(kc, w.dtype, dev))
            self.vc.append(_to_dev(vc, w.dtype, dev))
            self.tk.append(_to_dev(tk, w.dtype, dev))
            self.tv.append(_to_dev(tv, w.dtype, dev))
            self.out.append(torch.empty_like(self.q[-1]))
        self.lse = torch.empty(Bn, R, w.n_q_heads, dtype=torch.float32, device=dev)
        dt = B.EAGLE_F32 if w.dtype == "f32" else B.EAGLE_BF16
        self.attn_desc = B.AttnDesc(Bn, R, w.n_q_heads, w.n_kv_heads, w.head_dim, w.max_seq,
                                    1.0 / math.sqrt(w.head_dim), dt, num_splits, dt, precision)
        self.attn_ws = torch.zeros(B.workspace_size(B.EAGLE_WS_TREE_ATTN, self.attn_desc), dtype=torch.uint8,
                                   device=dev)
        prop = B.EAGLE_PROPOSAL_SAMPLED if w.proposal == "sampled" else B.EAGLE_PROPOSAL_DELTA
        self.acc_desc = B.AcceptDesc(Bn, R, w.vocab, float(w.temperature), prop, dt, self.max_depth)
        self.acc_ws = torch.zeros(B.workspace_size(B.EAGLE_WS_ACCEPT, self.acc_desc), dtype=torch.uint8, device=dev)
        self.acc = B.AcceptBuffers.allocate(Bn, self.max_depth, dev)
        self.commit_desc = B.CommitDesc(L, Bn, w.n_kv_heads, w.head_dim, R, w.max_seq, self.max_depth, dt, 0, dt)
        self.layers = B.LayerPointers(self.kc, self.vc, self.tk, self.tv)
        self.commit_pos = torch.zeros(Bn, self.max_depth + 1, dtype=torch.int32, device=dev)
        self.variants = [dict(tokens=self.tokens, parent=self.parent, anc_mask=self.anc_mask, target=self.target,
                              draft=self.draft, u_accept=self.u_accept, u_final=self.u_final)]

    # ------------------------------------------------------------------ step variants
    def add_variants(self, n: int):
        """n more verify steps of the same workload over the same caches and queries: each
        has its own root token, draft tree (built on the GPU from the synthetic LM's rows),
        logits at its nodes and uniforms (seeded by the step index), so replaying them in
        turn accepts drafts at the workload's own rate.  Variant 0 is the step built in
        the constructor."""
        w, Bn, dev = self.w, self.B, torch.device(self.device)
        i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(dev)
        lm = synth.hash_lm(w)
        for k in range(1, n + 1):
            g = synth.rng(w.config_id, 9100, k, Bn)
            root_tok = g.integers(0, w.vocab, size=Bn).astype(np.int32)
            root_h = [synth.root_hash(w.config_id, b, 1000 + k) for b in range(Bn)]
            ua, uf, ud = synth.step_uniforms(w, Bn, w.rows, step=1000 + k)
            tree, _ = build_tree(w, Bn, root_tok, root_h, self.seq_len0,
                                 ud if w.tree_mode == "static_sampled" else None, self.device)
            if tree["tokens"].shape[1] != self.R or int(tree["depth"].max()) > self.max_depth:
                continue  # a variant must fit the step's shapes (rows, path length)
            hs = node_hashes(tree["tokens"], tree["parent"], root_h)
            tgt = synth.as_dtype_bytes(np.stack([lm.rows(hs[b], "target") for b in range(Bn)]), w.dtype)
            v = dict(tokens=i32(tree["tokens"]), parent=i32(tree["parent"]),
                     anc_mask=torch.from_numpy(np.ascontiguousarray(tree["anc_mask"]).view(np.int64)).to(dev),
                     target=_to_dev(tgt, w.dtype, dev), draft=None, u_accept=torch.from_numpy(ua).to(dev),
                     u_final=torch.from_numpy(uf).to(dev))
            if self.draft is not None:
                dft = synth.as_dtype_bytes(np.stack([lm.rows(hs[b], "draft") for b in range(Bn)]), w.dtype)
                v["draft"] = _to_dev(dft, w.dtype, dev)
            self.variants.append(v)
        return len(self.variants)

    def use_variant(self, k: int):
        """Point the step's calls at variant k's tree, logits and uniforms."""
        v = self.variants[k]
        self.tokens, self.parent, self.anc_mask = v["tokens"], v["parent"], v["anc_mask"]
        self.target, self.draft = v["target"], v["draft"]
        self.u_accept, self.u_final = v["u_accept"], v["u_final"]

    # ------------------------------------------------------------------ calls
    def attn_layer(self, l: int, stream=None, lse: bool = False):
        B.eagle_tree_attn(self.attn_desc, self.q[l], self.kc[l], self.vc[l], self.tk[l], self.tv[l], self.seq_len,
                          self.anc_mask, self.out[l], self.lse if lse else None, self.attn_ws, stream)

    def accept(self, stream=None):
        B.eagle_accept(self.acc_desc, self.target, self.draft, self.tokens, self.parent, self.u_accept, self.u_final,
                       self.acc, self.acc_ws, stream)

    def commit(self, stream=None):
        B.eagle_kv_commit(self.commit_desc, self.layers, self.acc.n_acc, self.acc.path, self.seq_len,
                          self.commit_pos, status=self.acc.status, stream=stream)

    def reset(self):
        """Restore seq_len so that the next run repeats the same step."""
        self.seq_len.copy_(self.seq_len_init)

    def run(self, stream=None, reset: bool = True):
        if reset:
            self.reset()
        for l in range(self.L):
            self.attn_layer(l, stream)
        self.accept(stream)
        self.commit(stream)

    # ------------------------------------------------------------------ accounting
    def kv_bytes_per_layer(self) -> int:
        """Algorithmic K/V bytes one tree-attention launch must read: prefix + tree rows."""
        esz = 4 if self.w.dtype == "f32" else 2
        rows = int(self.seq_len0.sum()) + self.B * self.R
        return 2 * rows * self.w.n_kv_heads * self.w.head_dim * esz

    def logit_bytes_visited(self, n_acc: np.ndarray) -> int:
        """Target rows the acceptance walk visits (n_acc + 1 per request), plus draft rows when sampled."""
        esz = 4 if self.w.dtype == "f32" else 2
        rows = int(np.sum(n_acc + 1))
        per = self.w.vocab * esz
        return rows * per * (2 if self.draft is not None else 1)
