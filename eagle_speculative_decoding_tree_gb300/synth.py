"""Seeded synthetic inputs for the EAGLE draft-tree verify step.

This module only *draws numbers*: logit rows, Q/K/V, uniforms, prefix lengths and
the token-path hash that keys a synthetic language model's rows.  It holds none of
the verify step's arithmetic (no softmax, no top-k, no acceptance rule, no
attention), so the CUDA path and the CPU oracle can both take their inputs from it
without sharing any of the method.

Everything is keyed by numpy's Philox counter-based generator.  A stream is named
by ``(config_id, tag, *indices)`` on top of the master seed ``0xEA61E000``, so the
same name always yields the same bytes on any machine.

Workload shapes follow the pages' workloads: 7B/8B-class attention shapes, 32K and
128K vocabularies, 60-node dynamic trees, a 10-node static tree, an 8-token chain
and 1K-128K contexts (EAGLE review, sections 3.1 and 4; EAGLE-2 dynamic tree; Didi
EAGLE-3 practice, section 7).  Public benchmark prompts are not used: seeded
Gaussian or Zipf(1.1) logit rows stand in for them.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np

MASTER_SEED = 0xEA61E000
_MASK64 = (1 << 64) - 1
GOLDEN64 = 0x9E3779B97F4A7C15

# stream tags (first key word after the config id)
TAG_Q, TAG_K, TAG_V, TAG_TREE_K, TAG_TREE_V = 1, 2, 3, 4, 5
TAG_U_ACCEPT, TAG_U_FINAL, TAG_U_DRAFT, TAG_PREFIX, TAG_ROOT = 6, 7, 8, 9, 10
TAG_TARGET_ROW, TAG_DRAFT_ROW, TAG_FEAT, TAG_MISC = 11, 12, 13, 14


def rng(config_id: int, *key: int) -> np.random.Generator:
    """A Philox stream named by (config_id, *key) under the master seed."""
    ss = np.random.SeedSequence([MASTER_SEED + int(config_id)] + [int(k) & 0xFFFFFFFF for k in key])
    return np.random.Generator(np.random.Philox(ss))


def rng_for_hash(h: int, tag: int) -> np.random.Generator:
    """A Philox stream keyed directly by a 64-bit path hash (Philox key = [h, tag])."""
    return np.random.Generator(np.random.Philox(key=np.array([h & _MASK64, tag & _MASK64], dtype=np.uint64)))


# ----------------------------------------------------------------------------- bf16 bytes
def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest, ties to even); return the uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_value(bits: np.ndarray) -> np.ndarray:
    """The float32 value of bfloat16 bits (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def as_dtype_bytes(x: np.ndarray, dtype: str) -> np.ndarray:
    """Store float32 values as the given element type: 'f32' -> float32, 'bf16' -> uint16 bits."""
    if dtype == "f32":
        return np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "bf16":
        return bf16_bits(x)
    raise ValueError(dtype)


# ----------------------------------------------------------------------------- uniforms
def uniforms(gen: np.random.Generator, shape) -> np.ndarray:
    """Uniforms in [0, 1) on the 2^-24 grid: (uint32 >> 8) * 2^-24, exact in fp32 and fp64."""
    w = gen.integers(0, 1 << 32, size=shape, dtype=np.uint64)
    return ((w >> np.uint64(8)).astype(np.float64) * (2.0 ** -24)).astype(np.float32)


# ----------------------------------------------------------------------------- logit rows
def normal_row(gen: np.random.Generator, shape, sigma: float) -> np.ndarray:
    return (gen.standard_normal(size=shape, dtype=np.float32) * np.float32(sigma)).astype(np.float32)


def zipf_row(gen: np.random.Generator, vocab: int, s: float = 1.1) -> np.ndarray:
    """Zipf(s)-skewed logits: logit_v = -s * ln(rank_v), rank a seeded permutation of 1..V."""
    rank = gen.permutation(vocab).astype(np.float64) + 1.0
    return (-s * np.log(rank)).astype(np.float32)


# ----------------------------------------------------------------------------- path hash
def splitmix64(x: int) -> int:
    """SplitMix64 finaliser (Steele, Lea and Flood, 2014) on a Python int."""
    z = (x + GOLDEN64) & _MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
    return z ^ (z >> 31)


def child_hash(h_parent: int, tok: int) -> int:
    """Hash of the path (parent path, tok): splitmix64(h_parent xor (tok+1)*phi64)."""
    return splitmix64((h_parent ^ (((int(tok) + 1) * GOLDEN64) & _MASK64)) & _MASK64)


def root_hash(config_id: int, request: int, step: int = 0) -> int:
    return splitmix64(((MASTER_SEED + config_id) << 32) ^ (request << 16) ^ step)


class HashLM:
    """A synthetic language model whose logit rows are a pure function of the token path.

    The target row at a node is drawn from a Philox stream keyed by the node's path
    hash; the draft row is the target row plus N(0, draft_sigma^2) noise keyed by the
    same hash.  The same path therefore always yields the same rows, which lets a
    speculative decode be checked token for token against plain decoding.
    """

    def __init__(self, vocab: int, kind: str = "normal", sigma: float = 3.0,
                 draft_sigma: float = 0.5, dtype: str = "f32"):
        self.vocab, self.kind, self.sigma, self.draft_sigma, self.dtype = vocab, kind, sigma, draft_sigma, dtype

    def _target_f32(self, h: int) -> np.ndarray:
        g = rng_for_hash(h, TAG_TARGET_ROW)
        if self.kind == "zipf":
            return zipf_row(g, self.vocab, 1.1)
        return normal_row(g, (self.vocab,), self.sigma)

    def target_row(self, h: int) -> np.ndarray:
        """Target logit row, rounded to the element type (float32 values)."""
        x = self._target_f32(h)
        return bf16_value(bf16_bits(x)) if self.dtype == "bf16" else x

    def draft_row(self, h: int) -> np.ndarray:
        x = self._target_f32(h) + normal_row(rng_for_hash(h, TAG_DRAFT_ROW), (self.vocab,), self.draft_sigma)
        return bf16_value(bf16_bits(x)) if self.dtype == "bf16" else x.astype(np.float32)

    def rows(self, hashes: Sequence[int], which: str) -> np.ndarray:
        f = self.target_row if which == "target" else self.draft_row
        return np.stack([f(h) for h in hashes]).astype(np.float32)


class BigramLM:
    """A tiny synthetic LM whose next-token logits depend only on the last token.

    Used for the many-trial distribution tests: target row = T[last], draft row =
    T[last] + noise table.  Rows for a whole batch come from one fancy index.
    """

    def __init__(self, vocab: int, sigma: float, draft_sigma: float, seed_key: int = 0):
        g = rng(0, TAG_MISC, 0xB16, seed_key)
        self.vocab = vocab
        self.target = normal_row(g, (vocab, vocab), sigma)
        self.draft = (self.target + normal_row(g, (vocab, vocab), draft_sigma)).astype(np.float32)


# ----------------------------------------------------------------------------- workloads
@dataclasses.dataclass(frozen=True)
class Workload:
    """One verify-step workload.  Sizes are the configuration's; see WORKLOADS."""
    config_id: int
    name: str
    dtype: str                 # element type of Q/K/V and logits: "f32" or "bf16"
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    vocab: int
    prefix: int                # prefix length (or the upper bound when ragged)
    prefix_min: int            # == prefix unless the batch is ragged
    tree_mode: str             # "dynamic", "static_topk", "static_sampled"
    depth: int                 # draft levels
    top_k: int                 # dynamic tree: children per frontier node and frontier width
    total_tokens: int          # dynamic tree: drafts kept (rows = total_tokens + 1)
    static_choices: tuple      # static tree: paths of child ranks, ordered by depth
    logits: str                # "normal" or "zipf"
    sigma: float               # target logit scale (normal)
    draft_sigma: float
    temperature: float
    batch: int
    layers: int

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def rows(self) -> int:
        if self.tree_mode == "dynamic":
            return self.total_tokens + 1
        return len(self.static_choices) + 1

    @property
    def proposal(self) -> str:
        return "sampled" if self.tree_mode == "static_sampled" else "delta"

    @property
    def max_seq(self) -> int:
        """Cache capacity per request: the prefix plus room for one step's commit, rounded to 64."""
        return ((self.prefix + self.depth + 1 + 63) // 64) * 64

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The 10-node depth-3 static tree (root k=4; higher-ranked branches deeper and wider).
TINY_STATIC_CHOICES = ((0,), (1,), (2,), (3,), (0, 0), (0, 1), (1, 0), (2, 0), (0, 0, 0), (0, 0, 1))
CHAIN7 = tuple(tuple([0] * d) for d in range(1, 8))

WORKLOADS = {
    "tiny": Workload(1, "tiny", "f32", 4, 4, 64, 1000, 128, 128, "static_sampled", 3, 4, 10,
                     TINY_STATIC_CHOICES, "normal", 2.0, 0.5, 1.0, 1, 2),
    "vicuna7b": Workload(2, "vicuna7b", "bf16", 32, 32, 128, 32000, 2048, 2048, "dynamic", 6, 10, 60,
                         (), "normal", 3.0, 0.7, 0.0, 1, 32),
    "llama8b": Workload(3, "llama8b", "bf16", 32, 8, 128, 128256, 8192, 8192, "dynamic", 7, 8, 60,
                        (), "zipf", 0.0, 0.5, 1.0, 1, 32),
    "long128k": Workload(4, "long128k", "bf16", 32, 8, 128, 128256, 131072, 131072, "static_sampled", 7, 1, 7,
                         CHAIN7, "normal", 3.0, 1.0, 1.0, 1, 32),
    "concurrency": Workload(5, "concurrency", "bf16", 32, 8, 128, 128256, 16384, 1024, "dynamic", 6, 8, 60,
                            (), "zipf", 0.0, 0.5, 1.0, 8, 32),
}


def static_parents(choices: Sequence[Sequence[int]]) -> np.ndarray:
    """Parent index per node (node 0 = root) of a static tree given as child-rank paths."""
    index = {(): 0}
    par = [-1]
    for i, path in enumerate(choices, start=1):
        path = tuple(path)
        index[path] = i
        par.append(index[path[:-1]])
    return np.asarray(par, dtype=np.int32)


def prefix_lengths(w: Workload, batch: Optional[int] = None) -> np.ndarray:
    b = w.batch if batch is None else batch
    if w.prefix_min == w.prefix:
        return np.full(b, w.prefix, dtype=np.int32)
    g = rng(w.config_id, TAG_PREFIX, b)
    return g.integers(w.prefix_min, w.prefix + 1, size=b).astype(np.int32)


def attn_tensors(w: Workload, layer: int, batch: int, seq_len: np.ndarray, rows: int, q_scale: float = 1.0):
    """Q [B][R][Hq][D], K/V cache [B][Hkv][P_max][D], tree K/V [B][Hkv][R][D], all N(0,1).

    Returned in the workload's element type (float32 or bf16 bits).  Cache slots at
    or beyond a request's prefix length are zero.
    """
    P = w.max_seq
    D, Hq, Hkv = w.head_dim, w.n_q_heads, w.n_kv_heads
    gq = rng(w.config_id, TAG_Q, layer, batch)
    q = normal_row(gq, (batch, rows, Hq, D), q_scale)
    kc = np.zeros((batch, Hkv, P, D), np.float32)
    vc = np.zeros((batch, Hkv, P, D), np.float32)
    for b in range(batch):
        n = int(seq_len[b])
        kc[b, :, :n] = normal_row(rng(w.config_id, TAG_K, layer, b), (Hkv, n, D), 1.0)
        vc[b, :, :n] = normal_row(rng(w.config_id, TAG_V, layer, b), (Hkv, n, D), 1.0)
    tk = normal_row(rng(w.config_id, TAG_TREE_K, layer, batch), (batch, Hkv, rows, D), 1.0)
    tv = normal_row(rng(w.config_id, TAG_TREE_V, layer, batch), (batch, Hkv, rows, D), 1.0)
    cvt = lambda x: as_dtype_bytes(x, w.dtype)
    return cvt(q), cvt(kc), cvt(vc), cvt(tk), cvt(tv)


def step_uniforms(w: Workload, batch: int, rows: int, step: int = 0):
    """u_accept [B][R] (one per node test), u_final [B], u_draft [B][R] (sampled children)."""
    ua = uniforms(rng(w.config_id, TAG_U_ACCEPT, batch, step), (batch, rows))
    uf = uniforms(rng(w.config_id, TAG_U_FINAL, batch, step), (batch,))
    ud = uniforms(rng(w.config_id, TAG_U_DRAFT, batch, step), (batch, rows))
    return ua, uf, ud


def root_tokens(w: Workload, batch: int) -> np.ndarray:
    return rng(w.config_id, TAG_ROOT, batch).integers(0, w.vocab, size=batch).astype(np.int32)


def hash_lm(w: Workload) -> HashLM:
    return HashLM(w.vocab, w.logits, w.sigma, w.draft_sigma, w.dtype)


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def mask_words(rows: int) -> int:
    return max(1, math.ceil(rows / 64))
