"""Shared helpers for the GPU parity tests (marked `gpu`)."""
import math

import numpy as np
import torch

from eagle_speculative_decoding_tree_gb300 import binding as B
from eagle_speculative_decoding_tree_gb300 import synth

BF16_TOL = 2e-3  # max abs error, bf16 inputs with fp32 accumulation
F32_TOL = 1e-5   # max abs error, fp32 inputs


def dev(x: np.ndarray, dtype: str) -> torch.Tensor:
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()


def random_tree(rows: int, seed: int, chain: bool = False):
    """A random draft-tree shape (parent[i] < i) and its ancestor masks."""
    g = synth.rng(0, 4242, seed, rows)
    par = np.full(rows, -1, np.int32)
    for i in range(1, rows):
        par[i] = i - 1 if chain else int(g.integers(max(0, i - 12), i))
    W = max(1, -(-rows // 64))
    mask = np.zeros((rows, W), np.uint64)
    for i in range(rows):
        if i > 0:
            mask[i] = mask[par[i]]
        mask[i, i // 64] |= np.uint64(1) << np.uint64(i % 64)
    return par, mask


def run_attn(w: synth.Workload, batch: int, seq_len: np.ndarray, rows: int, parent: np.ndarray,
             mask: np.ndarray, layer: int = 0, q_scale: float = 1.0, num_splits: int = 0, out_f32: bool = False,
             precision: int = B.EAGLE_ATTN_PRECISE, engine: int = B.EAGLE_ENGINE_AUTO, n_nodes=None,
             fault_test: int = 0, ws=None):
    """Generate one layer's inputs and run eagle_tree_attn; returns host inputs and outputs
    (n_nodes: per-request tree sizes; ws: a workspace to reuse, else a zeroed one)."""
    q, kc, vc, tk, tv = synth.attn_tensors(w, layer, batch, seq_len, rows, q_scale)
    dt = B.EAGLE_F32 if w.dtype == "f32" else B.EAGLE_BF16
    odt = B.EAGLE_F32 if (out_f32 or w.dtype == "f32") else B.EAGLE_BF16
    desc = B.AttnDesc(batch, rows, w.n_q_heads, w.n_kv_heads, w.head_dim, w.max_seq, 1.0 / math.sqrt(w.head_dim),
                      dt, num_splits, odt, precision, engine, fault_test)
    if ws is None:
        ws = torch.zeros(B.workspace_size(B.EAGLE_WS_TREE_ATTN, desc), dtype=torch.uint8, device="cuda")
    tq = dev(q, w.dtype)
    out = torch.full(tq.shape, float("nan"), dtype=torch.float32 if odt == B.EAGLE_F32 else torch.bfloat16,
                     device="cuda")
    lse = torch.empty(batch, rows, w.n_q_heads, dtype=torch.float32, device="cuda")
    am = torch.from_numpy(np.broadcast_to(mask, (batch,) + mask.shape[-2:]).copy().view(np.int64)).cuda()
    B.eagle_tree_attn(desc, tq, dev(kc, w.dtype), dev(vc, w.dtype), dev(tk, w.dtype), dev(tv, w.dtype),
                      torch.from_numpy(np.asarray(seq_len, np.int32)).cuda(), am, out, lse, ws,
                      n_nodes=None if n_nodes is None else torch.from_numpy(np.asarray(n_nodes, np.int32)).cuda())
    torch.cuda.synchronize()
    if ws.numel() >= 4 and not fault_test:  # the tensor-core kernel's error word (bounded waits that gave up)
        assert int(ws[:4].view(torch.int32).item()) == 0 or not is_tc(desc), "tcgen05 kernel wait timed out"
    return (q, kc, vc, tk, tv), out.float().cpu().numpy(), lse.cpu().numpy()


def is_tc(desc) -> bool:
    """Whether a descriptor runs the tcgen05 kernel (bf16, head_dim 128, G divides 128, auto engine)."""
    G = desc.n_q_heads // desc.n_kv_heads
    return desc.dtype == B.EAGLE_BF16 and desc.head_dim == 128 and 128 % G == 0 and desc.engine == B.EAGLE_ENGINE_AUTO


def head_slice(inputs, h: int, G: int, b: int):
    """Inputs restricted to request b and KV head h (and its G query heads)."""
    q, kc, vc, tk, tv = inputs
    return (np.ascontiguousarray(q[b:b + 1, :, h * G:(h + 1) * G]), np.ascontiguousarray(kc[b:b + 1, h:h + 1]),
            np.ascontiguousarray(vc[b:b + 1, h:h + 1]), np.ascontiguousarray(tk[b:b + 1, h:h + 1]),
            np.ascontiguousarray(tv[b:b + 1, h:h + 1]))
