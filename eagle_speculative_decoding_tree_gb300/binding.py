"""Thin Python binding of libeagle's C ABI (include/eagle.h).

Argument marshalling only: every function here checks that tensors live on the GPU
with the expected dtype and layout, passes their data pointers and the current
CUDA stream to the library, and raises on a non-zero status.  All computation
happens in the library's CUDA kernels.  There is no fallback: if libeagle.so has
not been built, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional, Sequence

import torch

from . import build as _build

# ----------------------------------------------------------------------------- constants
EAGLE_OK = 0
EAGLE_ERR_INVALID_ARG, EAGLE_ERR_UNSUPPORTED, EAGLE_ERR_ALIGNMENT, EAGLE_ERR_WORKSPACE, EAGLE_ERR_CUDA = 1, 2, 3, 4, 5
EAGLE_F32, EAGLE_BF16 = 0, 1
EAGLE_TREE_DYNAMIC, EAGLE_TREE_STATIC_TOPK, EAGLE_TREE_STATIC_SAMPLED = 0, 1, 2
EAGLE_PROPOSAL_DELTA, EAGLE_PROPOSAL_SAMPLED = 0, 1
EAGLE_WS_TREE_BUILD, EAGLE_WS_TREE_ATTN, EAGLE_WS_ACCEPT = 1, 2, 3
EAGLE_ATTN_PRECISE, EAGLE_ATTN_FAST = 0, 1
EAGLE_ENGINE_AUTO, EAGLE_ENGINE_MMA_SYNC = 0, 1
EAGLE_STATUS_BAD_TREE, EAGLE_STATUS_PATH_OVERFLOW, EAGLE_STATUS_CACHE_FULL, EAGLE_STATUS_BAD_TOKEN = 1, 2, 4, 8

EXPORTED_SYMBOLS = ("eagle_tree_build", "eagle_tree_attn", "eagle_accept", "eagle_kv_commit",
                    "eagle_workspace_size", "eagle_status_string", "eagle_version",
                    "eagle_tree_frontier_rows", "eagle_tree_max_frontier", "eagle_last_cuda_error",
                    "eagle_last_cuda_error_string", "eagle_tree_attn_plan", "eagle_accept_noalloc",
                    "eagle_selftest_ff_log", "eagle_lmhead_stats", "eagle_ttt_attn", "eagle_tree_build_head")


class TreeDesc(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("vocab", ctypes.c_int32), ("mode", ctypes.c_int32),
                ("depth", ctypes.c_int32), ("top_k", ctypes.c_int32), ("total_tokens", ctypes.c_int32),
                ("n_static", ctypes.c_int32), ("static_parent", ctypes.POINTER(ctypes.c_int32)),
                ("dtype", ctypes.c_int32), ("temperature", ctypes.c_float)]


class TreeOut(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("tokens", "parent", "depth", "pos_id", "anc_mask", "score",
                                               "frontier_tok", "frontier_slot", "near_tie")]


class AttnDesc(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("rows", ctypes.c_int32), ("n_q_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("max_seq", ctypes.c_int32),
                ("scale", ctypes.c_float), ("dtype", ctypes.c_int32), ("num_splits", ctypes.c_int32),
                ("out_dtype", ctypes.c_int32), ("precision", ctypes.c_int32), ("engine", ctypes.c_int32),
                ("fault_test", ctypes.c_int32)]


class AcceptDesc(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("rows", ctypes.c_int32), ("vocab", ctypes.c_int32),
                ("temperature", ctypes.c_float), ("proposal", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("max_depth", ctypes.c_int32)]


class AcceptOut(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("n_acc", "path", "out_tok", "near_tie", "status")]


class LmHeadDesc(ctypes.Structure):
    _fields_ = [("rows", ctypes.c_int32), ("tree_rows", ctypes.c_int32), ("hidden", ctypes.c_int32),
                ("vocab", ctypes.c_int32), ("temperature", ctypes.c_float)]


EAGLE_LMHEAD_TILE = 128
EAGLE_WS_TTT_ATTN = 4


class TttDesc(ctypes.Structure):
    _fields_ = [("steps", ctypes.c_int32), ("seq", ctypes.c_int32), ("n_q_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("scale", ctypes.c_float),
                ("out_dtype", ctypes.c_int32)]
EAGLE_STATUS_TIMEOUT = 0x10


class CommitDesc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("layers", "batch", "n_kv_heads", "head_dim", "rows", "max_seq",
                                              "max_depth", "dtype", "feat_dim", "feat_dtype")]


# ----------------------------------------------------------------------------- loading
_lib = None


def lib_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Load libeagle.so.  Raises if it has not been built: there is no fallback."""
    global _lib
    if _lib is None:
        if not os.path.exists(_build.LIB):
            raise ImportError(f"libeagle.so is not built ({_build.LIB}); run __graft_entry__.build() "
                              "or python -m eagle_speculative_decoding_tree_gb300.build")
        L = ctypes.CDLL(_build.LIB)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        L.eagle_tree_build.argtypes = [ctypes.POINTER(TreeDesc), i32, vp, vp, vp, vp, vp, sz, ctypes.POINTER(TreeOut), vp]
        L.eagle_tree_attn.argtypes = [ctypes.POINTER(AttnDesc), vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.eagle_accept.argtypes = [ctypes.POINTER(AcceptDesc), vp, vp, vp, vp, vp, vp, ctypes.POINTER(AcceptOut), vp,
                                   sz, vp]
        L.eagle_accept_noalloc.argtypes = [ctypes.POINTER(AcceptDesc), vp, vp, vp, vp, vp, vp,
                                           ctypes.POINTER(AcceptOut), vp]
        L.eagle_kv_commit.argtypes = [ctypes.POINTER(CommitDesc), vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.eagle_selftest_ff_log.argtypes = [vp, vp, vp, vp, i32, vp]
        L.eagle_lmhead_stats.argtypes = [ctypes.POINTER(LmHeadDesc), vp, vp, vp, vp, vp, vp, vp, vp]
        L.eagle_ttt_attn.argtypes = [ctypes.POINTER(TttDesc), vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.eagle_tree_build_head.argtypes = [ctypes.POINTER(TreeDesc), i32, vp, vp, i32, vp, vp, vp, sz,
                                            ctypes.POINTER(TreeOut), vp, vp]
        L.eagle_workspace_size.argtypes = [i32, vp]
        L.eagle_workspace_size.restype = sz
        L.eagle_status_string.argtypes = [i32]
        L.eagle_status_string.restype = ctypes.c_char_p
        L.eagle_version.restype = ctypes.c_char_p
        L.eagle_last_cuda_error.restype = ctypes.c_int
        L.eagle_last_cuda_error_string.restype = ctypes.c_char_p
        L.eagle_tree_frontier_rows.argtypes = [ctypes.POINTER(TreeDesc), i32]
        L.eagle_tree_max_frontier.argtypes = [ctypes.POINTER(TreeDesc)]
        L.eagle_tree_attn_plan.argtypes = [ctypes.POINTER(AttnDesc), ctypes.POINTER(ctypes.c_int32),
                                           ctypes.POINTER(ctypes.c_int32)]
        for f in (L.eagle_tree_build, L.eagle_tree_build_head, L.eagle_tree_attn, L.eagle_accept, L.eagle_kv_commit,
                  L.eagle_tree_frontier_rows, L.eagle_tree_max_frontier, L.eagle_tree_attn_plan,
                  L.eagle_accept_noalloc):
            f.restype = ctypes.c_int
        _lib = L
    return _lib


class EagleError(RuntimeError):
    def __init__(self, fn: str, status: int):
        msg = f"{fn}: {load().eagle_status_string(status).decode()} (status {status})"
        if status == EAGLE_ERR_CUDA:
            msg += f": {load().eagle_last_cuda_error_string().decode()}"
        super().__init__(msg)
        self.status = status


def _check(fn: str, status: int):
    if status != EAGLE_OK:
        raise EagleError(fn, status)


def _ptr(t: Optional[torch.Tensor], dtype=None, name: str = "tensor") -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (libeagle runs on the GPU only)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def dtype_code(t: torch.dtype) -> int:
    if t == torch.float32:
        return EAGLE_F32
    if t == torch.bfloat16:
        return EAGLE_BF16
    raise ValueError(f"unsupported element type {t}")


FLOATS = (torch.float32, torch.bfloat16)


# ----------------------------------------------------------------------------- descriptors
def tree_desc(batch, vocab, mode, depth, top_k=0, total_tokens=0, static_parent: Sequence[int] = (),
              dtype=EAGLE_BF16, temperature=1.0) -> TreeDesc:
    d = TreeDesc(batch, vocab, mode, depth, top_k, total_tokens, 0, None, dtype, temperature)
    if mode != EAGLE_TREE_DYNAMIC:
        arr = (ctypes.c_int32 * len(static_parent))(*[int(x) for x in static_parent])
        d.n_static = len(static_parent) - 1
        d.static_parent = ctypes.cast(arr, ctypes.POINTER(ctypes.c_int32))
        d._keep = arr  # the HOST array must outlive the descriptor
    return d


def workspace_size(which: int, desc) -> int:
    return int(load().eagle_workspace_size(which, ctypes.cast(ctypes.pointer(desc), ctypes.c_void_p)))


def tree_attn_plan(desc: AttnDesc) -> tuple:
    """(splits, kernel launches per call) eagle_tree_attn uses for desc on this device."""
    sp, kn = ctypes.c_int32(0), ctypes.c_int32(0)
    st = load().eagle_tree_attn_plan(ctypes.byref(desc), ctypes.byref(sp), ctypes.byref(kn))
    if st != EAGLE_OK:
        raise EagleError("eagle_tree_attn_plan", st)
    return sp.value, kn.value


def tree_frontier_rows(desc: TreeDesc, level: int) -> int:
    return int(load().eagle_tree_frontier_rows(ctypes.byref(desc), level))


def tree_max_frontier(desc: TreeDesc) -> int:
    return int(load().eagle_tree_max_frontier(ctypes.byref(desc)))


@dataclass
class TreeBuffers:
    """Device outputs of eagle_tree_build (allocated by torch; the library allocates nothing)."""
    tokens: torch.Tensor
    parent: torch.Tensor
    depth: torch.Tensor
    pos_id: torch.Tensor
    anc_mask: torch.Tensor
    score: torch.Tensor
    frontier_tok: torch.Tensor
    frontier_slot: torch.Tensor
    near_tie: torch.Tensor

    @staticmethod
    def allocate(desc: TreeDesc, device="cuda") -> "TreeBuffers":
        B = desc.batch
        R = desc.total_tokens + 1 if desc.mode == EAGLE_TREE_DYNAMIC else desc.n_static + 1
        W = max(1, -(-R // 64))
        F = max(1, tree_max_frontier(desc))
        i32 = dict(dtype=torch.int32, device=device)
        return TreeBuffers(torch.zeros(B, R, **i32), torch.zeros(B, R, **i32), torch.zeros(B, R, **i32),
                           torch.zeros(B, R, **i32), torch.zeros(B, R, W, dtype=torch.int64, device=device),
                           torch.zeros(B, R, dtype=torch.float32, device=device), torch.zeros(B, F, **i32),
                           torch.zeros(B, F, **i32), torch.zeros(B, **i32))

    def c_struct(self) -> TreeOut:
        return TreeOut(*[_ptr(getattr(self, f[0]), name=f[0]) for f in TreeOut._fields_])


@dataclass
class AcceptBuffers:
    n_acc: torch.Tensor
    path: torch.Tensor
    out_tok: torch.Tensor
    near_tie: torch.Tensor
    status: torch.Tensor

    @staticmethod
    def allocate(batch: int, max_depth: int, device="cuda") -> "AcceptBuffers":
        i32 = dict(dtype=torch.int32, device=device)
        return AcceptBuffers(torch.zeros(batch, **i32), torch.zeros(batch, max_depth + 1, **i32),
                             torch.zeros(batch, max_depth + 1, **i32), torch.zeros(batch, **i32),
                             torch.zeros(1, **i32))

    def c_struct(self) -> AcceptOut:
        return AcceptOut(*[_ptr(getattr(self, f[0]), name=f[0]) for f in AcceptOut._fields_])


# ----------------------------------------------------------------------------- entry points
def eagle_tree_build(desc: TreeDesc, level: int, frontier_logits: torch.Tensor, u_draft: Optional[torch.Tensor],
                     root_tok: torch.Tensor, seq_len: torch.Tensor, ws: torch.Tensor, out: TreeBuffers,
                     stream=None) -> None:
    """One draft level of the tree build (see eagle.h: eagle_tree_build)."""
    o = out.c_struct()
    _check("eagle_tree_build", load().eagle_tree_build(
        ctypes.byref(desc), level, _ptr(frontier_logits, FLOATS, "frontier_logits"),
        _ptr(u_draft, torch.float32, "u_draft"), _ptr(root_tok, torch.int32, "root_tok"),
        _ptr(seq_len, torch.int32, "seq_len"), _ptr(ws, name="ws"), ws.numel() * ws.element_size(),
        ctypes.byref(o), _stream(stream)))


def eagle_tree_build_head(desc: TreeDesc, level: int, hidden: torch.Tensor, head_weight: torch.Tensor,
                          root_tok: torch.Tensor, seq_len: torch.Tensor, ws: torch.Tensor, out: TreeBuffers,
                          status: torch.Tensor, stream=None) -> None:
    """One draft level from the frontier rows' hidden states [B][F][h] and the LM head
    [V][h], both bf16 (see eagle.h: eagle_tree_build_head)."""
    o = out.c_struct()
    _check("eagle_tree_build_head", load().eagle_tree_build_head(
        ctypes.byref(desc), level, _ptr(hidden, torch.bfloat16, "hidden"),
        _ptr(head_weight, torch.bfloat16, "head_weight"), int(hidden.shape[-1]), _ptr(root_tok, torch.int32, "root_tok"),
        _ptr(seq_len, torch.int32, "seq_len"), _ptr(ws, name="ws"), ws.numel() * ws.element_size(), ctypes.byref(o),
        _ptr(status, torch.int32, "status"), _stream(stream)))


def eagle_tree_attn(desc: AttnDesc, q, k_cache, v_cache, tree_k, tree_v, seq_len, anc_mask, out,
                    lse: Optional[torch.Tensor], ws: Optional[torch.Tensor], stream=None,
                    n_nodes: Optional[torch.Tensor] = None) -> None:
    """One layer of tree attention (see eagle.h: eagle_tree_attn); n_nodes [B] int32
    gives each request's tree size (None: every request has desc.rows rows)."""
    ws_ptr = _ptr(ws, name="ws") if ws is not None else None
    ws_bytes = ws.numel() * ws.element_size() if ws is not None else 0
    _check("eagle_tree_attn", load().eagle_tree_attn(
        ctypes.byref(desc), _ptr(q, FLOATS, "q"), _ptr(k_cache, FLOATS, "k_cache"), _ptr(v_cache, FLOATS, "v_cache"),
        _ptr(tree_k, FLOATS, "tree_k"), _ptr(tree_v, FLOATS, "tree_v"), _ptr(seq_len, torch.int32, "seq_len"),
        _ptr(n_nodes, torch.int32, "n_nodes"),
        _ptr(anc_mask, torch.int64, "anc_mask"), _ptr(out, FLOATS, "out"), _ptr(lse, torch.float32, "lse"),
        ws_ptr, ws_bytes, _stream(stream)))


def eagle_accept(desc: AcceptDesc, target_logits, draft_logits, tree_tokens, tree_parent, u_accept, u_final,
                 out: AcceptBuffers, ws: torch.Tensor, stream=None) -> None:
    """Multi-round speculative sampling down the tree (see eagle.h: eagle_accept)."""
    o = out.c_struct()
    _check("eagle_accept", load().eagle_accept(
        ctypes.byref(desc), _ptr(target_logits, FLOATS, "target_logits"), _ptr(draft_logits, FLOATS, "draft_logits"),
        _ptr(tree_tokens, torch.int32, "tree_tokens"), _ptr(tree_parent, torch.int32, "tree_parent"),
        _ptr(u_accept, torch.float32, "u_accept"), _ptr(u_final, torch.float32, "u_final"), ctypes.byref(o),
        _ptr(ws, name="ws"), ws.numel() * ws.element_size(), _stream(stream)))


def eagle_accept_noalloc(desc: AcceptDesc, target_logits, draft_logits, tree_tokens, tree_parent, u_accept,
                         u_final, out: AcceptBuffers, stream=None) -> None:
    """eagle_accept with the library's fixed device scratch instead of a workspace (see
    eagle.h: eagle_accept_noalloc)."""
    o = out.c_struct()
    _check("eagle_accept_noalloc", load().eagle_accept_noalloc(
        ctypes.byref(desc), _ptr(target_logits, FLOATS, "target_logits"), _ptr(draft_logits, FLOATS, "draft_logits"),
        _ptr(tree_tokens, torch.int32, "tree_tokens"), _ptr(tree_parent, torch.int32, "tree_parent"),
        _ptr(u_accept, torch.float32, "u_accept"), _ptr(u_final, torch.float32, "u_final"), ctypes.byref(o),
        _stream(stream)))


class LayerPointers:
    """HOST arrays of per-layer device pointers for eagle_kv_commit (built once, reused)."""

    def __init__(self, k_cache: Sequence[torch.Tensor], v_cache: Sequence[torch.Tensor],
                 tree_k: Sequence[torch.Tensor], tree_v: Sequence[torch.Tensor]):
        n = len(k_cache)
        mk = lambda ts, nm: (ctypes.c_void_p * n)(*[_ptr(t, FLOATS, nm) for t in ts])
        self.k, self.v = mk(k_cache, "k_cache"), mk(v_cache, "v_cache")
        self.tk, self.tv = mk(tree_k, "tree_k"), mk(tree_v, "tree_v")
        self.tensors = (list(k_cache), list(v_cache), list(tree_k), list(tree_v))


def eagle_kv_commit(desc: CommitDesc, layers: LayerPointers, n_acc, path, seq_len, commit_pos,
                    feat_cache=None, tree_feat=None, status=None, stream=None) -> None:
    """Commit the accepted path's K/V (see eagle.h: eagle_kv_commit)."""
    _check("eagle_kv_commit", load().eagle_kv_commit(
        ctypes.byref(desc), layers.k, layers.v, layers.tk, layers.tv, _ptr(n_acc, torch.int32, "n_acc"),
        _ptr(path, torch.int32, "path"), _ptr(seq_len, torch.int32, "seq_len"),
        _ptr(commit_pos, torch.int32, "commit_pos"), _ptr(feat_cache, FLOATS, "feat_cache"),
        _ptr(tree_feat, FLOATS, "tree_feat"), _ptr(status, torch.int32, "status"), _stream(stream)))


def version() -> str:
    return load().eagle_version().decode()


def selftest_ff_log(z_hi: torch.Tensor, z_lo: torch.Tensor):
    """The tree build's float-float logarithm on device values (see eagle.h:
    eagle_selftest_ff_log); returns (hi, lo) device tensors."""
    out_hi, out_lo = torch.empty_like(z_hi), torch.empty_like(z_lo)
    _check("eagle_selftest_ff_log", load().eagle_selftest_ff_log(
        _ptr(z_hi, torch.float32, "z_hi"), _ptr(z_lo, torch.float32, "z_lo"), _ptr(out_hi, torch.float32, "out_hi"),
        _ptr(out_lo, torch.float32, "out_lo"), z_hi.numel(), _stream(None)))
    return out_hi, out_lo


def eagle_lmhead_stats(desc: LmHeadDesc, hidden, weight, tree_tokens, tree_parent, records, child_logit, status,
                       stream=None) -> None:
    """Vocabulary statistics at every tree node from hidden states and the LM head (see
    eagle.h: eagle_lmhead_stats).  records: an int32 tensor [M][tiles][4] (max, argmax,
    sum_hi, sum_lo as 32-bit words)."""
    _check("eagle_lmhead_stats", load().eagle_lmhead_stats(
        ctypes.byref(desc), _ptr(hidden, torch.bfloat16, "hidden"), _ptr(weight, torch.bfloat16, "weight"),
        _ptr(tree_tokens, torch.int32, "tree_tokens"), _ptr(tree_parent, torch.int32, "tree_parent"),
        _ptr(records, torch.int32, "records"), _ptr(child_logit, torch.float32, "child_logit"),
        _ptr(status, torch.int32, "status"), _stream(stream)))


def eagle_ttt_attn(desc: TttDesc, q, k_trunk, v_trunk, k_branch, v_branch, out, lse: Optional[torch.Tensor],
                   ws: torch.Tensor, stream=None) -> None:
    """Training-time-test attention (see eagle.h: eagle_ttt_attn)."""
    _check("eagle_ttt_attn", load().eagle_ttt_attn(
        ctypes.byref(desc), _ptr(q, torch.bfloat16, "q"), _ptr(k_trunk, torch.bfloat16, "k_trunk"),
        _ptr(v_trunk, torch.bfloat16, "v_trunk"), _ptr(k_branch, torch.bfloat16, "k_branch"),
        _ptr(v_branch, torch.bfloat16, "v_branch"), _ptr(out, FLOATS, "out"), _ptr(lse, torch.float32, "lse"),
        _ptr(ws, name="ws"), ws.numel() * ws.element_size(), _stream(stream)))
