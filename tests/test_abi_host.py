"""The C-ABI library on the host (no GPU needed): it builds, loads, exports every
function include/eagle.h declares, and rejects bad arguments before launching.

No test here makes a call that would pass validation: with no GPU such a call
could only fail at launch, and on a GPU machine fake pointers must never reach a
kernel.  Pointers below are aligned or misaligned integers that the library
only inspects on the host.
"""
import ctypes
import os
import re
import subprocess

import pytest

from eagle_speculative_decoding_tree_gb300 import binding as B
from eagle_speculative_decoding_tree_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "eagle.h")
A = 0x100000  # an aligned fake device address (never dereferenced: every call below fails validation)


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return B.load()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(eagle_[a-z_]+)\s*\(", text)))


def test_library_exports_every_declared_function(lib):
    names = _declared()
    assert {"eagle_tree_build", "eagle_tree_attn", "eagle_accept", "eagle_kv_commit"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", build_mod.LIB], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (eagle_\w+)", out))
    assert set(names) <= exported, set(names) - exported
    assert set(B.EXPORTED_SYMBOLS) == set(names)


def test_status_strings_and_version(lib):
    for code in range(6):
        assert B.load().eagle_status_string(code).startswith(b"EAGLE_")
    assert b"sm_103a" in lib.eagle_version()


def _attn(**kw):
    d = dict(batch=1, rows=61, n_q_heads=32, n_kv_heads=8, head_dim=128, max_seq=8256, scale=0.088, dtype=1,
             num_splits=0, out_dtype=1, precision=0)
    d.update(kw)
    return B.AttnDesc(**d)


def _call_attn(lib, desc, q=A, ws=A, ws_bytes=0, lse=None):
    return lib.eagle_tree_attn(ctypes.byref(desc), q, A, A, A, A, A, None, A, A, lse, ws, ws_bytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(head_dim=96), B.EAGLE_ERR_UNSUPPORTED),
    (dict(n_q_heads=12, n_kv_heads=8), B.EAGLE_ERR_UNSUPPORTED),
    (dict(rows=129), B.EAGLE_ERR_UNSUPPORTED),
    (dict(dtype=7), B.EAGLE_ERR_UNSUPPORTED),
    (dict(batch=0), B.EAGLE_ERR_INVALID_ARG),
    (dict(scale=0.0), B.EAGLE_ERR_INVALID_ARG),
    (dict(num_splits=-1), B.EAGLE_ERR_INVALID_ARG),
    (dict(dtype=0, out_dtype=1), B.EAGLE_ERR_UNSUPPORTED),
    (dict(precision=2), B.EAGLE_ERR_INVALID_ARG),
    (dict(fault_test=2), B.EAGLE_ERR_INVALID_ARG),
])
def test_attn_rejects_bad_descriptors(lib, kw, code):
    assert _call_attn(lib, _attn(**kw)) == code


def test_attn_rejects_null_misaligned_and_small_workspace(lib):
    d = _attn()
    assert _call_attn(lib, d, q=None) == B.EAGLE_ERR_INVALID_ARG
    assert _call_attn(lib, d, q=A + 2) == B.EAGLE_ERR_ALIGNMENT
    need = B.workspace_size(B.EAGLE_WS_TREE_ATTN, d)
    assert need > 16  # split partials
    assert _call_attn(lib, d, ws=A, ws_bytes=need - 1) == B.EAGLE_ERR_WORKSPACE
    assert _call_attn(lib, d, ws=None, ws_bytes=0) == B.EAGLE_ERR_WORKSPACE


def _acc(**kw):
    d = dict(batch=1, rows=61, vocab=128256, temperature=1.0, proposal=0, dtype=1, max_depth=7)
    d.update(kw)
    return B.AcceptDesc(**d)


def _call_acc(lib, desc, draft=None, ws_bytes=0, out_ok=True):
    o = B.AcceptOut(A, A, A, A, A) if out_ok else B.AcceptOut(A, None, A, A, A)
    return lib.eagle_accept(ctypes.byref(desc), A, draft, A, A, A, A, ctypes.byref(o), A, ws_bytes, None)


def test_accept_validation(lib):
    assert _call_acc(lib, _acc(temperature=-1.0)) == B.EAGLE_ERR_INVALID_ARG
    assert _call_acc(lib, _acc(temperature=float("nan"))) == B.EAGLE_ERR_INVALID_ARG
    assert _call_acc(lib, _acc(proposal=1)) == B.EAGLE_ERR_INVALID_ARG  # sampled needs draft logits
    assert _call_acc(lib, _acc(proposal=5)) == B.EAGLE_ERR_INVALID_ARG
    assert _call_acc(lib, _acc(rows=200)) == B.EAGLE_ERR_UNSUPPORTED
    assert _call_acc(lib, _acc(), out_ok=False) == B.EAGLE_ERR_INVALID_ARG
    d = _acc()
    need = B.workspace_size(B.EAGLE_WS_ACCEPT, d)
    # 256 bytes of per-request barrier counters, then one 24-byte record per (row,
    # 4096-token chunk): the larger of the two launch forms' record areas
    assert need == 256 + 61 * 32 * 24
    assert _call_acc(lib, d, ws_bytes=need - 1) == B.EAGLE_ERR_WORKSPACE
    ds = _acc(proposal=1)
    assert B.workspace_size(B.EAGLE_WS_ACCEPT, ds) == 256 + 2 * 61 * 32 * 24  # target and draft records


def _call_build(lib, desc, level=1, ws_bytes=0, u=None):
    o = B.TreeOut(*([A] * 9))
    return lib.eagle_tree_build(ctypes.byref(desc), level, A, u, A, A, A, ws_bytes, ctypes.byref(o), None)


def test_tree_build_validation(lib):
    dyn = lambda **kw: B.tree_desc(**{**dict(batch=1, vocab=128256, mode=B.EAGLE_TREE_DYNAMIC, depth=7, top_k=8,
                                              total_tokens=60), **kw})
    assert _call_build(lib, dyn(), level=0) == B.EAGLE_ERR_INVALID_ARG
    assert _call_build(lib, dyn(), level=8) == B.EAGLE_ERR_INVALID_ARG
    assert _call_build(lib, dyn(top_k=17)) == B.EAGLE_ERR_UNSUPPORTED
    assert _call_build(lib, dyn(total_tokens=128)) == B.EAGLE_ERR_UNSUPPORTED
    assert _call_build(lib, dyn(depth=2, top_k=3, total_tokens=13)) == B.EAGLE_ERR_INVALID_ARG  # pool is 12
    assert _call_build(lib, dyn(top_k=16, depth=10)) == B.EAGLE_ERR_UNSUPPORTED  # pool > 2048
    assert B.workspace_size(B.EAGLE_WS_TREE_BUILD, dyn(vocab=128 * 4096)) > 0  # largest vocabulary
    assert _call_build(lib, dyn(vocab=128 * 4096 + 1)) == B.EAGLE_ERR_UNSUPPORTED
    need = B.workspace_size(B.EAGLE_WS_TREE_BUILD, dyn())
    assert need > 0
    assert _call_build(lib, dyn(), ws_bytes=need - 1) == B.EAGLE_ERR_WORKSPACE
    st = lambda par, **kw: B.tree_desc(**{**dict(batch=1, vocab=1000, mode=B.EAGLE_TREE_STATIC_SAMPLED, depth=3,
                                                 static_parent=par), **kw})
    assert _call_build(lib, st([-1, 0, 0, 1]), u=None) == B.EAGLE_ERR_INVALID_ARG  # sampled needs u_draft
    assert _call_build(lib, st([-1, 0, 2, 1]), u=A) == B.EAGLE_ERR_INVALID_ARG  # parent not earlier
    assert _call_build(lib, st([-1, 0, 1, 0]), u=A) == B.EAGLE_ERR_INVALID_ARG  # not ordered by depth
    assert _call_build(lib, st([-1] + [0] * 17), u=A) == B.EAGLE_ERR_UNSUPPORTED  # 17 children
    assert _call_build(lib, st([-1, 0, 1], temperature=0.0), u=A) == B.EAGLE_ERR_INVALID_ARG


def _call_build_head(lib, desc, level=1, hidden_dim=4096, ws_bytes=1 << 40, status=A):
    o = B.TreeOut(*([A] * 9))
    lib.eagle_tree_build_head.argtypes = [ctypes.POINTER(B.TreeDesc), ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                          ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                          ctypes.c_size_t, ctypes.POINTER(B.TreeOut), ctypes.c_void_p, ctypes.c_void_p]
    return lib.eagle_tree_build_head(ctypes.byref(desc), level, A, A, hidden_dim, A, A, A, ws_bytes, ctypes.byref(o),
                                     status, None)


def test_tree_build_head_validation(lib):
    dyn = lambda **kw: B.tree_desc(**{**dict(batch=1, vocab=128256, mode=B.EAGLE_TREE_DYNAMIC, depth=7, top_k=8,
                                              total_tokens=60), **kw})
    assert _call_build_head(lib, dyn(), level=0) == B.EAGLE_ERR_INVALID_ARG
    assert _call_build_head(lib, dyn(), hidden_dim=0) == B.EAGLE_ERR_INVALID_ARG
    assert _call_build_head(lib, dyn(), hidden_dim=96) == B.EAGLE_ERR_UNSUPPORTED  # not a multiple of 64
    assert _call_build_head(lib, dyn(batch=17)) == B.EAGLE_ERR_UNSUPPORTED  # 17 x 8 rows > 128
    assert _call_build_head(lib, dyn(), status=None) == B.EAGLE_ERR_INVALID_ARG
    need = B.workspace_size(B.EAGLE_WS_TREE_BUILD, dyn())
    assert _call_build_head(lib, dyn(), ws_bytes=need - 1) == B.EAGLE_ERR_WORKSPACE
    sampled = B.tree_desc(1, 1000, B.EAGLE_TREE_STATIC_SAMPLED, 3, static_parent=[-1, 0, 0, 1], temperature=1.0)
    assert _call_build_head(lib, sampled) == B.EAGLE_ERR_UNSUPPORTED  # draws read the logits


def test_tree_frontier_rows(lib):
    d = B.tree_desc(1, 1000, B.EAGLE_TREE_STATIC_SAMPLED, 3, static_parent=[-1, 0, 0, 0, 0, 1, 1, 2, 3, 5, 5])
    assert [B.tree_frontier_rows(d, l) for l in (1, 2, 3)] == [1, 4, 4]
    assert B.tree_frontier_rows(d, 4) == -1
    assert B.tree_max_frontier(d) == 4
    dd = B.tree_desc(2, 32000, B.EAGLE_TREE_DYNAMIC, 6, 10, 60)
    assert [B.tree_frontier_rows(dd, l) for l in (1, 2, 6)] == [1, 10, 10]


def test_kv_commit_validation(lib):
    arr = (ctypes.c_void_p * 2)(A, A)
    bad = (ctypes.c_void_p * 2)(A, None)
    mis = (ctypes.c_void_p * 2)(A, A + 8)
    d = lambda **kw: B.CommitDesc(**{**dict(layers=2, batch=1, n_kv_heads=8, head_dim=128, rows=61, max_seq=8256,
                                            max_depth=7, dtype=1, feat_dim=0, feat_dtype=1), **kw})
    call = lambda desc, k=arr: lib.eagle_kv_commit(ctypes.byref(desc), k, arr, arr, arr, A, A, A, A, None, None,
                                                    A, None)
    assert call(d(layers=0)) == B.EAGLE_ERR_INVALID_ARG
    assert call(d(layers=129)) == B.EAGLE_ERR_UNSUPPORTED
    assert call(d(head_dim=12)) == B.EAGLE_ERR_UNSUPPORTED  # 24-byte rows
    assert call(d(), k=bad) == B.EAGLE_ERR_INVALID_ARG
    assert call(d(), k=mis) == B.EAGLE_ERR_ALIGNMENT
    assert call(d(feat_dim=64)) == B.EAGLE_ERR_INVALID_ARG  # feature rows requested without buffers


def test_workspace_size_zero_on_bad_desc(lib):
    assert B.workspace_size(B.EAGLE_WS_TREE_ATTN, _attn(head_dim=80)) == 0
    assert B.workspace_size(99, _attn()) == 0


def test_binding_refuses_cpu_tensors(lib):
    import torch
    d = _attn(rows=2, n_q_heads=1, n_kv_heads=1, head_dim=64, max_seq=4)
    x = torch.zeros(1, 2, 1, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        B.eagle_tree_attn(d, x, x, x, x, x, torch.zeros(1, dtype=torch.int32), torch.zeros(1, 2, 1, dtype=torch.int64),
                          x, None, None)


@pytest.mark.parametrize("kw,splits,kernels", [
    (dict(), 9, 1),                                                       # llama8b: 16 groups x 9 splits, one wave
    (dict(n_kv_heads=32, max_seq=2048 + 61), 4, 1),                       # vicuna7b (MHA): 32 groups x 4
    (dict(rows=8, max_seq=131072 + 8), 19, 1),                            # long128k chain: 8 groups x 19
    (dict(batch=8, max_seq=16384), 5, 2),                                 # 128 groups: 32-tile splits + combine
    (dict(batch=32, max_seq=16384), 3, 2),                                # 512 groups: 64-tile splits + combine
    (dict(batch=16, max_seq=1 << 20), 64, 2),                            # 1M-token cache: 129-tile pieces
    (dict(num_splits=7), 7, 1),                                           # forced, still one wave
    (dict(num_splits=20), 20, 2),                                         # forced past one wave
    (dict(dtype=0, out_dtype=0, head_dim=64), 1, 1),                      # fp32: one kernel, no splits
])
def test_attention_launch_plan(lib, kw, splits, kernels):
    """The plan the attention kernels get on 152 SMs (this host has no GPU, so the library
    plans for a GB300's count): even splits merged in the kernel while the grid fits one wave;
    for batched requests, fixed-size key splits merged by a second kernel."""
    assert B.tree_attn_plan(_attn(**kw)) == (splits, kernels)
