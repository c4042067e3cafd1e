"""GPU parity: eagle_tree_attn against the oracle's tree attention.

Small cases span several 64-key tiles with a ragged tail; the full-size cases use
the workloads' own shapes (prefix 2048 / 8192 / 131072, 61 or 8 tree rows, MHA and
GQA-4, ragged batches) in the launch configuration the benchmark uses, and check
whole KV heads against the oracle.  Tolerance: max abs error 2e-3 for bf16 inputs
(fp32 accumulation), plus the one rounding of a bf16 output (2^-8 |O|); 1e-5 for
fp32.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from eagle_speculative_decoding_tree_gb300 import binding as B
from eagle_speculative_decoding_tree_gb300 import synth
from gpu_helpers import BF16_TOL, F32_TOL, dev, head_slice, random_tree, run_attn

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS


def _refs(w, batch, seq_len, par, heads, inputs, n_nodes=None):
    """Oracle outputs (O, lse) of each checked (request, KV head), computed once per case."""
    G = w.group
    refs = {}
    for b, h in heads:
        sub = head_slice(inputs, h, G, b)
        n = sub[3].shape[2]
        if n_nodes is not None:  # request b's tree is its first n_nodes[b] rows
            n = int(n_nodes[b])
            q, kc, vc, tk, tv = sub
            sub = (np.ascontiguousarray(q[:, :n]), kc, vc, np.ascontiguousarray(tk[:, :, :n]),
                   np.ascontiguousarray(tv[:, :, :n]))
        refs[(b, h)] = (oracle.tree_attn(*sub, seq_len[b:b + 1], par[None, :n], 1.0 / np.sqrt(w.head_dim)), sub, n)
    return refs


def _compare(w, out, lse, refs, bound_fn, what):
    G = w.group
    tol = F32_TOL if w.dtype == "f32" else BF16_TOL
    worst = 0.0
    for (b, h), ((ref, ref_lse), sub, n) in refs.items():
        err = np.abs(out[b:b + 1, :n, h * G:(h + 1) * G] - ref)
        bound = bound_fn(ref, sub)
        assert (err <= bound).all(), (f"b={b} h={h} {what}: max abs error {err.max():.3e}, "
                                      f"worst excess {(err - bound).max():.3e}")
        worst = max(worst, float(err.max()))
        lerr = float(np.abs(lse[b:b + 1, :n, h * G:(h + 1) * G] - ref_lse).max())
        assert lerr < tol, f"b={b} h={h} {what}: lse max abs error {lerr}"
    return worst


def _check(w, batch, seq_len, rows, par, mask, heads, q_scale=1.0, num_splits=0, n_nodes=None):
    """Check one case against the oracle (the reference is computed once).

    fp32 inputs: max abs error < 1e-5.
    bf16 inputs (fp32 accumulation), four launches:
      * the benchmark's launch -- the tensor-core kernel where it applies, precise PV
        path (the default), bf16 output: max abs error <= 2e-3 + u |O|, where
        u = 2^-8 is the unit roundoff of the one rounding of O to bf16;
      * the same with fp32 output: max abs error < 2e-3;
      * the legacy warp-MMA kernel, precise, bf16 output: 2e-3 + u |O|;
      * the fast PV path (P rounded to bf16 once, an opt-in outside the stated bound):
        rounding P moves O by at most u/(1-u) * 2 max|v|, plus u |O| for the output.
    Returns the worst error of the benchmark's launch.
    """
    inputs = None
    runs = []
    if w.dtype == "f32":
        runs.append(("fp32", dict(out_f32=True), lambda ref, sub: F32_TOL))
    else:
        u = 2.0 ** -8

        def strict(ref, sub):
            return BF16_TOL + u * np.abs(ref)

        def fast(ref, sub):
            vmax = max(np.abs(synth.bf16_value(sub[2])).max(), np.abs(synth.bf16_value(sub[4])).max())
            return BF16_TOL + u / (1 - u) * 2 * vmax + u * np.abs(ref)

        runs += [("bench launch (auto engine, precise, bf16 out)", dict(), strict),
                 ("precise, fp32 out", dict(out_f32=True), lambda ref, sub: BF16_TOL),
                 ("mma.sync engine, precise, bf16 out", dict(engine=B.EAGLE_ENGINE_MMA_SYNC), strict),
                 ("fast P, bf16 out", dict(precision=B.EAGLE_ATTN_FAST), fast)]
    refs = None
    first = None
    for what, kw, bound_fn in runs:
        inputs, out, lse = run_attn(w, batch, seq_len, rows, par, mask, q_scale=q_scale, num_splits=num_splits,
                                    n_nodes=n_nodes, **kw)
        if refs is None:
            refs = _refs(w, batch, seq_len, par, heads, inputs, n_nodes)
        worst = _compare(w, out, lse, refs, bound_fn, what)
        if first is None:
            first = worst
    return first


@pytest.mark.parametrize("name,kw,prefix,rows,q_scale,splits", [
    ("tiny-f32", {}, 128, 11, 1.0, 0),
    ("tiny-f32-long", dict(prefix=700, prefix_min=700), 700, 11, 1.0, 0),
    ("mha-bf16-ragged", dict(prefix=1000, prefix_min=1000), 1000, 61, 1.0, 0),
    ("gqa-bf16", dict(prefix=777, prefix_min=777), 777, 61, 1.0, 0),
    ("gqa-bf16-forced-splits", dict(prefix=1500, prefix_min=1500), 1500, 61, 1.0, 7),
    ("gqa-bf16-20-splits", dict(prefix=3000, prefix_min=3000), 3000, 61, 1.0, 20),
    ("gqa-bf16-one-split", dict(prefix=300, prefix_min=300), 300, 61, 1.0, 1),
    ("gqa-bf16-128rows", dict(prefix=200, prefix_min=200), 200, 128, 1.0, 0),
    ("gqa-bf16-65rows", dict(prefix=129, prefix_min=129), 129, 65, 1.0, 0),
    ("chain-bf16", dict(prefix=3000, prefix_min=3000), 3000, 8, 1.0, 0),
    ("empty-prefix", dict(prefix=64, prefix_min=64), 0, 61, 1.0, 0),
])
def test_tree_attention_small(name, kw, prefix, rows, q_scale, splits):
    base = {"tiny-f32": "tiny", "tiny-f32-long": "tiny", "mha-bf16-ragged": "vicuna7b",
            "chain-bf16": "long128k"}.get(name, "llama8b")
    w = W[base].with_(**kw) if kw else W[base]
    par, mask = random_tree(rows, seed=len(name), chain=(base == "long128k"))
    seq_len = np.array([prefix], np.int32)
    heads = [(0, 0), (0, w.n_kv_heads - 1)]
    _check(w, 1, seq_len, rows, par, mask, heads, q_scale, splits)


@pytest.mark.parametrize("head_dim", [128, 64])
def test_tree_attention_peaked_rows(head_dim):
    """Q scaled by 4: sharply peaked softmax rows that exercise the online rescaling."""
    w = W["llama8b"].with_(prefix=500, prefix_min=500, head_dim=head_dim)
    par, mask = random_tree(61, seed=9)
    _check(w, 1, np.array([500], np.int32), 61, par, mask, [(0, 0), (0, 3), (0, 7)], q_scale=4.0)


def test_tree_attention_head_dim_64():
    w = W["llama8b"].with_(head_dim=64, prefix=333, prefix_min=333)
    par, mask = random_tree(61, seed=64)
    _check(w, 1, np.array([333], np.int32), 61, par, mask, [(0, 0), (0, 7)])


def test_tree_attention_ragged_batch():
    w = W["concurrency"].with_(prefix=1500, prefix_min=20, batch=5)
    seq_len = synth.prefix_lengths(w, 5)
    seq_len[2] = 0
    par, mask = random_tree(61, seed=5)
    _check(w, 5, seq_len, 61, par, mask, [(b, b % 8) for b in range(5)])


def test_tree_attention_ragged_fixed_splits():
    """More (request, KV head, row block) groups than SMs: fixed-size key splits of 32
    tiles per CTA, requests dispatched longest first, one request with no prefix."""
    w = W["concurrency"].with_(prefix=5000, prefix_min=1, batch=10)
    seq_len = synth.prefix_lengths(w, 10)
    seq_len[3] = 0
    seq_len[6] = 5000
    par, mask = random_tree(61, seed=17)
    _check(w, 10, seq_len, 61, par, mask, [(0, 1), (3, 5), (6, 7), (9, 0)])


@pytest.mark.parametrize("name", ["vicuna7b", "llama8b", "long128k"])
def test_tree_attention_full_size(name):
    """The benchmark's shapes and launch configuration; whole KV heads checked."""
    w = W[name]
    rows = w.rows
    par, mask = random_tree(rows, seed=11, chain=(name == "long128k"))
    seq_len = synth.prefix_lengths(w, 1)
    heads = [(0, 0)] if name == "long128k" else [(0, 0), (0, w.n_kv_heads - 1)]
    _check(w, 1, seq_len, rows, par, mask, heads)


def test_tree_attention_full_size_concurrency_batch8():
    w = W["concurrency"].with_(batch=8)
    seq_len = synth.prefix_lengths(w, 8)
    par, mask = random_tree(w.rows, seed=12)
    _check(w, 8, seq_len, w.rows, par, mask, [(0, 0), (7, 7), (3, 2)])


def test_tree_attention_full_size_concurrency_batch32():
    """The batch-32 benchmark shape: 64-tile key pieces, longest requests first; the
    longest and shortest requests among the checked heads."""
    w = W["concurrency"].with_(batch=32)
    seq_len = synth.prefix_lengths(w, 32)
    par, mask = random_tree(w.rows, seed=13)
    heads = [(0, 0), (31, 7), (int(np.argmax(seq_len)), 3), (int(np.argmin(seq_len)), 5)]
    _check(w, 32, seq_len, w.rows, par, mask, heads)


@pytest.mark.gpu
def test_tree_attention_workspace_reuse():
    """Calls on one workspace: identical outputs, group counters back at zero, no timeouts."""
    w = W["llama8b"]
    rows = w.rows
    par, mask = random_tree(rows, seed=21)
    seq_len = synth.prefix_lengths(w, 1)
    q, kc, vc, tk, tv = synth.attn_tensors(w, 0, 1, seq_len, rows, 1.0)
    desc = B.AttnDesc(1, rows, w.n_q_heads, w.n_kv_heads, w.head_dim, w.max_seq, 1.0 / math.sqrt(w.head_dim),
                      B.EAGLE_BF16, 0, B.EAGLE_BF16, B.EAGLE_ATTN_PRECISE, B.EAGLE_ENGINE_AUTO)
    splits, kernels = B.tree_attn_plan(desc)
    ws = torch.zeros(B.workspace_size(B.EAGLE_WS_TREE_ATTN, desc), dtype=torch.uint8, device="cuda")
    args = [dev(x, w.dtype) for x in (q, kc, vc, tk, tv)]
    sl = torch.from_numpy(np.asarray(seq_len, np.int32)).cuda()
    am = torch.from_numpy(np.ascontiguousarray(mask).view(np.int64)).cuda().reshape(1, rows, -1)
    outs = []
    for _ in range(3):
        out = torch.empty_like(args[0])
        lse = torch.empty(1, rows, w.n_q_heads, dtype=torch.float32, device="cuda")
        B.eagle_tree_attn(desc, *args, sl, am, out, lse, ws)
        torch.cuda.synchronize()
        outs.append((out.clone(), lse.clone()))
    for o, l in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(l, outs[0][1])
    assert int(ws[:4].view(torch.int32).item()) == 0
    if kernels == 1 and splits > 1:  # merged in the kernel: counters live after the error word
        assert int(ws[256:512].count_nonzero().item()) == 0


def test_tree_attention_ragged_tree_sizes():
    """Requests whose trees differ in size share one call (n_nodes): rows past a
    request's tree stay untouched and keys past it are ignored, even where mask bits
    are set."""
    w = W["concurrency"].with_(prefix=900, prefix_min=300, batch=4)
    seq_len = synth.prefix_lengths(w, 4)
    rows = 61
    par, mask = random_tree(rows, seed=23)
    n_nodes = np.array([61, 17, 1, 40], np.int32)
    inputs, out, lse = run_attn(w, 4, seq_len, rows, par, mask, n_nodes=n_nodes)
    refs = _refs(w, 4, seq_len, par, [(0, 0), (1, 3), (2, 5), (3, 7)], inputs, n_nodes)
    u = 2.0 ** -8
    _compare(w, out, lse, refs, lambda ref, sub: BF16_TOL + u * np.abs(ref), "ragged n_nodes")
    for b, n in enumerate(n_nodes):  # rows past the tree were not written (the buffer held NaN)
        assert np.isnan(out[b, n:]).all(), b

    # every mask bit set and 5 rows per request: row i must see the prefix and tree
    # keys 0..4 only -- the attention of the last row of a 5-node chain whose last
    # query is row i's
    ones = np.full_like(mask, ~np.uint64(0))
    inputs, out, lse = run_attn(w, 4, seq_len, rows, par, ones, n_nodes=np.full(4, 5, np.int32))
    assert np.isnan(out[:, 5:]).all()
    q, kc, vc, tk, tv = inputs
    G, h = w.group, 2
    chain = np.array([[-1, 0, 1, 2, 3]], np.int32)
    for b in range(4):
        for i in range(5):
            qi = np.repeat(q[b:b + 1, i:i + 1, h * G:(h + 1) * G], 5, axis=1)
            ref, _ = oracle.tree_attn(qi, kc[b:b + 1, h:h + 1], vc[b:b + 1, h:h + 1],
                                      np.ascontiguousarray(tk[b:b + 1, h:h + 1, :5]),
                                      np.ascontiguousarray(tv[b:b + 1, h:h + 1, :5]), seq_len[b:b + 1], chain,
                                      1.0 / np.sqrt(w.head_dim))
            got = out[b, i, h * G:(h + 1) * G]
            assert (np.abs(got - ref[0, 4]) <= BF16_TOL + u * np.abs(ref[0, 4])).all(), (b, i)


def test_tree_attention_group_wait_gives_up():
    """The in-kernel split merge's bounded wait, driven to its limit through the test
    hook: every group waits for a split that never comes, gives up after 1 ms and sets
    bit 0x100 of the error word; the group counters return to zero, TMEM is released
    (the next launches allocate it again), and on a re-zeroed workspace the same call
    is correct."""
    w = W["llama8b"]
    rows = w.rows
    par, mask = random_tree(rows, seed=31)
    seq_len = synth.prefix_lengths(w, 1)
    desc = B.AttnDesc(1, rows, w.n_q_heads, w.n_kv_heads, w.head_dim, w.max_seq, 1.0 / math.sqrt(w.head_dim),
                      B.EAGLE_BF16, 0, B.EAGLE_BF16, B.EAGLE_ATTN_PRECISE, B.EAGLE_ENGINE_AUTO, 1)
    splits, kernels = B.tree_attn_plan(desc)
    assert splits > 1 and kernels == 1, "the llama8b shape merges its splits in the kernel"
    ws = torch.zeros(B.workspace_size(B.EAGLE_WS_TREE_ATTN, desc), dtype=torch.uint8, device="cuda")
    for _ in range(2):  # twice: the first failure must leave the device usable
        run_attn(w, 1, seq_len, rows, par, mask, fault_test=1, ws=ws)
        err = int(ws[:4].view(torch.int32).item())
        assert err & 0x100, f"error word {err:#x}: the group wait did not give up"
        assert err & ~0x100 == 0, f"error word {err:#x}: another wait gave up"
        assert int(ws[256:512].count_nonzero().item()) == 0, "group counters not returned to zero"
        ws.zero_()
    inputs, out, lse = run_attn(w, 1, seq_len, rows, par, mask, ws=ws)
    assert int(ws[:4].view(torch.int32).item()) == 0
    refs = _refs(w, 1, seq_len, par, [(0, 0), (0, 7)], inputs)
    u = 2.0 ** -8
    _compare(w, out, lse, refs, lambda ref, sub: BF16_TOL + u * np.abs(ref), "after the failure test")
