"""GPU parity of whole verify steps, chained: tree build -> tree attention over L
layers -> acceptance -> commit -> next step from the emitted token.

The GPU chain and the oracle chain run side by side for 20 steps: trees, accepted
paths and emitted tokens must agree exactly, attention within the bf16 / fp32
tolerance, and the committed caches byte for byte (they grow by n_acc + 1 rows per
step).  A step in which either side reports a near-tie is counted and its
comparisons from that decision on are skipped; both chains then continue from the
oracle's decisions (its tree, its accepted path committed on both sides), so the
chain keeps going and every later step is compared again.  At most 2 of the 20
steps may hit a near-tie.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from eagle_speculative_decoding_tree_gb300 import binding as B
from eagle_speculative_decoding_tree_gb300 import synth
from eagle_speculative_decoding_tree_gb300.step import GpuTreeBuilder
from conftest import record_near_ties
from gpu_helpers import BF16_TOL, F32_TOL, dev
from spec_helpers import OracleDynamicBuilder, OracleStaticBuilder, node_hashes

pytestmark = pytest.mark.gpu

STEPS = 20


def _bytes_of(t, dtype):
    return t.view(torch.int16).cpu().numpy().view(np.uint16) if dtype == "bf16" else t.cpu().numpy()


@pytest.mark.parametrize("name,kw,batch,layers", [
    ("tiny", dict(prefix=128, prefix_min=128), 1, 2),
    ("llama8b", dict(vocab=8192, prefix=300, prefix_min=300), 2, 2),
    ("vicuna7b", dict(vocab=4096, prefix=200, prefix_min=200, temperature=0.0), 1, 2),
    ("llama8b", dict(prefix=1000, prefix_min=1000), 1, 1),  # the full 128256-token vocabulary
])
def test_chained_verify_steps(name, kw, batch, layers):
    w = synth.WORKLOADS[name].with_(**kw)
    cap = w.with_(prefix=w.prefix + 8 * STEPS + 64)  # cache capacity for the whole chain
    P = cap.max_seq
    R = w.rows
    dt = B.EAGLE_F32 if w.dtype == "f32" else B.EAGLE_BF16
    lm = synth.hash_lm(w)
    seq_len = synth.prefix_lengths(w, batch)
    root_tok = synth.root_tokens(w, batch)
    root_h = [synth.root_hash(w.config_id, b, 9) for b in range(batch)]
    # persistent caches: GPU tensors and the oracle's host copies
    caches = [synth.attn_tensors(cap, l, batch, seq_len, R)[1:3] for l in range(layers)]
    host_k = np.stack([c[0] for c in caches])
    host_v = np.stack([c[1] for c in caches])
    gk = [dev(host_k[l], w.dtype) for l in range(layers)]
    gv = [dev(host_v[l], w.dtype) for l in range(layers)]
    proposal = oracle.SAMPLED if w.proposal == "sampled" else oracle.DELTA
    steps_done, near_steps = 0, 0
    for s in range(STEPS):
        # ---- tree build (GPU and oracle on the same draft rows)
        gb = GpuTreeBuilder(w, batch)
        gb.set_context(root_tok, seq_len)
        if w.tree_mode == "dynamic":
            ob = OracleDynamicBuilder(batch, w.vocab, w.depth, w.top_k, w.total_tokens)
        else:
            ob = OracleStaticBuilder(batch, w.vocab, synth.static_parents(w.static_choices), True, w.temperature)
        ua, uf, ud = synth.step_uniforms(w, batch, R, step=s + 1)
        front = [[h] for h in root_h]
        near = False  # a near-tie in this step: later comparisons of the step are skipped
        for level in range(1, gb.depth + 1):
            rows = synth.as_dtype_bytes(np.stack([lm.rows(front[b], "draft") for b in range(batch)]), w.dtype)
            gt, gs = gb.expand(level, rows, ud)
            ot, os_ = ob.expand(level, rows, ud)
            near |= bool((ob.t.near_tie > 0).any())
            if not near:
                assert np.array_equal(gt, ot) and np.array_equal(gs, os_), (s, level)
            # both builders go on with the oracle's frontier rows
            front = [[synth.child_hash(front[b][int(os_[b, j])], int(ot[b, j])) for j in range(ot.shape[1])]
                     for b in range(batch)]
        tg, to = gb.finalize(root_tok, seq_len), ob.finalize(root_tok, seq_len)
        near |= bool((to["near_tie"] > 0).any() or (tg["near_tie"] > 0).any())
        for key in ("tokens", "parent", "anc_mask", "pos_id") if not near else ():
            assert np.array_equal(tg[key], to[key]), (s, key)
        tree = to
        # ---- tree attention, every layer
        sl_dev = torch.from_numpy(seq_len.copy()).cuda()
        am = torch.from_numpy(tree["anc_mask"].view(np.int64).copy()).cuda()
        desc = B.AttnDesc(batch, R, w.n_q_heads, w.n_kv_heads, w.head_dim, P, 1.0 / math.sqrt(w.head_dim), dt, 0, dt,
                          0)
        ws = torch.zeros(B.workspace_size(B.EAGLE_WS_TREE_ATTN, desc), dtype=torch.uint8, device="cuda")
        tks, tvs = [], []
        for l in range(layers):
            q, _, _, tk, tv = synth.attn_tensors(w.with_(prefix=1, prefix_min=1), 1000 * (s + 1) + l, batch,
                                                 np.ones(batch, np.int32), R)
            tks.append(tk)
            tvs.append(tv)
            out = torch.empty(q.shape, dtype=torch.float32 if w.dtype == "f32" else torch.bfloat16, device="cuda")
            B.eagle_tree_attn(desc, dev(q, w.dtype), gk[l], gv[l], dev(tk, w.dtype), dev(tv, w.dtype), sl_dev, am, out,
                              None, ws)
            torch.cuda.synchronize()
            ref, _ = oracle.tree_attn(q, host_k[l], host_v[l], tk, tv, seq_len, tree["parent"],
                                      1.0 / math.sqrt(w.head_dim))
            err = np.abs(out.float().cpu().numpy() - ref)
            # bf16 output: the 2e-3 bound plus one bf16 rounding of O (u = 2^-8)
            bound = F32_TOL if w.dtype == "f32" else BF16_TOL + 2.0 ** -8 * np.abs(ref)
            assert (err <= bound).all(), (s, l, float(err.max()))
        # ---- acceptance
        hs = node_hashes(tree, root_h)
        target = synth.as_dtype_bytes(np.stack([lm.rows(hs[b], "target") for b in range(batch)]), w.dtype)
        draft = synth.as_dtype_bytes(np.stack([lm.rows(hs[b], "draft") for b in range(batch)]), w.dtype) \
            if proposal == oracle.SAMPLED else None
        max_depth = int(tree["depth"].max())
        r = oracle.accept(target, tree["tokens"], tree["parent"], ua, uf, w.temperature, proposal, max_depth + 1,
                          draft=draft)
        adesc = B.AcceptDesc(batch, R, w.vocab, float(w.temperature), proposal, dt, max_depth)
        aws = torch.zeros(B.workspace_size(B.EAGLE_WS_ACCEPT, adesc), dtype=torch.uint8, device="cuda")
        acc = B.AcceptBuffers.allocate(batch, max_depth)
        i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()
        B.eagle_accept(adesc, dev(target, w.dtype), None if draft is None else dev(draft, w.dtype),
                       i32(tree["tokens"]), i32(tree["parent"]), torch.from_numpy(ua).cuda(),
                       torch.from_numpy(uf).cuda(), acc, aws)
        torch.cuda.synchronize()
        near |= bool((r["near_tie"] > 0).any() or (acc.near_tie.cpu().numpy() > 0).any())
        if not near:
            for key in ("n_acc", "path", "out_tok"):
                assert np.array_equal(getattr(acc, key).cpu().numpy(), r[key]), (s, key)
        # the GPU commits the oracle's decisions (identical unless a near-tie intervened)
        n_acc_dev, path_dev = i32(r["n_acc"]), i32(r["path"])
        # ---- commit (GPU into its caches, oracle into the host copies)
        tkd = [dev(t, w.dtype) for t in tks]
        tvd = [dev(t, w.dtype) for t in tvs]
        cdesc = B.CommitDesc(layers, batch, w.n_kv_heads, w.head_dim, R, P, max_depth, dt, 0, dt)
        pos = torch.zeros(batch, max_depth + 1, dtype=torch.int32, device="cuda")
        B.eagle_kv_commit(cdesc, B.LayerPointers(gk, gv, tkd, tvd), n_acc_dev, path_dev, sl_dev, pos,
                          status=acc.status)
        torch.cuda.synchronize()
        new_len, ref_pos = oracle.kv_commit(host_k, host_v, np.stack(tks), np.stack(tvs), r["n_acc"], r["path"],
                                            seq_len)
        assert np.array_equal(sl_dev.cpu().numpy(), new_len) and np.array_equal(pos.cpu().numpy(), ref_pos)
        for l in range(layers):
            assert _bytes_of(gk[l], w.dtype).tobytes() == host_k[l].tobytes(), (s, l)
            assert _bytes_of(gv[l], w.dtype).tobytes() == host_v[l].tobytes(), (s, l)
        assert int(acc.status.cpu()[0]) == 0
        # ---- next step: the emitted token is the new root
        for b in range(batch):
            na = int(r["n_acc"][b])
            emitted = int(r["out_tok"][b, na])
            root_h[b] = synth.child_hash(hs[b][int(r["path"][b, na])], emitted)
            root_tok[b] = emitted
        seq_len = new_len
        steps_done += 1
        near_steps += int(near)
    record_near_ties(f"chained steps {name} V={w.vocab}", near_steps, steps_done)
    assert steps_done == STEPS
    assert near_steps <= 2, f"{near_steps} of {STEPS} steps hit a near-tie"
