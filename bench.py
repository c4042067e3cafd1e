"""Benchmark: EAGLE draft-tree verify steps per second on one GB300 (or N replicas).

A step is one pass of the verify hot path over one batch: tree attention for
every layer, acceptance, KV commit (eagle_tree_attn x L, eagle_accept,
eagle_kv_commit), captured in one CUDA graph and replayed.  The default workload
is the LLaMA-3.1-8B-shaped one at 8K context (32 q / 8 kv heads x 128, vocab
128256, 61-row dynamic tree, 32 layers); --config picks another.

Output: one JSON line (rank 0).  `value` is whole-job verify steps/s with inputs
resident in HBM; `e2e` is the same metric through the C ABI with the step's
inputs copied from pinned host memory and its result read back inside the timed
region; `roofline` rates the tree-attention launch against the measured HBM
bandwidth; `cpu_baseline` times the CPU oracle on every host core.

--impl reference times the CPU oracle itself (as it stands, on every host core) on
the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import tempfile
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")
ATTN_SRCS = [os.path.join(ROOT, "eagle_speculative_decoding_tree_gb300", "csrc", f)
             for f in ("tree_attn_tc.cu", "sm100.cuh")]
L2_BYTES = 129 * 1024 * 1024


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            m = json.load(f)
        return float(m["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(value: float, world_size: int, device: str = "cpu") -> float:
    """Max of a per-rank value over all ranks of the current process group."""
    if world_size <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world_size: int, steps: int, ms: float) -> float:
    """Whole-job steps/s: every rank runs `steps` steps of its own replica in `ms` (max over ranks)."""
    return world_size * steps / (ms / 1e3)


def _workload_desc(w, batch):
    return {"workload": f"{w.name}: {w.n_q_heads}q/{w.n_kv_heads}kv x {w.head_dim} {w.dtype}, vocab {w.vocab}, "
                        f"prefix {w.prefix_min if w.prefix_min != w.prefix else w.prefix}"
                        f"{'-' + str(w.prefix) if w.prefix_min != w.prefix else ''}, "
                        f"{w.tree_mode} tree {w.rows} rows depth {w.depth}, T={w.temperature}, batch {batch}, "
                        f"{w.layers} layers",
            "batch": batch, "layers": w.layers, "tree_rows": w.rows, "prefix": int(w.prefix),
            "vocab": w.vocab, "heads": f"{w.n_q_heads}/{w.n_kv_heads}x{w.head_dim}"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"eagle_bench_clocks_{os.getpid()}.csv")

    def __enter__(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            p = [x.strip() for x in line.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                mx.append(float(p[2]))
            except ValueError:
                continue
            for n, v in zip(names, p[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)), "samples": len(sm),
                "reasons": sorted(reasons)}


def _kernel_sha(srcs) -> str:
    h = hashlib.sha256()
    for p in srcs:
        h.update(open(p, "rb").read())
    return h.hexdigest()


def _traffic_for(kernel_srcs, workload: str):
    """dram bytes per launch from the committed ncu summary, if the kernel is unchanged."""
    try:
        with open(PROFILE_TRAFFIC) as f:
            t = json.load(f)
        e = t.get(workload)
        if e and e.get("source_sha256") == _kernel_sha(kernel_srcs):
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


# ----------------------------------------------------------------------------- CPU oracle timing
def _oracle_attn_task(args):
    """Worker process: the oracle's tree attention for one (layer, KV head) pair, inputs
    read from the files the main process wrote; returns the seconds the call took."""
    root, d, layer, h, G, scale = args
    if root not in sys.path:
        sys.path.insert(0, root)
    import oracle
    ld = lambda n: np.load(os.path.join(d, f"{n}{layer}.npy"), mmap_mode="r")
    q, kc, vc, tk, tv = (ld(n) for n in ("q", "kc", "vc", "tk", "tv"))
    seq_len = np.load(os.path.join(d, "seq_len.npy"))
    parent = np.load(os.path.join(d, "parent.npy"))
    ins = (np.ascontiguousarray(q[:, :, h * G:(h + 1) * G]), np.ascontiguousarray(kc[:, h:h + 1]),
           np.ascontiguousarray(vc[:, h:h + 1]), np.ascontiguousarray(tk[:, h:h + 1]),
           np.ascontiguousarray(tv[:, h:h + 1]))
    t0 = time.perf_counter()
    oracle.tree_attn(*ins, seq_len, parent, scale)
    return time.perf_counter() - t0


def _pool_warm(_):
    import oracle  # noqa: F401  (loads the oracle library in the worker)
    return os.getpid()


class OracleBaseline:
    """The CPU oracle timed on every host core: tree attention of each (layer, KV head)
    pair in a pool of worker processes (one per core, started with spawn), then the
    acceptance and the commit in this process.  The layers' inputs are written once to
    a scratch directory and memory-mapped by the workers."""

    def __init__(self, w, layers, seq_len, parent, target, draft, tokens, ua, uf, max_path):
        import multiprocessing as mp
        import oracle
        oracle.build()
        self.w, self.layers = w, layers
        self.seq_len, self.parent = np.asarray(seq_len, np.int32), np.asarray(parent, np.int32)
        self.target, self.draft, self.tokens, self.ua, self.uf, self.max_path = target, draft, tokens, ua, uf, max_path
        self.dir = tempfile.mkdtemp(prefix="eagle_oracle_")
        for l, (q, kc, vc, tk, tv) in enumerate(layers):
            for n, a in (("q", q), ("kc", kc), ("vc", vc), ("tk", tk), ("tv", tv)):
                np.save(os.path.join(self.dir, f"{n}{l}.npy"), a)
        np.save(os.path.join(self.dir, "seq_len.npy"), self.seq_len)
        np.save(os.path.join(self.dir, "parent.npy"), self.parent)
        # the commit's caches and tree rows, every layer (the commit writes the same path
        # rows each step)
        self.kc = np.stack([c[1] for c in layers])
        self.vc = np.stack([c[2] for c in layers])
        self.tk = np.stack([c[3] for c in layers])
        self.tv = np.stack([c[4] for c in layers])
        self.cores = os.cpu_count() or 1
        self.pool = mp.get_context("spawn").Pool(self.cores)
        self.pool.map(_pool_warm, range(self.cores))

    def close(self):
        self.pool.terminate()
        import shutil
        shutil.rmtree(self.dir, ignore_errors=True)

    def step(self, budget_s: float = 1e9):
        """One verify step of the oracle; layers are processed in turn until `budget_s`
        of wall time has gone into attention (at least one layer), the rest extrapolated.
        Returns (seconds per full step, seconds spent, description, extrapolated)."""
        import oracle
        scale = 1.0 / math.sqrt(self.w.head_dim)
        G = self.w.group
        n_layers = len(self.layers)
        t0 = time.perf_counter()
        done = 0
        for l in range(n_layers):
            tasks = [(ROOT, self.dir, l, h, G, scale) for h in range(self.w.n_kv_heads)]
            self.pool.map(_oracle_attn_task, tasks, chunksize=1)
            done += 1
            if time.perf_counter() - t0 >= budget_s:
                break
        t_attn = time.perf_counter() - t0
        t1 = time.perf_counter()
        prop = oracle.SAMPLED if self.w.proposal == "sampled" else oracle.DELTA
        res = oracle.accept(self.target, self.tokens, self.parent, self.ua, self.uf, self.w.temperature, prop,
                            self.max_path, draft=self.draft)
        oracle.kv_commit(self.kc, self.vc, self.tk, self.tv, res["n_acc"], res["path"], self.seq_len)
        t_rest = time.perf_counter() - t1
        full = t_attn * n_layers / done + t_rest
        desc = (f"oracle on {self.cores} host cores: tree attention for {done * self.w.n_kv_heads} of the "
                f"{n_layers * self.w.n_kv_heads} (layer, KV head) pairs in worker processes"
                + ("" if done == n_layers else f" (extrapolated x{n_layers / done:g})")
                + f", then acceptance and the commit of all {n_layers} layers in one process, "
                  f"batch {self.seq_len.shape[0]}")
        return full, t_attn + t_rest, desc, done < n_layers


# ----------------------------------------------------------------------------- main arms
def run_ours(args):
    import torch
    import torch.distributed as dist

    from eagle_speculative_decoding_tree_gb300 import binding as B
    from eagle_speculative_decoding_tree_gb300 import synth
    from eagle_speculative_decoding_tree_gb300.step import VerifyStep

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    if ws > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    w = synth.WORKLOADS[args.config]
    batch = args.batch or w.batch
    w = w.with_(batch=batch, layers=args.layers or w.layers)
    B.load()
    t_setup = time.perf_counter()
    need_host = rank == 0 and not args.skip_cpu_baseline
    st = VerifyStep(w, batch=batch, keep_host=need_host)
    # distinct seeded steps (own root, tree, logits and uniforms over the same caches and
    # queries), replayed in turn so that the timed steps accept drafts at the workload's rate
    n_var = st.add_variants(args.variants - 1) if args.variants > 1 else 1
    torch.cuda.synchronize()
    t_setup = time.perf_counter() - t_setup

    stream = torch.cuda.Stream()
    graphs = []
    accepted = []
    with torch.cuda.stream(stream):
        for k in range(n_var):
            st.use_variant(k)
            for _ in range(2):  # warm the launch path before capture
                st.run(stream)
            stream.synchronize()
            accepted.append(st.acc.n_acc.cpu().numpy().copy())
            if not args.no_graph:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    st.run(stream)
                graphs.append(g)
        st.use_variant(0)
    counter = [0]

    def step():
        k = counter[0] % n_var
        counter[0] += 1
        if graphs:
            graphs[k].replay()
        else:
            st.use_variant(k)
            st.run(stream)
    attn_splits, per_layer_launches = B.tree_attn_plan(st.attn_desc)
    launches_per_step = st.L * per_layer_launches + 2 + 2

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    stream.synchronize()
    kv_total = st.kv_bytes_per_layer() * st.L
    l2_note = (f"inputs larger than L2: {kv_total / 1e9:.2f} GB of K/V read per step" if kv_total > L2_BYTES else
               "L2 flushed between steps")
    flush = None if kv_total > L2_BYTES else torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device="cuda")

    # ---- timed region: K graph replays
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        with torch.cuda.stream(stream):
            e0.record(stream)
            if flush is None:
                for _ in range(args.steps):
                    step()
            else:
                # L2 flush between steps is timed separately and subtracted
                for _ in range(args.steps):
                    flush.zero_()
                    step()
            e1.record(stream)
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    if flush is not None:
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            f0.record(stream)
            for _ in range(args.steps):
                flush.zero_()
            f1.record(stream)
        torch.cuda.synchronize()
        ms -= f0.elapsed_time(f1)
    if ws > 1:
        dist.barrier()
    ms = reduce_max(ms, ws, "cuda")
    clocks = clk.summary()
    ms_per_step = ms / args.steps
    value = job_value(ws, args.steps, ms)
    n_acc_all = np.stack(accepted)  # [variant][request]

    # ---- roofline of the dominant kernel: tree attention, timed alone (graph of L layers)
    ga = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        st.reset()
        for l in range(st.L):
            st.attn_layer(l, stream)
        stream.synchronize()
        with torch.cuda.graph(ga, stream=stream):
            for l in range(st.L):
                st.attn_layer(l, stream)
        for _ in range(3):
            ga.replay()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = max(5, args.steps // 4)
        a0.record(stream)
        for _ in range(reps):
            ga.replay()
        a1.record(stream)
    torch.cuda.synchronize()
    attn_ms = a0.elapsed_time(a1) / (reps * st.L)
    peak, peak_kind = _peaks()
    bytes_layer = st.kv_bytes_per_layer()
    achieved = bytes_layer / (attn_ms / 1e3) / 1e9
    traffic = _traffic_for(ATTN_SRCS, args.config)
    roofline = {"kernel": f"tree_attn_tc_kernel ({per_layer_launches} launch(es) per layer, {attn_splits} splits)",
                "bound": "hbm",
                "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                else "fallback 6.8 TB/s", "traffic": traffic, "algorithmic_bytes_per_launch": bytes_layer,
                "us_per_launch": round(attn_ms * 1e3, 2)}
    accept_t, commit_t = time_accept_commit(st, stream, n_var, n_acc_all, max(5, args.steps // 16), peak)
    tree_build = time_tree_build(st, stream, max(20, args.steps // 2))
    lmhead = time_lmhead(st, stream, max(10, args.steps // 4), peak)
    tree_head = time_tree_head(st, stream, max(5, args.steps // 8), peak)
    ttt = time_ttt(stream, 5) if args.config in ("llama8b", "vicuna7b") else {"skipped": "run with the 8B workloads"}
    step_bytes = kv_total + float(np.mean([st.logit_bytes_visited(a) for a in n_acc_all]))
    step_frac = step_bytes / (ms_per_step / 1e3) / 1e9 / peak

    # ---- e2e through the C ABI with host buffers (pinned), copies inside the timed region
    e2e = e2e_run(st, stream, args, ws)

    line = {"metric": "verify steps/s (tree attention x L + accept + commit), 1 GB300", "value": round(value, 2),
            "unit": "steps/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms_per_step, 5), "us_per_step": round(ms_per_step * 1e3, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": {**_workload_desc(w, batch), "l2": l2_note, "graph": g is not None, "attn_splits": attn_splits,
                       "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
            "step_roofline_frac": round(step_frac, 4), "step_algorithmic_bytes": int(step_bytes),
            "mean_accept_length": round(float(np.mean(n_acc_all + 1)), 4), "step_variants": int(n_var),
            "roofline": roofline, "accept": accept_t, "commit": commit_t, "tree_build": tree_build,
            "tree_build_head": tree_head, "lmhead_stats": lmhead,
            "ttt_attention": ttt, "e2e": e2e,
            "gpu_launches": int(launches_per_step * args.steps), "clocks": clocks,
            "setup_s": round(t_setup, 1)}
    if need_host:
        base = OracleBaseline(w, st.host, st.seq_len0, st.parent.cpu().numpy(), st.target_host, st.draft_host,
                              st.tokens.cpu().numpy(), st.u_accept.cpu().numpy(), st.u_final.cpu().numpy(),
                              st.max_depth + 1)
        try:
            per_step, spent, desc, extrap = base.step(budget_s=15.0)
        finally:
            base.close()
        line["cpu_baseline"] = {"value": round(1.0 / per_step, 6), "unit": "steps/s", "cores": base.cores,
                                "kind": "oracle", "sample": desc, "seconds": round(spent, 2),
                                "extrapolated": bool(extrap)}
    if ws > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def time_accept_commit(st, stream, n_var: int, n_acc_all, reps: int, peak: float):
    """Acceptance and commit, each timed alone over the step variants (graphs replayed in
    turn), against the bytes each must move: acceptance reads the target rows its walk
    visits (n_acc + 1 per request; their draft rows too for drawn proposals), the commit
    reads and writes the accepted path's K/V rows of every layer (n_acc + 1 rows per
    request, K and V)."""
    import torch
    ga, gc = [], []
    with torch.cuda.stream(stream):
        for k in range(n_var):
            st.use_variant(k)
            st.reset()
            st.accept(stream)
            st.commit(stream)
            stream.synchronize()
            g1, g2 = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
            with torch.cuda.graph(g1, stream=stream):
                st.accept(stream)
            with torch.cuda.graph(g2, stream=stream):
                st.reset()
                st.commit(stream)
            ga.append(g1)
            gc.append(g2)
        st.use_variant(0)

        def timed(gs):
            for g in gs:
                g.replay()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                for g in gs:
                    g.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) * 1e3 / (reps * len(gs))

        us_acc = timed(ga)
        # a commit moves the rows its own acceptance accepted: each variant's commit is
        # timed after that variant's acceptance
        us_com = 0.0
        for k in range(n_var):
            ga[k].replay()
            us_com += timed([gc[k]]) / n_var
        # leave the accept outputs of variant 0 in place for later users of the step
        ga[0].replay()
        stream.synchronize()
    acc_bytes = float(np.mean([st.logit_bytes_visited(a) for a in n_acc_all]))
    esz = 4 if st.w.dtype == "f32" else 2
    rows = float(np.mean([np.sum(a + 1) for a in n_acc_all]))
    com_bytes = rows * st.L * st.w.n_kv_heads * st.w.head_dim * esz * 2 * 2
    return ({"us_per_step": round(us_acc, 2), "algorithmic_bytes": int(acc_bytes),
             "gbs": round(acc_bytes / us_acc / 1e3, 1), "frac": round(acc_bytes / us_acc / 1e3 / peak, 4),
             "bound": "latency (one group barrier per visited node)"},
            {"us_per_step": round(us_com, 2), "algorithmic_bytes": int(com_bytes),
             "gbs": round(com_bytes / us_com / 1e3, 1), "frac": round(com_bytes / us_com / 1e3 / peak, 4),
             "bound": "launch latency (two kernels, a 4-byte seq_len reset in the graph)"})


def time_tree_build(st, stream, reps: int):
    """The draft-tree build of the step, timed apart from the verify step: all draft
    levels (eagle_tree_build per level: one kernel, plus a memset before level 1) replayed
    from a CUDA graph with the levels' draft logits already on the device.  Reports
    the time per tree and the logit bytes the chunk passes read."""
    import torch

    bld = st.builder
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        bld.replay(stream)
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            bld.replay(stream)
        for _ in range(3):
            g.replay()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(reps):
            g.replay()
        t1.record(stream)
    torch.cuda.synchronize()
    us = t0.elapsed_time(t1) * 1e3 / reps
    logit_bytes = sum(lg.numel() * lg.element_size() for _, lg, _ in bld.levels)
    return {"us_per_tree": round(us, 2), "levels": len(bld.levels), "launches_per_tree": len(bld.levels), "memsets_per_tree": 1,
            "logit_bytes_per_tree": int(logit_bytes), "gbs": round(logit_bytes / (us / 1e6) / 1e9, 1),
            "note": "timed apart from the verify step (not in value); inputs resident, L2 warm"}


def time_lmhead(st, stream, reps: int, peak: float):
    """The LM-head statistics at the step's tree nodes (eagle_lmhead_stats), timed apart
    from the verify step: hidden rows of the tree's nodes (4096 wide, N(0, 1)) times a
    random bf16 head of the workload's vocabulary (N(0, 1/4096)); the kernel reads the
    head once, so its roofline is the head's bytes over the time."""
    import torch
    from eagle_speculative_decoding_tree_gb300 import binding as B
    w = st.w
    M, R, h, V = st.B * st.R, st.R, 4096, w.vocab
    if M > 128 or w.dtype != "bf16":
        return {"skipped": f"{M} rows (the kernel takes up to 128) or fp32 workload"}
    g = torch.Generator(device="cuda").manual_seed(0xEA61E000 + w.config_id)
    hid = torch.randn(M, h, device="cuda", generator=g).to(torch.bfloat16)
    head = (torch.randn(V, h, device="cuda", generator=g) / 64.0).to(torch.bfloat16)
    desc = B.LmHeadDesc(M, R, h, V, float(w.temperature))
    rec = torch.zeros(M, -(-V // B.EAGLE_LMHEAD_TILE), 4, dtype=torch.int32, device="cuda")
    child = torch.zeros(M, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        B.eagle_lmhead_stats(desc, hid, head, st.tokens, st.parent, rec, child, status, stream)
        stream.synchronize()
        with torch.cuda.graph(gr, stream=stream):
            B.eagle_lmhead_stats(desc, hid, head, st.tokens, st.parent, rec, child, status, stream)
        for _ in range(3):
            gr.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            gr.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / reps
    byt = V * h * 2 + M * h * 2
    out = {"us_per_call": round(us, 2), "rows": M, "hidden": h, "vocab": V, "algorithmic_bytes": int(byt),
           "gbs": round(byt / us / 1e3, 1), "frac": round(byt / us / 1e3 / peak, 4), "status": int(status.item()),
           "note": "timed apart from the verify step (not in value): head bytes read once per call"}
    del head
    torch.cuda.empty_cache()
    return out


def time_tree_head(st, stream, reps: int, peak: float):
    """The draft-tree build from the draft's hidden states (eagle_tree_build_head: the
    draft LM head fused with tree expansion), timed apart from the verify step: every
    level's frontier hidden states (4096 wide, N(0, 1)) against a random bf16 head of the
    workload's vocabulary (N(0, 1/4096)), all levels replayed from a CUDA graph.  Each
    level reads the head once, so the roofline is the levels' head bytes over the time."""
    import torch
    from eagle_speculative_decoding_tree_gb300 import binding as B, synth
    from eagle_speculative_decoding_tree_gb300.step import GpuTreeBuilder
    w = st.w
    h, V = 4096, w.vocab
    if w.tree_mode == "static_sampled" or w.dtype != "bf16":
        return {"skipped": "sampled trees draw from the logits; bf16 workloads only"}
    bld = GpuTreeBuilder(w, st.B)
    if st.B * bld.desc.top_k > 128:
        return {"skipped": "more than 128 frontier rows"}
    g = np.random.default_rng(0xEA61E000 + w.config_id)
    head = (torch.randn(V, h, device="cuda", generator=torch.Generator(device="cuda").manual_seed(w.config_id))
            / 64.0).to(torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    bld.set_context(np.zeros(st.B, np.int32), np.asarray(st.seq_len0, np.int32))
    F, rows = 1, 0
    for level in range(1, bld.depth + 1):
        hid = synth.bf16_bits(g.normal(0, 1, (st.B, F, h)).astype(np.float32))
        tok, _ = bld.expand_head(level, hid, head, status)
        rows += st.B * F
        F = tok.shape[1]
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        bld.replay_head(head, status, stream)
        stream.synchronize()
        with torch.cuda.graph(gr, stream=stream):
            bld.replay_head(head, status, stream)
        for _ in range(3):
            gr.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            gr.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / reps
    levels = bld.depth
    byt = levels * V * h * 2 + rows * h * 2
    out = {"us_per_tree": round(us, 2), "levels": levels, "launches_per_tree": 2 * levels, "hidden": h, "vocab": V,
           "algorithmic_bytes": int(byt), "gbs": round(byt / us / 1e3, 1), "frac": round(byt / us / 1e3 / peak, 4),
           "status": int(status.item()),
           "note": "timed apart from the verify step (not in value): the draft head read once per level"}
    del head
    torch.cuda.empty_cache()
    return out


def time_ttt(stream, reps: int):
    """EAGLE-3 training-time-test attention (eagle_ttt_attn) for an 8B-shaped draft layer
    in training: 32 q / 8 kv heads x 128, sequence 4096, 7 TTT steps, bf16 N(0, 1)
    inputs; timed apart from the verify step.  Its work is the causal trunk's products,
    2 * 128 * S (S + 1) flops per (step, query head) (QK^T and PV, the causal half), so
    its roofline is the tensor pipe (measured bf16 peak)."""
    import torch
    from eagle_speculative_decoding_tree_gb300 import binding as B
    K, S, Hq, Hkv, D = 7, 4096, 32, 8, 128
    g = torch.Generator(device="cuda").manual_seed(0xEA61E7)
    mk = lambda *shape: torch.randn(*shape, device="cuda", generator=g).to(torch.bfloat16)
    q, kt, vt, kb, vb = mk(K, S, Hq, D), mk(Hkv, S, D), mk(Hkv, S, D), mk(K, Hkv, S, D), mk(K, Hkv, S, D)
    out = torch.empty(K, S, Hq, D, dtype=torch.bfloat16, device="cuda")
    desc = B.TttDesc(K, S, Hq, Hkv, D, 1.0 / math.sqrt(D), B.EAGLE_BF16)
    ws = torch.zeros(B.workspace_size(B.EAGLE_WS_TTT_ATTN, desc), dtype=torch.uint8, device="cuda")
    with torch.cuda.stream(stream):
        for _ in range(2):
            B.eagle_ttt_attn(desc, q, kt, vt, kb, vb, out, None, ws, stream)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            B.eagle_ttt_attn(desc, q, kt, vt, kb, vb, out, None, ws, stream)
        e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    flops = K * Hq * 2.0 * D * S * (S + 1)
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            tpeak = float(json.load(f)["bf16_tflops"])
    except Exception:
        tpeak = 1900.0
    tf = flops / (ms / 1e3) / 1e12
    res = {"shape": f"{Hq}q/{Hkv}kv x {D}, sequence {S}, {K} TTT steps", "ms_per_call": round(ms, 3),
           "bound": "tensor", "achieved": round(tf, 1), "peak": tpeak, "unit": "TFLOP/s", "frac": round(tf / tpeak, 4),
           "algorithmic_flops": flops, "error_word": int(ws[:4].view(torch.int32).item()),
           "note": "timed apart from the verify step; P enters PV as two bf16 terms (1.5x the MMAs of the flops counted)"}
    del q, kt, vt, kb, vb, out
    torch.cuda.empty_cache()
    return res


def e2e_run(st, stream, args, ws):
    """The same step through the public API with host inputs: every step copies the
    step's inputs (queries and tree K/V of all layers, logits, uniforms, tree) from
    pinned host memory, runs the step, and reads the accepted tokens back.  The inputs
    live in one device arena mirrored by one pinned host buffer, so a step's upload is a
    single copy; the step's C-ABI calls are replayed from a CUDA graph, as a decode loop
    would run them."""
    import torch
    names = [("q", l) for l in range(st.L)] + [("tk", l) for l in range(st.L)] + [("tv", l) for l in range(st.L)]
    names += [(n, None) for n in ("target", "u_accept", "u_final", "tokens", "parent", "anc_mask")]
    if st.draft is not None:
        names.append(("draft", None))
    get = lambda n, l: getattr(st, n)[l] if l is not None else getattr(st, n)
    ins = [get(n, l) for n, l in names]
    offs, total = [], 0
    for t in ins:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    dev = torch.empty(total, dtype=torch.uint8, device="cuda")
    host = torch.empty(total, dtype=torch.uint8, pin_memory=True)
    views = [dev[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape) for o, t in zip(offs, ins)]
    for v, t in zip(views, ins):
        v.copy_(t)
    host.copy_(dev)
    saved = {n: (list(getattr(st, n)) if isinstance(getattr(st, n), list) else getattr(st, n)) for n, _ in names}
    for (n, l), v in zip(names, views):  # the step reads its inputs from the arena
        if l is None:
            setattr(st, n, v)
        else:
            getattr(st, n)[l] = v
    outs = [st.acc.n_acc, st.acc.out_tok]
    host_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
    h2d = sum(t.numel() * t.element_size() for t in ins)
    d2h = sum(t.numel() * t.element_size() for t in outs)
    n = max(3, args.steps // 4)
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            st.run(stream)
            stream.synchronize()
            with torch.cuda.graph(g, stream=stream):
                st.run(stream)

            def one():
                dev.copy_(host, non_blocking=True)
                g.replay()
                for h, d in zip(host_out, outs):
                    h.copy_(d, non_blocking=True)

            for _ in range(2):
                one()
            stream.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(n):
                one()
            e1.record(stream)
        torch.cuda.synchronize()
    finally:
        for n_, v in saved.items():
            setattr(st, n_, v)
    ms = e0.elapsed_time(e1)
    return {"value": round(ws * n / (ms / 1e3), 2), "unit": "steps/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "steps": n, "ms_per_step": round(ms / n, 5),
            "copies_per_step": 1 + len(outs), "graph": True}


def run_reference(args):
    """The CPU oracle timed as the reference arm (rank 0 only): each step is the oracle's
    verify step on every host core (tree attention of each (layer, KV head) pair in a
    pool of worker processes, then acceptance and commit), measured; when a full step
    would not fit the run, a step processes the layers that fit in about 6 s and the
    rest is extrapolated (said in the line)."""
    ws, rank, local = _dist()
    if rank != 0:
        return
    from eagle_speculative_decoding_tree_gb300 import synth
    w = synth.WORKLOADS[args.config]
    batch = args.batch or w.batch
    w = w.with_(batch=batch)
    base = OracleBaseline(w, *reference_inputs(w, batch))
    try:
        per, spent_all, desc, extrap = [], 0.0, "", False
        for i in range(args.warmup + args.steps):
            full, spent, desc, ex = base.step(budget_s=6.0)
            if i >= args.warmup:
                per.append(full)
                spent_all += spent
                extrap |= ex
    finally:
        base.close()
    sec = float(np.mean(per))
    value = 1.0 / sec
    line = {"impl": "reference", "metric": "verify steps/s (tree attention x L + accept + commit), 1 GB300",
            "value": round(value, 6), "unit": "steps/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            # the time each timed step took (its sample, when the rest is extrapolated)
            "ms_per_step": round(spent_all / args.steps * 1e3, 3),
            "full_step_ms": round(sec * 1e3, 3), "extrapolated": bool(extrap),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": w.dtype, "data": "synthetic", "config": _workload_desc(w, batch),
            "cpu_baseline": {"value": round(value, 6), "unit": "steps/s", "cores": base.cores, "kind": "oracle",
                             "sample": desc, "seconds": round(spent_all, 1), "extrapolated": bool(extrap)},
            "e2e": {"value": round(value, 6), "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def reference_inputs(w, batch):
    """Host inputs for the reference arm: every layer's attention tensors and a tree of
    the workload's shape (the oracle builds it), logits at its nodes."""
    import oracle
    from eagle_speculative_decoding_tree_gb300 import synth
    seq_len = synth.prefix_lengths(w, batch)
    root_tok = synth.root_tokens(w, batch)
    root_h = [synth.root_hash(w.config_id, b) for b in range(batch)]
    lm = synth.hash_lm(w)
    ua, uf, ud = synth.step_uniforms(w, batch, w.rows)
    if w.tree_mode == "dynamic":
        t = oracle.DynamicTree(batch, w.vocab, w.depth, w.top_k, w.total_tokens)
        front = [[h] for h in root_h]
        for level in range(1, w.depth + 1):
            rows = synth.as_dtype_bytes(np.stack([lm.rows(front[b], "draft") for b in range(batch)]), w.dtype)
            prev = None if level == 1 else t.frontier.copy()
            t.expand(rows)
            slot = t.frontier_parent_slot(prev)
            tok = t.frontier_tokens()
            front = [[synth.child_hash(front[b][int(slot[b, j])], int(tok[b, j])) for j in range(tok.shape[1])]
                     for b in range(batch)]
        tree = t.finalize(root_tok, seq_len)
    else:
        par = synth.static_parents(w.static_choices)
        t = oracle.StaticTree(batch, w.vocab, par, w.tree_mode == "static_sampled", w.temperature)
        hs = [[h] + [0] * (len(par) - 1) for h in root_h]
        for level in range(1, int(t.depths.max()) + 1):
            nodes = t.frontier_nodes(level)
            rows = synth.as_dtype_bytes(np.stack([[lm.draft_row(hs[b][n]) for n in nodes] for b in range(batch)]),
                                        w.dtype)
            t.expand(rows, ud)
            for b in range(batch):
                for i in np.nonzero(t.depths == level)[0]:
                    hs[b][i] = synth.child_hash(hs[b][par[i]], int(t.tokens[b, i]))
        tree = t.finalize(root_tok, seq_len)
    hs = []
    for b in range(batch):
        h = [root_h[b]]
        for i in range(1, tree["tokens"].shape[1]):
            h.append(synth.child_hash(h[tree["parent"][b, i]], int(tree["tokens"][b, i])))
        hs.append(h)
    target = synth.as_dtype_bytes(np.stack([lm.rows(hs[b], "target") for b in range(batch)]), w.dtype)
    draft = synth.as_dtype_bytes(np.stack([lm.rows(hs[b], "draft") for b in range(batch)]), w.dtype) \
        if w.proposal == "sampled" else None
    R = tree["tokens"].shape[1]
    layers = [synth.attn_tensors(w, l, batch, seq_len, R) for l in range(w.layers)]
    return (layers, seq_len, tree["parent"], target, draft, tree["tokens"], ua, uf, int(tree["depth"].max()) + 1)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="llama8b",
                    choices=["tiny", "vicuna7b", "llama8b", "long128k", "concurrency"])
    ap.add_argument("--batch", type=int, default=0, help="override the workload's batch (concurrency: 1/8/32)")
    ap.add_argument("--layers", type=int, default=0, help="override the layer count (small profiling cases)")
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--skip-cpu-baseline", action="store_true")
    ap.add_argument("--variants", type=int, default=16,
                    help="distinct seeded verify steps replayed in turn (trees, logits, uniforms)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
