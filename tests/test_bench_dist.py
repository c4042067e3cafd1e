"""The benchmark's multi-process logic on CPU (gloo, world size 2).

Each rank runs its own replica; the job's time is the max over ranks and the
job's value is world_size * steps / that time.  The reference arm runs on rank 0
only; the other ranks exit without output.
"""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = 100.0 + 50.0 * rank  # rank 1 is slower
    mx = bench.reduce_max(ms, world)
    buf = io.StringIO()
    with redirect_stdout(buf):
        if rank != 0:  # the reference arm is rank 0's job only
            class A:
                config, batch, steps, warmup = "tiny", 0, 1, 3
            bench.run_reference(A())
    dist.destroy_process_group()
    q.put((rank, mx, bench.job_value(world, 20, mx), buf.getvalue()))


def test_two_rank_max_and_job_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, mx, value, out in res:
        assert mx == 150.0
        assert abs(value - 2 * 20 / 0.150) < 1e-9
        if rank == 1:
            assert out == ""


def test_reference_arm_json_line():
    """bench.py --impl reference (the CPU oracle arm) prints one JSON line with the
    contract's keys; it needs no GPU."""
    import json
    import subprocess
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "tiny",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "steps/s" and d["higher_is_better"]
    assert d["steps"] == 1 and d["warmup"] == 3 and d["n_gpus"] == 1 and d["vs_baseline"] is None
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
