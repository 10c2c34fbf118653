"""The multi-rank path of bench.py on CPU: world_size-2 gloo process groups.

The block has no exchange between GPUs on this path (each rank runs its own replica), so
the only cross-rank logic is the job's step time (the slowest rank's), the whole-job
throughput, and the reference arm running on rank 0 alone.
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
    try:
        q.put((rank, _run(rank, world, port)))
    except Exception as e:  # reported to the parent at once instead of a queue timeout
        q.put((rank, {"error": repr(e)}))
        raise


def _run(rank, world, port):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import torch
    out = {"max": bench.reduce_max(1.5 + rank, torch.device("cpu"), world)}
    out["tflops"] = bench.job_tflops(2e12, world, 10.0)
    args = type("A", (), dict(workload=1, tp=None, tokens=None, warmup=0, steps=1,
                              grad_accum=False, branch=False, recompute=False,
                              fp8=False))()
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(args, rank, world)
    out["printed"] = buf.getvalue()
    dist.barrier()
    dist.destroy_process_group()
    return out


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q), daemon=True) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=300) for _ in procs)
    for r in range(2):
        assert "error" not in res[r], f"rank {r}: {res[r].get('error')}"
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(2):
        assert res[r]["max"] == 2.5                 # the slowest rank's time, on every rank
        assert abs(res[r]["tflops"] - 400.0) < 1e-9  # 2 ranks x 2e12 flop / 10 ms
    assert '"impl": "reference"' in res[0]["printed"] and res[0]["printed"].count("\n") == 1
    assert res[1]["printed"] == ""                  # the reference arm runs on rank 0 only
