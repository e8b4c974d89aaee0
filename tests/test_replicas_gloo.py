"""The replica path of bench.py on CPU: two gloo ranks run the same
rendezvous, barrier and max / sum reductions that the timed region uses
under NCCL (replicas only: the attention path has no exchange step, so these
reductions of timings and byte counts are the only collectives)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench
    r, w, local = bench.dist_setup(None)
    bench.barrier(w)
    # ms per step: the slowest rank's time; bytes: every rank's units
    ms = bench.max_over_ranks(1.5 + rank, w)
    total = bench.sum_over_ranks(1000.0 * (rank + 1), w)
    q.put((r, w, local, ms, total))
    dist.destroy_process_group()


def test_two_gloo_ranks_reduce_timing_and_bytes():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        got = sorted(q.get(timeout=120) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert [p.exitcode for p in procs] == [0, 0]
    assert got == [(0, 2, 0, 2.5, 3000.0), (1, 2, 1, 2.5, 3000.0)]


def test_reference_arm_other_ranks_do_no_work():
    import bench
    assert bench.run_reference(None, 1, 2, 1) is None


def test_reference_arm_line_on_the_host():
    """Rank 0 of the reference arm times the float64 oracle on the host
    cores: a bench line with the contract's keys and the oracle as its CPU
    baseline, from a process that never maps the CUDA library."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = (
        "import json, sys, types\n"
        "import bench\n"
        "line = bench.run_reference(types.SimpleNamespace(steps=2, warmup=1), 0, 1, 0)\n"
        "maps = open('/proc/self/maps').read()\n"
        "print(json.dumps({'line': line, 'mapped': 'libpagedattn' in maps}))\n")
    out = subprocess.run([sys.executable, "-c", code], cwd=root, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    res = json.loads(out.stdout.strip().splitlines()[-1])
    line = res["line"]
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["dtype"] == "f64" and line["steps"] == 2
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    assert not res["mapped"]
