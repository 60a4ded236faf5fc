"""The multi-process path of bench.py on CPU (gloo, world size 2, 127.0.0.1).

bench.py runs one process per GPU under torchrun; on this path the work is
replicated (no collective on the data path) and only the timing is combined:
a barrier on both sides of the timed region and the maximum over ranks.  These
tests run that host logic with two gloo ranks, and the reference arm end to end
under torchrun (rank 0 prints one JSON line, the other rank exits 0).
"""
import importlib.util
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _load_bench():
    spec = importlib.util.spec_from_file_location("bench_mp", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _rank_main(rank, world, port, values, out_q):
    import torch.distributed as dist
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    bench = _load_bench()
    w, r, local = bench.dist_setup()
    try:
        bench.barrier(w)
        m = bench.max_over_ranks(w, values[r])
        out_q.put((r, w, local, m))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    values = [3.25, 7.5]
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, values, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 2, 0, 7.5), (1, 2, 1, 7.5)]


def test_single_process_needs_no_group():
    bench = _load_bench()
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        os.environ.pop(k, None)
    assert bench.dist_setup() == (1, 0, 0)
    assert bench.max_over_ranks(1, 2.5) == 2.5


def test_reference_arm_under_torchrun_two_ranks():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "3", "--workload", "b2_c24_15x17_k3", "--dtype", "float32"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["unit"] == "Mpixel/s"
    assert d["value"] > 0 and d["e2e"]["value"] == d["value"]
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1


@pytest.mark.parametrize("step", ["forward", "filter", "filter_train"])
def test_reference_arm_times_each_step_kind(step):
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--step", step, "--steps", "1", "--warmup", "3",
           "--workload", "b2_c24_15x17_k3", "--dtype", "float32"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        env.pop(k, None)
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads([l for l in r.stdout.splitlines() if l.startswith("{")][-1])
    bench = _load_bench()
    assert d["impl"] == "reference" and d["metric"] == bench.STEP_METRIC[step] and d["value"] > 0
