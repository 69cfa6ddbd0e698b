"""The N > 1 path of bench.py on the host (world size 2, gloo, CPU): the
replicas share no data path, so what N > 1 adds is the rank environment, the
barrier around the timed region and the max over ranks of the timed seconds
(value = all ranks' tokens / that time), with rank 0 alone printing.  The
reference arm under the launcher: rank 0 prints one line, the other rank
exits 0 without work."""
import importlib.util
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _rank(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    bench = _bench()
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        bench.barrier(w)
        seconds = [1.5, 2.25][rank]           # this rank's timed region
        mx = bench.max_over_ranks(seconds, w)
        bench.barrier(w)
        q.put((rank, r, w, local, mx))
    finally:
        dist.destroy_process_group()


def test_rank_environment_barrier_and_max_over_ranks_under_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, r, w, local, mx in got:
        assert (r, w, local) == (rank, 2, rank)
        assert mx == 2.25                      # the slower rank sets the job time


def test_max_over_ranks_is_the_identity_for_one_rank():
    assert _bench().max_over_ranks(3.5, 1) == 3.5


def test_reference_arm_under_the_launcher_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--steps", "1", "--warmup", "3", "--workload", "tiny"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["config"]["workload"] == "tiny"


def test_gpus_flag_without_a_launcher_spawns_the_replicas():
    """bench.py --gpus 2 run directly re-launches itself under
    torch.distributed.run with two processes; still one line, from rank 0."""
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "3", "--workload", "tiny"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2
