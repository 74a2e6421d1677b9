"""The N-replica path on the CPU: two gloo ranks (no GPU).

Requests are independent, so N GPUs run N replicas with no data exchange;
the ranks only meet for a barrier and a max of the step time.  These tests
run that plumbing with gloo, and the reference arm under torchrun, where
rank 0 alone works and prints.
"""

import importlib.util
import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    bench = _bench()
    ranks = bench.Ranks(world, torch.device("cpu"), backend="gloo")
    ranks.barrier()
    step_ms = [2.0, 5.0][rank]  # rank 1 is the slow one
    ms = ranks.max(step_ms)
    out[rank] = (ms, bench.aggregate_value(world, ms), bench.replica_seed(20260004, rank))
    ranks.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_step_and_their_own_seeds():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 5.0
    assert res[0][1] == res[1][1] == 2 * 1000.0 / 5.0  # weak scaling: both ranks' rounds count
    assert res[0][2] != res[1][2]                         # each replica its own batch


def test_single_rank_needs_no_process_group():
    bench = _bench()
    r = bench.Ranks(1)
    r.barrier()
    assert r.max(3.5) == 3.5 and bench.aggregate_value(1, 4.0) == 250.0


def test_reference_arm_under_torchrun_prints_once_from_rank_zero():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "2",
           "--warmup", "1", "--workload", "b1_k4_v1024_f32_gauss"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
