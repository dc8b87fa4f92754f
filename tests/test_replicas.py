"""The multi-GPU path is replicas only: every rank runs the whole layer on its own
batch and the ranks meet only around the timed region.  These CPU tests run that
host logic (delta_rule_recurrent_gated_gb300/replicas.py, used by bench.py) as two
gloo processes on 127.0.0.1: the barrier, the maximum of the per-rank times, the
per-rank seeds (different batches), the whole-job unit count, rank 0 alone
reporting, a rank that fails before joining surfacing as an error on the other,
and the reference arm under a launcher (rank 1 exits at once without output)."""
import json
import os
import socket
import subprocess
import sys
import time

import pytest
import torch
import torch.multiprocessing as mp

from delta_rule_recurrent_gated_gb300 import inputs
from delta_rule_recurrent_gated_gb300.replicas import Replicas

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir, delays):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    rep = Replicas.from_env()
    rep.init("gloo")
    w = inputs.small("gdn", B=1, T=16, H=1, dk=16, dv=16, h0=False, dhT=False)
    x = inputs.make(w, seed=rep.seed())
    rep.barrier()
    t0 = time.perf_counter()
    time.sleep(delays[rank])  # stands in for this rank's timed steps
    mine = time.perf_counter() - t0
    rep.barrier()
    slowest = rep.max_over_ranks(mine)
    res = {"rank": rank, "mine": mine, "slowest": slowest, "root": rep.is_root,
           "total": rep.total_units(w.tokens), "q0": float(x["q"].float().flatten()[0])}
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump(res, f)
    rep.shutdown()


def test_two_gloo_replicas(tmp_path):
    world, port = 2, free_port()
    mp.start_processes(_worker, args=(world, port, str(tmp_path), [0.05, 0.30]), nprocs=world,
                       join=True, start_method="spawn")
    r = [json.load(open(tmp_path / f"r{i}.json")) for i in range(world)]
    assert r[0]["root"] and not r[1]["root"]
    # both ranks see the slowest rank's time
    assert r[0]["slowest"] == r[1]["slowest"] == max(r[0]["mine"], r[1]["mine"])
    assert r[1]["slowest"] >= 0.30
    assert r[0]["total"] == r[1]["total"] == 2 * 16
    assert r[0]["q0"] != r[1]["q0"]  # each replica draws its own batch


def _failing_worker(rank, world, port):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    if rank == 1:
        raise RuntimeError("replica 1 failed before joining")
    import datetime
    import torch.distributed as dist
    dist.init_process_group("gloo", timeout=datetime.timedelta(seconds=5))
    dist.barrier()


def test_a_failed_replica_is_an_error_not_a_hang():
    """A rank that dies before joining makes the launch fail (the others time out on
    the host), with no GPU involved."""
    port = free_port()
    with pytest.raises(Exception):
        mp.start_processes(_failing_worker, args=(2, port), nprocs=2, join=True,
                           start_method="spawn")


def test_single_process_needs_no_group():
    rep = Replicas()
    rep.init("gloo")
    assert rep.backend is None and rep.is_root
    rep.barrier()
    assert rep.max_over_ranks(1.5) == 1.5
    assert rep.total_units(7) == 7
    rep.shutdown()


def test_reference_arm_rank1_exits_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    t0 = time.time()
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--gpus", "2", "--steps", "1", "--warmup", "3"],
                         env=env, capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stderr
    assert out.stdout.strip() == ""
    assert time.time() - t0 < 60
