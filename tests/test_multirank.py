"""The N > 1 path on CPU: two gloo ranks.

Every (batch row, KV head) unit is independent, so ranks shard whole units
(weak scaling: each rank decodes its own batch) and the only cross-rank
traffic is a barrier and the max of the ranks' times.  These tests run that
host logic, and the oracle reference arm of bench.py under
torch.distributed.run, with world size 2 on the gloo backend.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    from bit_kv_cache_kvq_gb300.workloads import WORKLOADS
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # the slowest rank's time reaches every rank
        slowest = bench.max_over_ranks(10.0 + 5.0 * rank, world)
        w = bench.rank_workload(WORKLOADS["llama8b_gqa_32k_b16"], rank)
        dist.barrier()
        out[rank] = (slowest, w.seed, w.B, w.Hkv)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_the_slowest_time_and_own_their_units():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 15.0          # max over ranks, on every rank
    assert res[0][1] != res[1][1]                  # distinct inputs per rank
    assert res[0][2:] == res[1][2:]                # same shape: weak scaling


def test_max_over_ranks_is_identity_for_one_rank():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25


def test_reference_arm_under_torchrun_prints_one_line_from_rank_zero():
    import oracle
    oracle.build()   # built once here, not raced by the ranks
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--workload", "tiny_1head_1k", "--steps", "2", "--warmup", "1"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, capture_output=True, text=True, cwd=ROOT, env=env, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference"
    assert line["n_gpus"] == 2
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
