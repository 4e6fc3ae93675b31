"""Host logic of bench.py's N>1 path on CPU with gloo, world_size 2.

The path has no exchange step: each rank runs its own replica, and the job's
throughput is every rank's units over the slowest rank's time.
"""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    dev = torch.device("cpu")
    local_ms = 10.0 * (rank + 1)           # rank 1 is the slow one
    value, t = bench.aggregate(1e9, 10, local_ms, world, dev)
    bench.barrier(dev)
    m = bench.reduce_max(float(rank), dev)
    results[rank] = (value, t, m)
    dist.destroy_process_group()


def test_two_rank_aggregation_uses_slowest_rank():
    world = 2
    mgr = mp.Manager()
    results = mgr.dict()
    mp.spawn(_worker, args=(world, _free_port(), results), nprocs=world, join=True)
    for r in range(world):
        value, t, m = results[r]
        assert t == pytest.approx(20.0)
        assert m == 1.0
        # 2 ranks x 10 steps x 1e9 bytes over 20 ms
        assert value == pytest.approx(2 * 10 * 1e9 / 0.020)


def test_reference_arm_only_rank0_works(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    assert bench.main(["--impl", "reference", "--steps", "3", "--warmup", "3"]) is None
    assert capsys.readouterr().out == ""


def test_single_process_has_no_group():
    import bench
    assert bench.reduce_max(3.5, torch.device("cpu")) == 3.5
    v, t = bench.aggregate(100.0, 4, 8.0, 1, torch.device("cpu"))
    assert t == 8.0 and v == pytest.approx(100.0 * 4 / 0.008)


def test_algorithmic_counts_match_closed_forms():
    import numpy as np

    import bench
    from paged_kv_cache_03_gb300 import synth
    inp = synth.workload("tiny")
    # visible pairs per head: L*(S-L) + L(L+1)/2 for S = 13 and 40, L = 5
    assert bench.visible_pairs(inp) == (5 * 8 + 15) + (5 * 35 + 15)
    assert bench.algorithmic_flops(inp) == 4 * 4 * 128 * 245
    kv = 2 * 2 * 128 * 2 * (13 + 40)
    qo = 2 * inp.query.size * 2
    assert bench.algorithmic_bytes(inp) == kv + qo + 4 * (1 + 3) + 4 * 2
    assert np.int64(bench.visible_pairs(synth.workload("prefill"))) == 4 * 2048 * 2049 // 2


def test_torchrun_two_ranks_print_one_line():
    """The driver's N>1 launch (torch.distributed.run, 127.0.0.1) of the
    reference arm: both ranks exit 0 and only rank 0 prints its JSON line."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(root, "bench.py"), "--gpus", "2", "--impl", "reference", "--workload",
           "tiny", "--steps", "3", "--warmup", "3", "--ref-budget", "1"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
