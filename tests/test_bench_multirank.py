"""bench.py's multi-GPU aggregation, exercised with two gloo ranks on the CPU: the timed region is
the max over ranks and the value is all ranks' units over that time (weak scaling)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    elapsed = [3.5, 7.25][rank]                       # per-rank timed region, ms
    m = bench.max_over_ranks(elapsed, dist, torch.device("cpu"))
    v = bench.aggregate(world, 1000.0, 10, m)
    q.put((rank, m, v))
    dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, m, v in res:
        assert m == 7.25
        assert v == pytest.approx(2 * 1000.0 * 10 / 7.25e-3)


def test_single_rank_identity():
    assert bench.max_over_ranks(4.0, None, None) == 4.0
    assert bench.aggregate(1, 150994944, 100, 4.0) == pytest.approx(150994944 * 100 / 4.0e-3)


def _reference_line(env_extra):
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, **env_extra)
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], capture_output=True, text=True, timeout=600, env=env, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    return [json.loads(l) for l in lines]


def test_reference_arm_line():
    """The reference arm times the oracle on the host cores and prints the contract's line."""
    (d,) = _reference_line({})
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["steps"] == 1 and d["warmup"] == 3 and d["n_gpus"] == 1


def test_reference_arm_other_ranks_print_nothing():
    """Under a multi-rank launch only rank 0 runs the reference arm."""
    assert _reference_line({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}) == []
