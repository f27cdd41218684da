"""Host logic of bench.py's multi-GPU mode (replicas), on CPU: two gloo ranks
with different step times reduce to the whole-job line the driver expects —
the slowest rank's time, the bytes of all ranks, per-GPU roofline — and the
reference arm under torchrun runs on rank 0 only."""
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


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _line(ms, us_e2e):
    return {"metric": "m", "value": 0.0, "unit": "GB/s", "n_gpus": 1, "steps": 10, "warmup": 3,
            "ms_per_step": ms, "us_per_call": ms * 1e3,
            "config": {"workload": "w", "bytes_per_call": 17_043_456},
            "roofline": {"bound": "hbm", "achieved": 0.0, "peak": 6747.0, "unit": "GB/s", "frac": 0.0,
                         "traffic": None},
            "e2e": {"value": 0.0, "unit": "GB/s", "us_per_call": us_e2e, "h2d_bytes_per_step": 131072,
                    "d2h_bytes_per_step": 131072},
            "gpu_launches": 10}


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)

    def all_reduce_max(v):
        t = torch.tensor([float(v)], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return t.item()
    out = bench.aggregate_over_ranks(_line(0.010 + 0.002 * rank, 20.0 + 5.0 * rank), world, all_reduce_max)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, out))


def test_aggregate_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    bpc = 17_043_456
    for rank in (0, 1):
        out = res[rank]
        assert out["n_gpus"] == 2
        assert out["ms_per_step"] == pytest.approx(0.012)            # the slower rank
        assert out["value"] == pytest.approx(round(2 * bpc / 12e-6 / 1e9, 1))
        assert out["roofline"]["achieved"] == pytest.approx(round(bpc / 12e-6 / 1e9, 1))
        assert out["roofline"]["frac"] == pytest.approx(round(bpc / 12e-6 / 1e9 / 6747.0, 4))
        assert out["e2e"]["us_per_call"] == pytest.approx(25.0)
        assert out["e2e"]["value"] == pytest.approx(round(2 * bpc / 25e-6 / 1e9, 1))
        assert out["gpu_launches"] == 20


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
