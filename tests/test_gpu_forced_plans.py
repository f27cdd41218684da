"""GPU parity of the decode stream kernel under forced launch plans.

The planner normally gives each cluster one or two 128-row weight tiles, so the
paths that only run with many tiles per cluster (receive buffers reused every
other tile, the weight ring refilled through its last stages, including the
stages the tcgen05 body takes over from the activation area) see little use.
`R9Q_PLAN=S,G,stages` (read once per process) forces the split count, the tile
groups and the ring depth, so each case runs in a fresh process with a plan of
one cluster (G = 1) walking every tile through a two-stage ring, and is
compared with the oracle exactly as in test_gpu_parity.py.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TESTS = os.path.join(ROOT, "tests")

# (id, plan, python statements run with `t` = test_gpu_parity and `lib` = the binding)
CASES = [
    # W8A8, 16-row tile (tcgen05 body): 8 tiles a cluster, 4 k-blocks a tile
    ("w8a8_M16_tc", "2,1,2", "t._w8a8_case(lib, 16, 1024, 1024, 0.01, 20.0, 31)"),
    # W8A8, 32-row tile (tcgen05 body), ragged M
    ("w8a8_M20_tc", "2,1,2", "t._w8a8_case(lib, 20, 1024, 1024, 0.01, 20.0, 32)"),
    # W8A8, 8-row tile (mma.sync body)
    ("w8a8_M3_sync", "2,1,2", "t._w8a8_case(lib, 3, 1024, 1024, 0.01, 20.0, 33)"),
    # weight-only (mma.sync body)
    ("w8bf16_M16_sync", "2,1,2", "t._w8bf16_case(lib, 16, 1024, 1024, 34)"),
    # fused expert MLP, W8A8 (tcgen05 gate_up with the SwiGLU epilogue, tcgen05 down;
    # the unfused chain's down GEMM reads pre-quantised rows) and weight-only
    ("mlp_w8a8_M16", "2,1,2", "t.test_mlp_fused_vs_unfused_and_oracle(lib, False, 16, 512, 256, 512)"),
    ("mlp_wonly_M8", "2,1,2", "t.test_mlp_fused_vs_unfused_and_oracle(lib, True, 8, 512, 256, 512)"),
    # grouped experts: 16- and 64-row token tiles, 3 tiles a cluster
    ("grouped_w8a8", "2,1,2", "t._grouped_case(lib, [3, 0, 1, 16, 5], 384, 512, 0, 35)"),
    ("grouped_w8a8_M70", "2,1,2", "t._grouped_case(lib, [70, 3], 384, 512, 0, 36)"),
]


@pytest.mark.parametrize("case,plan,stmt", CASES, ids=[c[0] for c in CASES])
def test_forced_plan_matches_oracle(case, plan, stmt):
    code = ("import sys; sys.path.insert(0, %r); sys.path.insert(0, %r)\n"
            "import __graft_entry__; __graft_entry__.build()\n"
            "import block_scaled_fp8_x128_gb300 as lib\n"
            "import test_gpu_parity as t\n"
            "%s\n"
            "print('ok')\n" % (ROOT, TESTS, stmt))
    env = dict(os.environ, R9Q_PLAN=plan)
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), (case, r.stdout[-2000:], r.stderr[-4000:])
