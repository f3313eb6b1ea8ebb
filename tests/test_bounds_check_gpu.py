"""The bounds-checked debug build (-DCOLI_BOUNDS_CHECK) on ordinary inputs: the FP4 GEMM checks every
tile record against the buffers and would record kErrBounds and skip the tile; on valid inputs it
records nothing and gives the oracle's results. Runs in a child process so that the debug library
is the one loaded."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys
sys.path.insert(0, ROOT)
from routed_moe_fp4_gb300 import build, colimoe as cm
cm.load(build.build(bounds_check=True))
from oracle.oracle import Oracle
from routed_moe_fp4_gb300 import synthetic as S
from tests import parity as P
import dataclasses
oracle = Oracle()
cases = ["tiny", "decode", dataclasses.replace(S.WORKLOADS["tiny"], name="bc_big", T=200, H=512, E=8, top_k=2, I=256,
                                               I_s=384)]
for name in cases:
    inputs = S.make_inputs(name)
    outs, routing, launches = P.run_gpu(inputs)   # asserts a clear device error word
    rep = P.check(oracle, inputs, outs[0], routing, None, launches)
    assert rep.ok and rep.routing_bit_exact, rep
    print("bounds-checked", inputs.workload.name, "ok", rep.rel_err)
"""


def test_bounds_checked_build_runs_clean():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    r = subprocess.run([sys.executable, "-c", CHILD.replace("ROOT", repr(ROOT))], capture_output=True, text=True,
                       timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert r.stdout.count("ok") == 3, r.stdout
