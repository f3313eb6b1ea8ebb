"""Failure detection without a fault (needs a GB300).

The FP4 path's barrier waits are bounded. With a limit far below one memory latency a wait runs
out: the kernel records a code in the device error word, lets its copies and MMAs in flight
land, frees TMEM and returns. The context must stay usable, and the next forward with the
default limit must match the oracle, with a clear error word.
"""
import numpy as np
import pytest

from routed_moe_fp4_gb300 import synthetic as S
from tests import parity as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from routed_moe_fp4_gb300 import build, colimoe
    build.build()
    colimoe.load()


@pytest.mark.parametrize("name", ["decode", "prefill"])
def test_wait_runs_out_and_context_survives(oracle, name):
    import torch
    from routed_moe_fp4_gb300 import colimoe as cm
    inputs = S.make_inputs(name)
    layer = cm.MoELayer(inputs)
    x = torch.from_numpy(inputs.x.view(np.int16)).cuda()
    out = torch.empty_like(x)
    layer.set_wait_limit(1000)                  # 1 us: below the latency of one weight stage
    layer.forward(x, out)
    assert layer.ffn_path() == cm.COLI_FFN_GEMM_MXF4
    code = layer.device_error()                 # synchronises: raises if the context were lost
    assert code in (1, 2, 4), f"expected a pipeline wait to run out, got code {code}"
    layer.set_wait_limit(0)
    outs, routing, launches = P.run_gpu(inputs, layer=layer)   # asserts a clear error word
    T = inputs.x.shape[0]
    tokens = None if T <= 8 else P.sample_tokens(routing, T, 8)
    rep = P.check(oracle, inputs, outs[0], routing, tokens, launches)
    assert rep.routing_bit_exact and rep.rel_err <= P.OUT_TOL, rep
    layer.close()


def test_wait_limit_rejects_negative():
    from routed_moe_fp4_gb300 import colimoe as cm
    layer = cm.MoELayer(S.make_inputs("tiny"))
    with pytest.raises(cm.ColiError):
        layer.set_wait_limit(-1)
    layer.close()
