"""coli_moe_route_static: routing for callers that cannot allocate device memory.

Those callers (code running under CUDA graph capture, runtimes whose own pool owns every byte of
device memory, loops that cannot afford a first-call allocation) get a routing call whose scratch
lives in a fixed array inside the library. Its results must equal what coli_moe_forward routes
for the same inputs, call after call. This file sorts last so that a run stopping at the first
failure has already run every other test.
"""
import numpy as np
import pytest

from routed_moe_fp4_gb300 import synthetic as S

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from routed_moe_fp4_gb300 import build, colimoe
    build.build()
    return colimoe


@pytest.mark.parametrize("name", ["decode", "sweep_T64", "prefill"])
def test_route_static_matches_forward(lib, name):
    import torch
    cm = lib
    inputs = S.make_inputs(name)
    wl = inputs.workload
    layer = cm.MoELayer(inputs)
    x = torch.from_numpy(inputs.x.view(np.int16)).cuda()
    out = torch.empty_like(x)
    layer.forward(x, out)
    torch.cuda.synchronize()
    ref = layer.routing(wl.T)            # the existing entry point's routing
    for call in range(2):                # two calls in a row share the static scratch
        idx = torch.full((wl.T, wl.top_k), -1, dtype=torch.int32, device="cuda")
        w = torch.full((wl.T, wl.top_k), -1.0, dtype=torch.float32, device="cuda")
        cm.coli_moe_route_static(x, wl.T, wl.H, layer.router_w, layer.router_b, wl.E, wl.top_k, idx, w)
        torch.cuda.synchronize()
        assert np.array_equal(idx.cpu().numpy(), ref["idx"]), f"call {call}: expert indices differ"
        assert np.array_equal(w.cpu().numpy().view(np.uint32), ref["weights"].view(np.uint32)), \
            f"call {call}: weights differ"
    layer.close()


def test_route_static_rejects_oversize(lib):
    import torch
    cm = lib
    x = torch.zeros((2048, 256), dtype=torch.int16, device="cuda")
    wr = torch.zeros((256, 256), dtype=torch.float32, device="cuda")
    idx = torch.zeros((2048, 8), dtype=torch.int32, device="cuda")
    w = torch.zeros((2048, 8), dtype=torch.float32, device="cuda")
    with pytest.raises(cm.ColiError) as e:       # 2048 * 256 > 262144
        cm.coli_moe_route_static(x, 2048, 256, wr, None, 256, 8, idx, w)
    assert e.value.code == cm.COLI_ERR_INVALID_ARG and "scratch limit" in str(e.value)
