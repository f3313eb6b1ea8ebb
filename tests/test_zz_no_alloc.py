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


# Shapes where a split count chosen from the size of the partial-logit buffer would differ
# between the two calls: few experts with many tokens, a layer created for more tokens than it
# routes, and T * E exactly at the fixed limit (1024 x 256 and 2048 x 128). Small experts (I = 128)
# keep the weights cheap; routing does not read them.
_EXTRA = {
    "na_e64_t1024": (S.Workload("na_e64_t1024", 1024, 4096, 64, 8, 128, 128, "normal"), None),
    "na_e256_t1024_max4096": (S.Workload("na_e256_t1024", 1024, 4096, 256, 8, 128, 128, "normal"), 4096),
    "na_e128_t2048": (S.Workload("na_e128_t2048", 2048, 2048, 128, 6, 128, 0, "normal"), None),
}


@pytest.mark.parametrize("name", ["decode", "sweep_T64", "prefill", *_EXTRA])
def test_route_static_matches_forward(lib, name):
    import torch
    cm = lib
    wl, max_tokens = _EXTRA.get(name, (name, None))
    inputs = S.make_inputs(wl)
    wl = inputs.workload
    layer = cm.MoELayer(inputs, max_tokens=max_tokens)
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
