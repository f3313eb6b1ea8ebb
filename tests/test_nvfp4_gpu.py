"""The NVFP4 variant of the layer on the GPU against the oracle's NVFP4 forward: routing bit-exact
from the GPU's scores, outputs within 2e-2 x RMS beyond half a bf16 ulp."""
import dataclasses

import numpy as np
import pytest

from routed_moe_fp4_gb300 import synthetic as S
from tests import parity as P

pytestmark = pytest.mark.gpu


def _run(inputs, T=None):
    import torch
    from routed_moe_fp4_gb300 import colimoe as cm
    T = inputs.workload.T if T is None else T
    layer = cm.NvMoELayer(inputs, max_tokens=max(T, 1))
    x = torch.from_numpy(inputs.x[:T].view(np.int16)).cuda()
    out = torch.full((T, inputs.workload.H), -1, dtype=torch.int16, device="cuda")
    layer.forward(x, out, T)
    torch.cuda.synchronize()
    routing = layer.routing(T)
    assert layer.device_error() == 0
    layer.close()
    return out.cpu().numpy().view(np.uint16), routing


def _check(oracle, inputs, got, routing, tokens):
    wl = inputs.workload
    idx_o, w_o = oracle.route(routing["scores"], inputs.router_b, wl.top_k)
    assert np.array_equal(idx_o, routing["idx"]) and np.array_equal(w_o.view(np.uint32),
                                                                    routing["weights"].view(np.uint32))
    tokens = sorted(set(int(t) for t in tokens))
    ref_bits, ref64 = oracle.tokens_output_nv(inputs.x, routing["idx"], routing["weights"], inputs.experts,
                                              inputs.shared, tokens)
    g = P.bf16_bits_to_f32(got[tokens]).astype(np.float64)
    rms = float(np.sqrt((ref64 ** 2).mean()))
    err = float(max((np.abs(g - ref64) - P.half_ulp_bf16(ref64)).max(), 0.0)) / rms
    assert err <= P.OUT_TOL, f"max error beyond half a bf16 ulp: {err:.3e} x RMS"
    return err


def test_nvfp4_tiny(oracle):
    inputs = S.make_nv_inputs("tiny")
    got, routing = _run(inputs)
    _check(oracle, inputs, got, routing, range(inputs.workload.T))


def test_nvfp4_decode_all_tokens(oracle):
    inputs = S.make_nv_inputs("decode")
    got, routing = _run(inputs)
    _check(oracle, inputs, got, routing, range(inputs.workload.T))


@pytest.mark.parametrize("T", [1, 63, 64, 130])
def test_nvfp4_token_counts(oracle, T):
    """Small-T and large-T routing paths, 16- and 32-token tiles, ragged tails."""
    inputs = S.make_nv_inputs("decode", T=T)
    got, routing = _run(inputs)
    _check(oracle, inputs, got, routing, P.sample_tokens(routing, T, min(T, 6)))


def test_nvfp4_prefill_sampled(oracle):
    inputs = S.make_nv_inputs("prefill")
    got, routing = _run(inputs)
    _check(oracle, inputs, got, routing, P.sample_tokens(routing, inputs.workload.T, 6))


def test_nvfp4_hidden_7168(oracle):
    """The larger hidden size (7168 = 448 groups of 16)."""
    inputs = S.make_nv_inputs("sweep_T4")
    got, routing = _run(inputs)
    _check(oracle, inputs, got, routing, range(inputs.workload.T))


def test_nvfp4_scale_edges(oracle):
    """Extreme E4M3 weight scales: the largest (448), subnormal, zero (a zeroed block), and a tiny
    matrix scale."""
    inputs = S.make_nv_inputs("tiny")
    ex = dataclasses.replace(inputs.experts)
    gs = ex.gate_up_scales.copy()
    gs[0, 0, 0] = 0x7E
    gs[0, 1, :] = 0x01
    gs[1, 2, 3] = 0x00
    ds = ex.down_scales.copy()
    ds[2, 5, 1] = 0x7E
    gg = ex.gate_up_global.copy()
    gg[3] = np.float32(2.0 ** -20)
    ex = dataclasses.replace(ex, gate_up_scales=gs, down_scales=ds, gate_up_global=gg)
    inputs = dataclasses.replace(inputs, experts=ex)
    got, routing = _run(inputs)
    _check(oracle, inputs, got, routing, range(inputs.workload.T))
