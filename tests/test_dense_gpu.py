"""The FP8 dense projection on the GPU against the oracle: every output of the small cases,
sampled outputs of the decode and prefill shapes, ragged token counts and a rectangular matrix."""
import dataclasses

import numpy as np
import pytest

from routed_moe_fp4_gb300 import synthetic as S
from tests import parity as P

pytestmark = pytest.mark.gpu

# x enters as two E4M3 terms (about 2^-9 relative per element) and the sums are fp32: far inside
# the layer's bar of 2e-2 x RMS beyond half a bf16 ulp.
TOL = 2e-2


def _run(inputs, T=None):
    import torch
    from routed_moe_fp4_gb300 import colimoe as cm
    T = inputs.workload.T if T is None else T
    layer = cm.DenseLayer(inputs, max_tokens=max(T, 1))
    x = torch.from_numpy(inputs.x[:T].view(np.int16)).cuda()
    out = torch.full((T, inputs.workload.N), -1, dtype=torch.int16, device="cuda")
    layer.forward(x, out, T)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    got = out.cpu().numpy().view(np.uint16)
    layer.close()
    return got


def _check(oracle, inputs, got, rows=None):
    x = inputs.x if rows is None else inputs.x[rows]
    ref_bits, ref64 = oracle.fp8_linear(np.ascontiguousarray(x), inputs.w, inputs.w_scale)
    g = P.bf16_bits_to_f32(got if rows is None else got[rows]).astype(np.float64)
    rms = float(np.sqrt((ref64 ** 2).mean()))
    excess = np.abs(g - ref64) - P.half_ulp_bf16(ref64)
    err = float(max(excess.max(), 0.0)) / rms
    assert err <= TOL, f"max error beyond half a bf16 ulp: {err:.3e} x RMS"
    agree = float((g == P.bf16_bits_to_f32(ref_bits)).mean())
    return err, agree


def test_dense_tiny_all_outputs(oracle):
    inputs = S.make_dense_inputs("dense_tiny")
    err, agree = _check(oracle, inputs, _run(inputs))
    assert agree > 0.9, agree


@pytest.mark.parametrize("T", [1, 7, 16, 17, 40, 64, 65, 130])
def test_dense_ragged_tokens(oracle, T):
    """Token counts around the 16/64/128-token tiles and their ragged tails (K 512, N 384)."""
    wl = S.DenseWorkload(f"dense_r{T}", T, 512, 384)
    inputs = S.make_dense_inputs(wl)
    _check(oracle, inputs, _run(inputs))


def test_dense_decode(oracle):
    inputs = S.make_dense_inputs("dense_decode")
    _check(oracle, inputs, _run(inputs))


def test_dense_prefill_sampled(oracle):
    inputs = S.make_dense_inputs("dense_prefill")
    got = _run(inputs)
    rows = np.array([0, 1, 127, 128, 255, 300, 511])
    _check(oracle, inputs, got, rows)


def test_dense_rectangular(oracle):
    """A wide matrix (N 1024 x K 7168, the larger hidden size) and a tall one (N 7168 x K 1024)."""
    for K, N in ((7168, 1024), (1024, 7168)):
        inputs = S.make_dense_inputs(S.DenseWorkload(f"dense_{K}x{N}", 9, K, N))
        _check(oracle, inputs, _run(inputs))


def test_dense_scale_edges(oracle):
    """Extreme codes (max 448, subnormals, both zeros) and power-of-two and odd block scales."""
    inputs = S.make_dense_inputs("dense_tiny")
    w = inputs.w.copy()
    w[0, :] = 0x7E
    w[1, :] = 0xFE
    w[2, ::2] = 0x01
    w[3, :] = 0x80
    sc = inputs.w_scale.copy()
    sc[0, 0] = 2.0 ** -20
    sc[1, 2] = 3.0e-3
    inputs = dataclasses.replace(inputs, w=w, w_scale=sc)
    _check(oracle, inputs, _run(inputs))


def test_dense_rejects_bad_shapes():
    import torch
    from routed_moe_fp4_gb300 import colimoe as cm
    d = cm.coli_dense_create(4, 256)
    x = torch.zeros((4, 256), dtype=torch.int16, device="cuda")
    w = torch.zeros((128, 256), dtype=torch.uint8, device="cuda")
    sc = torch.ones((1, 2), dtype=torch.float32, device="cuda")
    out = torch.zeros((4, 128), dtype=torch.int16, device="cuda")
    for args in ((5, 256, 128), (4, 384, 128), (4, 200, 128), (4, 256, 100)):
        with pytest.raises(cm.ColiError):
            cm.coli_dense_forward(d, x, args[0], args[1], w, sc, args[2], out)
    cm.coli_dense_forward(d, x, 4, 256, w, sc, 128, out)
    torch.cuda.synchronize()
    assert int(out.abs().max()) == 0
    cm.coli_dense_destroy(d)
