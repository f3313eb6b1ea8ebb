"""The FP8 dense projection on the GPU against the oracle: every output of the small cases,
sampled outputs of the decode and prefill shapes, ragged token counts and a rectangular matrix."""
import dataclasses

import numpy as np
import pytest

from routed_moe_fp4_gb300 import synthetic as S
from tests import parity as P

pytestmark = pytest.mark.gpu

# Tensor-core path: x enters as two E4M3 terms (about 2^-9 relative per element) and the sums are
# fp32. CUDA-core path: exact products, fp32 sums. Both far inside the layer's bar of 2e-2 x RMS
# beyond half a bf16 ulp.
TOL = 2e-2
AUTO, CORES, TENSOR = 0, 1, 2


def _run(inputs, T=None, path=AUTO, expect=None):
    """Runs the projection on `path` (forced unless AUTO); `expect` is the path the forward must
    report having taken."""
    import torch
    from routed_moe_fp4_gb300 import colimoe as cm
    T = inputs.workload.T if T is None else T
    layer = cm.DenseLayer(inputs, max_tokens=max(T, 1))
    if path != AUTO:
        layer.set_path(path)
    x = torch.from_numpy(inputs.x[:T].view(np.int16)).cuda()
    out = torch.full((T, inputs.workload.N), -1, dtype=torch.int16, device="cuda")
    layer.forward(x, out, T)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    ran = layer.last_path()
    assert ran == (expect if expect is not None else path if path != AUTO else ran), ran
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


@pytest.mark.parametrize("path", [CORES, TENSOR])
def test_dense_tiny_all_outputs(oracle, path):
    inputs = S.make_dense_inputs("dense_tiny")
    err, agree = _check(oracle, inputs, _run(inputs, path=path))
    assert agree > (0.99 if path == CORES else 0.9), agree


@pytest.mark.parametrize("T", [1, 7, 16, 17, 40, 64, 65, 130])
def test_dense_ragged_tokens(oracle, T):
    """Token counts around the 16/64/128-token tiles and their ragged tails (K 512, N 384); for this
    small matrix the automatic choice takes the CUDA-core kernel up to 8 tokens."""
    wl = S.DenseWorkload(f"dense_r{T}", T, 512, 384)
    inputs = S.make_dense_inputs(wl)
    _check(oracle, inputs, _run(inputs, expect=CORES if T <= 8 else TENSOR))


@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 8, 9, 16, 17])
def test_dense_cuda_cores_tokens(oracle, T):
    """The CUDA-core kernel at every tokens-per-pass size (1, 2, 4, 8) and with two or three passes."""
    wl = S.DenseWorkload(f"dense_c{T}", T, 512, 384)
    inputs = S.make_dense_inputs(wl)
    err, agree = _check(oracle, inputs, _run(inputs, path=CORES))
    assert agree > 0.99, agree


@pytest.mark.parametrize("path", [CORES, TENSOR])
def test_dense_decode(oracle, path):
    inputs = S.make_dense_inputs("dense_decode")
    _check(oracle, inputs, _run(inputs, path=path))


@pytest.mark.parametrize("T,K,N,expect", [(8, 4096, 4096, TENSOR), (1, 4096, 4096, TENSOR), (8, 7168, 512, CORES),
                                           (4, 7168, 1024, CORES), (8, 7168, 1024, TENSOR), (2, 7168, 2048, CORES),
                                           (4, 7168, 2048, TENSOR)])
def test_dense_auto_path(T, K, N, expect):
    """The automatic choice: the CUDA-core kernel for few tokens on small matrices, where it measured
    faster, the tensor-core GEMM otherwise."""
    inputs = S.make_dense_inputs(S.DenseWorkload(f"dense_a{T}_{K}_{N}", T, K, N))
    _run(inputs, expect=expect)


def test_dense_prefill_sampled(oracle):
    inputs = S.make_dense_inputs("dense_prefill")
    got = _run(inputs)
    rows = np.array([0, 1, 127, 128, 255, 300, 511])
    _check(oracle, inputs, got, rows)


@pytest.mark.parametrize("path", [CORES, TENSOR])
def test_dense_rectangular(oracle, path):
    """A wide matrix (N 1024 x K 7168, the larger hidden size) and a tall one (N 7168 x K 1024); on
    the CUDA-core kernel K 7168 takes 4 tokens per pass, so 9 tokens make three passes."""
    for K, N in ((7168, 1024), (1024, 7168)):
        inputs = S.make_dense_inputs(S.DenseWorkload(f"dense_{K}x{N}", 9, K, N))
        _check(oracle, inputs, _run(inputs, path=path))


@pytest.mark.parametrize("path", [CORES, TENSOR])
def test_dense_scale_edges(oracle, path):
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
    _check(oracle, inputs, _run(inputs, path=path))


@pytest.mark.parametrize("path", [CORES, TENSOR])
def test_dense_nan_codes(oracle, path):
    """A NaN code (S.1111.111) in a weight row makes that row's outputs NaN for every token, as the
    oracle's exact sum does; the other rows are unaffected."""
    inputs = S.make_dense_inputs("dense_tiny")
    w = inputs.w.copy()
    w[5, 17] = 0x7F
    w[130, 300] = 0xFF
    w[w == 0x7F] = 0x7E                 # no other NaN codes
    w[w == 0xFF] = 0xFE
    w[5, 17], w[130, 300] = 0x7F, 0xFF
    inputs = dataclasses.replace(inputs, w=w)
    got = _run(inputs, path=path)
    ref_bits, ref64 = oracle.fp8_linear(inputs.x, inputs.w, inputs.w_scale)
    g = P.bf16_bits_to_f32(got).astype(np.float64)
    assert np.array_equal(np.isnan(g), np.isnan(ref64)) and np.isnan(ref64[:, [5, 130]]).all()
    ok = ~np.isnan(ref64)
    rms = float(np.sqrt((ref64[ok] ** 2).mean()))
    excess = np.abs(g[ok] - ref64[ok]) - P.half_ulp_bf16(ref64[ok])
    assert float(max(excess.max(), 0.0)) / rms <= TOL


def test_dense_path_argument_checks():
    """An unknown path is refused; a forced CUDA-core path refuses a shape it cannot hold (K above
    8192) and the tensor-core path still runs it."""
    import torch
    from routed_moe_fp4_gb300 import colimoe as cm
    d = cm.coli_dense_create(2, 8448)
    with pytest.raises(cm.ColiError):
        cm.coli_dense_set_path(d, 3)
    x = torch.zeros((2, 8448), dtype=torch.int16, device="cuda")
    w = torch.zeros((128, 8448), dtype=torch.uint8, device="cuda")
    sc = torch.ones((1, 66), dtype=torch.float32, device="cuda")
    out = torch.full((2, 128), -1, dtype=torch.int16, device="cuda")
    cm.coli_dense_set_path(d, CORES)
    with pytest.raises(cm.ColiError) as e:
        cm.coli_dense_forward(d, x, 2, 8448, w, sc, 128, out)
    assert "8192" in str(e.value)
    cm.coli_dense_set_path(d, AUTO)
    cm.coli_dense_forward(d, x, 2, 8448, w, sc, 128, out)
    torch.cuda.synchronize()
    assert cm.coli_dense_last_path(d) == TENSOR and int(out.abs().max()) == 0
    cm.coli_dense_destroy(d)


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
