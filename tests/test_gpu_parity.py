"""CUDA path vs the oracle (needs a GB300). Every case goes through the C ABI."""
import dataclasses

import numpy as np
import pytest

from routed_moe_fp4_gb300 import synthetic as S
from tests import parity as P

pytestmark = pytest.mark.gpu

GEMV, AUTO, MXF4 = 1, 0, 2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from routed_moe_fp4_gb300 import build, colimoe
    build.build()
    colimoe.load()


def _assert_ok(rep, literal=True):
    """The parity bar; `literal` also holds the output to max|out - ref64| <= 2e-2 RMS with the bf16
    rounding included (the default FP4 path; the GEMV keeps h in bf16 and is held to the bar beyond
    the half ulp only)."""
    print(f"\nPARITY T={rep.T} tokens={rep.tokens_checked} score_err={rep.max_score_err:.2e} "
          f"routing_exact={rep.routing_bit_exact} own_diffs={rep.own_routing_diffs} "
          f"beyond_half_ulp={rep.rel_err:.3e} literal={rep.rel_err_literal:.3e} "
          f"vs_rounded_ref={rep.rel_err_bf16:.3e} launches={rep.launches}")
    assert rep.routing_bit_exact, "routing/permutation differ from the oracle on identical scores"
    assert rep.max_score_err <= P.SCORE_TOL, rep
    assert rep.rel_err <= P.OUT_TOL, rep
    if literal:
        assert rep.rel_err_literal <= P.OUT_TOL, rep


def _run(oracle, inputs, path, n_tokens=None, repeats=1):
    outs, routing, launches = P.run_gpu(inputs, path=path, repeats=repeats)
    T = inputs.x.shape[0]
    tokens = None if n_tokens is None or n_tokens >= T else P.sample_tokens(routing, T, n_tokens)
    rep = P.check(oracle, inputs, outs[0], routing, tokens, launches)
    return rep, outs, routing


@pytest.mark.parametrize("path", [GEMV, AUTO])
def test_tiny_all_tokens(oracle, path):
    inputs = S.make_inputs("tiny")
    rep, outs, _ = _run(oracle, inputs, path)
    _assert_ok(rep, literal=path != GEMV)
    assert rep.launches > 0


def test_tiny_matches_oracle_forward_exactly_routed(oracle):
    """The full oracle forward (its own scores) agrees with the GPU on routing for the tiny case."""
    inputs = S.make_inputs("tiny")
    outs, routing, _ = P.run_gpu(inputs)
    ref = oracle.moe_forward(inputs.x, inputs.router_w, inputs.router_b, 2, inputs.experts, inputs.shared)
    assert np.array_equal(ref["idx"], routing["idx"])
    got = P.bf16_bits_to_f32(outs[0]).astype(np.float64)
    excess = np.abs(got - ref["out_f64"]) - P.half_ulp_bf16(ref["out_f64"])
    assert excess.max() <= P.OUT_TOL * np.sqrt((ref["out_f64"] ** 2).mean())


def test_decode_all_tokens(oracle):
    inputs = S.make_inputs("decode")
    rep, _, _ = _run(oracle, inputs, AUTO)
    _assert_ok(rep)
    assert rep.own_routing_diffs == 0      # the margin workload has no near-ties


@pytest.mark.parametrize("T", list(S.SWEEP_T))
def test_sweep(oracle, T):
    inputs = S.make_inputs(f"sweep_T{T}")
    rep, _, _ = _run(oracle, inputs, AUTO, n_tokens=6)
    _assert_ok(rep)


def test_prefill_all_tokens(oracle):
    """All 512 tokens of the prefill chunk against the oracle."""
    inputs = S.make_inputs("prefill")
    rep, _, _ = _run(oracle, inputs, AUTO)
    _assert_ok(rep)
    assert rep.tokens_checked == 512


def test_v4pro_decode_all_tokens(oracle):
    """The V4-Pro shape (E = 384, H = 7168): every token against the oracle."""
    inputs = S.make_inputs("v4pro_decode")
    rep, _, _ = _run(oracle, inputs, AUTO)
    _assert_ok(rep)


def test_skewed_sampled(oracle):
    """256 of the 4096 tokens: the first and last rows of the Zipf head expert, the lightest
    expert, last rows of partial tiles of each box height, and a seeded sample; routing and the
    permutation are compared on every token."""
    inputs = S.make_inputs("skewed")
    outs, routing, launches = P.run_gpu(inputs)
    named = P.structured_tokens(routing, inputs.workload.T, 256)
    print("\nskewed tokens: " + ", ".join(f"{k}={v}" for k, v in named.items() if not k.startswith("sample")))
    assert {"heavy_first_row", "heavy_last_row", "lightest_expert", "partial_tile_1_16",
            "partial_tile_17_32", "partial_tile_33_47"} <= set(named)
    rep = P.check(oracle, inputs, outs[0], routing, list(named.values()), launches)
    _assert_ok(rep)
    assert rep.tokens_checked >= 256
    assert routing["cnt"][:-1].max() > 3000      # the Zipf head expert


def test_skewed_e32_sampled(oracle):
    """About 256 rows per expert at hidden 7168: the big-tile launches on a production shape."""
    inputs = S.make_inputs("skewed_e32")
    rep, _, _ = _run(oracle, inputs, AUTO, n_tokens=12)
    _assert_ok(rep)


def test_repeatable_bitwise(oracle):
    """Two forwards on the same inputs give bit-identical outputs (fixed-order reductions)."""
    inputs = S.make_inputs("sweep_T16")
    outs, _, _ = P.run_gpu(inputs, repeats=2)
    assert np.array_equal(outs[0], outs[1])


@pytest.mark.parametrize("name", ["sweep_T1", "sweep_T4", "decode"])
def test_graph_replay_matches_eager(name):
    """A forward captured in a CUDA graph and replayed on new inputs gives the eager forward's bytes:
    at 4 and 8 tokens the down launch starts per expert on counters that every forward's x-term
    kernel zeroes, at one token it waits for the whole gate/up launch."""
    import torch
    from routed_moe_fp4_gb300 import colimoe as cm
    inputs = S.make_inputs(name)
    wl = inputs.workload
    stream = torch.cuda.Stream()
    layer = cm.MoELayer(inputs, stream=stream)
    xs = [torch.from_numpy(S.x_batch(0, wl.name, 100 + i, wl.T, wl.H).view(np.int16)).cuda() for i in range(3)]
    x = xs[0].clone()
    out = torch.empty_like(x)
    eager = []
    for xi in xs:
        layer.forward(xi, out)
        stream.synchronize()
        eager.append(out.cpu().numpy().copy())
    layer.forward(x, out)          # warm (kernel attributes and tensor maps) before the capture
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        layer.forward(x, out)
    for i, xi in enumerate(xs):
        with torch.cuda.stream(stream):
            x.copy_(xi)
            g.replay()
        stream.synchronize()
        assert np.array_equal(out.cpu().numpy(), eager[i]), f"replay {i} differs from the eager forward"
    assert layer.device_error() == 0
    del g
    layer.close()


def _custom(name, **kw):
    base = dataclasses.replace(S.WORKLOADS["tiny"], name=name)
    return dataclasses.replace(base, **kw)


@pytest.mark.parametrize("wl", [
    _custom("edge_k1", top_k=1),
    _custom("edge_E1", E=1, top_k=1),
    _custom("edge_noshared", I_s=0),
    _custom("edge_shared_wider", I_s=256),
    _custom("edge_ragged", T=37, H=384, E=16, top_k=3),
    _custom("edge_T1", T=1),
    _custom("edge_many_experts", T=9, E=300, top_k=8, H=256),
    _custom("edge_k32_T63", T=63, E=64, top_k=32),        # largest single-block routing (63 x 32 slots)
    _custom("edge_T64", T=64, E=16, top_k=4),             # smallest T of the multi-kernel routing
    _custom("edge_E1024", T=5, E=1024, top_k=8, H=256),   # widest expert set (NPL = 32)
], ids=lambda w: w.name)
def test_edge_cases(oracle, wl):
    inputs = S.make_inputs(wl)
    rep, _, _ = _run(oracle, inputs, AUTO)
    _assert_ok(rep)


@pytest.mark.parametrize("path", [MXF4, GEMV], ids=["mxf4", "gemv"])
@pytest.mark.parametrize("name", ["tiny", "decode", "sweep_T16", "sweep_T128"])
def test_ffn_paths(oracle, name, path):
    """Each FFN path, forced, against the oracle."""
    inputs = S.make_inputs(name)
    rep, _, _ = _run(oracle, inputs, path, n_tokens=8)
    _assert_ok(rep, literal=path != GEMV)


@pytest.mark.parametrize("wl", [
    _custom("gemm_ragged", T=37, H=384, E=16, top_k=3),
    _custom("gemm_shared_wider", I_s=256),
    _custom("gemm_noshared", I_s=0),
    _custom("gemm_many_rows", T=300, E=4, top_k=2),
    _custom("gemm_half_stages", T=21, H=640, I=384, I_s=256, E=12, top_k=3),
    # a small batch (x terms per token) with 32-token gate/up tiles: the shared expert's 40 rows
    # take one 32-row and one 16-row box
    _custom("gemm_small_gu32", T=40, H=512, E=8, top_k=8, I=256, I_s=256),
    # 48 or more rows per expert on average with H a multiple of 256: both launches take 48-token
    # tiles with two weight matrices each (ragged last tiles, a wider shared expert, K = 3 x 256)
    _custom("big_ragged", T=200, H=512, E=8, top_k=2, I=256, I_s=384),
    _custom("big_many_rows", T=400, H=768, E=6, top_k=3, I=384, I_s=128),
    # H, I and I_s multiples of 512: the scale bytes come by TMA with each stage, for big tiles
    # and for small ones with a shared expert twice as wide as the routed ones
    _custom("sft_big", T=200, H=512, E=8, top_k=2, I=512, I_s=512),
    _custom("sft_shared_wider", T=21, H=512, E=12, top_k=3, I=512, I_s=1024),
], ids=lambda w: w.name)
@pytest.mark.parametrize("path", [MXF4, GEMV], ids=["mxf4", "gemv"])
def test_gemm_edge_cases(oracle, wl, path):
    inputs = S.make_inputs(wl)
    rep, _, _ = _run(oracle, inputs, path)
    _assert_ok(rep, literal=path != GEMV)


@pytest.mark.parametrize("path", [MXF4], ids=["mxf4"])
def test_gemm_matches_gemv(oracle, path):
    """The two FFN paths agree with each other within the parity bar on the same routing."""
    inputs = S.make_inputs("sweep_T64")
    o1, r1, _ = P.run_gpu(inputs, path=GEMV)
    o2, r2, _ = P.run_gpu(inputs, path=path)
    assert np.array_equal(r1["idx"], r2["idx"])
    a = P.bf16_bits_to_f32(o1[0]).astype(np.float64)
    b = P.bf16_bits_to_f32(o2[0]).astype(np.float64)
    rms = np.sqrt((a ** 2).mean())
    assert np.abs(a - b).max() <= 2 * P.OUT_TOL * rms


def test_zero_tokens_is_noop():
    import torch
    from routed_moe_fp4_gb300 import colimoe as cm
    inputs = S.make_inputs("tiny")
    layer = cm.MoELayer(inputs)
    x = torch.zeros((1, 256), dtype=torch.int16, device="cuda")
    out = torch.full((1, 256), 7, dtype=torch.int16, device="cuda")
    layer.forward(x, out, T=0)
    torch.cuda.synchronize()
    assert int(out[0, 0]) == 7 and layer.launches() == 0
    layer.close()


def test_bad_arguments_rejected():
    import torch
    from routed_moe_fp4_gb300 import colimoe as cm
    inputs = S.make_inputs("tiny")
    layer = cm.MoELayer(inputs)
    x = torch.zeros((4, 256), dtype=torch.int16, device="cuda")
    out = torch.zeros_like(x)
    with pytest.raises(cm.ColiError) as e:
        cm.coli_moe_forward(layer.h, x, 5, layer.router_w, None, layer.experts.struct, None, 2, out)
    assert e.value.code == cm.COLI_ERR_INVALID_ARG and "max_tokens" in str(e.value)
    with pytest.raises(cm.ColiError):
        cm.coli_moe_forward(layer.h, x, 4, layer.router_w, None, layer.experts.struct, None, 3, out)
    with pytest.raises(cm.ColiError):
        cm.coli_moe_forward(layer.h, x, 4, layer.router_w, None, layer.experts.struct, None, 2, x)
    # out may not overlap x even in part; adjacent buffers are fine
    buf = torch.zeros((8, 256), dtype=torch.int16, device="cuda")
    with pytest.raises(cm.ColiError) as e:
        cm.coli_moe_forward(layer.h, buf[:4], 4, layer.router_w, None, layer.experts.struct, None, 2, buf[2:6])
    assert e.value.code == cm.COLI_ERR_INVALID_ARG and "overlap" in str(e.value)
    cm.coli_moe_forward(layer.h, buf[:4], 4, layer.router_w, None, layer.experts.struct, None, 2, buf[4:])
    torch.cuda.synchronize()
    layer.close()


@pytest.mark.parametrize("pinned", [True, False], ids=["mapped", "pageable"])
def test_forward_host_matches_device(oracle, pinned):
    """Host buffers give the device forward's bits, read in place when page-locked, else copied."""
    import torch
    from routed_moe_fp4_gb300 import colimoe as cm
    inputs = S.make_inputs("sweep_T4")
    outs, _, _ = P.run_gpu(inputs)
    layer = cm.MoELayer(inputs)
    x_host = torch.from_numpy(inputs.x.view(np.int16).copy())
    out_host = torch.zeros_like(x_host)
    if pinned:
        x_host, out_host = x_host.pin_memory(), out_host.pin_memory()
    for _ in range(2):
        out_host.zero_()
        layer.forward_host(x_host, out_host)
        assert np.array_equal(out_host.numpy().view(np.uint16), outs[0])
    layer.close()


def test_auto_path_is_mxf4():
    """The automatic choice on a GB300 is the FP4 x FP4 block-scaled GEMM, and the handle reports it."""
    import torch
    from routed_moe_fp4_gb300 import colimoe as cm
    inputs = S.make_inputs("tiny")
    layer = cm.MoELayer(inputs)
    assert layer.ffn_path() == cm.COLI_FFN_AUTO
    x = torch.from_numpy(inputs.x.view(np.int16)).cuda()
    out = torch.empty_like(x)
    layer.forward(x, out)
    torch.cuda.synchronize()
    assert layer.ffn_path() == cm.COLI_FFN_GEMM_MXF4
    layer.set_ffn_path(cm.COLI_FFN_GEMV)
    layer.forward(x, out)
    assert layer.ffn_path() == cm.COLI_FFN_GEMV
    layer.close()
