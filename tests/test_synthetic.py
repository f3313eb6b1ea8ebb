"""The seeded input generator: published SplitMix64 output, determinism, distributions."""
import numpy as np

from routed_moe_fp4_gb300 import synthetic as S


def test_splitmix64_published_first_output():
    # SplitMix64 from state 0: the first output is 0xE220A8397B1DCDAF (reference C code).
    assert int(S.u64_stream(0, 1)[0]) == 0xE220A8397B1DCDAF


def test_counter_based_streams():
    k = S.stream_key(0, "a", 1)
    full = S.u64_stream(k, 100)
    assert np.array_equal(full[40:60], S.u64_stream(k, 20, start=40))
    assert S.stream_key(0, "a", 1) != S.stream_key(0, "a", 2) != S.stream_key(1, "a", 1)


def test_bf16_rounding_ties_to_even():
    v = np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 1.0 + 2 ** -8 + 2 ** -20], np.float32)
    assert S.f32_to_bf16_bits(v).tolist() == [0x3F80, 0x3F82, 0xC020, 0x3F81]


def test_value_distributions():
    inp = S.make_inputs("tiny", 0)
    wl = inp.workload
    x = (inp.x.astype(np.uint32) << 16).view(np.float32)
    assert abs(x.mean()) < 0.1 and abs(x.std() - 1.0) < 0.1
    assert abs(inp.router_w.std() - 0.02) < 0.002
    assert inp.router_b is None
    sc = inp.experts.gate_up_scales
    assert sc.min() == 121 and sc.max() == 125
    nib = np.concatenate([inp.experts.down_codes.reshape(-1) & 15, inp.experts.down_codes.reshape(-1) >> 4])
    counts = np.bincount(nib, minlength=16)
    assert counts.min() > 0.8 * nib.size / 16
    assert inp.experts.gate_up_codes.shape == (wl.E, 2 * wl.I, wl.H // 2)
    assert inp.shared.down_scales.shape == (1, wl.H, wl.I_s // 32)


def test_deterministic_and_row_streams():
    a = S.make_inputs("tiny", 0)
    b = S.make_inputs("tiny", 0)
    assert np.array_equal(a.x, b.x) and np.array_equal(a.experts.down_codes, b.experts.down_codes)
    c = S.make_inputs("tiny", 1)
    assert not np.array_equal(a.x, c.x)
    # T override keeps each row's stream
    d = S.make_inputs("tiny", 0, T=2, with_experts=False)
    assert np.array_equal(d.x, a.x[:2])


def test_zipf_rank_is_permutation():
    r = S.zipf_rank(0, 256)
    assert sorted(r.tolist()) == list(range(256))


def test_calibration_present():
    cal = S.calibration()
    wl = S.WORKLOADS["skewed"]
    assert len(cal["decode_row_attempts"]) == S.WORKLOADS["decode"].T
    assert len(cal["skewed_router_bias"]) == wl.E
    slots = np.array(cal["skewed_slots_by_rank"], np.float64)
    target = np.array(cal["skewed_target_slots_by_rank"], np.float64)
    assert slots.sum() == wl.T * wl.top_k
    # popularity follows the Zipf(1.1) targets: within 20% (log) for every rank
    assert np.abs(np.log(slots + 1) - np.log(target + 1)).max() < 0.2
    # a Zipf law: log-log slope of slots vs rank over ranks 2..200 is close to -1.1
    r = np.arange(2, 201)
    slope = np.polyfit(np.log(r + 1.0), np.log(slots[r]), 1)[0]
    assert -1.25 < slope < -0.95, slope
    inp = S.make_inputs("skewed", 0, T=1, with_experts=False)
    assert np.array_equal(inp.router_b, np.array(cal["skewed_router_bias"], np.float32))


def test_dense_inputs_have_no_nan_codes_and_positive_scales():
    from routed_moe_fp4_gb300 import synthetic as S
    d = S.make_dense_inputs("dense_tiny")
    assert d.w.shape == (256, 384) and d.w_scale.shape == (2, 3) and d.x.shape == (5, 384)
    assert not np.any((d.w & 0x7F) == 0x7F), "E4M3 NaN code in the weights"
    assert np.all(d.w_scale > 0) and np.all(np.isfinite(d.w_scale))
    assert np.array_equal(d.w, S.make_dense_inputs("dense_tiny").w), "not seeded"


def test_nvfp4_experts_scale_bytes():
    from routed_moe_fp4_gb300 import synthetic as S
    ex = S.make_nv_experts(0, "t", 2, 256, 128)
    assert ex.gate_up_scales.shape == (2, 256, 16) and ex.down_scales.shape == (2, 256, 8)
    e = (ex.gate_up_scales >> 3) & 15
    assert e.min() >= 4 and e.max() <= 8 and not np.any(ex.gate_up_scales & 0x80)
    assert np.all((ex.gate_up_global >= 2.0 ** -6) & (ex.gate_up_global < 2.0 ** -5))


def test_x_batches_are_distinct_streams():
    from routed_moe_fp4_gb300 import synthetic as S
    a = S.x_batch(0, "decode", 1, 4, 256)
    b = S.x_batch(0, "decode", 2, 4, 256)
    assert a.shape == (4, 256) and not np.array_equal(a, b)
    assert np.array_equal(a, S.x_batch(0, "decode", 1, 4, 256))
