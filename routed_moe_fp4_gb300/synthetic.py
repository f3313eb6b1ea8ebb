"""Seeded synthetic inputs for the routed MXFP4 MoE layer.

This module only draws numbers. It holds none of the layer's arithmetic (no
logits, no sigmoid, no top-k, no matmul); both the CUDA path and the CPU oracle
consume the arrays it returns.

Random source: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014), used as a counter-based generator: element i of a
stream with key K is mix64(K + (i + 1) * 0x9E3779B97F4A7C15). A stream key is
mix64 of the FNV-1a 64-bit hash of a text tag (seed, tensor name, indices), so
every tensor, expert and token row has its own stream and any single row can be
redrawn without touching the others.

Value recipes (the shapes and distributions of the DeepSeek-V4 expert layer as
described on "DeepSeek V4 Flash CPU inference with NVMe expert streaming": hidden
4096 x moe_inter 2048, 256 experts, FP4 E2M1 experts with UE8M0 group-32 scales):
  * x      : N(0, 1) drawn in float64, rounded to float32, then RNE to bf16.
  * router : N(0, 0.02^2), float32.
  * bias   : zero, N(0, 0.01^2), or the stored per-expert bias of the skewed workload, under
             which expert popularity (routed slots by seeded rank) follows Zipf(1.1).
  * codes  : uniform bytes, i.e. two uniform E2M1 nibbles (the -0 code included).
  * scales : UE8M0 bytes 127 + U{-6..-2}.
Normals use the Box-Muller transform on two independent streams.
"""
from __future__ import annotations

import concurrent.futures as _cf
import dataclasses
import json
import math
import os
from typing import Dict, List, Optional

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_MASK64 = (1 << 64) - 1


def _mix64_int(z: int) -> int:
    z &= _MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
    return z ^ (z >> 31)


def _fnv1a64(text: str) -> int:
    h = 0xCBF29CE484222325
    for b in text.encode("utf-8"):
        h ^= b
        h = (h * 0x100000001B3) & _MASK64
    return h


def stream_key(seed: int, *tags) -> int:
    """64-bit key of the stream named by (seed, tags)."""
    return _mix64_int(_fnv1a64("/".join([str(seed)] + [str(t) for t in tags])))


def u64_stream(key: int, count: int, start: int = 0) -> np.ndarray:
    """Elements [start, start+count) of the SplitMix64 stream with this key."""
    with np.errstate(over="ignore"):
        i = np.arange(start + 1, start + 1 + count, dtype=np.uint64)
        z = np.uint64(key) + i * _GOLDEN
        z ^= z >> np.uint64(30)
        z *= _M1
        z ^= z >> np.uint64(27)
        z *= _M2
        z ^= z >> np.uint64(31)
    return z


def uniform01(key: int, count: int) -> np.ndarray:
    """Uniform doubles in [0, 1) with 53 random bits."""
    return (u64_stream(key, count) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normal(key: int, count: int) -> np.ndarray:
    """Standard normals by Box-Muller from two independent uniform streams."""
    u1 = ((u64_stream(_mix64_int(key ^ 0xA5A5A5A5A5A5A5A5), count) >> np.uint64(11))
          .astype(np.float64) + 1.0) * (2.0 ** -53)          # (0, 1]
    u2 = uniform01(_mix64_int(key ^ 0x5A5A5A5A5A5A5A5A), count)  # [0, 1)
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (round to nearest, ties to even); returns uint16 bits."""
    b = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    return ((b + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def random_bytes(key: int, count: int) -> np.ndarray:
    """`count` uniform bytes: byte j of stream element i is bits [8j, 8j+8)."""
    n = (count + 7) // 8
    return u64_stream(key, n).astype("<u8").view(np.uint8)[:count].copy()


def scale_bytes(key: int, count: int) -> np.ndarray:
    """UE8M0 scale bytes 127 + e with e uniform in {-6, ..., -2} (Lemire's multiply-shift)."""
    hi = u64_stream(key, count) >> np.uint64(32)
    return (np.uint64(121) + ((hi * np.uint64(5)) >> np.uint64(32))).astype(np.uint8)


# --------------------------------------------------------------------------------------
# Workloads


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    E: int
    top_k: int
    I: int
    I_s: int          # shared-expert intermediate size; 0 = no shared expert
    bias: str         # "zero" | "normal" | "zipf"
    margin: float = 0.0   # > 0: token rows are redrawn until the top-k key gaps exceed it


WORKLOADS: Dict[str, Workload] = {
    "tiny": Workload("tiny", 4, 256, 8, 2, 128, 128, "zero"),
    "decode": Workload("decode", 8, 4096, 256, 8, 2048, 2048, "normal", margin=1e-3),
    "prefill": Workload("prefill", 512, 4096, 256, 8, 2048, 2048, "normal"),
    "skewed": Workload("skewed", 4096, 7168, 256, 8, 2048, 2048, "zipf"),
    # the larger V4 shape of the pages (hidden 7168, 384 experts, same MXFP4 layout); top-8 and
    # I = I_s = 2048 as in the other workloads (the pages give neither for it)
    "v4pro_decode": Workload("v4pro_decode", 8, 7168, 384, 8, 2048, 2048, "normal"),
    # a reduced stand-in for the skewed prefill's heavy experts, small enough for a counter capture
    # (33 experts, 0.77 GB): hidden 7168 with about 256 rows per expert, so the expert GEMMs run in
    # the compute-heavy regime of the large groups
    "skewed_e32": Workload("skewed_e32", 1024, 7168, 32, 8, 2048, 2048, "normal"),
}
SWEEP_T = (1, 2, 4, 16, 64, 128)
for _t in SWEEP_T:
    WORKLOADS[f"sweep_T{_t}"] = Workload(f"sweep_T{_t}", _t, 7168, 256, 8, 2048, 2048, "normal")

_CALIBRATION_FILE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "workload_calibration.json")


def calibration() -> dict:
    """Input-recipe constants written by oracle/calibrate_workloads.py (row redraw counts
    for the margin workload, the skewed workload's router bias)."""
    if not os.path.exists(_CALIBRATION_FILE):
        return {}
    with open(_CALIBRATION_FILE) as f:
        return json.load(f)


def zipf_rank(seed: int, E: int) -> np.ndarray:
    """A seeded permutation: rank[e] is expert e's popularity rank (0 = most popular)."""
    order = np.argsort(u64_stream(stream_key(seed, "zipf_perm", E), E), kind="stable")
    rank = np.empty(E, dtype=np.int64)
    rank[order] = np.arange(E)
    return rank


@dataclasses.dataclass
class MXFP4Experts:
    """Host arrays in the library's packed layout (K-major rows, low nibble = even k)."""
    gate_up_codes: np.ndarray   # uint8 [E, 2I, H/2]: gate rows then up rows
    gate_up_scales: np.ndarray  # uint8 [E, 2I, H/32]
    down_codes: np.ndarray      # uint8 [E, H, I/2]
    down_scales: np.ndarray     # uint8 [E, H, I/32]

    @property
    def nbytes(self) -> int:
        return sum(a.nbytes for a in (self.gate_up_codes, self.gate_up_scales,
                                      self.down_codes, self.down_scales))


@dataclasses.dataclass
class MoEInputs:
    workload: Workload
    x: np.ndarray               # uint16 bf16 bits [T, H]
    router_w: np.ndarray        # float32 [E, H]
    router_b: Optional[np.ndarray]  # float32 [E] or None (zero bias)
    experts: MXFP4Experts
    shared: Optional[MXFP4Experts]  # E = 1


def x_row(seed: int, wl_name: str, t: int, H: int, attempt: int = 0) -> np.ndarray:
    """Token row t as bf16 bits; `attempt` selects a redraw of that row."""
    z = normal(stream_key(seed, wl_name, "x", t, attempt), H)
    return f32_to_bf16_bits(z.astype(np.float32))


def x_batch(seed: int, wl_name: str, batch: int, T: int, H: int) -> np.ndarray:
    """A further batch of T token rows (bf16 bits [T, H]) of a workload, batch >= 1: a stream of
    distinct batches, as successive forwards of a layer see them."""
    if T == 0:
        return np.zeros((0, H), np.uint16)
    return np.stack([f32_to_bf16_bits(normal(stream_key(seed, wl_name, "x-batch", batch, t), H).astype(np.float32))
                     for t in range(T)])


def _expert_arrays(seed: int, tag: str, e: int, H: int, I: int):
    gu_c = random_bytes(stream_key(seed, tag, e, "gate_up_codes"), 2 * I * H // 2).reshape(2 * I, H // 2)
    gu_s = scale_bytes(stream_key(seed, tag, e, "gate_up_scales"), 2 * I * H // 32).reshape(2 * I, H // 32)
    d_c = random_bytes(stream_key(seed, tag, e, "down_codes"), H * I // 2).reshape(H, I // 2)
    d_s = scale_bytes(stream_key(seed, tag, e, "down_scales"), H * I // 32).reshape(H, I // 32)
    return gu_c, gu_s, d_c, d_s


def make_experts(seed: int, tag: str, E: int, H: int, I: int, threads: Optional[int] = None) -> MXFP4Experts:
    """E experts of shape (H, I); tag "experts" or "shared". Experts are drawn in parallel."""
    out = MXFP4Experts(np.empty((E, 2 * I, H // 2), np.uint8), np.empty((E, 2 * I, H // 32), np.uint8),
                       np.empty((E, H, I // 2), np.uint8), np.empty((E, H, I // 32), np.uint8))

    def fill(e):
        gu_c, gu_s, d_c, d_s = _expert_arrays(seed, tag, e, H, I)
        out.gate_up_codes[e] = gu_c
        out.gate_up_scales[e] = gu_s
        out.down_codes[e] = d_c
        out.down_scales[e] = d_s

    n = threads or min(16, os.cpu_count() or 1)
    if E == 1 or n == 1:
        for e in range(E):
            fill(e)
    else:
        with _cf.ThreadPoolExecutor(n) as ex:
            list(ex.map(fill, range(E)))
    return out


def make_inputs(name, seed: int = 0, T: Optional[int] = None, with_experts: bool = True,
                unbiased: bool = False) -> MoEInputs:
    """All inputs of a workload (a name in WORKLOADS or a Workload). `T` overrides the token count
    (rows keep their streams). `unbiased` returns no router bias (used when the stored bias is
    being fitted)."""
    wl = WORKLOADS[name] if isinstance(name, str) else name
    if T is not None:
        wl = dataclasses.replace(wl, T=T)
    cal = calibration()
    attempts: List[int] = [0] * wl.T
    if wl.margin > 0:
        redraw = cal.get(f"{wl.name}_row_attempts", [])
        for t in range(min(wl.T, len(redraw))):
            attempts[t] = int(redraw[t])
    x = np.stack([x_row(seed, wl.name, t, wl.H, attempts[t]) for t in range(wl.T)]) if wl.T > 0 \
        else np.zeros((0, wl.H), np.uint16)
    router_w = (0.02 * normal(stream_key(seed, wl.name, "router_w"), wl.E * wl.H)).astype(np.float32)
    router_w = router_w.reshape(wl.E, wl.H)
    if wl.bias == "zero" or unbiased:
        router_b = None
    elif wl.bias == "normal":
        router_b = (0.01 * normal(stream_key(seed, wl.name, "router_b"), wl.E)).astype(np.float32)
    elif wl.bias == "zipf":
        stored = cal.get(f"{wl.name}_router_bias")
        if stored is None or len(stored) != wl.E or seed != 0:
            raise ValueError(f"no stored Zipf router bias for workload {wl.name} with seed {seed}")
        router_b = np.asarray(stored, np.float32)
    else:
        raise ValueError(wl.bias)
    if with_experts:
        experts = make_experts(seed, wl.name + "/experts", wl.E, wl.H, wl.I)
        shared = make_experts(seed, wl.name + "/shared", 1, wl.H, wl.I_s) if wl.I_s > 0 else None

    else:
        experts = shared = None
    return MoEInputs(wl, x, router_w, router_b, experts, shared)


def expert_bytes(H: int, I: int) -> int:
    """Bytes of one MXFP4 expert (gate, up and down matrices with their scales)."""
    return 3 * H * I // 2 + 3 * H * I // 32


# --------------------------------------------------------------------------------------
# FP8 dense projections (y = x W^T, W E4M3 with one fp32 scale per 128 x 128 block)


@dataclasses.dataclass(frozen=True)
class DenseWorkload:
    name: str
    T: int
    K: int            # input features (x columns, W columns)
    N: int            # output features (W rows)


# One per-layer dense projection of the hidden-4096 model (a 4096 x 4096 matrix: the pages name
# the five projections but not their sizes), in decode and prefill, plus a small ragged case.
DENSE_WORKLOADS: Dict[str, DenseWorkload] = {
    "dense_tiny": DenseWorkload("dense_tiny", 5, 384, 256),
    "dense_decode": DenseWorkload("dense_decode", 8, 4096, 4096),
    "dense_prefill": DenseWorkload("dense_prefill", 512, 4096, 4096),
    # a narrow projection out of the larger hidden size: 3.5 MiB of weights, the size class where
    # the CUDA-core kernel is the automatic choice for up to 8 tokens
    "dense_narrow": DenseWorkload("dense_narrow", 8, 7168, 512),
}


@dataclasses.dataclass
class DenseInputs:
    workload: DenseWorkload
    x: np.ndarray          # uint16 bf16 bits [T, K]
    w: np.ndarray          # uint8 E4M3 codes [N, K]
    w_scale: np.ndarray    # float32 [ceil(N/128), ceil(K/128)]


def e4m3_codes(key: int, count: int) -> np.ndarray:
    """E4M3 bytes shaped like block-quantised weights, built from their bit fields: a random sign,
    exponent field 14 - floor(|N(0, 2.5)|) clipped to [0, 14], a uniform 3-bit mantissa."""
    z = np.abs(normal(key, count))
    e = np.clip(14 - np.floor(2.5 * z), 0, 14).astype(np.uint8)
    r = random_bytes(_mix64_int(key ^ 0x3C3C3C3C3C3C3C3C), count)
    return ((r & np.uint8(0x80)) | (e << np.uint8(3)) | (r & np.uint8(7))).astype(np.uint8)


def make_dense_inputs(name, seed: int = 0, T: Optional[int] = None) -> DenseInputs:
    wl = DENSE_WORKLOADS[name] if isinstance(name, str) else name
    if T is not None:
        wl = dataclasses.replace(wl, T=T)
    x = np.stack([x_row(seed, wl.name, t, wl.K) for t in range(wl.T)]) if wl.T > 0 \
        else np.zeros((0, wl.K), np.uint16)
    w = e4m3_codes(stream_key(seed, wl.name, "w"), wl.N * wl.K).reshape(wl.N, wl.K)
    nb, kb = -(-wl.N // 128), -(-wl.K // 128)
    u = uniform01(stream_key(seed, wl.name, "w_scale_m"), nb * kb)
    p = np.floor(uniform01(stream_key(seed, wl.name, "w_scale_e"), nb * kb) * 5)
    sc = ((1.0 + u) * 2.0 ** (-14 + p)).astype(np.float32).reshape(nb, kb)
    return DenseInputs(wl, x, w, sc)


# --------------------------------------------------------------------------------------
# NVFP4 experts (the format variant): E2M1 codes, an E4M3 scale per 16 elements along K and
# one fp32 scale per matrix.


@dataclasses.dataclass
class NVFP4Experts:
    gate_up_codes: np.ndarray   # uint8 [E, 2I, H/2]
    gate_up_scales: np.ndarray  # uint8 [E, 2I, H/16] E4M3
    gate_up_global: np.ndarray  # float32 [E]
    down_codes: np.ndarray      # uint8 [E, H, I/2]
    down_scales: np.ndarray     # uint8 [E, H, I/16] E4M3
    down_global: np.ndarray     # float32 [E]

    @property
    def nbytes(self) -> int:
        return sum(a.nbytes for a in (self.gate_up_codes, self.gate_up_scales, self.gate_up_global,
                                      self.down_codes, self.down_scales, self.down_global))


def e4m3_scale_bytes(key: int, count: int) -> np.ndarray:
    """Positive E4M3 scale bytes from their fields: exponent field uniform in 4..8 (2^-3 .. 2^1),
    mantissa uniform in 0..7."""
    r = u64_stream(key, count)
    e = np.uint64(4) + (((r >> np.uint64(32)) * np.uint64(5)) >> np.uint64(32))
    m = r & np.uint64(7)
    return ((e << np.uint64(3)) | m).astype(np.uint8)


def make_nv_experts(seed: int, tag: str, E: int, H: int, I: int) -> NVFP4Experts:
    gu_c = np.stack([random_bytes(stream_key(seed, tag, e, "nv_gate_up_codes"), I * H).reshape(2 * I, H // 2)
                     for e in range(E)])
    gu_s = np.stack([e4m3_scale_bytes(stream_key(seed, tag, e, "nv_gate_up_scales"), 2 * I * H // 16)
                     .reshape(2 * I, H // 16) for e in range(E)])
    d_c = np.stack([random_bytes(stream_key(seed, tag, e, "nv_down_codes"), H * I // 2).reshape(H, I // 2)
                    for e in range(E)])
    d_s = np.stack([e4m3_scale_bytes(stream_key(seed, tag, e, "nv_down_scales"), H * I // 16).reshape(H, I // 16)
                    for e in range(E)])
    g = (1.0 + uniform01(stream_key(seed, tag, "nv_global"), 2 * E)) * 2.0 ** -6
    return NVFP4Experts(gu_c, gu_s, g[:E].astype(np.float32), d_c, d_s, g[E:].astype(np.float32))


def make_nv_inputs(name, seed: int = 0, T: Optional[int] = None) -> MoEInputs:
    """A workload's tokens and router with NVFP4 experts in place of the MXFP4 ones."""
    base = make_inputs(name, seed=seed, T=T, with_experts=False)
    wl = base.workload
    experts = make_nv_experts(seed, wl.name + "/nv_experts", wl.E, wl.H, wl.I)
    shared = make_nv_experts(seed, wl.name + "/nv_shared", 1, wl.H, wl.I_s) if wl.I_s > 0 else None
    return dataclasses.replace(base, experts=experts, shared=shared)
