"""GPU-vs-oracle parity protocol (used by the -m gpu tests and the smoke check).

Routing is compared given identical fp32 scores: the GPU's scores must be within 1e-5 of the
oracle's fp64 sigmoid of fp64 logits; the oracle's key/top-k/renormalisation and permutation run
on the GPU's scores and must match the GPU's idx, w, cnt, off, src_token and inv_row bit for bit;
the oracle's expert FFN and combine then use those indices and weights, and the GPU output must
satisfy |out - ref| <= 2e-2 * RMS(ref) + ulp_bf16(ref)/2 for every output, ref being the oracle's
unrounded fp64 value: the bar bounds the computation's error, and the half ulp is the rounding
that the bf16 output format forces on any implementation (a single rounding flip at an output of
4x RMS is already 1 bf16 ulp > 2e-2 * RMS). The report also carries the literal bar,
max |out - ref| <= 2e-2 * RMS(ref) with the rounding included, which the default FP4 path is held
to as well. Tokens whose fp64-score routing differs from the GPU's must sit within 1e-5 of a key
tie at the k / k+1 boundary.
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Sequence

import numpy as np

SCORE_TOL = 1e-5
OUT_TOL = 2e-2          # max(|out - ref| - ulp_bf16(ref)/2) <= OUT_TOL * RMS(ref)
TIE_TOL = 1e-5


def half_ulp_bf16(v: np.ndarray) -> np.ndarray:
    """Half the bf16 spacing at |v|: the rounding error any bf16 output of v may carry."""
    a = np.abs(np.asarray(v, np.float64))
    _, e = np.frexp(a)                      # a = m * 2^e, m in [0.5, 1)
    ulp = np.ldexp(1.0, np.maximum(e - 8, -133))
    return 0.5 * ulp


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclasses.dataclass
class ParityReport:
    T: int
    tokens_checked: int
    max_score_err: float
    routing_bit_exact: bool
    own_routing_diffs: int
    max_err: float
    rms_ref: float
    rel_err: float
    launches: int
    rel_err_bf16: float = 0.0   # max |out - round_bf16(ref)| / RMS, for information
    rel_err_literal: float = 0.0   # max |out - ref| / RMS: the bar with the output rounding included

    @property
    def ok(self) -> bool:
        return (self.max_score_err <= SCORE_TOL and self.routing_bit_exact and self.rel_err <= OUT_TOL)


def run_gpu(inputs, path: int = 0, T: Optional[int] = None, repeats: int = 1, layer=None):
    """Runs the library on `inputs`; returns (out bf16 bits [T, H], routing dict, launches)."""
    import torch
    from routed_moe_fp4_gb300 import colimoe as cm
    T = inputs.x.shape[0] if T is None else T
    own = layer is None
    if own:
        layer = cm.MoELayer(inputs, max_tokens=max(T, 1))
    layer.set_ffn_path(path)
    x = torch.from_numpy(inputs.x[:T].view(np.int16)).cuda()
    outs = []
    for _ in range(repeats):
        out = torch.empty((T, inputs.workload.H), dtype=torch.int16, device="cuda")
        layer.forward(x, out, T)
        torch.cuda.synchronize()
        outs.append(out.cpu().numpy().view(np.uint16))
    routing = layer.routing(T)
    launches = layer.launches()
    assert layer.device_error() == 0, "a kernel wait ran out (device error word set)"
    if own:
        layer.close()
    return outs, routing, launches


def check(oracle, inputs, out_bits: np.ndarray, routing: dict, tokens: Optional[Sequence[int]] = None,
          launches: int = 0) -> ParityReport:
    wl = inputs.workload
    T = out_bits.shape[0]
    k = wl.top_k
    s_gpu = routing["scores"]
    # (ii) bit-exact routing and permutation from the GPU's scores
    idx_o, w_o = oracle.route(s_gpu, inputs.router_b, k)
    cnt_o, off_o, src_o, inv_o = oracle.permute(idx_o, wl.E, with_shared=inputs.shared is not None)
    exact = (np.array_equal(idx_o, routing["idx"]) and np.array_equal(w_o.view(np.uint32),
                                                                       routing["weights"].view(np.uint32))
             and np.array_equal(cnt_o, routing["cnt"]) and np.array_equal(off_o, routing["off"])
             and np.array_equal(src_o, routing["src_token"]) and np.array_equal(inv_o, routing["inv_row"]))
    if tokens is None:
        tokens = list(range(T))
    tokens = np.asarray(sorted(set(int(t) for t in tokens)), np.int32)
    # (i) scores against fp64 sigmoid of fp64 logits, on the checked tokens
    s_ref = oracle.scores(np.ascontiguousarray(inputs.x[tokens]), inputs.router_w)
    max_score_err = float(np.abs(s_ref.astype(np.float64) - s_gpu[tokens].astype(np.float64)).max())
    # (iv) the oracle's own routing: differences only at near-ties
    idx_own, _ = oracle.route(s_ref, inputs.router_b, k)
    diffs = 0
    for n, t in enumerate(tokens):
        if set(idx_own[n].tolist()) != set(routing["idx"][t].tolist()):
            key = s_ref[n].astype(np.float64) + (0 if inputs.router_b is None else inputs.router_b)
            srt = np.sort(key)[::-1]
            assert srt[k - 1] - srt[k] < TIE_TOL, f"token {t}: own routing differs away from a tie"
            diffs += 1
    # (iii) output: oracle FFN + combine with the GPU's (== oracle's) indices and weights
    ref_bits, ref64 = oracle.tokens_output(inputs.x, routing["idx"], routing["weights"], inputs.experts,
                                           inputs.shared, tokens)
    got = bf16_bits_to_f32(out_bits[tokens]).astype(np.float64)
    ref = bf16_bits_to_f32(ref_bits).astype(np.float64)
    excess = np.abs(got - ref64) - half_ulp_bf16(ref64)
    err = float(max(excess.max(), 0.0))
    rms = float(np.sqrt((ref64 ** 2).mean()))
    err_bf16 = float(np.abs(got - ref).max())
    err_lit = float(np.abs(got - ref64).max())
    rel = lambda e: e / rms if rms > 0 else e
    return ParityReport(T, len(tokens), max_score_err, bool(exact), diffs, err, rms, rel(err), launches,
                        rel(err_bf16), rel(err_lit))


def structured_tokens(routing: dict, T: int, n: int, tile: int = 48, seed: int = 0) -> dict:
    """Named tokens that reach the GEMM tiling's corners, plus a seeded sample up to n tokens:
    the first and last rows of the heaviest expert, the lightest touched expert, and the last row of
    an expert whose last `tile`-row tile is partial with 1-16, 17-32 and 33-47 rows (the three box
    heights of a ragged tile). Returns {name: token} with the sample under "sample_i"."""
    cnt, off, src = routing["cnt"][:-1], routing["off"], routing["src_token"]
    touched = np.where(cnt > 0)[0]
    named = {}
    heavy = int(touched[np.argmax(cnt[touched])])
    named["heavy_first_row"] = int(src[off[heavy]])
    named["heavy_last_row"] = int(src[off[heavy] + cnt[heavy] - 1])
    light = int(touched[np.argmin(cnt[touched])])
    named["lightest_expert"] = int(src[off[light]])
    for lo, hi in ((1, 16), (17, 32), (33, tile - 1)):
        for e in touched:
            r = int(cnt[e]) % tile
            if lo <= r <= hi:
                named[f"partial_tile_{lo}_{hi}"] = int(src[off[e] + cnt[e] - 1])
                break
    rng = np.random.Generator(np.random.PCG64(seed))
    rest = [int(t) for t in rng.permutation(T) if int(t) not in named.values()]
    for i, t in enumerate(rest[:max(0, n - len(named))]):
        named[f"sample_{i}"] = t
    return named


def sample_tokens(routing: dict, T: int, n: int, seed: int = 0) -> list:
    """A seeded token sample that includes tokens routed to the heaviest and lightest touched experts."""
    rng = np.random.Generator(np.random.PCG64(seed))
    idx = routing["idx"]
    cnt = routing["cnt"][:-1]
    touched = np.where(cnt > 0)[0]
    picks = set()
    if len(touched):
        heavy, light = touched[np.argmax(cnt[touched])], touched[np.argmin(cnt[touched])]
        for e in (heavy, light):
            picks.add(int(np.where((idx == e).any(1))[0][0]))
    picks.update(int(t) for t in rng.choice(T, size=min(n, T), replace=False))
    picks.update({0, T - 1})
    return sorted(picks)
