"""Writes routed_moe_fp4_gb300/workload_calibration.json from the oracle (run once).

Two input-recipe constants need the layer's routing to be found, so they come from the
oracle, never from the CUDA path:
  * decode workload: its token rows are redrawn (attempt 0, 1, ...) until the gaps between
    consecutive keys among each token's k+1 largest keys exceed 1e-3; keys are the fp32
    key = s + b the oracle routes on. The attempt index per token is stored.
  * skewed workload: a per-expert router bias under which the routed-slot count of the
    expert with popularity rank r follows Zipf(1.1): c_r = min(T, lam * (r+1)^-1.1), lam
    such that the counts sum to T*k (top-k routing gives an expert at most one slot per
    token). Ranks are a seeded permutation of the experts. The bias is fitted by iterating
    b_e += lr * (ln(c_e + 1) - ln(count_e + 1)) with the oracle's routing; the bias vector
    and the realised counts are stored.
Usage: python -m oracle.calibrate_workloads
"""
from __future__ import annotations

import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from oracle.oracle import Oracle  # noqa: E402
from routed_moe_fp4_gb300 import synthetic as S  # noqa: E402


def margin_attempts(o: Oracle, seed: int = 0):
    wl = S.WORKLOADS["decode"]
    inp = S.make_inputs("decode", seed, with_experts=False)
    attempts = []
    for t in range(wl.T):
        a = 0
        while True:
            row = S.x_row(seed, wl.name, t, wl.H, a)[None, :]
            s = o.scores(row, inp.router_w)
            key = (s + inp.router_b[None, :]).astype(np.float32)[0]
            top = np.sort(key.astype(np.float64))[::-1][: wl.top_k + 1]
            if np.all(-np.diff(top) > wl.margin):
                break
            a += 1
        attempts.append(a)
    return attempts


def zipf_targets(T: int, k: int, E: int, s_exp: float = 1.1) -> np.ndarray:
    """Slots per popularity rank: c_r = min(T, lam * (r+1)^-s), lam set so sum c = T*k
    (an expert can take at most one slot per token)."""
    p = (np.arange(E) + 1.0) ** -s_exp
    lo, hi = 0.0, float(T * k) / p.min()
    for _ in range(200):
        lam = 0.5 * (lo + hi)
        if np.minimum(T, lam * p).sum() < T * k:
            lo = lam
        else:
            hi = lam
    return np.minimum(T, 0.5 * (lo + hi) * p)


def zipf_bias_fit(o: Oracle, seed: int = 0, iters: int = 600):
    """Per-expert router bias whose routed-slot counts follow the Zipf(1.1) targets."""
    wl = S.WORKLOADS["skewed"]
    inp = S.make_inputs("skewed", seed, with_experts=False, unbiased=True)
    s = o.scores(inp.x, inp.router_w)
    rank = S.zipf_rank(seed, wl.E)
    target = zipf_targets(wl.T, wl.top_k, wl.E)[rank]
    b = np.zeros(wl.E, np.float64)
    best = None
    for it in range(iters):
        lr = 0.05 if it < iters // 2 else 0.01
        idx, _ = o.route(s, b.astype(np.float32), wl.top_k)
        cnt = np.bincount(idx.reshape(-1), minlength=wl.E)
        err = np.abs(np.log(cnt + 1.0) - np.log(target + 1.0)).max()
        if best is None or err < best[0]:
            best = (err, b.astype(np.float32).copy(), cnt.copy())
        b += lr * (np.log(target + 1.0) - np.log(cnt + 1.0))
        b -= b.max()
    err, bias, cnt = best
    return bias, target, cnt, err


def main():
    o = Oracle()
    out = {}
    out["decode_row_attempts"] = margin_attempts(o)
    bias, target, cnt, err = zipf_bias_fit(o)
    rank = S.zipf_rank(0, S.WORKLOADS["skewed"].E)
    order = np.argsort(rank)
    out["skewed_router_bias"] = [float(v) for v in bias]
    out["skewed_target_slots_by_rank"] = [round(float(v), 2) for v in target[order]]
    out["skewed_slots_by_rank"] = [int(v) for v in cnt[order]]
    out["skewed_max_abs_log_error"] = float(err)
    path = S._CALIBRATION_FILE
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
    print("decode attempts", out["decode_row_attempts"], "max |log err|", out["skewed_max_abs_log_error"])
    print("slots by rank (first 12):", out["skewed_slots_by_rank"][:12], "last 6:", out["skewed_slots_by_rank"][-6:])
    print("target by rank (first 12):", out["skewed_target_slots_by_rank"][:12], "last 6:",
          out["skewed_target_slots_by_rank"][-6:])


if __name__ == "__main__":
    main()
