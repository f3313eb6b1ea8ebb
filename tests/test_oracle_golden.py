"""The oracle and the generator reproduce the stored tiny-workload result exactly."""
import json
import os

import numpy as np

from routed_moe_fp4_gb300 import synthetic as S
from tests.golden.make_golden import OUT, input_digest


def test_tiny_matches_stored(oracle):
    with open(OUT) as f:
        doc = json.load(f)
    inp = S.make_inputs("tiny", 0)
    assert input_digest(inp) == doc["input_sha256"]
    r = oracle.moe_forward(inp.x, inp.router_w, inp.router_b, inp.workload.top_k, inp.experts, inp.shared)
    assert r["idx"].tolist() == doc["idx"]
    assert r["w"].view(np.uint32).tolist() == doc["w_bits"]
    assert r["cnt"].tolist() == doc["cnt"] and r["off"].tolist() == doc["off"]
    assert r["src_token"].tolist() == doc["src_token"] and r["inv_row"].tolist() == doc["inv_row"]
    assert r["out"].tolist() == doc["out_bf16_bits"]


def test_decode_margin_holds(oracle):
    """The stored row redraws give every decode token top-(k+1) key gaps above 1e-3."""
    inp = S.make_inputs("decode", 0, with_experts=False)
    s = oracle.scores(inp.x, inp.router_w)
    key = (s + inp.router_b[None, :]).astype(np.float32).astype(np.float64)
    top = -np.sort(-key, axis=1)[:, : inp.workload.top_k + 1]
    assert np.all(-np.diff(top, axis=1) > 1e-3)
