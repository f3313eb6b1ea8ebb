"""The oracle and the generator reproduce the stored results of the small workloads exactly
(MXFP4 and NVFP4 layers, the FP8 projection and an expert-bank sequence)."""
import json
import os

import numpy as np

from routed_moe_fp4_gb300 import synthetic as S
from oracle.oracle import BankState, bank_plan
from tests.golden.make_golden import (BANK_OUT, BANK_SEQUENCE, BANK_SLOTS, DENSE_OUT, NV_OUT, OUT, digest,
                                      input_digest)


def _load(path):
    with open(path) as f:
        return json.load(f)


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


def test_nv_tiny_matches_stored(oracle):
    doc = _load(NV_OUT)
    inp = S.make_nv_inputs("tiny", 0)
    e, sh = inp.experts, inp.shared
    assert digest(inp.x, inp.router_w, e.gate_up_codes, e.gate_up_scales, e.gate_up_global, e.down_codes,
                  e.down_scales, e.down_global, sh.gate_up_codes, sh.gate_up_scales, sh.gate_up_global,
                  sh.down_codes, sh.down_scales, sh.down_global) == doc["input_sha256"]
    idx, w = oracle.route(oracle.scores(inp.x, inp.router_w), inp.router_b, inp.workload.top_k)
    assert idx.tolist() == doc["idx"] and w.view(np.uint32).tolist() == doc["w_bits"]
    out, _ = oracle.tokens_output_nv(inp.x, idx, w, e, sh, range(inp.workload.T))
    assert out.tolist() == doc["out_bf16_bits"]


def test_dense_tiny_matches_stored(oracle):
    doc = _load(DENSE_OUT)
    inp = S.make_dense_inputs("dense_tiny", 0)
    assert digest(inp.x, inp.w, inp.w_scale) == doc["input_sha256"]
    out, _ = oracle.fp8_linear(inp.x, inp.w, inp.w_scale)
    assert out.tolist() == doc["out_bf16_bits"]


def test_bank_sequence_matches_stored(oracle):
    doc = _load(BANK_OUT)
    assert doc["slots"] == BANK_SLOTS and doc["sequence"] == [list(p) for p in BANK_SEQUENCE]
    inp = S.make_inputs("tiny", 0, with_experts=False)
    wl = inp.workload
    state = BankState(wl.E, BANK_SLOTS)
    for (batch, T), want in zip(BANK_SEQUENCE, doc["steps"]):
        x = S.x_batch(0, wl.name, batch, T, wl.H)
        idx, _ = oracle.route(oracle.scores(x, inp.router_w), inp.router_b, wl.top_k)
        cnt, _, _, _ = oracle.permute(idx, wl.E)
        assert cnt[:wl.E].tolist() == want["cnt"]
        rnd, slot, cop = bank_plan(oracle, state, cnt, T, wl.top_k)
        assert rnd.tolist() == want["round_of"] and slot.tolist() == want["slot_for"]
        assert cop.tolist() == want["copied"]
        for key in ("slot_of", "expert_in", "usage", "last_use", "stats"):
            assert getattr(state, key).tolist() == want[key], key


def test_skewed_popularity_is_what_the_stored_bias_routes_to(oracle):
    """The stored Zipf bias, routed by the oracle over the skewed workload's 4096 tokens, gives
    exactly the stored slot counts per popularity rank."""
    cal = S.calibration()
    wl = S.WORKLOADS["skewed"]
    inp = S.make_inputs("skewed", 0, with_experts=False)
    idx, _ = oracle.route(oracle.scores(inp.x, inp.router_w), inp.router_b, wl.top_k)
    cnt = np.bincount(idx.reshape(-1), minlength=wl.E)
    order = np.argsort(S.zipf_rank(0, wl.E))
    assert cnt[order].tolist() == cal["skewed_slots_by_rank"]
