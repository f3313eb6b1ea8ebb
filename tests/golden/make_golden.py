"""Writes the oracle's results on the small workloads into tests/golden/:

  tiny_oracle.json        the MXFP4 layer on the tiny workload (routing and output)
  nv_tiny_oracle.json     the same tokens and router with NVFP4 experts
  dense_tiny_oracle.json  the FP8 E4M3 block-scaled projection of dense_tiny (5 x 384 -> 256)
  bank_tiny_oracle.json   the expert bank's state over a sequence of tiny forwards (8 experts,
                          3 slots: cache and transient forwards)

Calls only the oracle (and the seeded input generator for its inputs). The stored files
guard the oracle and the generator against silent change; the GPU tests compare with the
oracle directly. Usage: python -m tests.golden.make_golden
"""
import hashlib
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

from oracle.oracle import BankState, Oracle, bank_plan  # noqa: E402
from routed_moe_fp4_gb300 import synthetic as S  # noqa: E402

HERE = os.path.dirname(os.path.abspath(__file__))
OUT = os.path.join(HERE, "tiny_oracle.json")
NV_OUT = os.path.join(HERE, "nv_tiny_oracle.json")
DENSE_OUT = os.path.join(HERE, "dense_tiny_oracle.json")
BANK_OUT = os.path.join(HERE, "bank_tiny_oracle.json")
# the bank sequence: (batch, tokens) per forward; with top-2 over 8 experts and 3 slots, one token
# is a cache forward and two or more tokens are transient ones
BANK_SLOTS = 3
BANK_SEQUENCE = ((1, 1), (2, 1), (3, 4), (4, 1), (5, 2), (6, 1), (7, 1), (8, 3), (9, 1))


def input_digest(inp) -> str:
    h = hashlib.sha256()
    for a in (inp.x, inp.router_w, inp.experts.gate_up_codes, inp.experts.gate_up_scales,
              inp.experts.down_codes, inp.experts.down_scales, inp.shared.gate_up_codes,
              inp.shared.gate_up_scales, inp.shared.down_codes, inp.shared.down_scales):
        h.update(a.tobytes())
    return h.hexdigest()


def digest(*arrays) -> str:
    h = hashlib.sha256()
    for a in arrays:
        h.update(a.tobytes())
    return h.hexdigest()


def nv_tiny(o: Oracle) -> dict:
    inp = S.make_nv_inputs("tiny", 0)
    wl = inp.workload
    idx, w = o.route(o.scores(inp.x, inp.router_w), inp.router_b, wl.top_k)
    out, _ = o.tokens_output_nv(inp.x, idx, w, inp.experts, inp.shared, range(wl.T))
    e, sh = inp.experts, inp.shared
    return {
        "workload": "tiny with NVFP4 experts: T=4, H=256, E=8, top-2, I=I_s=128, seed 0",
        "input_sha256": digest(inp.x, inp.router_w, e.gate_up_codes, e.gate_up_scales, e.gate_up_global,
                               e.down_codes, e.down_scales, e.down_global, sh.gate_up_codes, sh.gate_up_scales,
                               sh.gate_up_global, sh.down_codes, sh.down_scales, sh.down_global),
        "idx": idx.tolist(),
        "w_bits": w.view("uint32").tolist(),
        "out_bf16_bits": out.tolist(),
    }


def dense_tiny(o: Oracle) -> dict:
    inp = S.make_dense_inputs("dense_tiny", 0)
    out, _ = o.fp8_linear(inp.x, inp.w, inp.w_scale)
    return {
        "workload": "dense_tiny: T=5, K=384, N=256, E4M3 with an fp32 scale per 128 x 128 block, seed 0",
        "input_sha256": digest(inp.x, inp.w, inp.w_scale),
        "out_bf16_bits": out.tolist(),
    }


def bank_tiny(o: Oracle) -> dict:
    inp = S.make_inputs("tiny", 0, with_experts=False)
    wl = inp.workload
    state = BankState(wl.E, BANK_SLOTS)
    steps = []
    for batch, T in BANK_SEQUENCE:
        x = S.x_batch(0, wl.name, batch, T, wl.H)
        idx, _ = o.route(o.scores(x, inp.router_w), inp.router_b, wl.top_k)
        cnt, _, _, _ = o.permute(idx, wl.E)
        rnd, slot, cop = bank_plan(o, state, cnt, T, wl.top_k)
        steps.append({"batch": batch, "T": T, "cnt": cnt[:wl.E].tolist(), "round_of": rnd.tolist(),
                      "slot_for": slot.tolist(), "copied": cop.tolist(), "slot_of": state.slot_of.tolist(),
                      "expert_in": state.expert_in.tolist(), "usage": state.usage.tolist(),
                      "last_use": state.last_use.tolist(), "stats": state.stats.tolist()})
    return {"workload": f"tiny router (E=8, top-2), {BANK_SLOTS} slots, token batches of x_batch(seed 0)",
            "slots": BANK_SLOTS, "sequence": [list(p) for p in BANK_SEQUENCE], "steps": steps}


def main():
    o = Oracle()
    for path, doc in ((NV_OUT, nv_tiny(o)), (DENSE_OUT, dense_tiny(o)), (BANK_OUT, bank_tiny(o))):
        with open(path, "w") as f:
            json.dump(doc, f)
        print("wrote", path)
    inp = S.make_inputs("tiny", 0)
    r = o.moe_forward(inp.x, inp.router_w, inp.router_b, inp.workload.top_k, inp.experts, inp.shared)
    doc = {
        "workload": "tiny: T=4, H=256, E=8, top-2, I=I_s=128, seed 0",
        "input_sha256": input_digest(inp),
        "idx": r["idx"].tolist(),
        "w_bits": r["w"].view("uint32").tolist(),
        "cnt": r["cnt"].tolist(),
        "off": r["off"].tolist(),
        "src_token": r["src_token"].tolist(),
        "inv_row": r["inv_row"].tolist(),
        "out_bf16_bits": r["out"].tolist(),
    }
    with open(OUT, "w") as f:
        json.dump(doc, f)
    print("wrote", OUT)


if __name__ == "__main__":
    main()
