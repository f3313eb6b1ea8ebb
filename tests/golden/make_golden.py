"""Writes tests/golden/tiny_oracle.json: the oracle's result on the tiny workload.

Calls only the oracle (and the seeded input generator for its inputs). The stored file
guards the oracle and the generator against silent change; the GPU tests compare with the
oracle directly. Usage: python -m tests.golden.make_golden
"""
import hashlib
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

from oracle.oracle import Oracle  # noqa: E402
from routed_moe_fp4_gb300 import synthetic as S  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_oracle.json")


def input_digest(inp) -> str:
    h = hashlib.sha256()
    for a in (inp.x, inp.router_w, inp.experts.gate_up_codes, inp.experts.gate_up_scales,
              inp.experts.down_codes, inp.experts.down_scales, inp.shared.gate_up_codes,
              inp.shared.gate_up_scales, inp.shared.down_codes, inp.shared.down_scales):
        h.update(a.tobytes())
    return h.hexdigest()


def main():
    inp = S.make_inputs("tiny", 0)
    r = Oracle().moe_forward(inp.x, inp.router_w, inp.router_b, inp.workload.top_k, inp.experts, inp.shared)
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
