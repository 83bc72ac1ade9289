"""Writes tests/golden/tiny_layer.json, tiny_q4k_layer.json and tiny_q3k_layer.json from the CPU
oracle (and nothing else).

The pages print no worked numeric example for this layer, so these fixtures are
regression records of the pinned oracle on the seeded tiny workloads (N=64,
D=256, E=8, top_k=2, norm_topk_prob off, seed 0; F=128 with Q8_0 expert
weights, F=256 with Q4_K and with Q3_K): they detect any later change of the
oracle's results and any difference between the x86 and Arm builds.
Run: python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

import oracle  # noqa: E402
from mixture_experts_ffn_top_gb300.workloads import WORKLOADS, make_inputs  # noqa: E402


FIXTURES = {"tiny": "tiny_layer.json", "tiny_q4k": "tiny_q4k_layer.json", "tiny_q3k": "tiny_q3k_layer.json"}


def write(name):
    wl = WORKLOADS[name]
    r = oracle.moe_ffn_inputs(make_inputs(wl), wl.top_k, wl.norm_topk_prob)
    fx = {
        "workload": wl.describe(),
        "source": "oracle/moe_oracle.c via tests/golden/make_golden.py",
        "topk_idx": r["topk_idx"].tolist(),
        "topk_w_first8": r["topk_w"][:8].tolist(),
        "expStart": r["expStart"].tolist(),
        "x_q_int_sum": int(r["x_q"].astype(np.int64).sum()),
        "x_q_abs_sum": int(np.abs(r["x_q"].astype(np.int64)).sum()),
        "x_d16_first8": r["x_d16"][0, :8].tolist(),
        "h_q_abs_sum": int(np.abs(r["h_q"].astype(np.int64)).sum()),
        "out_row0_first16": r["out"][0, :16].tolist(),
        "out_sum": float(r["out"].astype(np.float64).sum()),
        "out_l2": float(np.linalg.norm(r["out"].astype(np.float64))),
    }
    with open(os.path.join(HERE, FIXTURES[name]), "w") as f:
        f.write("{\n" + ",\n".join(f" {json.dumps(k)}: {json.dumps(v)}" for k, v in fx.items()) + "\n}\n")


def main():
    for name in FIXTURES:
        write(name)


if __name__ == "__main__":
    main()
