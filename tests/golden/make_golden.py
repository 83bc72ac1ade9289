"""Writes tests/golden/tiny_layer.json from the CPU oracle (and nothing else).

The pages print no worked numeric example for this layer, so this fixture is a
regression record of the pinned oracle on the seeded tiny workload (N=64,
D=256, E=8, top_k=2, F=128, norm_topk_prob off, seed 0): it detects any later
change of the oracle's results and any difference between the x86 and Arm
builds.  Run: python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

import oracle  # noqa: E402
from mixture_experts_ffn_top_gb300.workloads import WORKLOADS, make_inputs  # noqa: E402


def main():
    wl = WORKLOADS["tiny"]
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
    with open(os.path.join(HERE, "tiny_layer.json"), "w") as f:
        f.write("{\n" + ",\n".join(f" {json.dumps(k)}: {json.dumps(v)}" for k, v in fx.items()) + "\n}\n")


if __name__ == "__main__":
    main()
