"""Writes tests/golden/tiny_layer.json from the float64 oracle only.

The tiny layer is the 512/256/8-expert/top-2/16-token configuration (seed 0).
Route packing follows "MoE: Add fused additive EXL3 kernels" (exllamav3 #284),
"Summary" (stable route packing); the outputs follow "EXL3 linear and grouped
routed experts" (TensorFold #837), "What this changes" (grouped experts).
Run:  python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from oracle import exl3_oracle as O          # noqa: E402
from workloads import MoEWorkload, config, act_to_f64, rw_to_f64  # noqa: E402


def main():
    spec = config(0)
    w = MoEWorkload(spec)
    off, packed, tiles, nact = O.route_pack(w.ids, spec.E, 3)
    out = O.moe_forward(act_to_f64(w.x, spec.act), w.ids, rw_to_f64(w.rw, spec.rw_dtype),
                        w.projection)
    doc = {
        "source": "oracle/exl3_oracle.py via tests/golden/make_golden.py",
        "workload": "tiny layer: hidden 512, inter 256, 8 experts, top-2, 16 tokens, seed 0",
        "capacity": 3,
        "offsets": off.tolist(), "packed": packed.tolist(), "tiles": tiles.tolist(),
        "num_active": nact,
        "out_rows_0_1_cols_0_16": [[float(v) for v in out[r, :16]] for r in (0, 1)],
        "out_l2": float((out ** 2).sum() ** 0.5),
    }
    with open(os.path.join(HERE, "tiny_layer.json"), "w") as f:
        json.dump(doc, f, indent=1)


if __name__ == "__main__":
    main()
