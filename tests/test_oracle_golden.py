"""The oracle still reproduces its committed tiny-layer fixture (a guard against
unintended changes to its arithmetic; the fixture was written by the oracle)."""
import json
import os

import numpy as np

from oracle import exl3_oracle as O
from workloads import MoEWorkload, config, act_to_f64, rw_to_f64

GOLD = os.path.join(os.path.dirname(__file__), "golden", "tiny_layer.json")


def test_tiny_layer_fixture():
    g = json.load(open(GOLD))
    spec = config(0)
    w = MoEWorkload(spec)
    off, packed, tiles, nact = O.route_pack(w.ids, spec.E, g["capacity"])
    assert off.tolist() == g["offsets"] and packed.tolist() == g["packed"]
    assert tiles.tolist() == g["tiles"] and nact == g["num_active"]
    out = O.moe_forward(act_to_f64(w.x, spec.act), w.ids, rw_to_f64(w.rw, spec.rw_dtype),
                        w.projection, impl="numpy")
    assert np.allclose(out[:2, :16], np.array(g["out_rows_0_1_cols_0_16"]), rtol=1e-12, atol=1e-15)
    assert abs((out ** 2).sum() ** 0.5 - g["out_l2"]) < 1e-12 * g["out_l2"]
