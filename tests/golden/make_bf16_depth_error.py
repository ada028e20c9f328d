"""Write bf16_depth_error.json: the gradient error that bf16 activations
alone produce in the whole 1.3B-shape stack (24 layers, hidden 2048), from
tests/bf16_rounding_model.py against the float64 oracle (both CPU).  The
shape is the 1.3B workload with one sequence of 128 tokens (the error comes
from depth and width, not from the token count).  Run from the repo root:
    python tests/golden/make_bf16_depth_error.py
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import inputs  # noqa: E402
import oracle  # noqa: E402
from inputs import CONFIGS  # noqa: E402
from tests.bf16_rounding_model import step_bf16_activations  # noqa: E402
from tests.helpers import oracle_weights, rel_l2  # noqa: E402


def main():
    cfg = CONFIGS["1.3b"].with_(batch=1, seq=128)
    w = oracle_weights(cfg)
    tok, lab = inputs.tokens_and_labels(cfg)
    loss0, g0 = oracle.step(w, tok, lab, cfg)
    loss1, g1 = step_bf16_activations(w, tok, lab, cfg)
    per = {f"{i}.{k}": rel_l2(g1["layers"][i][k], g0["layers"][i][k])
           for i in range(cfg.n_layers) for k in g0["layers"][i]}
    out = {"workload": cfg.name, "batch": cfg.batch, "seq": cfg.seq,
           "loss_rel": abs(loss1 - loss0) / loss0,
           "lm_head": rel_l2(g1["lm_head"], g0["lm_head"]),
           "final_norm": rel_l2(g1["final_norm"], g0["final_norm"]),
           "layer_max": max(per.values()), "layer_median": float(np.median(list(per.values()))),
           "per_tensor": per}
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "bf16_depth_error.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1, sort_keys=True)
    print({k: v for k, v in out.items() if k != "per_tensor"})


if __name__ == "__main__":
    main()
