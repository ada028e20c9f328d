"""Write bf16_depth_error_<workload>.json: the gradient error that bf16
tensor-core operands alone produce in a whole decoder stack, from
tests/bf16_rounding_model.py against the oracle (both CPU, nothing from the
CUDA path), at the full depth and width of the workload.

The stacks run layer by layer (oracle.step_streamed): each layer's weights
are regenerated from the seeded generator when needed, so memory holds the
activations, not the weights.  Each gradient tensor is compared on a fixed
sample of at most 2^20 of its elements (the same sample for both runs), the
small ones whole.  The token count is the workload's sequence length with
batch 1 (the per-tensor error does not grow with the number of sequences:
each sequence adds independent rounding noise and independent signal).

Run from the repo root (minutes per workload; 8b needs ~40 GB of memory):
    python tests/golden/make_bf16_depth_error.py 1.3b 8b 123b-slice [--float32]
"""
import json
import os
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import inputs  # noqa: E402
import oracle  # noqa: E402
from inputs import CONFIGS, UNIT_EMBED, UNIT_FINAL_NORM, UNIT_LM_HEAD  # noqa: E402
from tests import bf16_rounding_model as model  # noqa: E402
from tests.helpers import rel_l2  # noqa: E402

SAMPLE = 1 << 20


def sample_index(n, key):
    if n <= SAMPLE:
        return None
    rng = np.random.default_rng(1000 + key)
    return np.sort(rng.choice(n, SAMPLE, replace=False))


def run(step_fn, cfg, dtype, idx):
    """One streamed step; returns (loss, {tensor: sampled gradient})."""
    def layer(i):  # rounded tensor by tensor: smaller temporaries than the whole layer
        return {k: oracle.bf16_round(v) for k, v in inputs.split_layer(cfg, inputs.layer_master(cfg, i)).items()}

    out = {}

    def keep(i, g):
        for k, v in g.items():
            v = np.asarray(v).reshape(-1)
            ix = idx.get(k)
            out[f"{i}.{k}"] = (v if ix is None else v[ix]).astype(np.float64)

    d, V = cfg.hidden, cfg.vocab
    E = oracle.bf16_round(inputs.unit_master(cfg, UNIT_EMBED)).reshape(V, d)
    gf = oracle.bf16_round(inputs.unit_master(cfg, UNIT_FINAL_NORM))
    Wlm = oracle.bf16_round(inputs.unit_master(cfg, UNIT_LM_HEAD)).reshape(V, d)
    tok, lab = inputs.tokens_and_labels(cfg)
    loss, g = step_fn(layer, cfg.n_layers, E, gf, Wlm, tok, lab, cfg, dtype=dtype,
                      on_layer_grads=keep)
    for k, ix in (("lm_head", idx["lm_head"]), ("embed", idx["embed"])):
        v = np.asarray(g[k]).reshape(-1)
        out[k] = (v if ix is None else v[ix]).astype(np.float64)
    out["final_norm"] = np.asarray(g["final_norm"], np.float64)
    return float(loss), out


def make(name, dtype):
    cfg = CONFIGS[name].with_(batch=1)
    from inputs.configs import layer_tensor_shapes
    idx = {k: sample_index(int(np.prod(s)), j) for j, (k, s) in enumerate(layer_tensor_shapes(cfg))}
    idx["lm_head"] = sample_index(cfg.vocab * cfg.hidden, 90)
    idx["embed"] = sample_index(cfg.vocab * cfg.hidden, 91)
    t0 = time.time()
    loss0, g0 = run(oracle.step_streamed, cfg, dtype, idx)
    loss1, g1 = run(model.step_streamed, cfg, dtype, idx)
    per = {k: rel_l2(g1[k], g0[k]) for k in g0 if k not in ("lm_head", "embed", "final_norm")}
    vals = np.array(list(per.values()))
    out = {"workload": cfg.name, "batch": cfg.batch, "seq": cfg.seq,
           "dtype": np.dtype(dtype).name, "sampled_elements_per_tensor": SAMPLE,
           "loss_rel": abs(loss1 - loss0) / loss0,
           "lm_head": rel_l2(g1["lm_head"], g0["lm_head"]),
           "final_norm": rel_l2(g1["final_norm"], g0["final_norm"]),
           "embed": rel_l2(g1["embed"], g0["embed"]),
           "layer_max": float(vals.max()), "layer_median": float(np.median(vals)),
           "per_tensor": per}
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)),
                        f"bf16_depth_error_{name}.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1, sort_keys=True)
    print({k: v for k, v in out.items() if k != "per_tensor"}, f"{time.time() - t0:.0f}s", flush=True)


def main():
    dtype = np.float32 if "--float32" in sys.argv else np.float64
    names = [a for a in sys.argv[1:] if not a.startswith("--")] or ["1.3b"]
    for n in names:
        make(n, dtype)


if __name__ == "__main__":
    main()
