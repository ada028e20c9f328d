"""Shared test helpers: inputs for both sides and the comparison metrics."""
from __future__ import annotations

import numpy as np

import inputs
from inputs import UNIT_EMBED, UNIT_FINAL_NORM, UNIT_LM_HEAD
from oracle import ModelWeights, bf16_round

# Tolerances of the parity bar: loss relative error and per-tensor relative L2
# error of bf16-compute / fp32-accumulate gradients against the oracle.
LOSS_RTOL = 1e-3
GRAD_RL2 = 2e-2
ZERO_ATOL = 1e-6


def rel_l2(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nb = np.linalg.norm(b)
    if nb == 0.0:
        return float(np.abs(a).max()) if a.size else 0.0
    return float(np.linalg.norm(a - b) / nb)


def masters(cfg):
    """fp32 master arrays per unit, as the library receives them (no LM-head
    unit when it is tied to the embedding)."""
    m = {l: inputs.unit_master(cfg, l) for l in range(cfg.n_layers)}
    for u in (UNIT_EMBED, UNIT_FINAL_NORM, UNIT_LM_HEAD):
        if inputs.unit_numel(cfg, u):
            m[u] = inputs.unit_master(cfg, u)
    return m


def oracle_weights(cfg, mast=None, round_bf16=True) -> ModelWeights:
    """The weights the step computes with: the bf16 (round-to-nearest-even)
    values of the fp32 masters."""
    if mast is None:
        mast = masters(cfg)
    r = bf16_round if round_bf16 else (lambda a: a)
    layers = [{k: r(v) for k, v in inputs.split_layer(cfg, mast[l]).items()}
              for l in range(cfg.n_layers)]
    d, V = cfg.hidden, cfg.vocab
    return ModelWeights(layers=layers,
                        embed=r(mast[UNIT_EMBED]).reshape(V, d),
                        final_norm=r(mast[UNIT_FINAL_NORM]),
                        lm_head=None if cfg.tie_embeddings else r(mast[UNIT_LM_HEAD]).reshape(V, d))


def flat_layer_grads(cfg, g: dict) -> np.ndarray:
    """Concatenate a layer's grads in unit order."""
    from inputs.configs import layer_tensor_shapes
    return np.concatenate([np.asarray(g[n]).reshape(-1) for n, _ in layer_tensor_shapes(cfg)])
