"""How much error do bf16 activations alone cause at depth?

TEST INFRASTRUCTURE.  The oracle's step (float64) with one change: values are
rounded to bfloat16 (nearest even) at the points where the CUDA path stores
them in bf16 -- the inputs of every projection (RMSNorm outputs, attention
output, SwiGLU output), the Q/K/V projections before and after the rotary
embedding, the gate/up outputs, and in the backward the bf16 copies of the
residual gradient and the dm, dab, dO, dQKV products.  Everything else stays
float64.  Comparing this model with the plain oracle measures the error that
bf16 storage of activations produces by itself; the CUDA path cannot be
expected to beat it, so it sets the tolerance of deep-stack parity tests.
Uses only oracle functions and numpy (nothing from the CUDA path).
"""
import numpy as np

from oracle import bf16_round
from oracle import llama_step as ls


def _r(a):
    return bf16_round(np.asarray(a, np.float32)).astype(np.float64)


def _layer_fwd(x, p, cfg, cos, sin):
    B, S, d = x.shape
    T = B * S
    Hq, Hkv, hd = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
    xf = x.reshape(T, d)
    u, c1 = ls.rmsnorm_fwd(xf, p["g1"], cfg.rms_eps)
    u = _r(u)
    q = _r(ls.rope_fwd(_r(u @ p["wq"].T).reshape(B, S, Hq, hd), cos, sin))
    k = _r(ls.rope_fwd(_r(u @ p["wk"].T).reshape(B, S, Hkv, hd), cos, sin))
    v = _r(u @ p["wv"].T).reshape(B, S, Hkv, hd)
    o, _ = ls.attention_fwd(q, k, v)
    of = _r(o.reshape(T, -1))
    h = xf + of @ p["wo"].T
    w2, c2 = ls.rmsnorm_fwd(h, p["g2"], cfg.rms_eps)
    w2 = _r(w2)
    a, b = _r(w2 @ p["wg"].T), _r(w2 @ p["wu"].T)
    m = _r(ls.swiglu_fwd(a, b))
    out = h + m @ p["wd"].T
    return out.reshape(B, S, d), dict(u=u, c1=c1, q=q, k=k, v=v, of=of, w2=w2, c2=c2, a=a, b=b, m=m)


def _layer_bwd(dout, p, c, cfg, cos, sin):
    T, d = dout.shape
    Hq, hd = cfg.n_heads, cfg.head_dim
    B, S = c["q"].shape[:2]
    gr = {}
    doutb = _r(dout)
    gr["wd"] = doutb.T @ c["m"]
    dm = _r(doutb @ p["wd"])
    da, db = ls.swiglu_bwd(dm, c["a"], c["b"])
    da, db = _r(da), _r(db)
    gr["wg"], gr["wu"] = da.T @ c["w2"], db.T @ c["w2"]
    dhn, gr["g2"] = ls.rmsnorm_bwd(da @ p["wg"] + db @ p["wu"], p["g2"], c["c2"])
    dh = dout + dhn
    dhb = _r(dh)
    gr["wo"] = dhb.T @ c["of"]
    do = _r(dhb @ p["wo"]).reshape(B, S, Hq, hd)
    dq, dk, dv = ls.attention_bwd(do, c["q"], c["k"], c["v"])
    dq = _r(ls.rope_bwd(dq, cos, sin).reshape(T, -1))
    dk = _r(ls.rope_bwd(dk, cos, sin).reshape(T, -1))
    dv = _r(dv.reshape(T, -1))
    u = c["u"]
    gr["wq"], gr["wk"], gr["wv"] = dq.T @ u, dk.T @ u, dv.T @ u
    dxn, gr["g1"] = ls.rmsnorm_bwd(dq @ p["wq"] + dk @ p["wk"] + dv @ p["wv"], p["g1"], c["c1"])
    return dh + dxn, gr


def step_bf16_activations(w, tokens, labels, cfg):
    """(loss, grads) like oracle.step, with bf16 storage of activations."""
    tokens = np.asarray(tokens)
    B, S = tokens.shape
    T, d = B * S, cfg.hidden
    layers = [{k: np.asarray(v, np.float64) for k, v in lp.items()} for lp in w.layers]
    E, gf, Wlm = (np.asarray(a, np.float64) for a in (w.embed, w.final_norm, w.lm_head))
    cos, sin = ls.rope_tables(S, cfg.head_dim, cfg.rope_base)
    x = E[tokens]
    caches = []
    for p in layers:
        x, c = _layer_fwd(x, p, cfg, cos, sin)
        caches.append(c)
    hf, cf = ls.rmsnorm_fwd(x.reshape(T, d), gf, cfg.rms_eps)
    hf = _r(hf)
    z = _r(hf @ Wlm.T)
    loss, dz, _ = ls.cross_entropy_fwd_bwd(z, labels)
    dz = _r(dz)
    g_lm = dz.T @ hf
    dx, g_gf = ls.rmsnorm_bwd(dz @ Wlm, gf, cf)
    g_layers = [None] * len(layers)
    for i in range(len(layers) - 1, -1, -1):
        dx, g_layers[i] = _layer_bwd(dx, layers[i], caches[i], cfg, cos, sin)
    return loss, dict(layers=g_layers, lm_head=g_lm, final_norm=g_gf)
