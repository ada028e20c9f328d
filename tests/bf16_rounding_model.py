"""How much error must any bf16-operand tensor-core implementation make?

TEST INFRASTRUCTURE.  The oracle's step with one change: values are rounded
to bfloat16 (nearest even) at exactly the points where every implementation
that feeds bf16 operands to the tensor cores has to round them, and nowhere
else:
  * forward: the inputs of every projection (the RMSNorm outputs u, w2 and
    the final hf, the attention output o, the SwiGLU output m); the attention
    operands Q and K (after the rotation) and V; the attention probabilities
    P that multiply V;
  * backward: the upstream gradient of every projection (the residual-stream
    gradient entering the down and output projections, da and db, dZ); the
    attention backward's operand dO and its internal P (the operand of dV)
    and dS (the operand of dQ and dK); dQ, dK (after the inverse rotation)
    and dV, the operands of the Q/K/V projection's products;
  * the gradients that leave the GPU: every weight gradient and the input
    gradient dX0 are cast to bf16 (the method's gradient cast and pack).
Everything else stays at the working precision: the residual stream and its
gradient, the norm statistics, the logits and the softmax, the gate and up
outputs a, b and dm = dY Wd.  So the distance between this model and the
plain oracle is the error that bf16 operands alone produce: a bound that no
implementation of the bf16-compute step can be expected to beat, and the
tolerance of the deep-stack parity tests where it exceeds their stated bar.

Uses only oracle functions and numpy (nothing from the CUDA path).  The
attention rounds P = exp(s - m) with m the row maximum; an online softmax
rounds it against a running maximum, which moves individual roundings but
not their statistics.
"""
import numpy as np

from oracle import bf16_round
from oracle import llama_step as ls


def _r(a):
    return bf16_round(np.asarray(a, np.float32)).astype(np.asarray(a).dtype)


def attention_fwd(q, k, v):
    """ls.attention_fwd with P rounded to bf16 before it multiplies V (the row
    sum l of the normaliser stays unrounded)."""
    B, S, Hq, hd = q.shape
    grp = Hq // k.shape[2]
    scale = 1.0 / np.sqrt(hd)
    future = np.triu(np.ones((S, S), dtype=bool), 1)
    o = np.empty_like(q)
    lse = np.empty((B, Hq, S), dtype=q.dtype)
    for b in range(B):
        for h in range(Hq):
            g = h // grp
            sc = (q[b, :, h, :] @ k[b, :, g, :].T) * scale
            sc[future] = -np.inf
            m = sc.max(axis=1, keepdims=True)
            e = np.exp(sc - m)
            l = e.sum(axis=1, keepdims=True)
            o[b, :, h, :] = (_r(e) @ v[b, :, g, :]) / l
            lse[b, h, :] = (m + np.log(l))[:, 0]
    return o, lse


def attention_bwd(do, q, k, v, o, lse):
    """ls.attention_bwd with P rounded for dV = P^T dO and dS rounded for
    dQ = dS K and dK = dS^T Q; P comes from the forward's lse and the row term
    is sum(dO * O) over the (bf16) forward output."""
    B, S, Hq, hd = q.shape
    grp = Hq // k.shape[2]
    scale = 1.0 / np.sqrt(hd)
    future = np.triu(np.ones((S, S), dtype=bool), 1)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for b in range(B):
        for h in range(Hq):
            g = h // grp
            sc = (q[b, :, h, :] @ k[b, :, g, :].T) * scale
            sc[future] = -np.inf
            p = np.exp(sc - lse[b, h, :, None])
            dv[b, :, g, :] += _r(p).T @ do[b, :, h, :]
            dp = do[b, :, h, :] @ v[b, :, g, :].T
            delta = np.sum(do[b, :, h, :] * o[b, :, h, :], axis=1, keepdims=True)
            ds = _r(p * (dp - delta))
            dq[b, :, h, :] = (ds @ k[b, :, g, :]) * scale
            dk[b, :, g, :] += (ds.T @ q[b, :, h, :]) * scale
    return dq, dk, dv


def layer_fwd(x, p, cfg, cos, sin):
    B, S, d = x.shape
    T = B * S
    Hq, Hkv, hd = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
    xf = x.reshape(T, d)
    u, c1 = ls.rmsnorm_fwd(xf, p["g1"], cfg.rms_eps)
    u = _r(u)
    q, k, v = u @ p["wq"].T, u @ p["wk"].T, u @ p["wv"].T
    if "bq" in p:
        q, k, v = q + p["bq"], k + p["bk"], v + p["bv"]
    q = _r(ls.rope_fwd(q.reshape(B, S, Hq, hd), cos, sin))
    k = _r(ls.rope_fwd(k.reshape(B, S, Hkv, hd), cos, sin))
    v = _r(v).reshape(B, S, Hkv, hd)
    o, lse = attention_fwd(q, k, v)
    o = _r(o)
    of = o.reshape(T, -1)
    h = xf + of @ p["wo"].T
    w2, c2 = ls.rmsnorm_fwd(h, p["g2"], cfg.rms_eps)
    w2 = _r(w2)
    a, b = w2 @ p["wg"].T, w2 @ p["wu"].T
    m = _r(ls.swiglu_fwd(a, b))
    out = h + m @ p["wd"].T
    cache = dict(u=u, c1=c1, q=q, k=k, v=v, o=o, lse=lse, of=of, w2=w2, c2=c2, a=a, b=b, m=m)
    return out.reshape(B, S, d), cache


def layer_bwd(dout, p, c, cfg, cos, sin):
    T, d = dout.shape
    Hq, hd = cfg.n_heads, cfg.head_dim
    B, S = c["q"].shape[:2]
    gr = {}
    doutb = _r(dout)
    gr["wd"] = doutb.T @ c["m"]
    da, db = ls.swiglu_bwd(doutb @ p["wd"], c["a"], c["b"])
    da, db = _r(da), _r(db)
    gr["wg"], gr["wu"] = da.T @ c["w2"], db.T @ c["w2"]
    dhn, gr["g2"] = ls.rmsnorm_bwd(da @ p["wg"] + db @ p["wu"], p["g2"], c["c2"])
    dh = dout + dhn
    dhb = _r(dh)
    gr["wo"] = dhb.T @ c["of"]
    do = _r(dhb @ p["wo"]).reshape(B, S, Hq, hd)
    dq, dk, dv = attention_bwd(do, c["q"], c["k"], c["v"], c["o"], c["lse"])
    dq = _r(ls.rope_bwd(dq, cos, sin).reshape(T, -1))
    dk = _r(ls.rope_bwd(dk, cos, sin).reshape(T, -1))
    dv = _r(dv.reshape(T, -1))
    u = c["u"]
    gr["wq"], gr["wk"], gr["wv"] = dq.T @ u, dk.T @ u, dv.T @ u
    if "bq" in p:
        gr["bq"], gr["bk"], gr["bv"] = dq.sum(axis=0), dk.sum(axis=0), dv.sum(axis=0)
    dxn, gr["g1"] = ls.rmsnorm_bwd(dq @ p["wq"] + dk @ p["wk"] + dv @ p["wv"], p["g1"], c["c1"])
    return dh + dxn, {k_: _r(v_) for k_, v_ in gr.items()}


def step_streamed(get_layer, n_layers, embed, final_norm, lm_head, tokens, labels, cfg,
                  dtype=np.float64, on_layer_grads=None):
    """(loss, grads) like oracle.step_streamed, with bf16 operands."""
    tokens = np.asarray(tokens)
    B, S = tokens.shape
    T, d = B * S, cfg.hidden
    cast = lambda a: np.asarray(a, dtype=dtype)
    E, gf = cast(embed), cast(final_norm)
    Wlm = E if lm_head is None else cast(lm_head)
    cos, sin = ls.rope_tables(S, cfg.head_dim, cfg.rope_base, dtype)
    x = E[tokens]
    caches = []
    for i in range(n_layers):
        p = {k: cast(v) for k, v in get_layer(i).items()}
        x, c = layer_fwd(x, p, cfg, cos, sin)
        caches.append(c)
    hf, cf = ls.rmsnorm_fwd(x.reshape(T, d), gf, cfg.rms_eps)
    hf = _r(hf)
    loss, dz, _ = ls.cross_entropy_fwd_bwd(hf @ Wlm.T, labels)
    dz = _r(dz)
    g_lm = _r(dz.T @ hf)
    dx, g_gf = ls.rmsnorm_bwd(dz @ Wlm, gf, cf)
    g_layers = None if on_layer_grads else [None] * n_layers
    for i in range(n_layers - 1, -1, -1):
        p = {k: cast(v) for k, v in get_layer(i).items()}
        dx, g = layer_bwd(dx, p, caches[i], cfg, cos, sin)
        caches[i] = None
        if on_layer_grads:
            on_layer_grads(i, g)
        else:
            g_layers[i] = g
    g_E = np.zeros_like(E)
    np.add.at(g_E, tokens.reshape(T), _r(dx))
    if lm_head is None:
        g_E, g_lm = g_E + g_lm, None
    return loss, dict(layers=g_layers, embed=g_E, final_norm=_r(g_gf), lm_head=g_lm)


def step_bf16_operands(w, tokens, labels, cfg, dtype=np.float64):
    """(loss, grads) like oracle.step, with bf16 operands."""
    return step_streamed(lambda i: w.layers[i], len(w.layers), w.embed, w.final_norm,
                         w.lm_head, tokens, labels, cfg, dtype=dtype)
