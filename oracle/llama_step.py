"""One training step of a pre-norm Llama-style decoder stack, written out plainly.

TEST INFRASTRUCTURE ONLY: imported by the tests, by the smoke check and by the
benchmark's CPU-baseline leg, never by the library.

What is computed, and where it comes from.  SlideFormer ("An Efficient
Heterogeneous Co-Design for Fine-Tuning on a Single GPU") fine-tunes Llama,
Qwen and Mistral models with their standard training objectives (gist.science
summary, section 4 "Betekenis en Impact"); it names RoPE, RMSNorm and SwiGLU as
the kernels it optimises and fuses the LM-head projection with the
cross-entropy loss without changing the result (section 2.C "Geintegreerde
Geavanceerde I/O en Kernels"); its optimizer is a per-layer Adam applied on the
host (section 2.A and 2.B "Layer-Adam Optimizer").  The pages print none of
these equations, so each function below is the standard Llama definition.
Readings taken where the pages are silent:
  * RoPE pairs feature j with j + head_dim/2 ("rotate half"), angle
    s * base^(-2j/head_dim) at position s, no frequency scaling.
  * RMSNorm: y = g * x / sqrt(mean(x^2) + eps), gain applied after normalising.
  * Causal mask includes the diagonal; softmax scale 1/sqrt(head_dim).
  * GQA: query head h reads kv head floor(h / (Hq / Hkv)) (contiguous groups).
  * Loss: mean of (logsumexp(z_t) - z_t[y_t]) over the whole batch's rows whose
    label is not IGNORE_INDEX; with no valid row the loss and all gradients are 0.
  * Embedding and LM head are separate tensors, unless the model ties them
    (then the LM head is the embedding matrix and its gradient is the sum of
    the two uses).
  * Qwen-family models add a bias to the Q, K and V projections, before RoPE.
  * Adam: bias-corrected, decoupled weight decay (AdamW form), no clipping.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

IGNORE_INDEX = -100


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); result as float32."""
    a = np.ascontiguousarray(x, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).reshape(a.shape)


# ---------------------------------------------------------------- RMSNorm
def rmsnorm_fwd(x, g, eps):
    """y = g * x / sqrt(mean_j x_j^2 + eps) over the last axis.  Returns y and
    the cache (x_hat, rstd) that the backward needs."""
    rstd = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    xhat = x * rstd
    return xhat * g, (xhat, rstd)


def rmsnorm_bwd(dy, g, cache):
    """Chain rule through rmsnorm_fwd: dx = rstd * (g dy - x_hat * mean(g dy x_hat)),
    dg = sum over rows of dy * x_hat."""
    xhat, rstd = cache
    dg = np.sum((dy * xhat).reshape(-1, dy.shape[-1]), axis=0)
    gdy = dy * g
    dx = rstd * (gdy - xhat * np.mean(gdy * xhat, axis=-1, keepdims=True))
    return dx, dg


# ---------------------------------------------------------------- RoPE
def rope_tables(seq, head_dim, base, dtype=np.float64):
    """cos and sin of the angles s * base^(-2j/head_dim), s < seq, j < head_dim/2."""
    j = np.arange(head_dim // 2, dtype=np.float64)
    inv_freq = float(base) ** (-2.0 * j / head_dim)
    ang = np.arange(seq, dtype=np.float64)[:, None] * inv_freq[None, :]
    return np.cos(ang).astype(dtype), np.sin(ang).astype(dtype)


def rope_fwd(x, cos, sin):
    """Rotate each pair (x_j, x_{j+hd/2}) of x [B, S, H, hd] by the angle of its
    position s:  x'_j = x_j cos - x_{j+hd/2} sin,  x'_{j+hd/2} = x_{j+hd/2} cos + x_j sin."""
    half = x.shape[-1] // 2
    c, s = cos[None, :, None, :], sin[None, :, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def rope_bwd(dy, cos, sin):
    """Transpose of rope_fwd (rotation by the opposite angle)."""
    half = dy.shape[-1] // 2
    c, s = cos[None, :, None, :], sin[None, :, None, :]
    d1, d2 = dy[..., :half], dy[..., half:]
    return np.concatenate([d1 * c + d2 * s, d2 * c - d1 * s], axis=-1)


# ---------------------------------------------------------------- attention
def _group(n_heads, n_kv_heads):
    assert n_heads % n_kv_heads == 0
    return n_heads // n_kv_heads


def attention_fwd(q, k, v):
    """Causal softmax attention.  q [B, S, Hq, hd]; k, v [B, S, Hkv, hd].
    o[s] = sum_{r<=s} softmax_r(q_s . k_r / sqrt(hd)) v_r for each query head,
    using kv head h // (Hq/Hkv).  Returns o [B, S, Hq, hd] and the row
    log-sum-exp lse [B, Hq, S] of the scaled scores."""
    B, S, Hq, hd = q.shape
    grp = _group(Hq, k.shape[2])
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
            o[b, :, h, :] = (e / l) @ v[b, :, g, :]
            lse[b, h, :] = (m + np.log(l))[:, 0]
    return o, lse


def attention_bwd(do, q, k, v):
    """Gradients of attention_fwd.  With P the attention matrix of one head:
    dV = P^T dO, dP = dO V^T, dS = P * (dP - rowsum(dP * P)), dQ = dS K / sqrt(hd),
    dK = dS^T Q / sqrt(hd); dK and dV are summed over the query heads that share
    a kv head."""
    B, S, Hq, hd = q.shape
    grp = _group(Hq, k.shape[2])
    scale = 1.0 / np.sqrt(hd)
    future = np.triu(np.ones((S, S), dtype=bool), 1)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for h in range(Hq):
            g = h // grp
            sc = (q[b, :, h, :] @ k[b, :, g, :].T) * scale
            sc[future] = -np.inf
            p = np.exp(sc - sc.max(axis=1, keepdims=True))
            p /= p.sum(axis=1, keepdims=True)
            dv[b, :, g, :] += p.T @ do[b, :, h, :]
            dp = do[b, :, h, :] @ v[b, :, g, :].T
            ds = p * (dp - np.sum(dp * p, axis=1, keepdims=True))
            dq[b, :, h, :] = (ds @ k[b, :, g, :]) * scale
            dk[b, :, g, :] += (ds.T @ q[b, :, h, :]) * scale
    return dq, dk, dv


# ---------------------------------------------------------------- SwiGLU
def swiglu_fwd(a, b):
    """m = silu(a) * b with silu(a) = a / (1 + exp(-a))."""
    return a / (1.0 + np.exp(-a)) * b


def swiglu_bwd(dm, a, b):
    """da = dm * b * sigma(a) * (1 + a (1 - sigma(a))),  db = dm * silu(a)."""
    sig = 1.0 / (1.0 + np.exp(-a))
    return dm * b * sig * (1.0 + a * (1.0 - sig)), dm * a * sig


# ---------------------------------------------------------------- loss
def cross_entropy_fwd_bwd(z, labels):
    """Mean token cross-entropy over rows whose label is not IGNORE_INDEX, on the
    full (unfused) logits z [N, V].  Returns (loss, dz, lse) where
    dz = (softmax(z) - onehot(label)) / n_valid on valid rows and 0 elsewhere."""
    labels = np.asarray(labels).reshape(-1)
    valid = labels != IGNORE_INDEX
    n_valid = int(valid.sum())
    m = z.max(axis=1, keepdims=True)
    lse = m[:, 0] + np.log(np.sum(np.exp(z - m), axis=1))
    if n_valid == 0:
        return 0.0, np.zeros_like(z), lse
    rows = np.nonzero(valid)[0]
    loss = float(np.sum(lse[rows] - z[rows, labels[rows]]) / n_valid)
    dz = np.exp(z - lse[:, None])
    dz[rows, labels[rows]] -= 1.0
    dz[~valid] = 0.0
    return loss, dz / n_valid, lse


# ---------------------------------------------------------------- one layer
def layer_fwd(x, p, cfg, cos, sin):
    """Pre-norm decoder layer on x [B, S, d]:
    h = x + Attn(RoPE(RMSNorm(x; g1) Wq^T), RoPE(. Wk^T), . Wv^T) Wo^T,
    out = h + (silu(RMSNorm(h; g2) Wg^T) * (RMSNorm(h; g2) Wu^T)) Wd^T."""
    B, S, d = x.shape
    T = B * S
    Hq, Hkv, hd = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
    xf = x.reshape(T, d)
    u, c1 = rmsnorm_fwd(xf, p["g1"], cfg.rms_eps)
    q, k, v = u @ p["wq"].T, u @ p["wk"].T, u @ p["wv"].T
    if "bq" in p:  # projection biases, added before the rotation
        q, k, v = q + p["bq"], k + p["bk"], v + p["bv"]
    q = rope_fwd(q.reshape(B, S, Hq, hd), cos, sin)
    k = rope_fwd(k.reshape(B, S, Hkv, hd), cos, sin)
    v = v.reshape(B, S, Hkv, hd)
    o, _ = attention_fwd(q, k, v)
    of = o.reshape(T, Hq * hd)
    h = xf + of @ p["wo"].T
    w2, c2 = rmsnorm_fwd(h, p["g2"], cfg.rms_eps)
    a = w2 @ p["wg"].T
    b = w2 @ p["wu"].T
    m = swiglu_fwd(a, b)
    out = h + m @ p["wd"].T
    cache = dict(u=u, c1=c1, q=q, k=k, v=v, of=of, w2=w2, c2=c2, a=a, b=b, m=m)
    return out.reshape(B, S, d), cache


def layer_bwd(dout, p, cache, cfg, cos, sin):
    """Backward of layer_fwd.  dout [T, d] -> (dx [T, d], grads by tensor name)."""
    T, d = dout.shape
    Hq, Hkv, hd = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
    q, k, v = cache["q"], cache["k"], cache["v"]
    B, S = q.shape[0], q.shape[1]
    gr = {}
    gr["wd"] = dout.T @ cache["m"]
    dm = dout @ p["wd"]
    da, db = swiglu_bwd(dm, cache["a"], cache["b"])
    gr["wg"] = da.T @ cache["w2"]
    gr["wu"] = db.T @ cache["w2"]
    dw2 = da @ p["wg"] + db @ p["wu"]
    dhn, gr["g2"] = rmsnorm_bwd(dw2, p["g2"], cache["c2"])
    dh = dout + dhn
    gr["wo"] = dh.T @ cache["of"]
    do = (dh @ p["wo"]).reshape(B, S, Hq, hd)
    dq, dk, dv = attention_bwd(do, q, k, v)
    dq = rope_bwd(dq, cos, sin).reshape(T, Hq * hd)
    dk = rope_bwd(dk, cos, sin).reshape(T, Hkv * hd)
    dv = dv.reshape(T, Hkv * hd)
    u = cache["u"]
    gr["wq"], gr["wk"], gr["wv"] = dq.T @ u, dk.T @ u, dv.T @ u
    if "bq" in p:
        gr["bq"], gr["bk"], gr["bv"] = dq.sum(axis=0), dk.sum(axis=0), dv.sum(axis=0)
    du = dq @ p["wq"] + dk @ p["wk"] + dv @ p["wv"]
    dxn, gr["g1"] = rmsnorm_bwd(du, p["g1"], cache["c1"])
    return dh + dxn, gr


# ---------------------------------------------------------------- full step
@dataclass
class ModelWeights:
    """Weights the step computes with (already rounded to bf16 by the caller
    where the compared path uses bf16).  layers[i] maps g1, wq, wk, wv, wo, g2,
    wg, wu, wd (and bq, bk, bv when the model has projection biases) to arrays
    in nn.Linear [out, in] layout.  lm_head None: tied to the embedding."""
    layers: list
    embed: np.ndarray
    final_norm: np.ndarray
    lm_head: np.ndarray
    extras: dict = field(default_factory=dict)


def step(w: ModelWeights, tokens, labels, cfg, dtype=np.float64, return_hidden=False):
    """Forward and backward of the whole stack plus mean token cross-entropy.
    tokens, labels: int [B, S].  Returns (loss, grads) with grads = dict(
    layers=[{name: array}], embed, final_norm, lm_head).  With a tied LM head
    (w.lm_head None) grads["lm_head"] is None and grads["embed"] holds both
    uses of the embedding.  With return_hidden the per-layer inputs X_l, the
    final hidden states and the logits are returned too."""
    cast = lambda a: np.asarray(a, dtype=dtype)
    layers = [{k: cast(v) for k, v in lp.items()} for lp in w.layers]
    return step_streamed(lambda i: layers[i], len(layers), w.embed, w.final_norm, w.lm_head,
                         tokens, labels, cfg, dtype=dtype, return_hidden=return_hidden)


def step_streamed(get_layer, n_layers, embed, final_norm, lm_head, tokens, labels, cfg,
                  dtype=np.float64, on_layer_grads=None, return_hidden=False):
    """step() with the decoder layers' weights fetched one layer at a time:
    get_layer(i) returns layer i's weight dict (called once in the forward and
    once in the backward), so only the activations of the stack are held, not
    all of its weights.  When on_layer_grads is given, layer i's gradients go
    to on_layer_grads(i, grads) as the backward produces them (and
    grads["layers"] is None); otherwise they are collected as in step()."""
    tokens = np.asarray(tokens)
    B, S = tokens.shape
    T, d = B * S, cfg.hidden
    cast = lambda a: np.asarray(a, dtype=dtype)
    E, gf = cast(embed), cast(final_norm)
    tied = lm_head is None
    Wlm = E if tied else cast(lm_head)
    cos, sin = rope_tables(S, cfg.head_dim, cfg.rope_base, dtype)

    x = E[tokens]                                  # [B, S, d]
    xs, caches = [], []
    for i in range(n_layers):
        p = {k: cast(v) for k, v in get_layer(i).items()}
        xs.append(x)
        x, c = layer_fwd(x, p, cfg, cos, sin)
        caches.append(c)
        del p
    hf, cf = rmsnorm_fwd(x.reshape(T, d), gf, cfg.rms_eps)
    z = hf @ Wlm.T
    loss, dz, _ = cross_entropy_fwd_bwd(z, labels)

    g_lm = dz.T @ hf
    dx, g_gf = rmsnorm_bwd(dz @ Wlm, gf, cf)
    if not return_hidden:
        del z, dz
    g_layers = None if on_layer_grads else [None] * n_layers
    for i in range(n_layers - 1, -1, -1):
        p = {k: cast(v) for k, v in get_layer(i).items()}
        dx, g = layer_bwd(dx, p, caches[i], cfg, cos, sin)
        caches[i] = None
        del p
        if on_layer_grads:
            on_layer_grads(i, g)
        else:
            g_layers[i] = g
    g_E = np.zeros_like(E)
    np.add.at(g_E, tokens.reshape(T), dx)
    if tied:  # one tensor used twice: its gradient is the sum of both uses
        g_E, g_lm = g_E + g_lm, None
    grads = dict(layers=g_layers, embed=g_E, final_norm=g_gf, lm_head=g_lm, dx0=dx)
    if return_hidden:
        return loss, grads, dict(xs=xs, x_final=x.reshape(T, d), logits=z, hf=hf)
    return loss, grads


# ---------------------------------------------------------------- Adam
def adam_update(theta, g, m, v, t, lr, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0):
    """One bias-corrected Adam step with decoupled weight decay, at step count t >= 1:
    m <- b1 m + (1-b1) g;  v <- b2 v + (1-b2) g^2;
    theta <- theta - lr * wd * theta - lr * (m / (1-b1^t)) / (sqrt(v / (1-b2^t)) + eps).
    Returns new (theta, m, v)."""
    m = beta1 * m + (1.0 - beta1) * g
    v = beta2 * v + (1.0 - beta2) * g * g
    mhat = m / (1.0 - beta1 ** t)
    vhat = v / (1.0 - beta2 ** t)
    theta = theta - lr * weight_decay * theta - lr * mhat / (np.sqrt(vhat) + eps)
    return theta, m, v


# ---------------------------------------------------------------- Adam with 16-bit moments
# Optimizer-state compression: the moments are stored as bfloat16, rounded
# stochastically so that increments far below a bf16 step (v moves by
# (1 - beta2) = 0.1% of itself per step) survive in expectation.  The random
# bits are a counter-based hash of (step, unit, element index), so both
# implementations draw the same bits: one 32-bit word per element, its low
# half-word rounds the first moment and its high half-word the second.
_U32 = np.uint32


def lowbias32(x):
    """32-bit integer hash (Wellons' "lowbias32": xorshift-multiply rounds with
    the constants 0x7feb352d and 0x846ca68b), elementwise on uint32."""
    x = np.asarray(x, dtype=_U32)
    with np.errstate(over="ignore"):
        x = x ^ (x >> _U32(16))
        x = x * _U32(0x7FEB352D)
        x = x ^ (x >> _U32(15))
        x = x * _U32(0x846CA68B)
        x = x ^ (x >> _U32(16))
    return x


def sr_key(t, unit):
    """Stream key of step t >= 1 and unit (layer index, or -1 embedding, -2
    final norm, -3 LM head)."""
    with np.errstate(over="ignore"):
        mixed = lowbias32(_U32(t & 0xFFFFFFFF)) ^ (_U32(unit + 3) * _U32(0x9E3779B9))
    return lowbias32(mixed)


def sr_bits(key, index):
    """The random word of element `index` (its position in the unit's tensors,
    concatenated in unit order) in the stream `key`."""
    return lowbias32(np.asarray(index, dtype=np.uint64).astype(_U32) ^ _U32(key))


def bf16_round_stochastic(x, r):
    """Round float32 x to bfloat16 upwards (in magnitude) with probability
    (low 16 bits of x) / 2^16: add the low 16 bits of r to x's bits, then
    truncate.  E[result] = x for finite x.  Result as float32."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(_U32).astype(np.uint64)
    u = (u + (np.asarray(r, dtype=np.uint64) & np.uint64(0xFFFF))) & np.uint64(0xFFFF0000)
    return u.astype(_U32).view(np.float32).reshape(np.shape(x))


def adam_update_bf16_states(theta, g, m, v, t, lr, unit, beta1=0.9, beta2=0.999, eps=1e-8,
                            weight_decay=0.0, index0=0):
    """adam_update in float32 arithmetic with the moments m, v stored as
    bfloat16 (float32 arrays holding bf16 values): the new moments are
    computed in float32, used unrounded for this step's parameter update,
    then stored with bf16_round_stochastic: element i of the unit draws
    r = sr_bits(sr_key(t, unit), index0 + i), the first moment rounds with
    the low and the second with the high half-word of r.  Returns (theta, m, v)."""
    f = np.float32
    theta, g, m, v = (np.asarray(a, dtype=np.float32) for a in (theta, g, m, v))
    b1, b2, lr_, eps_, wd = f(beta1), f(beta2), f(lr), f(eps), f(weight_decay)
    # the scalar bias corrections in float64 (1 - b2^t cancels in float32)
    bc1 = f(1.0 - float(b1) ** t)
    bc2 = f(1.0 - float(b2) ** t)
    m1 = b1 * m + (f(1.0) - b1) * g
    v1 = b2 * v + (f(1.0) - b2) * g * g
    th = theta - lr_ * wd * theta - lr_ * (m1 / bc1) / (np.sqrt(v1 / bc2) + eps_)
    idx = index0 + np.arange(theta.size, dtype=np.uint64)
    r = sr_bits(sr_key(t, unit), idx).reshape(theta.shape)
    mq = bf16_round_stochastic(m1, r)
    vq = bf16_round_stochastic(v1, r >> _U32(16))
    return th.astype(np.float32), mq, vq
