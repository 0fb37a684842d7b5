"""Full-batch fp64 training step: the definition that GPipe reproduces exactly.

TEST INFRASTRUCTURE ONLY (see the package docstring): never imported by the
product path.

What is computed, and where it comes from:

* GPipe technical review (zzz0906.github.io), "Preliminaries 6" and "Pipeline
  flow, phase 3": gradients of all micro-batches are accumulated and applied
  once, which is mathematically the single-device full-batch step.  So this
  module takes the whole mini-batch at once.
* "Preliminaries 2: the memory wall" names RMSProp as the optimizer (about
  12 bytes per parameter).  Its form is the common one: v <- rho v + (1-rho) g^2,
  w <- w - lr g / (sqrt(v) + eps), v starts at 0; no momentum, centring, decay.
* "Batch Normalization" section: LayerNorm normalises inside each sample, so
  micro-batching does not change it.  LN uses eps = 1e-5 and the biased
  (divide-by-d) variance.
* The block is the pre-LN Transformer block the review's Transformer
  experiments use (Vaswani et al. is its reference):
      h1 = x + W_o Attn(LN1(x)) + b_o
      y  = h1 + W_2 GELU(W_1 LN2(h1) + b_1) + b_2
  with exact erf GELU, causal softmax attention scaled by 1/sqrt(d_head), no
  positional term, a final LN before the tied-embedding head, and next-token
  cross-entropy averaged over all N(seq-1) predicted tokens.
  The FFN-only block (kind 0) is y = x + W_2 GELU(W_1 LN(x) + b_1) + b_2 with
  the MSE loss (1/(N d)) sum (y - t)^2.
* "Training stability": logit clipping, read as clamping every logit to
  [-c, c] before the softmax (so the loss sees the clamped logits and the
  gradient is zero where a logit lies outside the interval).  c is the
  workload's threshold in thousandths, v / 1000 rounded to fp32 (the value the
  step is given); v = 0 means no clipping.

All arithmetic is fp64; inputs (fp32 arrays from ``synth``) are promoted.
"""
from __future__ import annotations

import numpy as np
from scipy.special import erf

LN_EPS = 1e-5
_SQRT2 = np.sqrt(2.0)
_INV_SQRT_2PI = 1.0 / np.sqrt(2.0 * np.pi)


# --------------------------------------------------------------------------
# Elementary layers (forward returns the value and what backward needs)
# --------------------------------------------------------------------------

def layer_norm(x, g, b):
    """LayerNorm over the last axis: ((x - mean) / sqrt(var + eps)) * g + b."""
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    rstd = 1.0 / np.sqrt(var + LN_EPS)
    xhat = (x - mu) * rstd
    return xhat * g + b, (xhat, rstd)


def layer_norm_backward(dy, cache, g):
    """Gradients of layer_norm w.r.t. x, g and b."""
    xhat, rstd = cache
    d = xhat.shape[-1]
    dxhat = dy * g
    dx = rstd * (dxhat - dxhat.mean(axis=-1, keepdims=True)
                 - xhat * (dxhat * xhat).mean(axis=-1, keepdims=True))
    dg = (dy * xhat).reshape(-1, d).sum(axis=0)
    db = dy.reshape(-1, d).sum(axis=0)
    return dx, dg, db


def gelu(z):
    """Exact GELU: z * Phi(z), Phi the standard normal CDF."""
    return 0.5 * z * (1.0 + erf(z / _SQRT2))


def gelu_grad(z):
    """d GELU / dz = Phi(z) + z * phi(z)."""
    return 0.5 * (1.0 + erf(z / _SQRT2)) + z * _INV_SQRT_2PI * np.exp(-0.5 * z * z)


def linear(x, w, b=None):
    """x @ W^T (+ b), W stored [out, in]."""
    y = x @ w.T
    return y if b is None else y + b


def causal_attention(q, k, v):
    """softmax(q k^T / sqrt(dh) + causal mask) v for q, k, v of shape [N, H, S, dh].

    Position i attends to positions j <= i.  Returns the output and the
    probabilities P (needed by backward).
    """
    dh = q.shape[-1]
    s = (q @ np.swapaxes(k, -1, -2)) / np.sqrt(dh)
    S = s.shape[-1]
    future = np.triu(np.ones((S, S), dtype=bool), k=1)
    s = np.where(future, -np.inf, s)
    s = s - s.max(axis=-1, keepdims=True)
    p = np.exp(s)
    p = p / p.sum(axis=-1, keepdims=True)
    return p @ v, p


def causal_attention_backward(do, q, k, v, p):
    """Gradients of causal_attention w.r.t. q, k, v."""
    dh = q.shape[-1]
    scale = 1.0 / np.sqrt(dh)
    dv = np.swapaxes(p, -1, -2) @ do
    dp = do @ np.swapaxes(v, -1, -2)
    ds = p * (dp - (dp * p).sum(axis=-1, keepdims=True))
    dq = (ds @ k) * scale
    dk = (np.swapaxes(ds, -1, -2) @ q) * scale
    return dq, dk, dv


def _split_heads(t, heads):
    n, s, d = t.shape
    return t.reshape(n, s, heads, d // heads).transpose(0, 2, 1, 3)


def _merge_heads(t):
    n, h, s, dh = t.shape
    return t.transpose(0, 2, 1, 3).reshape(n, s, h * dh)


# --------------------------------------------------------------------------
# Blocks
# --------------------------------------------------------------------------

def block_forward(kind, p, pre, x, heads):
    """One residual block.  ``p`` maps names to fp64 arrays, ``pre`` is 'l<i>.'."""
    if kind == 0:
        u, c = layer_norm(x, p[pre + "ln_g"], p[pre + "ln_b"])
        z1 = linear(u, p[pre + "w1"], p[pre + "b1"])
        g = gelu(z1)
        y = x + linear(g, p[pre + "w2"], p[pre + "b2"])
        return y, dict(u=u, c=c, z1=z1, g=g)
    u, c1 = layer_norm(x, p[pre + "ln1_g"], p[pre + "ln1_b"])
    qkv = linear(u, p[pre + "w_qkv"], p[pre + "b_qkv"])
    d = x.shape[-1]
    q, k, v = (_split_heads(qkv[..., i * d:(i + 1) * d], heads) for i in range(3))
    o, prob = causal_attention(q, k, v)
    a = _merge_heads(o)
    h1 = x + linear(a, p[pre + "w_o"], p[pre + "b_o"])
    u2, c2 = layer_norm(h1, p[pre + "ln2_g"], p[pre + "ln2_b"])
    z1 = linear(u2, p[pre + "w1"], p[pre + "b1"])
    g = gelu(z1)
    y = h1 + linear(g, p[pre + "w2"], p[pre + "b2"])
    return y, dict(u=u, c1=c1, q=q, k=k, v=v, prob=prob, a=a, u2=u2, c2=c2, z1=z1, g=g)


def _acc(grads, name, val):
    grads[name] = grads[name] + val if name in grads else val


def _wgrad(dy, x):
    """Gradient of x @ W^T w.r.t. W: sum over all leading axes of dy^T x."""
    return dy.reshape(-1, dy.shape[-1]).T @ x.reshape(-1, x.shape[-1])


def _bgrad(dy):
    return dy.reshape(-1, dy.shape[-1]).sum(axis=0)


def block_backward(kind, p, pre, x, cache, dy, grads):
    """Backward of block_forward; accumulates parameter grads, returns dx."""
    if kind == 0:
        _acc(grads, pre + "w2", _wgrad(dy, cache["g"]))
        _acc(grads, pre + "b2", _bgrad(dy))
        dz1 = (dy @ p[pre + "w2"]) * gelu_grad(cache["z1"])
        _acc(grads, pre + "w1", _wgrad(dz1, cache["u"]))
        _acc(grads, pre + "b1", _bgrad(dz1))
        du = dz1 @ p[pre + "w1"]
        dx, dg, db = layer_norm_backward(du, cache["c"], p[pre + "ln_g"])
        _acc(grads, pre + "ln_g", dg)
        _acc(grads, pre + "ln_b", db)
        return dx + dy
    # FFN half
    _acc(grads, pre + "w2", _wgrad(dy, cache["g"]))
    _acc(grads, pre + "b2", _bgrad(dy))
    dz1 = (dy @ p[pre + "w2"]) * gelu_grad(cache["z1"])
    _acc(grads, pre + "w1", _wgrad(dz1, cache["u2"]))
    _acc(grads, pre + "b1", _bgrad(dz1))
    du2 = dz1 @ p[pre + "w1"]
    dh1, dg2, db2 = layer_norm_backward(du2, cache["c2"], p[pre + "ln2_g"])
    _acc(grads, pre + "ln2_g", dg2)
    _acc(grads, pre + "ln2_b", db2)
    dh1 = dh1 + dy
    # attention half
    _acc(grads, pre + "w_o", _wgrad(dh1, cache["a"]))
    _acc(grads, pre + "b_o", _bgrad(dh1))
    da = dh1 @ p[pre + "w_o"]
    heads = cache["q"].shape[1]
    dq, dk, dv = causal_attention_backward(_split_heads(da, heads), cache["q"], cache["k"],
                                           cache["v"], cache["prob"])
    dqkv = np.concatenate([_merge_heads(dq), _merge_heads(dk), _merge_heads(dv)], axis=-1)
    _acc(grads, pre + "w_qkv", _wgrad(dqkv, cache["u"]))
    _acc(grads, pre + "b_qkv", _bgrad(dqkv))
    du = dqkv @ p[pre + "w_qkv"]
    dx, dg1, db1 = layer_norm_backward(du, cache["c1"], p[pre + "ln1_g"])
    _acc(grads, pre + "ln1_g", dg1)
    _acc(grads, pre + "ln1_b", db1)
    return dx + dh1


# --------------------------------------------------------------------------
# Losses
# --------------------------------------------------------------------------

def mse_loss(y, t, count):
    """sum (y - t)^2 / count and its gradient; count = N*d for the full batch."""
    r = y - t
    return (r * r).sum() / count, 2.0 * r / count


def logit_clip_threshold(w):
    """The clipping threshold c of workload ``w`` (0.0: none)."""
    v = getattr(w, "logit_clip_milli", 0)
    return float(np.float32(v / 1000.0)) if v else 0.0


def next_token_ce(z, tokens, count, clip=0.0):
    """Next-token softmax cross-entropy over logits z [N, S, V].

    Position t predicts tokens[:, t+1]; the last position predicts nothing.
    clip > 0: the loss is taken over min(max(z, -clip), clip), and dz is the
    gradient with respect to the unclipped z (zero where |z| > clip).
    Returns (sum of per-token losses / count, dz, per-token losses [N, S-1]).
    """
    n, s, vocab = z.shape
    raw = z
    if clip > 0:
        z = np.clip(z, -clip, clip)
    zp = z[:, :-1, :]
    tgt = tokens[:, 1:]
    m = zp.max(axis=-1, keepdims=True)
    ez = np.exp(zp - m)
    se = ez.sum(axis=-1, keepdims=True)
    lse = (m + np.log(se))[..., 0]
    zt = np.take_along_axis(zp, tgt[..., None], axis=-1)[..., 0]
    per_tok = lse - zt
    dz = np.zeros_like(z)
    dz[:, :-1, :] = ez / se
    np.put_along_axis(dz[:, :-1, :], tgt[..., None],
                      np.take_along_axis(dz[:, :-1, :], tgt[..., None], axis=-1) - 1.0, axis=-1)
    if clip > 0:
        dz = np.where(np.abs(raw) <= clip, dz, 0.0)
    return per_tok.sum() / count, dz / count, per_tok


# --------------------------------------------------------------------------
# Full step
# --------------------------------------------------------------------------

def _f64(params):
    return {k: np.asarray(v, dtype=np.float64) for k, v in params.items()}


def loss_and_grads(w, params, batch, count=None):
    """Loss and exact gradients of the mini-batch in ``batch``.

    ``count`` is the normaliser (N*d for kind 0, N*(seq-1) for kind 1); by
    default the batch's own.  Passing the full batch's count for a slice gives
    that slice's contribution to the full-batch loss.
    Returns (loss, grads dict, extras dict with per-sequence losses for kind 1).
    """
    p = _f64(params)
    kind, L = w.kind, w.L
    grads = {}
    extras = {}
    if kind == 0:
        x = np.asarray(batch["x"], dtype=np.float64)
        t = np.asarray(batch["targets"], dtype=np.float64)
        if count is None:
            count = x.shape[0] * x.shape[1]
        xs, caches = [x], []
        for l in range(L):
            y, c = block_forward(0, p, f"l{l}.", xs[-1], 0)
            xs.append(y)
            caches.append(c)
        loss, dy = mse_loss(xs[-1], t, count)
        for l in reversed(range(L)):
            dy = block_backward(0, p, f"l{l}.", xs[l], caches[l], dy, grads)
        extras["dx0"] = dy
        return float(loss), grads, extras
    tok = np.asarray(batch["tokens"])
    n, s = tok.shape
    if count is None:
        count = n * (s - 1)
    emb = p["emb"]
    x = emb[tok]
    xs, caches = [x], []
    for l in range(L):
        y, c = block_forward(1, p, f"l{l}.", xs[-1], w.heads)
        xs.append(y)
        caches.append(c)
    hf, cf = layer_norm(xs[-1], p["lnf_g"], p["lnf_b"])
    z = hf @ emb.T
    loss, dz, per_tok = next_token_ce(z, tok, count, clip=logit_clip_threshold(w))
    extras["per_seq_loss"] = per_tok.sum(axis=1) / (s - 1)
    _acc(grads, "emb", _wgrad(dz, hf))
    dhf = dz @ emb
    dy, dgf, dbf = layer_norm_backward(dhf, cf, p["lnf_g"])
    _acc(grads, "lnf_g", dgf)
    _acc(grads, "lnf_b", dbf)
    for l in reversed(range(L)):
        dy = block_backward(1, p, f"l{l}.", xs[l], caches[l], dy, grads)
    dembg = np.zeros_like(emb)
    np.add.at(dembg, tok.reshape(-1), dy.reshape(-1, dy.shape[-1]))
    grads["emb"] = grads["emb"] + dembg
    return float(loss), grads, extras


def forward_loss(w, params, batch, count=None):
    """Loss only, keeping one layer's activations alive at a time.

    Used where the full backward does not fit: the value equals the loss of
    ``loss_and_grads``.  For kind 1 also returns per-sequence mean losses.
    """
    p = _f64(params)
    if w.kind == 0:
        x = np.asarray(batch["x"], dtype=np.float64)
        t = np.asarray(batch["targets"], dtype=np.float64)
        if count is None:
            count = x.shape[0] * x.shape[1]
        for l in range(w.L):
            x, _ = block_forward(0, p, f"l{l}.", x, 0)
        loss, _ = mse_loss(x, t, count)
        return float(loss), {}
    tok = np.asarray(batch["tokens"])
    n, s = tok.shape
    if count is None:
        count = n * (s - 1)
    x = p["emb"][tok]
    for l in range(w.L):
        x, _ = block_forward(1, p, f"l{l}.", x, w.heads)
    hf, _ = layer_norm(x, p["lnf_g"], p["lnf_b"])
    z = hf @ p["emb"].T
    loss, _, per_tok = next_token_ce(z, tok, count, clip=logit_clip_threshold(w))
    return float(loss), {"per_seq_loss": per_tok.sum(axis=1) / (s - 1)}


def rmsprop(params, grads, v, lr, decay, eps):
    """One RMSProp update of every parameter; returns (new params, new v)."""
    new_p, new_v = {}, {}
    for name, w0 in params.items():
        g = grads[name]
        vv = decay * np.asarray(v[name], dtype=np.float64) + (1.0 - decay) * g * g
        new_v[name] = vv
        new_p[name] = np.asarray(w0, dtype=np.float64) - lr * g / (np.sqrt(vv) + eps)
    return new_p, new_v


def step(w, params, batch, v=None):
    """One synchronous training step on the whole mini-batch.

    Returns dict(loss, grads, params (updated), v (updated), extras).
    ``v`` defaults to zeros (the first step).
    """
    loss, grads, extras = loss_and_grads(w, params, batch)
    if v is None:
        v = {k: np.zeros(np.shape(a)) for k, a in params.items()}
    new_p, new_v = rmsprop(params, grads, v, w.lr, w.decay, w.eps)
    return dict(loss=loss, grads=grads, params=new_p, v=new_v, extras=extras)
