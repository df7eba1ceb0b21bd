"""fp64 CPU oracle for the backward pass of the parallel transformer block
(PTB) with causal sliding-window attention (SWA).

TEST INFRASTRUCTURE ONLY, like ptb_oracle: used by the tests and nowhere in
the product path; it shares no code with the CUDA path.

The pages' workload is training: MegaScale counts 6N FLOPs per token, 2N for
the forward pass and 4N for the backward pass (MegaScale study notes,
ai-yanyi-papers.pages.dev/papers/18-megascale.html, ch.2 §2.1, MFU
definition).  The backward pass is not written out on the pages; it is the
chain rule applied to the forward definition of the PTB (§2.2, PTB row)

    u = LN(x)
    q, k, v = u W_q^T, u W_k^T, u W_v^T       ctx = SWA_w(q, k, v) per head
    z = u W_up^T      g = gelu_tanh(z)
    y = x + ctx W_o^T + g W_down^T

for an upstream gradient dy = dL/dy.  Every step below is that derivative
written out in float64, one formula per intermediate, with full matrix
products through numpy and the attention as a dense masked softmax.
Pins (CPU tests): central finite differences of L = sum(y * dy) for every
gradient, the closed-form special cases W_o = W_down = 0 and w = 1, and
planted mistakes that those checks must catch.  Not "parity unpinned".
"""
from __future__ import annotations

import math

import numpy as np

from .ptb_oracle import (GELU_C, GELU_CUBIC, LN_EPS, _f64, band_mask, gelu_tanh, layer_norm,
                         swa_weights)


def gelu_tanh_grad(z) -> np.ndarray:
    """d/dz of 0.5 z (1 + tanh(c (z + a z^3))):
    0.5 (1 + t) + 0.5 z (1 - t^2) c (1 + 3 a z^2), t = tanh(c (z + a z^3))."""
    z = _f64(z)
    t = np.tanh(GELU_C * (z + GELU_CUBIC * z ** 3))
    return 0.5 * (1.0 + t) + 0.5 * z * (1.0 - t * t) * GELU_C * (1.0 + 3.0 * GELU_CUBIC * z * z)


def layer_norm_backward(x, gamma, du, eps: float = LN_EPS):
    """Gradients of u = (x - mean) / sqrt(var + eps) * gamma + beta over the
    last axis, given du = dL/du.  With xh = (x - mean) * r, r = 1/sqrt(var + eps)
    and g = du * gamma:
        dx = r * (g - mean(g) - xh * mean(g * xh))
        dgamma = sum over rows of du * xh,   dbeta = sum over rows of du.
    Returns (dx, dgamma, dbeta)."""
    x = _f64(x)
    du = _f64(du)
    mu = x.mean(axis=-1, keepdims=True)
    r = 1.0 / np.sqrt(((x - mu) ** 2).mean(axis=-1, keepdims=True) + eps)
    xh = (x - mu) * r
    g = du * _f64(gamma)
    dx = r * (g - g.mean(axis=-1, keepdims=True) - xh * (g * xh).mean(axis=-1, keepdims=True))
    rows = tuple(range(du.ndim - 1))
    return dx, (du * xh).sum(axis=rows), du.sum(axis=rows)


def swa_backward(q, k, v, do, window: int, scale: float | None = None):
    """Gradients of o = P v, P = softmax_band(q k^T * scale), for do = dL/do.
    Shapes [..., s, d].  With the softmax Jacobian written out:
        dv = P^T do,   dP = do v^T,   dS = P * (dP - rowsum(dP * P)),
        dq = dS k * scale,   dk = dS^T q * scale.
    Entries outside the band have P = 0 and so dS = 0.  Returns (dq, dk, dv)."""
    q, k, v, do = (_f64(a) for a in (q, k, v, do))
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    p = swa_weights(q, k, window, scale)
    dv = np.swapaxes(p, -1, -2) @ do
    dp = do @ np.swapaxes(v, -1, -2)
    ds = p * (dp - (dp * p).sum(axis=-1, keepdims=True))
    dq = (ds @ k) * scale
    dk = (np.swapaxes(ds, -1, -2) @ q) * scale
    return dq, dk, dv


def ptb_backward(x, ln_gamma, ln_beta, w_qkv, w_o, w_up, w_down, heads: int, window: int, dy,
                 eps: float = LN_EPS) -> dict:
    """All gradients of the PTB layer for the upstream gradient dy [B, s, H].

    Weights in nn.Linear [out, in] form and head layout as in
    ptb_oracle.ptb_forward.  Returns a dict with dx [B, s, H], dln_gamma,
    dln_beta [H], dw_qkv [3H, H], dw_o [H, H], dw_up [F, H], dw_down [H, F]."""
    x, dy = _f64(x), _f64(dy)
    w_qkv, w_o, w_up, w_down = (_f64(w) for w in (w_qkv, w_o, w_up, w_down))
    bsz, seq, hidden = x.shape
    d = hidden // heads

    # Forward intermediates (the definitions of ptb_oracle, on all rows).
    u = layer_norm(x, ln_gamma, ln_beta, eps)                      # [B, s, H]
    qkv = u @ w_qkv.T                                              # [B, s, 3H]

    def heads_of(t):  # [B, s, H] -> [B, heads, s, d]
        return t.reshape(bsz, seq, heads, d).transpose(0, 2, 1, 3)

    def merge(t):     # [B, heads, s, d] -> [B, s, H]
        return t.transpose(0, 2, 1, 3).reshape(bsz, seq, hidden)

    q, k, v = (heads_of(qkv[..., i * hidden:(i + 1) * hidden]) for i in range(3))
    scale = 1.0 / math.sqrt(d)
    ctx = merge(swa_weights(q, k, window, scale) @ v)              # [B, s, H]
    z = u @ w_up.T                                                 # [B, s, F]
    g = gelu_tanh(z)

    def flat(t):      # [B, s, n] -> [B*s, n]
        return t.reshape(-1, t.shape[-1])

    # y = x + ctx W_o^T + g W_down^T
    dw_o = flat(dy).T @ flat(ctx)
    dw_down = flat(dy).T @ flat(g)
    dctx = dy @ w_o
    dg = dy @ w_down
    # g = gelu(z), z = u W_up^T
    dz = dg * gelu_tanh_grad(z)
    dw_up = flat(dz).T @ flat(u)
    # ctx = SWA(q, k, v), [q | k | v] = u W_qkv^T
    dq, dk, dv = swa_backward(q, k, v, heads_of(dctx), window, scale)
    dqkv = np.concatenate([merge(dq), merge(dk), merge(dv)], axis=-1)
    dw_qkv = flat(dqkv).T @ flat(u)
    du = dqkv @ w_qkv + dz @ w_up
    # u = LN(x); y also holds x itself
    dx_ln, dgamma, dbeta = layer_norm_backward(x, ln_gamma, du, eps)
    return dict(dx=dy + dx_ln, dln_gamma=dgamma, dln_beta=dbeta, dw_qkv=dw_qkv, dw_o=dw_o,
                dw_up=dw_up, dw_down=dw_down)


def backward_flops(batch: int, seq: int, hidden: int, ffn: int, window: int) -> dict:
    """Algorithmic backward FLOPs of one PTB layer.

    GEMMs: each forward GEMM has an input-gradient and a weight-gradient GEMM
    of the same size, 2 x the forward GEMM FLOPs.  Attention: dV = P^T dO,
    dP = dO V^T, dQ = dS K, dK = dS^T Q over the in-band pairs, 8*B*H*band."""
    t = batch * seq
    band = int(band_mask(np.arange(seq), np.arange(seq), window).sum())
    gemm = 2 * (2 * t * hidden * (3 * hidden + ffn) + 2 * t * (hidden + ffn) * hidden)
    attn = 8 * batch * hidden * band
    return {"gemm": gemm, "attn": attn, "total": gemm + attn}
