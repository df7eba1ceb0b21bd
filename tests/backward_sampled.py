"""Sampled entries of the PTB layer's gradients, for full-size parity checks.

Composes the fp64 oracle's functions (oracle.layer_norm, swa_weights,
swa_backward, gelu_tanh, gelu_tanh_grad, layer_norm_backward) on subsets:
every returned entry is the same formula as oracle.ptb_backward, evaluated
only where it is needed -- dx at a few sequence rows, and the weight
gradients at a few heads, FFN columns and output rows.  Batch entries are
summed as in the full oracle.
"""
import math

import numpy as np

import oracle


def _f64(t):
    return t.detach().to("cpu").double().numpy() if hasattr(t, "detach") else np.asarray(t, np.float64)


def sampled_backward(x, ln_gamma, ln_beta, w_qkv, w_o, w_up, w_down, heads, window, dy, rows,
                     head_sel, f_sel, r_sel):
    """Returns a dict of expected values:
      dx       [B, len(rows), H]
      dw_o     [len(r_sel), len(head_sel) * d]   (columns of the selected heads)
      dw_down  [len(r_sel), len(f_sel)]
      dw_up    [len(f_sel), H]
      dw_qkv   [3 * len(head_sel) * d, H]        (q rows, then k rows, then v rows
                                                  of the selected heads)"""
    x, dy = _f64(x), _f64(dy)
    w_qkv, w_o, w_up, w_down = (_f64(w) for w in (w_qkv, w_o, w_up, w_down))
    bsz, seq, hidden = x.shape
    d = hidden // heads
    scale = 1.0 / math.sqrt(d)
    rows = np.asarray(rows)
    u = oracle.layer_norm(x, ln_gamma, ln_beta)                       # [B, s, H]
    qkv = u @ w_qkv.T                                                 # [B, s, 3H]
    dctx = dy @ w_o                                                   # [B, s, H]

    def head(t, i, h):  # [B, s, 3H or H] -> [B, s, d] of block i, head h
        return t[..., i * hidden + h * d: i * hidden + (h + 1) * d]

    dq_rows = np.zeros((bsz, len(rows), hidden))
    dk_rows = np.zeros_like(dq_rows)
    dv_rows = np.zeros_like(dq_rows)
    ctx_sel, dqkv_sel = [], []
    for h in range(heads):
        q, k, v, g = head(qkv, 0, h), head(qkv, 1, h), head(qkv, 2, h), head(dctx, 0, h)
        dq, dk, dv = oracle.swa_backward(q, k, v, g, window, scale)
        dq_rows[..., h * d:(h + 1) * d] = dq[:, rows]
        dk_rows[..., h * d:(h + 1) * d] = dk[:, rows]
        dv_rows[..., h * d:(h + 1) * d] = dv[:, rows]
        if h in head_sel:
            ctx_sel.append(oracle.swa_weights(q, k, window, scale) @ v)
            dqkv_sel.append((dq, dk, dv))

    # dx at the sampled rows: dxn = [dq | dk | dv | dz] [W_qkv ; W_up]
    z_rows = u[:, rows] @ w_up.T
    dz_rows = (dy[:, rows] @ w_down) * oracle.gelu_tanh_grad(z_rows)
    dxn = np.concatenate([dq_rows, dk_rows, dv_rows], axis=-1) @ w_qkv + dz_rows @ w_up
    dx = dy[:, rows] + oracle.layer_norm_backward(x[:, rows], ln_gamma, dxn)[0]

    def tsum(a, b):  # sum over batch and sequence of a^T b
        return np.einsum("bsi,bsj->ij", a, b)

    r_sel, f_sel = np.asarray(r_sel), np.asarray(f_sel)
    dw_o = tsum(dy[..., r_sel], np.concatenate(ctx_sel, axis=-1))
    z_sel = u @ w_up[f_sel].T
    dw_down = tsum(dy[..., r_sel], oracle.gelu_tanh(z_sel))
    dz_sel = (dy @ w_down[:, f_sel]) * oracle.gelu_tanh_grad(z_sel)
    dw_up = tsum(dz_sel, u)
    dw_qkv = np.concatenate([tsum(t[i], u) for i in range(3) for t in dqkv_sel], axis=0)
    return dict(dx=dx, dw_o=dw_o, dw_down=dw_down, dw_up=dw_up, dw_qkv=dw_qkv)


def gathered(g, hidden, heads, rows, head_sel, f_sel, r_sel):
    """The same entries picked out of full gradient tensors (host numpy)."""
    d = hidden // heads
    cols = np.concatenate([np.arange(h * d, (h + 1) * d) for h in head_sel])
    qkv_rows = np.concatenate([i * hidden + np.arange(h * d, (h + 1) * d)
                               for i in range(3) for h in head_sel])
    r_sel, f_sel = np.asarray(r_sel), np.asarray(f_sel)
    return dict(dx=g["dx"][:, rows], dw_o=g["dw_o"][np.ix_(r_sel, cols)],
                dw_down=g["dw_down"][np.ix_(r_sel, f_sel)], dw_up=g["dw_up"][f_sel],
                dw_qkv=g["dw_qkv"][qkv_rows])
