"""fp64 CPU oracle for the parallel transformer block (PTB) forward pass with
causal sliding-window attention (SWA).

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import or call this
module; only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` use it.  It shares no code with the CUDA path: it takes numpy
arrays (the bf16 inputs already upcast by the caller) and returns numpy fp64.

Sources (MegaScale study notes, ai-yanyi-papers.pages.dev/papers/18-megascale.html):
  * ch.2 §2.2 (paper §3.1), algorithm-change table, PTB row:
        y = x + MLP(LN(x)) + Attention(LN(x))
    -- one LayerNorm shared by both branches, the two branch outputs summed
    with the residual.
  * same table, SWA row: every token attends only to a fixed window of w
    positions, cost O(s*w) instead of O(s*s).
  * ch.2 §2.2, "common misreadings" (1): PTB keeps the residual structure and
    the output space of the serial block.
Constants the pages leave open (fixed by the workload definition and restated
here): the window is causal and contains the token itself, so row i sees keys
max(0, i-w+1) .. i; softmax scale 1/sqrt(d); tanh-approximated GELU; LayerNorm
eps 1e-5 with the biased variance; no biases, dropout or positional terms.

Every function computes its definition directly in float64: full matrix
products through numpy (a library primitive), the attention as a masked
softmax over all key positions.  No blocking, online softmax or fusion.
Parity pins: all functions here are pinned by the CPU tests (closed forms,
library special cases, brute force) -- none is "parity unpinned".
"""
from __future__ import annotations

import math

import numpy as np

LN_EPS = 1e-5
GELU_C = math.sqrt(2.0 / math.pi)
GELU_CUBIC = 0.044715


def _f64(a) -> np.ndarray:
    """float64 numpy copy of an array; torch tensors of any dtype (bf16
    included, which numpy lacks) are converted on the host first."""
    if hasattr(a, "detach"):
        a = a.detach().to("cpu").double().numpy()
    return np.asarray(a, dtype=np.float64)


def layer_norm(x, gamma, beta, eps: float = LN_EPS) -> np.ndarray:
    """LayerNorm over the last axis: (x - mean) / sqrt(var + eps) * gamma + beta.

    var is the biased (population) variance, eps sits inside the square root
    and the affine step follows the normalisation.  The PTB formula applies
    LN(x) once and feeds the same result to both branches (MegaScale notes,
    §2.2, PTB row)."""
    x = _f64(x)
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps) * _f64(gamma) + _f64(beta)


def gelu_tanh(z) -> np.ndarray:
    """gelu(z) = z/2 * (1 + tanh(sqrt(2/pi) * (z + 0.044715 z^3))).

    The pages name GeLU only as a fused operator (MegaScale notes, §2.5,
    Table 3, efficient-operators row); the tanh form is the workload's choice."""
    z = _f64(z)
    return 0.5 * z * (1.0 + np.tanh(GELU_C * (z + GELU_CUBIC * z ** 3)))


def band_mask(q_pos, k_pos, window: int) -> np.ndarray:
    """Boolean [len(q_pos), len(k_pos)] mask of the causal sliding window.

    Query position i may see key position j iff i - window < j <= i: the
    token itself and at most window-1 predecessors (MegaScale notes, §2.2,
    SWA row; causal, self-inclusive reading)."""
    if window < 1:
        raise ValueError("window must be >= 1")
    i = np.asarray(q_pos, dtype=np.int64)[:, None]
    j = np.asarray(k_pos, dtype=np.int64)[None, :]
    return (j <= i) & (j > i - window)


def attended_counts(seq: int, window: int) -> np.ndarray:
    """Number of keys each query row of a length-`seq` sequence attends to,
    read off the mask itself (row sums of band_mask)."""
    pos = np.arange(seq)
    return band_mask(pos, pos, window).sum(axis=1).astype(np.int64)


def swa_weights(q, k, window: int, scale: float | None = None,
                q_pos=None, k_pos=None) -> np.ndarray:
    """Softmax weights of causal sliding-window attention.

    q: [..., R, d] queries at positions q_pos (default 0..R-1);
    k: [..., S, d] keys at positions k_pos (default 0..S-1).
    Scores q.k * scale are set to -inf outside the band, then normalised with
    a max-subtracted softmax over the key axis.  Returns [..., R, S]."""
    q = _f64(q)
    k = _f64(k)
    d = q.shape[-1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if q_pos is None:
        q_pos = np.arange(q.shape[-2])
    if k_pos is None:
        k_pos = np.arange(k.shape[-2])
    mask = band_mask(q_pos, k_pos, window)
    scores = (q @ np.swapaxes(k, -1, -2)) * scale
    scores = np.where(mask, scores, -np.inf)
    m = scores.max(axis=-1, keepdims=True)
    e = np.exp(scores - m)
    return e / e.sum(axis=-1, keepdims=True)


def swa(q, k, v, window: int, scale: float | None = None,
        q_pos=None, k_pos=None) -> np.ndarray:
    """Causal sliding-window attention o = softmax_band(q k^T * scale) v.

    Shapes [..., R, d] for q and [..., S, d] for k and v (e.g. [B, heads, s, d]).
    When q_pos is a subset of rows, k_pos must contain every key position in
    the window of each of those rows."""
    if q_pos is not None and k_pos is not None:
        need = set()
        for i in np.asarray(q_pos):
            need.update(range(max(0, int(i) - window + 1), int(i) + 1))
        missing = need.difference(int(j) for j in np.asarray(k_pos))
        if missing:
            raise ValueError(f"k_pos misses {len(missing)} in-window keys")
    p = swa_weights(q, k, window, scale, q_pos, k_pos)
    return p @ _f64(v)


def linear(a, w) -> np.ndarray:
    """a @ w.T for an nn.Linear weight w of shape [out, in] (no bias).

    w is upcast to float64 a slab of output rows at a time so that the
    530B-shaped weights need not exist twice in fp64; every output element
    is still one full-length dot product."""
    a = _f64(a)
    out = np.empty(a.shape[:-1] + (w.shape[0],), dtype=np.float64)
    step = 8192
    for r0 in range(0, w.shape[0], step):
        out[..., r0:r0 + step] = a @ _f64(w[r0:r0 + step]).T
    return out


def needed_key_positions(rows, window: int) -> np.ndarray:
    """Sorted union of the key positions inside the windows of `rows`."""
    need = set()
    for i in rows:
        need.update(range(max(0, int(i) - window + 1), int(i) + 1))
    return np.array(sorted(need), dtype=np.int64)


def attention_branch(u_q, u_k, w_qkv, w_o, heads: int, window: int,
                     q_pos, k_pos) -> np.ndarray:
    """Attn(u) = concat_h(SWA(u W_q,h^T, u W_k,h^T, u W_v,h^T)) W_o^T.

    u_q: normalised rows at the query positions q_pos, [B, R, H];
    u_k: normalised rows at the key positions k_pos, [B, S, H].
    w_qkv [3H, H] holds all query heads, then all key heads, then all value
    heads (head h at rows h*d .. h*d+d-1 of each third); w_o [H, H] takes its
    input columns ordered by head.  Causal window `window`, scale 1/sqrt(d)
    (MegaScale notes, §2.2, SWA row)."""
    bsz, _, hidden = u_q.shape
    d = hidden // heads
    q = linear(u_q, w_qkv[0:hidden])
    k = linear(u_k, w_qkv[hidden:2 * hidden])
    v = linear(u_k, w_qkv[2 * hidden:3 * hidden])

    def split_heads(t):  # [B, n, H] -> [B, heads, n, d]
        return t.reshape(bsz, t.shape[1], heads, d).transpose(0, 2, 1, 3)

    ctx = swa(split_heads(q), split_heads(k), split_heads(v), window,
              1.0 / math.sqrt(d), q_pos, k_pos)                 # [B, heads, R, d]
    ctx = ctx.transpose(0, 2, 1, 3).reshape(bsz, len(q_pos), hidden)
    return linear(ctx, w_o)


def mlp_branch(u, w_up, w_down) -> np.ndarray:
    """MLP(u) = gelu_tanh(u W_up^T) W_down^T, no biases."""
    return linear(gelu_tanh(linear(u, w_up)), w_down)


def ptb_forward(x, ln_gamma, ln_beta, w_qkv, w_o, w_up, w_down,
                heads: int, window: int, rows=None, eps: float = LN_EPS
                ) -> np.ndarray:
    """Parallel transformer block y = x + MLP(LN(x)) + Attn(LN(x))
    (MegaScale notes, §2.2, PTB row): one LayerNorm, both branches fed from
    it, their outputs summed with the residual.

    x: [B, s, H]; weights in nn.Linear [out, in] form: w_qkv [3H, H],
    w_o [H, H], w_up [F, H], w_down [H, F] (layout as in attention_branch).

    rows: optional list of sequence positions; if given, y is returned only
    for those positions ([B, len(rows), H]), computing keys and values only
    at the positions inside their windows.  The arithmetic per output row is
    the same as for the full layer."""
    x = _f64(x)
    _, seq, hidden = x.shape
    if hidden % heads:
        raise ValueError("hidden must be a multiple of heads")
    q_pos = np.arange(seq) if rows is None else np.asarray(rows, dtype=np.int64)
    k_pos = np.arange(seq) if rows is None else needed_key_positions(q_pos, window)
    xn_q = layer_norm(x[:, q_pos], ln_gamma, ln_beta, eps)
    xn_k = xn_q if rows is None else layer_norm(x[:, k_pos], ln_gamma, ln_beta, eps)
    attn = attention_branch(xn_q, xn_k, w_qkv, w_o, heads, window, q_pos, k_pos)
    mlp = mlp_branch(xn_q, w_up, w_down)
    return x[:, q_pos] + attn + mlp


def serial_block(x, ln1_gamma, ln1_beta, ln2_gamma, ln2_beta, w_qkv, w_o,
                 w_up, w_down, heads: int, window: int, rows=None,
                 eps: float = LN_EPS) -> np.ndarray:
    """The serial block that PTB replaces: h = x + Attn(LN1(x)),
    y = h + MLP(LN2(h)).

    The notes print the serial form with the attention residual missing
    (MegaScale notes, §2.2, PTB row); this is the standard pre-LN reading.
    rows: optional sequence positions, as in ptb_forward (the MLP half is
    row-local, so only the attention half needs the window's keys)."""
    x = _f64(x)
    seq = x.shape[1]
    q_pos = np.arange(seq) if rows is None else np.asarray(rows, dtype=np.int64)
    k_pos = np.arange(seq) if rows is None else needed_key_positions(q_pos, window)
    u1_q = layer_norm(x[:, q_pos], ln1_gamma, ln1_beta, eps)
    u1_k = u1_q if rows is None else layer_norm(x[:, k_pos], ln1_gamma, ln1_beta, eps)
    h = x[:, q_pos] + attention_branch(u1_q, u1_k, w_qkv, w_o, heads, window, q_pos, k_pos)
    u2 = layer_norm(h, ln2_gamma, ln2_beta, eps)
    return h + mlp_branch(u2, w_up, w_down)


def layer_flops(batch: int, seq: int, hidden: int, ffn: int, window: int
                ) -> dict:
    """Algorithmic forward FLOPs of one PTB layer.

    GEMMs: 2*T*H*(3H + F) for [QKV | up] plus 2*T*(H + F)*H for [out | down].
    Attention: 4*B*H*sum_i min(i+1, w) (QK^T and PV over in-band keys only;
    the work the window removes is not counted)."""
    t = batch * seq
    band = int(attended_counts(seq, window).sum())
    gemm = 2 * t * hidden * (3 * hidden + ffn) + 2 * t * (hidden + ffn) * hidden
    attn = 4 * batch * hidden * band
    return {"gemm": gemm, "attn": attn, "total": gemm + attn, "band_keys": band}


def mfu(tokens_per_s: float, params: float, n_gpus: int, peak_flops: float,
        flops_per_token_per_param: float = 6.0) -> float:
    """Model FLOPs utilisation: observed model FLOP/s over the aggregate peak,
    with 6N FLOPs per trained token (2N forward + 4N backward, attention term
    ignored) -- MegaScale notes, §2.1 (paper §2), MFU definition."""
    return tokens_per_s * flops_per_token_per_param * params / (n_gpus * peak_flops)
