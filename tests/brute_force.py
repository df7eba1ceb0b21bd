"""A second, naive PTB + SWA implementation in pure-Python loops.

Written independently of the oracle (no numpy, no masks): per token it
normalises the row, walks the window of keys explicitly for every head and
sums the three terms of the PTB output (MegaScale study notes, §2.2, PTB and
SWA rows).  Only for tiny shapes; it pins the oracle by brute force.
"""
import math


def _dot(a, b):
    return math.fsum(x * y for x, y in zip(a, b))


def _matvec(w, vec):
    """w is [out][in]; returns w @ vec."""
    return [_dot(row, vec) for row in w]


def _layer_norm_row(row, gamma, beta, eps):
    n = len(row)
    mu = math.fsum(row) / n
    var = math.fsum((v - mu) ** 2 for v in row) / n
    inv = 1.0 / math.sqrt(var + eps)
    return [(row[c] - mu) * inv * gamma[c] + beta[c] for c in range(n)]


def _gelu(u):
    return 0.5 * u * (1.0 + math.tanh(math.sqrt(2.0 / math.pi) * (u + 0.044715 * u * u * u)))


def window_keys(i, window):
    """Key positions row i attends to: itself and up to window-1 before it."""
    return list(range(max(0, i - window + 1), i + 1))


def attend_row(q, keys, vals, scale):
    """softmax(q.k * scale) over the listed keys, applied to vals."""
    scores = [_dot(q, k) * scale for k in keys]
    top = max(scores)
    e = [math.exp(s - top) for s in scores]
    z = math.fsum(e)
    d = len(vals[0])
    return [math.fsum(e[n] * vals[n][c] for n in range(len(vals))) / z for c in range(d)]


def ptb(x, gamma, beta, w_qkv, w_o, w_up, w_down, heads, window, eps=1e-5):
    """x: nested lists [B][s][H]; weights nested lists in [out][in] form."""
    out = []
    for seq in x:
        s = len(seq)
        hidden = len(seq[0])
        d = hidden // heads
        xn = [_layer_norm_row(seq[t], gamma, beta, eps) for t in range(s)]
        qkv = [_matvec(w_qkv, xn[t]) for t in range(s)]
        rows = []
        for t in range(s):
            ctx = []
            for h in range(heads):
                q = qkv[t][h * d:(h + 1) * d]
                ks = [qkv[j][hidden + h * d: hidden + (h + 1) * d] for j in window_keys(t, window)]
                vs = [qkv[j][2 * hidden + h * d: 2 * hidden + (h + 1) * d] for j in window_keys(t, window)]
                ctx.extend(attend_row(q, ks, vs, 1.0 / math.sqrt(d)))
            attn = _matvec(w_o, ctx)
            mlp = _matvec(w_down, [_gelu(u) for u in _matvec(w_up, xn[t])])
            rows.append([seq[t][c] + attn[c] + mlp[c] for c in range(hidden)])
        out.append(rows)
    return out


def swa(q, k, v, window, scale=None):
    """q, k, v nested lists [B][heads][s][d]."""
    res = []
    for qb, kb, vb in zip(q, k, v):
        hs = []
        for qh, kh, vh in zip(qb, kb, vb):
            d = len(qh[0])
            sc = scale if scale is not None else 1.0 / math.sqrt(d)
            hs.append([attend_row(qh[i], [kh[j] for j in window_keys(i, window)],
                                  [vh[j] for j in window_keys(i, window)], sc)
                       for i in range(len(qh))])
        res.append(hs)
    return res


def serial(x, g1, b1, g2, b2, w_qkv, w_o, w_up, w_down, heads, window, eps=1e-5):
    """The serial pre-LN block h = x + Attn(LN1(x)), y = h + MLP(LN2(h)), by
    looping: the attention half is the PTB with a zero MLP, the MLP half is
    written out row by row."""
    zeros_down = [[0.0] * len(w_down[0]) for _ in w_down]
    h = ptb(x, g1, b1, w_qkv, w_o, w_up, zeros_down, heads, window, eps)
    out = []
    for seq in h:
        rows = []
        for row in seq:
            u = _layer_norm_row(row, g2, b2, eps)
            mlp = _matvec(w_down, [_gelu(a) for a in _matvec(w_up, u)])
            rows.append([row[c] + mlp[c] for c in range(len(row))])
        out.append(rows)
    return out
