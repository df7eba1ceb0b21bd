"""Pins for the fp64 oracle, on the CPU only.

The pages print no numeric PTB or SWA output, so the oracle is pinned by
what the definitions and the mathematics fix (MegaScale study notes, §2.2,
PTB and SWA rows):
  * closed forms: the attended-key count min(i+1, w); w = 1 gives o = v;
    the sum of min(i+1, w) over a sequence; gelu(z) - gelu(-z) = z;
  * library special cases: full causal attention (w >= s) and the banded
    case against torch's fp64 scaled_dot_product_attention with its own
    mask; LayerNorm and tanh-GELU against torch's fp64 functions;
  * invariants: convex attention rows, LN shift invariance, head permutation;
  * the PTB's special cases against the serial block;
  * brute force on tiny inputs against a pure-Python loop implementation.
Each check is a function that raises AssertionError, so the mutation tests at
the bottom can plant a mistake in the oracle and show that a pin catches it.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import ptb_oracle
from tests import brute_force

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _rand_ptb(seed, batch, seq, hidden, heads, ffn, std=0.3):
    r = _rng(seed)
    return dict(
        x=r.standard_normal((batch, seq, hidden)),
        ln_gamma=1.0 + 0.1 * r.standard_normal(hidden),
        ln_beta=0.1 * r.standard_normal(hidden),
        w_qkv=std * r.standard_normal((3 * hidden, hidden)),
        w_o=std * r.standard_normal((hidden, hidden)),
        w_up=std * r.standard_normal((ffn, hidden)),
        w_down=std * r.standard_normal((hidden, ffn)),
    )


def _sdpa_band(q, k, v, window, scale):
    """torch fp64 SDPA with a band mask built from triangular matrices."""
    s = q.shape[-2]
    ones = torch.ones(s, s, dtype=torch.bool)
    keep = torch.tril(ones) & ~torch.tril(ones, diagonal=-window)
    t = [torch.from_numpy(np.ascontiguousarray(a)) for a in (q, k, v)]
    return F.scaled_dot_product_attention(*t, attn_mask=keep, scale=scale).numpy()


# ---------------------------------------------------------------- checks --

def check_counts_closed_form():
    for s in (1, 2, 7, 64, 129, 300):
        for w in (1, 2, 3, 31, 64, 128, 299, 300, 301, 1000):
            got = oracle.attended_counts(s, w)
            want = np.minimum(np.arange(s) + 1, w)
            assert np.array_equal(got, want), (s, w)
            # sum_i min(i+1, w) = w(w+1)/2 + (s-w)w for w <= s, else s(s+1)/2
            total = w * (w + 1) // 2 + (s - w) * w if w <= s else s * (s + 1) // 2
            assert int(got.sum()) == total


def check_window1_is_v():
    r = _rng(1)
    q, k, v = (r.standard_normal((2, 3, 37, 16)) for _ in range(3))
    o = oracle.swa(q, k, v, 1)
    assert np.array_equal(o, v)


def check_full_causal_vs_sdpa():
    r = _rng(2)
    for s, d in ((1, 8), (17, 16), (96, 32)):
        q, k, v = (r.standard_normal((2, 3, s, d)) for _ in range(3))
        tq, tk, tv = (torch.from_numpy(a) for a in (q, k, v))
        ref = F.scaled_dot_product_attention(tq, tk, tv, is_causal=True).numpy()
        for w in (s, s + 1, 4 * s):
            got = oracle.swa(q, k, v, w)
            assert np.allclose(got, ref, rtol=1e-12, atol=1e-12), (s, d, w)


def check_band_vs_sdpa():
    r = _rng(3)
    for s, d, w in ((40, 16, 1), (40, 16, 2), (40, 16, 7), (130, 32, 33), (130, 8, 129)):
        q, k, v = (r.standard_normal((2, 2, s, d)) for _ in range(3))
        scale = 1.0 / math.sqrt(d)
        got = oracle.swa(q, k, v, w, scale)
        ref = _sdpa_band(q, k, v, w, scale)
        assert np.allclose(got, ref, rtol=1e-12, atol=1e-12), (s, d, w)


def check_convex_rows():
    r = _rng(4)
    s, w = 50, 9
    q, k = r.standard_normal((3, s, 8)), r.standard_normal((3, s, 8))
    p = oracle.swa_weights(q, k, w)
    assert np.all(p >= 0)
    assert np.allclose(p.sum(-1), 1.0, rtol=0, atol=1e-12)
    nnz = (p > 0).sum(-1)
    assert np.array_equal(nnz, np.broadcast_to(np.minimum(np.arange(s) + 1, w), nnz.shape))


def check_layer_norm():
    r = _rng(5)
    x = 3.0 * r.standard_normal((4, 6, 64)) + 2.0
    g, b = 1.0 + r.standard_normal(64), r.standard_normal(64)
    got = oracle.layer_norm(x, g, b)
    ref = F.layer_norm(torch.from_numpy(x), (64,), torch.from_numpy(g),
                       torch.from_numpy(b), eps=1e-5).numpy()
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)
    # shift invariance and unit statistics with gamma = 1, beta = 0
    one, zero = np.ones(64), np.zeros(64)
    assert np.allclose(oracle.layer_norm(x + 7.5, one, zero),
                       oracle.layer_norm(x, one, zero), atol=1e-10)
    y = oracle.layer_norm(x, one, zero)
    assert np.allclose(y.mean(-1), 0.0, atol=1e-12)
    var = x.var(-1)
    assert np.allclose(y.var(-1), var / (var + 1e-5), atol=1e-12)


def check_gelu():
    z = np.linspace(-8, 8, 1601)
    g = oracle.gelu_tanh(z)
    assert oracle.gelu_tanh(np.array([0.0]))[0] == 0.0
    assert np.allclose(g - oracle.gelu_tanh(-z), z, rtol=0, atol=1e-13)
    ref = F.gelu(torch.from_numpy(z), approximate="tanh").numpy()
    assert np.allclose(g, ref, rtol=1e-13, atol=1e-14)


def check_brute_force_ptb():
    for seed, (b, s, h, nh, f, w) in enumerate(((2, 9, 8, 2, 12, 3),
                                               (1, 6, 12, 3, 8, 1),
                                               (1, 7, 8, 1, 16, 20))):
        p = _rand_ptb(seed, b, s, h, nh, f)
        got = oracle.ptb_forward(p["x"], p["ln_gamma"], p["ln_beta"], p["w_qkv"],
                                 p["w_o"], p["w_up"], p["w_down"], nh, w)
        ref = brute_force.ptb(p["x"].tolist(), p["ln_gamma"].tolist(),
                              p["ln_beta"].tolist(), p["w_qkv"].tolist(),
                              p["w_o"].tolist(), p["w_up"].tolist(),
                              p["w_down"].tolist(), nh, w)
        assert np.allclose(got, np.array(ref), rtol=1e-11, atol=1e-11), (b, s, h, nh, f, w)


def check_brute_force_swa():
    r = _rng(6)
    q, k, v = (r.standard_normal((1, 2, 11, 4)) for _ in range(3))
    for w in (1, 3, 11, 50):
        ref = np.array(brute_force.swa(q.tolist(), k.tolist(), v.tolist(), w))
        assert np.allclose(oracle.swa(q, k, v, w), ref, rtol=1e-12, atol=1e-12), w


def check_brute_force_serial():
    b, s, h, nh, f, w = 2, 7, 8, 2, 12, 3
    p = _rand_ptb(11, b, s, h, nh, f)
    r = _rng(12)
    g2, b2 = 1.0 + 0.1 * r.standard_normal(h), 0.1 * r.standard_normal(h)
    got = oracle.serial_block(p["x"], p["ln_gamma"], p["ln_beta"], g2, b2, p["w_qkv"], p["w_o"],
                              p["w_up"], p["w_down"], nh, w)
    ref = brute_force.serial(p["x"].tolist(), p["ln_gamma"].tolist(), p["ln_beta"].tolist(),
                             g2.tolist(), b2.tolist(), p["w_qkv"].tolist(), p["w_o"].tolist(),
                             p["w_up"].tolist(), p["w_down"].tolist(), nh, w)
    assert np.allclose(got, np.array(ref), rtol=1e-11, atol=1e-11)


def check_ptb_special_cases():
    b, s, h, nh, f, w = 2, 12, 16, 4, 24, 5
    p = _rand_ptb(7, b, s, h, nh, f)
    x, g, be = p["x"], p["ln_gamma"], p["ln_beta"]
    zo, zd = np.zeros_like(p["w_o"]), np.zeros_like(p["w_down"])
    u = oracle.layer_norm(x, g, be)
    # W_o = 0: y = x + MLP(LN(x)), which is also the serial block with W_o = 0.
    y = oracle.ptb_forward(x, g, be, p["w_qkv"], zo, p["w_up"], p["w_down"], nh, w)
    mlp_only = x + oracle.gelu_tanh(u @ p["w_up"].T) @ p["w_down"].T
    assert np.allclose(y, mlp_only, atol=1e-12)
    ser = oracle.serial_block(x, g, be, g, be, p["w_qkv"], zo, p["w_up"], p["w_down"], nh, w)
    assert np.allclose(y, ser, atol=1e-12)
    # W_down = 0: y = x + Attn(LN(x)), the serial block's first residual.
    y = oracle.ptb_forward(x, g, be, p["w_qkv"], p["w_o"], p["w_up"], zd, nh, w)
    ser = oracle.serial_block(x, g, be, g, be, p["w_qkv"], p["w_o"], p["w_up"], zd, nh, w)
    assert np.allclose(y, ser, atol=1e-12)
    q = u @ p["w_qkv"][:h].T
    k = u @ p["w_qkv"][h:2 * h].T
    v = u @ p["w_qkv"][2 * h:].T
    heads = lambda t: t.reshape(b, s, nh, h // nh).transpose(0, 2, 1, 3)  # noqa: E731
    ctx = _sdpa_band(heads(q), heads(k), heads(v), w, 1.0 / math.sqrt(h // nh))
    attn = ctx.transpose(0, 2, 1, 3).reshape(b, s, h) @ p["w_o"].T
    assert np.allclose(y, x + attn, atol=1e-12)
    # All weights zero: y = x.
    y = oracle.ptb_forward(x, g, be, 0 * p["w_qkv"], zo, 0 * p["w_up"], zd, nh, w)
    assert np.array_equal(y, x)
    # In general PTB and the serial block differ (same shapes, other function).
    y = oracle.ptb_forward(x, g, be, p["w_qkv"], p["w_o"], p["w_up"], p["w_down"], nh, w)
    ser = oracle.serial_block(x, g, be, g, be, p["w_qkv"], p["w_o"], p["w_up"], p["w_down"], nh, w)
    assert y.shape == ser.shape and not np.allclose(y, ser, atol=1e-6)


def check_head_permutation():
    b, s, h, nh, f, w = 1, 10, 12, 3, 16, 4
    d = h // nh
    p = _rand_ptb(8, b, s, h, nh, f)
    perm = [2, 0, 1]
    cols = np.concatenate([np.arange(ph * d, (ph + 1) * d) for ph in perm])
    wqkv = np.concatenate([p["w_qkv"][i * h:(i + 1) * h][cols] for i in range(3)])
    wo = p["w_o"][:, cols]
    y0 = oracle.ptb_forward(p["x"], p["ln_gamma"], p["ln_beta"], p["w_qkv"], p["w_o"],
                            p["w_up"], p["w_down"], nh, w)
    y1 = oracle.ptb_forward(p["x"], p["ln_gamma"], p["ln_beta"], wqkv, wo,
                            p["w_up"], p["w_down"], nh, w)
    assert np.allclose(y0, y1, atol=1e-12)


def check_row_sampling():
    b, s, h, nh, f, w = 2, 40, 16, 2, 32, 6
    p = _rand_ptb(9, b, s, h, nh, f)
    args = (p["x"], p["ln_gamma"], p["ln_beta"], p["w_qkv"], p["w_o"], p["w_up"], p["w_down"], nh, w)
    full = oracle.ptb_forward(*args)
    rows = [0, 1, 5, 6, 22, 39]
    part = oracle.ptb_forward(*args, rows=rows)
    assert np.allclose(part, full[:, rows], rtol=1e-13, atol=1e-13)
    assert list(oracle.needed_key_positions([0, 6, 39], w)) == [0, 1, 2, 3, 4, 5, 6, 34, 35, 36, 37, 38, 39]
    g2, b2 = p["ln_gamma"][::-1].copy(), p["ln_beta"][::-1].copy()
    sargs = (p["x"], p["ln_gamma"], p["ln_beta"], g2, b2, p["w_qkv"], p["w_o"], p["w_up"],
             p["w_down"], nh, w)
    sfull = oracle.serial_block(*sargs)
    assert np.allclose(oracle.serial_block(*sargs, rows=rows), sfull[:, rows], rtol=1e-13,
                       atol=1e-13)


def check_linear_slabs():
    """oracle.linear upcasts the weight a slab of 8192 output rows at a time.
    A selector weight pins every output column by a closed form: row r of w
    is (r + 1) times the unit vector e_(r mod K), so y[..., r] = (r + 1) *
    a[..., r mod K] exactly (every other product is an exact zero).  With
    2 * 8192 + 37 rows the check spans two full slabs and a ragged third, and
    a bf16 weight takes the torch upcast path."""
    k = 24
    n = 2 * 8192 + 37
    rng = np.random.default_rng(5)
    a = rng.standard_normal((2, 3, k))
    r = np.arange(n)
    w = np.zeros((n, k))
    w[r, r % k] = r + 1.0
    want = a[..., r % k] * (r + 1.0)
    assert np.array_equal(oracle.linear(a, w), want)
    wb = torch.from_numpy(w).to(torch.bfloat16)  # r + 1 <= 256 is exact in bf16
    small = w[:256]
    assert np.array_equal(oracle.linear(a, wb[:256]), a[..., np.arange(256) % k] * (np.arange(256) + 1.0))
    assert np.array_equal(oracle.linear(a, small), want[..., :256])


# ----------------------------------------------------------------- tests --

CHECKS = [check_linear_slabs, check_counts_closed_form, check_window1_is_v, check_full_causal_vs_sdpa,
          check_band_vs_sdpa, check_convex_rows, check_layer_norm, check_gelu,
          check_brute_force_ptb, check_brute_force_swa, check_brute_force_serial,
          check_ptb_special_cases,
          check_head_permutation, check_row_sampling]


@pytest.mark.parametrize("check", CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check):
    check()


def test_mfu_worked_example():
    """The notes' MFU hand check: 1984.0k tokens/s on 12,288 GPUs for a 175B
    model at 6N FLOPs per token and an assumed 312 TFLOP/s per GPU gives about
    54.3%; 1.984e6 tokens/s for 1.75 days is about 300B tokens."""
    with open(os.path.join(GOLDEN, "mfu_worked_example.json")) as fh:
        g = json.load(fh)
    m = oracle.mfu(g["tokens_per_s"], g["params"], g["n_gpus"], g["assumed_peak_flops_per_gpu"])
    assert abs(m - g["mfu_hand_check"]) < 5e-4
    assert abs(g["tokens_per_s"] * 6 * g["params"] - g["model_flops_per_s"]) / g["model_flops_per_s"] < 5e-3
    assert abs(g["n_gpus"] * g["assumed_peak_flops_per_gpu"] - g["cluster_peak_flops"]) / g["cluster_peak_flops"] < 5e-3
    assert abs(g["tokens_per_s"] * g["train_seconds"] - g["train_tokens"]) / g["train_tokens"] < 1e-2
    # The hand check lands below the reported 55.2%, as the notes remark.
    assert m < g["mfu_reported"]


def test_layer_flops_closed_form():
    # tiny: T = 128, H = 64, F = 256, w = 32
    f = oracle.layer_flops(1, 128, 64, 256, 32)
    assert f["band_keys"] == 32 * 33 // 2 + (128 - 32) * 32 == 3600
    assert f["gemm"] == 2 * 128 * 64 * (3 * 64 + 256) + 2 * 128 * (64 + 256) * 64
    assert f["attn"] == 4 * 64 * 3600
    # 175B shape: H = 12288, F = 4H, s = 2048, w = 1024
    f = oracle.layer_flops(1, 2048, 12288, 49152, 1024)
    assert f["band_keys"] == 1024 * 1025 // 2 + 1024 * 1024 == 1573376
    assert f["gemm"] == 2 * 2048 * 12288 * (7 * 12288) + 2 * 2048 * (5 * 12288) * 12288
    # attention FLOPs never exceed the dense causal count
    assert f["attn"] <= 4 * 12288 * 2048 * 2049 // 2


# ------------------------------------------------------ planted mistakes --

def _bad_mask_off_by_one(q_pos, k_pos, window):
    i = np.asarray(q_pos)[:, None]
    j = np.asarray(k_pos)[None, :]
    return (j <= i) & (j >= i - window)


def _bad_mask_not_causal(q_pos, k_pos, window):
    i = np.asarray(q_pos)[:, None]
    j = np.asarray(k_pos)[None, :]
    return np.abs(j - i) < window


def _bad_ln_unbiased(x, gamma, beta, eps=1e-5):
    x = np.asarray(x, dtype=np.float64)
    mu = x.mean(-1, keepdims=True)
    var = x.var(-1, ddof=1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps) * gamma + beta


def _bad_gelu_sign(z):
    z = np.asarray(z, dtype=np.float64)
    return 0.5 * z * (1.0 + np.tanh(math.sqrt(2 / math.pi) * (z - 0.044715 * z ** 3)))


def _bad_mlp_dropped(u, w_up, w_down):
    return np.zeros(u.shape[:-1] + (np.asarray(w_down).shape[0],))


def _bad_attn_transposed_wo(u_q, u_k, w_qkv, w_o, heads, window, q_pos, k_pos):
    return _ORIG_ATTN(u_q, u_k, w_qkv, np.asarray(w_o).T, heads, window, q_pos, k_pos)


_ORIG_ATTN = ptb_oracle.attention_branch


def _bad_linear_drops_ragged_slab(a, w):
    a = np.asarray(a, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    out = np.zeros(a.shape[:-1] + (w.shape[0],))
    step = 8192
    for r0 in range(0, w.shape[0] // step * step, step):
        out[..., r0:r0 + step] = a @ w[r0:r0 + step].T
    return out

MUTATIONS = [
    ("band_mask", _bad_mask_off_by_one, check_counts_closed_form),
    ("band_mask", _bad_mask_off_by_one, check_band_vs_sdpa),
    ("band_mask", _bad_mask_not_causal, check_full_causal_vs_sdpa),
    ("layer_norm", _bad_ln_unbiased, check_layer_norm),
    ("gelu_tanh", _bad_gelu_sign, check_gelu),
    ("mlp_branch", _bad_mlp_dropped, check_brute_force_ptb),
    ("mlp_branch", _bad_mlp_dropped, check_brute_force_serial),
    ("attention_branch", _bad_attn_transposed_wo, check_brute_force_ptb),
    ("linear", _bad_linear_drops_ragged_slab, check_linear_slabs),
]


@pytest.mark.parametrize("name,bad,check", MUTATIONS,
                         ids=[f"{m[0]}-{m[1].__name__}-{m[2].__name__}" for m in MUTATIONS])
def test_planted_mistake_is_caught(monkeypatch, name, bad, check):
    monkeypatch.setattr(ptb_oracle, name, bad)
    monkeypatch.setattr(oracle, name, bad, raising=False)
    with pytest.raises(AssertionError):
        check()
