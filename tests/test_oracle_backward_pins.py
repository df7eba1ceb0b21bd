"""Pins for the fp64 backward oracle, on the CPU only.

The pages print no gradient values; the backward pass is the chain rule of
the PTB's forward definition (MegaScale study notes, §2.2, PTB and SWA rows;
§2.1 counts it as 4N of the 6N FLOPs per token).  It is pinned by:
  * central finite differences of L = sum(y * dy), with y from the forward
    oracle, for every gradient the backward oracle returns;
  * library routines: torch fp64 autograd through scaled_dot_product_attention
    with a band mask, F.layer_norm and F.gelu(approximate="tanh");
  * closed forms: W_o = W_down = 0 gives dx = dy and zero input-side weight
    gradients; w = 1 gives dq = dk = 0 and dv = do;
and planted mistakes that these checks must catch.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import backward as pb

NAMES = ["x", "ln_gamma", "ln_beta", "w_qkv", "w_o", "w_up", "w_down"]
GRADS = ["dx", "dln_gamma", "dln_beta", "dw_qkv", "dw_o", "dw_up", "dw_down"]


def _layer(seed, batch=1, seq=7, hidden=8, heads=2, ffn=12, std=0.4):
    r = np.random.default_rng(seed)
    p = dict(x=r.standard_normal((batch, seq, hidden)),
             ln_gamma=1.0 + 0.2 * r.standard_normal(hidden),
             ln_beta=0.2 * r.standard_normal(hidden),
             w_qkv=std * r.standard_normal((3 * hidden, hidden)),
             w_o=std * r.standard_normal((hidden, hidden)),
             w_up=std * r.standard_normal((ffn, hidden)),
             w_down=std * r.standard_normal((hidden, ffn)))
    dy = r.standard_normal((batch, seq, hidden))
    return p, dy


def _loss(p, dy, heads, window):
    y = oracle.ptb_forward(*(p[n] for n in NAMES), heads, window)
    return float((y * dy).sum())


def check_finite_differences(window=3, seed=0, h=1e-5):
    heads = 2
    p, dy = _layer(seed)
    g = oracle.ptb_backward(*(p[n] for n in NAMES), heads, window, dy)
    for name, gname in zip(NAMES, GRADS):
        fd = np.zeros_like(p[name])
        flat = p[name].reshape(-1)
        out = fd.reshape(-1)
        for i in range(flat.size):
            keep = flat[i]
            flat[i] = keep + h
            lp = _loss(p, dy, heads, window)
            flat[i] = keep - h
            lm = _loss(p, dy, heads, window)
            flat[i] = keep
            out[i] = (lp - lm) / (2 * h)
        err = np.abs(fd - g[gname]).max()
        assert err <= 1e-7 * max(1.0, np.abs(fd).max()), (gname, err)


def check_finite_differences_full_window():
    check_finite_differences(window=50, seed=1)


def check_finite_differences_unit_window():
    check_finite_differences(window=1, seed=2)


def check_swa_backward_vs_autograd():
    r = np.random.default_rng(3)
    b, hd, s, d, w = 2, 3, 19, 8, 5
    q, k, v, do = (r.standard_normal((b, hd, s, d)) for _ in range(4))
    scale = 1.0 / math.sqrt(d)
    t = [torch.tensor(a, requires_grad=True) for a in (q, k, v)]
    ones = torch.ones(s, s, dtype=torch.bool)
    keep = torch.tril(ones) & ~torch.tril(ones, diagonal=-w)
    o = F.scaled_dot_product_attention(*t, attn_mask=keep, scale=scale)
    o.backward(torch.tensor(do))
    got = oracle.swa_backward(q, k, v, do, w, scale)
    for a, b_ in zip(got, t):
        assert np.abs(a - b_.grad.numpy()).max() < 1e-12


def check_layer_norm_backward_vs_autograd():
    r = np.random.default_rng(4)
    x = r.standard_normal((3, 5, 16)) * 2 + 1
    gam, bet = r.standard_normal(16), r.standard_normal(16)
    du = r.standard_normal((3, 5, 16))
    t = [torch.tensor(a, requires_grad=True) for a in (x, gam, bet)]
    F.layer_norm(t[0], (16,), t[1], t[2], eps=1e-5).backward(torch.tensor(du))
    got = oracle.layer_norm_backward(x, gam, du)
    for a, b_ in zip(got, t):
        assert np.abs(a - b_.grad.numpy()).max() < 1e-12


def check_gelu_grad_vs_autograd():
    z = torch.linspace(-8, 8, 2001, dtype=torch.float64, requires_grad=True)
    F.gelu(z, approximate="tanh").sum().backward()
    assert np.abs(oracle.gelu_tanh_grad(z.detach().numpy()) - z.grad.numpy()).max() < 1e-14


def check_zero_output_weights():
    """W_o = W_down = 0: nothing flows back into the branches, so dx = dy and
    the input-side gradients vanish; dW_o = dy^T ctx, dW_down = dy^T gelu(z)."""
    heads, window = 2, 4
    p, dy = _layer(5)
    p["w_o"][:] = 0.0
    p["w_down"][:] = 0.0
    g = oracle.ptb_backward(*(p[n] for n in NAMES), heads, window, dy)
    assert np.array_equal(g["dx"], dy)
    for n in ("dln_gamma", "dln_beta", "dw_qkv", "dw_up"):
        assert not g[n].any(), n
    u = oracle.layer_norm(p["x"], p["ln_gamma"], p["ln_beta"])
    pos = np.arange(u.shape[1])
    ctx = oracle.attention_branch(u, u, p["w_qkv"], np.eye(8), heads, window, pos, pos)
    assert np.allclose(g["dw_o"], dy[0].T @ ctx[0], rtol=1e-13, atol=1e-13)
    assert np.allclose(g["dw_down"], dy[0].T @ oracle.gelu_tanh(u[0] @ p["w_up"].T),
                       rtol=1e-13, atol=1e-13)


def check_unit_window_attention():
    """w = 1: each row attends only to itself with weight 1, so o = v and the
    scores get no gradient: dq = dk = 0 exactly, dv = do."""
    r = np.random.default_rng(6)
    q, k, v, do = (r.standard_normal((1, 2, 9, 4)) for _ in range(4))
    dq, dk, dv = oracle.swa_backward(q, k, v, do, 1)
    assert not dq.any() and not dk.any() and np.array_equal(dv, do)


def check_backward_flops_closed_form():
    fl = oracle.backward_flops(2, 100, 64, 256, 30)
    band = sum(min(i + 1, 30) for i in range(100))
    assert fl["attn"] == 8 * 2 * 64 * band
    assert fl["gemm"] == 2 * oracle.layer_flops(2, 100, 64, 256, 30)["gemm"]


CHECKS = [check_finite_differences, check_finite_differences_full_window,
          check_finite_differences_unit_window, check_swa_backward_vs_autograd,
          check_layer_norm_backward_vs_autograd, check_gelu_grad_vs_autograd,
          check_zero_output_weights, check_unit_window_attention,
          check_backward_flops_closed_form]


@pytest.mark.parametrize("check", CHECKS, ids=[c.__name__ for c in CHECKS])
def test_backward_oracle_pin(check):
    check()


# ------------------------------------------------------ planted mistakes --

_ORIG_SWA_BWD = pb.swa_backward
_ORIG_LN_BWD = pb.layer_norm_backward


def _bad_softmax_jacobian(q, k, v, do, window, scale=None):
    """Drops the rowsum(dP * P) term of the softmax Jacobian."""
    q, k, v, do = (np.asarray(a, np.float64) for a in (q, k, v, do))
    scale = 1.0 / math.sqrt(q.shape[-1]) if scale is None else scale
    p = oracle.swa_weights(q, k, window, scale)
    ds = p * (do @ np.swapaxes(v, -1, -2))
    return (ds @ k) * scale, (np.swapaxes(ds, -1, -2) @ q) * scale, np.swapaxes(p, -1, -2) @ do


def _bad_dk_unscaled(q, k, v, do, window, scale=None):
    dq, dk, dv = _ORIG_SWA_BWD(q, k, v, do, window, scale)
    return dq, dk / (1.0 / math.sqrt(np.asarray(q).shape[-1])), dv


def _bad_gelu_grad(z):
    z = np.asarray(z, np.float64)
    t = np.tanh(pb.GELU_C * (z + pb.GELU_CUBIC * z ** 3))
    return 0.5 * (1.0 + t) + 0.5 * z * (1.0 + t * t) * pb.GELU_C * (1.0 + 3 * pb.GELU_CUBIC * z * z)


def _bad_ln_no_projection(x, gamma, du, eps=1e-5):
    dx, dg, db = _ORIG_LN_BWD(x, gamma, du, eps)
    x = np.asarray(x, np.float64)
    r = 1.0 / np.sqrt(x.var(axis=-1, keepdims=True) + eps)
    return r * np.asarray(du) * gamma, dg, db


MUTATIONS = [
    ("swa_backward", _bad_softmax_jacobian, check_finite_differences),
    ("swa_backward", _bad_softmax_jacobian, check_swa_backward_vs_autograd),
    ("swa_backward", _bad_dk_unscaled, check_finite_differences),
    ("gelu_tanh_grad", _bad_gelu_grad, check_finite_differences),
    ("gelu_tanh_grad", _bad_gelu_grad, check_gelu_grad_vs_autograd),
    ("layer_norm_backward", _bad_ln_no_projection, check_finite_differences),
    ("layer_norm_backward", _bad_ln_no_projection, check_layer_norm_backward_vs_autograd),
]


@pytest.mark.parametrize("name,bad,check", MUTATIONS,
                         ids=[f"{m[0]}-{m[1].__name__}-{m[2].__name__}" for m in MUTATIONS])
def test_planted_backward_mistake_is_caught(monkeypatch, name, bad, check):
    monkeypatch.setattr(pb, name, bad)
    monkeypatch.setattr(oracle, name, bad)
    with pytest.raises(AssertionError):
        check()


def test_sampled_backward_helper_matches_full_oracle():
    """The full-size tests' sampled gradient entries (tests/backward_sampled)
    are the full backward oracle's entries."""
    from tests.backward_sampled import gathered, sampled_backward
    heads, window = 4, 5
    r = np.random.default_rng(9)
    p = dict(x=r.standard_normal((2, 23, 16)), ln_gamma=1 + 0.1 * r.standard_normal(16),
             ln_beta=0.1 * r.standard_normal(16), w_qkv=0.3 * r.standard_normal((48, 16)),
             w_o=0.3 * r.standard_normal((16, 16)), w_up=0.3 * r.standard_normal((40, 16)),
             w_down=0.3 * r.standard_normal((16, 40)))
    dy = r.standard_normal((2, 23, 16))
    args = [p[n] for n in NAMES] + [heads, window, dy]
    full = oracle.ptb_backward(*args)
    rows, head_sel, f_sel, r_sel = [0, 4, 5, 22], [1, 3], [0, 7, 39], [2, 15]
    want = gathered(full, 16, heads, rows, head_sel, f_sel, r_sel)
    got = sampled_backward(*args, rows, head_sel, f_sel, r_sel)
    for k in want:
        assert np.allclose(got[k], want[k], rtol=1e-12, atol=1e-12), k
