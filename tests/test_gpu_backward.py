"""Parity of the backward pass (through the C ABI) with the fp64 backward
oracle.

The pages' workload is training (MegaScale study notes, §2.1: 6N FLOPs per
token, 4N of them backward); the backward pass is the chain rule of the PTB
definition (§2.2, PTB and SWA rows).  Every case feeds identical seeded bf16
inputs and upstream gradient to both sides and compares each gradient
tensor element by element:
  * relative L2 error <= 1e-2;
  * max-abs error <= 3e-2 * max|oracle| -- the forward pass's absolute
    3e-2 bar, taken relative to the gradient's own scale, since gradients
    have no fixed magnitude (dy is N(0, 1) here).
The attention's per-row log-sum-exp, which the backward pass reads, is
checked against the oracle's softmax denominators directly.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from block_sliding_window_gb300 import workloads
from tests.parity import to_np

pytestmark = pytest.mark.gpu

REL_L2 = 1e-2
MAX_ABS_REL = 3e-2


@pytest.fixture(autouse=True)
def _status_clean(ptb_lib):
    ptb_lib.last_device_error()
    yield
    assert ptb_lib.last_device_error() == 0, "a kernel recorded a device-side error"


def grad_errors(got, want):
    g, w = to_np(got), to_np(want)
    assert g.shape == w.shape, (g.shape, w.shape)
    assert np.all(np.isfinite(g)), "non-finite gradient"
    scale = max(float(np.abs(w).max()), 1e-30)
    rel = float(np.linalg.norm(g - w) / max(np.linalg.norm(w), 1e-30))
    return rel, float(np.abs(g - w).max()) / scale


# Closed-form zeros (dq, dk at w = 1) come out as fp32 rounding residue: the
# kernel forms dP_ii = dO_i . v_i with the tensor cores and delta_i = the same
# dot product in another summation order, so dS = P (dP - delta) is a few
# fp32 ulps of |dO . v| rather than 0.
ZERO_TOL = 1e-4


def assert_grad_close(got, want, what):
    if not to_np(want).any():
        g = to_np(got)
        mx = float(np.abs(g).max()) if g.size else 0.0
        print(f"{what}: closed-form zero, max |got| {mx:.3e}")
        assert mx <= ZERO_TOL, f"{what}: max |got| {mx:.3e} where the gradient is 0"
        return
    rel, mx = grad_errors(got, want)
    print(f"{what}: rel-L2 {rel:.3e}, max-abs / max|want| {mx:.3e}")
    assert rel <= REL_L2 and mx <= MAX_ABS_REL, (
        f"{what}: rel-L2 {rel:.3e} (<= {REL_L2}), max-abs/max {mx:.3e} (<= {MAX_ABS_REL})")


# -------------------------------------------------------- SWA operator --

SWA_CASES = [  # batch, heads, seq, d, window
    (1, 2, 200, 64, 33),
    (2, 3, 257, 128, 100),
    (1, 4, 130, 96, 1),
    (1, 2, 300, 32, 1000),
    (2, 2, 64, 16, 7),
    (1, 1, 1, 64, 5),
    (1, 8, 1024, 128, 512),
]


@pytest.mark.parametrize("b,h,s,d,w", SWA_CASES, ids=[f"b{c[0]}h{c[1]}s{c[2]}d{c[3]}w{c[4]}"
                                                      for c in SWA_CASES])
def test_swa_backward_operator(ptb_lib, b, h, s, d, w):
    q, k, v = workloads.swa_inputs(b, h, s, d, seed=s + d + w)
    dout = workloads.normal_bf16((b, h, s, d), seed=s + w)
    qc, kc, vc, dc = (t.cuda() for t in (q, k, v, dout))
    o, lse = ptb_lib.swa_attention_lse(qc, kc, vc, w)
    dq, dk, dv = ptb_lib.swa_attention_backward(qc, kc, vc, o, dc, lse, w)
    torch.cuda.synchronize()
    # lse: log2 of the banded softmax denominator of the scaled scores
    scale = 1.0 / math.sqrt(d)
    qf, kf = to_np(q), to_np(k)
    sc = (qf @ np.swapaxes(kf, -1, -2)) * scale
    mask = oracle.band_mask(np.arange(s), np.arange(s), w)
    sc = np.where(mask, sc, -np.inf)
    m = sc.max(axis=-1, keepdims=True)
    want_lse = (m[..., 0] + np.log(np.exp(sc - m).sum(axis=-1))) / math.log(2.0)
    assert np.abs(to_np(lse) - want_lse).max() < 1e-3
    # gradients against the oracle, which takes the same bf16 o the kernel
    # produced as the forward output only through dout (o is recomputed)
    want = oracle.swa_backward(q, k, v, dout, w, scale)
    for name, got, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), want):
        assert_grad_close(got, ref, f"SWA b{b}h{h}s{s}d{d}w{w} {name}")


def test_swa_backward_window_at_int32_max(ptb_lib):
    """Any window >= s is plain causal attention: the backward pass with
    w = 2^31 - 1 gives the same bits as with w = s."""
    b, h, s, d = 1, 2, 300, 128
    q, k, v = (t.cuda() for t in workloads.swa_inputs(b, h, s, d, seed=32))
    dout = workloads.normal_bf16((b, h, s, d), seed=33).cuda()
    o, lse = ptb_lib.swa_attention_lse(q, k, v, s)
    got_big = ptb_lib.swa_attention_backward(q, k, v, o, dout, lse, 2**31 - 1)
    got_s = ptb_lib.swa_attention_backward(q, k, v, o, dout, lse, s)
    for name, g_big, g_s in zip(("dq", "dk", "dv"), got_big, got_s):
        assert torch.equal(g_big, g_s), name


def test_swa_backward_unit_window(ptb_lib):
    """w = 1: P is the identity, so dv = dout bit for bit and dq = dk = 0 up
    to the rounding residue described at ZERO_TOL."""
    q, k, v = workloads.swa_inputs(1, 2, 150, 64, seed=5)
    dout = workloads.normal_bf16((1, 2, 150, 64), seed=6)
    qc, kc, vc, dc = (t.cuda() for t in (q, k, v, dout))
    o, lse = ptb_lib.swa_attention_lse(qc, kc, vc, 1)
    dq, dk, dv = ptb_lib.swa_attention_backward(qc, kc, vc, o, dc, lse, 1)
    torch.cuda.synchronize()
    assert float(dq.abs().max()) <= ZERO_TOL and float(dk.abs().max()) <= ZERO_TOL
    assert torch.equal(dv, dc)


# ---------------------------------------------------------- PTB layer --

LAYERS = [
    workloads.PTB_CONFIGS["tiny"],
    workloads.small_ptb(2, 300, 256, 4, 1024, 100, seed=31),
    workloads.small_ptb(1, 257, 384, 4, 1536, 65, seed=32),
    workloads.small_ptb(3, 130, 128, 8, 512, 1, seed=33),
    workloads.small_ptb(1, 200, 512, 4, 2048, 1000, seed=34),
]

GRADS = ["dx", "dln_gamma", "dln_beta", "dw_qkv", "dw_o", "dw_up", "dw_down"]


def _layer(cfg, dy_seed):
    host = workloads.ptb_inputs(cfg)
    dy = workloads.normal_bf16(tuple(host["x"].shape), seed=dy_seed)
    return host, dy


@pytest.mark.parametrize("cfg", LAYERS, ids=lambda c: c.name)
def test_ptb_backward_small(ptb_lib, cfg):
    host, dy = _layer(cfg, cfg.seed + 100)
    d = {k: v.cuda() for k, v in host.items()}
    y, saved = ptb_lib.ptb_forward_train(d["x"], d["ln_gamma"], d["ln_beta"], d["w_qkv"],
                                         d["w_o"], d["w_up"], d["w_down"], cfg.heads, cfg.window)
    g = ptb_lib.ptb_backward(dy.cuda(), d["x"], d["ln_gamma"], d["w_qkv"], d["w_o"], d["w_up"],
                             d["w_down"], saved, cfg.heads, cfg.window)
    torch.cuda.synchronize()
    want = oracle.ptb_backward(host["x"], host["ln_gamma"], host["ln_beta"], host["w_qkv"],
                               host["w_o"], host["w_up"], host["w_down"], cfg.heads, cfg.window,
                               dy)
    for name in GRADS:
        assert_grad_close(g[name], want[name], f"{cfg.name} {name}")


def test_forward_train_matches_forward_and_backward_is_deterministic(ptb_lib):
    cfg = workloads.small_ptb(2, 300, 256, 4, 1024, 100, seed=31)
    host, dy = _layer(cfg, 7)
    d = {k: v.cuda() for k, v in host.items()}
    args = (d["x"], d["ln_gamma"], d["ln_beta"], d["w_qkv"], d["w_o"], d["w_up"], d["w_down"],
            cfg.heads, cfg.window)
    y0 = ptb_lib.ptb_forward(*args)
    y1, saved = ptb_lib.ptb_forward_train(*args)
    torch.cuda.synchronize()
    assert torch.equal(y0, y1)
    bargs = (dy.cuda(), d["x"], d["ln_gamma"], d["w_qkv"], d["w_o"], d["w_up"], d["w_down"], saved,
             cfg.heads, cfg.window)
    g0 = ptb_lib.ptb_backward(*bargs)
    g1 = ptb_lib.ptb_backward(*bargs)
    torch.cuda.synchronize()
    for name in GRADS:
        assert torch.equal(g0[name], g1[name]), name


def test_backward_zero_output_weights(ptb_lib):
    """W_o = W_down = 0: dx = dy bit for bit, and nothing reaches the
    input-side weights or the LayerNorm parameters."""
    cfg = workloads.small_ptb(1, 200, 256, 4, 1024, 50, seed=35)
    host, dy = _layer(cfg, 8)
    host["w_o"].zero_()
    host["w_down"].zero_()
    d = {k: v.cuda() for k, v in host.items()}
    _, saved = ptb_lib.ptb_forward_train(d["x"], d["ln_gamma"], d["ln_beta"], d["w_qkv"],
                                         d["w_o"], d["w_up"], d["w_down"], cfg.heads, cfg.window)
    g = ptb_lib.ptb_backward(dy.cuda(), d["x"], d["ln_gamma"], d["w_qkv"], d["w_o"], d["w_up"],
                             d["w_down"], saved, cfg.heads, cfg.window)
    torch.cuda.synchronize()
    assert torch.equal(g["dx"].cpu(), dy)
    for name in ("dln_gamma", "dln_beta", "dw_qkv", "dw_up"):
        assert not g[name].any(), name


# ------------------------------------------------------- full size --

def _train_on_device(ptb_lib, cfg, dy_seed):
    """forward_train + backward on the device with caller workspaces, as the
    training benchmark launches them; returns host copies of inputs, dy and
    the gradients."""
    d = workloads.ptb_inputs(cfg, device="cuda")
    dy = workloads.normal_bf16(tuple(d["x"].shape), seed=dy_seed, device="cuda")
    b, s, h, f = cfg.batch, cfg.seq, cfg.hidden, cfg.ffn
    ws_f = torch.empty(ptb_lib.workspace_size(b, s, h, f), dtype=torch.uint8, device="cuda")
    ws_b = torch.empty(ptb_lib.backward_workspace_size(b, s, h, f, cfg.heads), dtype=torch.uint8,
                       device="cuda")
    w = (d["w_qkv"], d["w_o"], d["w_up"], d["w_down"])
    _, saved = ptb_lib.ptb_forward_train(d["x"], d["ln_gamma"], d["ln_beta"], *w, cfg.heads,
                                         cfg.window, workspace=ws_f)
    g = ptb_lib.ptb_backward(dy, d["x"], d["ln_gamma"], *w, saved, cfg.heads, cfg.window,
                             workspace=ws_b)
    torch.cuda.synchronize()
    host = {k: v.cpu() for k, v in d.items()}
    g = {k: v.cpu() for k, v in g.items()}
    dy = dy.cpu()
    del d, ws_f, ws_b, saved, w
    torch.cuda.empty_cache()
    return host, dy, g


def test_ptb_backward_full_size_13b(ptb_lib):
    cfg = workloads.PTB_CONFIGS["13b"]
    host, dy, g = _train_on_device(ptb_lib, cfg, cfg.seed + 100)
    want = oracle.ptb_backward(host["x"], host["ln_gamma"], host["ln_beta"], host["w_qkv"],
                               host["w_o"], host["w_up"], host["w_down"], cfg.heads, cfg.window,
                               dy)
    for name in GRADS:
        assert_grad_close(g[name], want[name], f"13b {name}")


@pytest.mark.parametrize("name", ["175b"])
def test_ptb_backward_full_size_sampled(ptb_lib, name):
    """dx at sampled rows and the weight gradients at two heads, 48 FFN
    columns and 32 output rows, each against the oracle's formula on those
    entries (tests/backward_sampled)."""
    from tests.backward_sampled import gathered, sampled_backward
    cfg = workloads.PTB_CONFIGS[name]
    host, dy, g = _train_on_device(ptb_lib, cfg, cfg.seed + 100)
    rng = np.random.default_rng(cfg.seed)
    rows = workloads.sample_rows(cfg.seq, cfg.window)
    head_sel = [0, cfg.heads - 1]
    f_sel = sorted(rng.choice(cfg.ffn, 48, replace=False).tolist())
    r_sel = sorted(rng.choice(cfg.hidden, 32, replace=False).tolist())
    want = sampled_backward(host["x"], host["ln_gamma"], host["ln_beta"], host["w_qkv"],
                            host["w_o"], host["w_up"], host["w_down"], cfg.heads, cfg.window, dy,
                            rows, head_sel, f_sel, r_sel)
    got = gathered({k: to_np(v) for k, v in g.items()}, cfg.hidden, cfg.heads, rows, head_sel,
                   f_sel, r_sel)
    for k in want:
        assert_grad_close(got[k], want[k], f"{name} {k} (sampled)")


def test_swa_long_sequence_forward_and_backward(ptb_lib):
    """A long sequence (6144 positions, window 1500, d = 64): many query and
    key blocks per item range, both kernels' band edges far from the
    sequence ends.  Forward output, LSE and all three gradients against the
    oracle."""
    b, h, s, d, w = 1, 1, 6144, 64, 1500
    q, k, v = workloads.swa_inputs(b, h, s, d, seed=61)
    dout = workloads.normal_bf16((b, h, s, d), seed=62)
    qc, kc, vc, dc = (t.cuda() for t in (q, k, v, dout))
    o, lse = ptb_lib.swa_attention_lse(qc, kc, vc, w)
    dq, dk, dv = ptb_lib.swa_attention_backward(qc, kc, vc, o, dc, lse, w)
    torch.cuda.synchronize()
    scale = 1.0 / math.sqrt(d)
    assert_grad_close(o, oracle.swa(q, k, v, w, scale), "long SWA o")
    want = oracle.swa_backward(q, k, v, dout, w, scale)
    for name, got, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), want):
        assert_grad_close(got, ref, f"long SWA {name}")
