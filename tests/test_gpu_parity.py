"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Every case feeds identical seeded bf16 inputs to both sides and compares
element by element with relative L2 <= 1e-2 and max-abs <= 3e-2; the
attention mask is compared bit-exactly through the kernel's own per-row
attended-key counts and through the zero pattern of a one-hot value probe.
Full-size layers (13B-class, 175B and 530B shapes) run in the same launch
configuration the benchmark times and are checked on sampled rows that the
oracle computes one by one.
"""
import math
import time

import numpy as np
import pytest
import torch

import oracle
from block_sliding_window_gb300 import workloads
from tests.bf16_storage_model import (e4m3_codes_fp32, ptb_forward_bf16_storage,
                                     ptb_forward_fp8_storage, serial_bf16_storage)
from tests.parity import MAX_ABS, REL_L2, assert_close, errors, to_np

pytestmark = pytest.mark.gpu


def _cuda(d):
    return {k: v.cuda() for k, v in d.items()}


@pytest.fixture(autouse=True)
def _status_clean(ptb_lib):
    ptb_lib.last_device_error()
    yield
    assert ptb_lib.last_device_error() == 0, "a kernel recorded a device-side error"


# ------------------------------------------------------------- bounded wait --

def test_bounded_wait_gives_up_and_reports(ptb_lib):
    """A wait on an mbarrier nobody signals ends with PTB_ERR_TIMEOUT instead
    of hanging, and the context stays usable."""
    ptb_lib.wait_probe(20_000_000)  # 20 ms
    assert ptb_lib.last_device_error() == 6
    assert ptb_lib.last_device_error() == 0
    assert torch.ones(8, device="cuda").sum().item() == 8


def test_status_read_waits_for_its_own_stream_only(ptb_lib):
    """ptb_last_device_error(stream A) returns while a long kernel queued on
    stream B is still running: it synchronises stream A, not the device."""
    a, b = torch.cuda.Stream(), torch.cuda.Stream()
    assert ptb_lib.last_device_error(stream=a) == 0  # kernel loaded, stream A idle
    torch.cuda.synchronize()
    with torch.cuda.stream(b):
        torch.cuda._sleep(3_000_000_000)  # about 1.5 s at 2 GHz
    t0 = time.perf_counter()
    st = ptb_lib.last_device_error(stream=a)
    waited = time.perf_counter() - t0
    b_busy = not b.query()
    torch.cuda.synchronize()
    assert st == 0
    assert b_busy, f"the status read on stream A waited for stream B ({waited:.3f} s)"
    assert waited < 0.5, f"the status read on stream A took {waited:.3f} s"


# --------------------------------------------------------------- LayerNorm --

@pytest.mark.parametrize("rows,hidden", [(1, 64), (3, 8), (130, 5120), (17, 12288),
                                         (5, 20480), (2, 32768), (64, 96)])
def test_layernorm(ptb_lib, rows, hidden):
    x = workloads.normal_bf16((rows, hidden), seed=rows + hidden, std=2.0, mean=0.5)
    gamma = workloads.normal_bf16((hidden,), seed=1, std=0.1, mean=1.0)
    beta = workloads.normal_bf16((hidden,), seed=2, std=0.1)
    out = ptb_lib.layernorm(x.cuda(), gamma.cuda(), beta.cuda())
    assert_close(out, oracle.layer_norm(x, gamma, beta), f"LN {rows}x{hidden}")


# ----------------------------------------------------------- [QKV | up] GEMM --

GEMM_SHAPES = [(128, 64, 256), (600, 256, 1024), (257, 384, 1536), (1, 64, 64),
               (2048, 1024, 4096), (333, 192, 320)]


def _gemm_ws(ptb_lib, split, tokens, hidden, ffn):
    """Scratch that lets the GEMM split its last wave along K (None: unsplit)."""
    n = ptb_lib.gemm_workspace_size(tokens, hidden, ffn) if split else 0
    return torch.full((n,), 0x7F, dtype=torch.uint8, device="cuda") if n else None


@pytest.mark.parametrize("split", [False, True])
@pytest.mark.parametrize("tokens,hidden,ffn", GEMM_SHAPES)
def test_gemm_qkv_up(ptb_lib, tokens, hidden, ffn, split):
    xn = workloads.normal_bf16((tokens, hidden), seed=3)
    w_qkv = workloads.normal_bf16((3 * hidden, hidden), seed=4, std=1.0 / math.sqrt(hidden))
    w_up = workloads.normal_bf16((ffn, hidden), seed=5, std=1.0 / math.sqrt(hidden))
    u = ptb_lib.gemm_qkv_up(xn.cuda(), w_qkv.cuda(), w_up.cuda(),
                            workspace=_gemm_ws(ptb_lib, split, tokens, hidden, ffn))
    want = np.concatenate([oracle.linear(xn, w_qkv),
                           oracle.gelu_tanh(oracle.linear(xn, w_up))], axis=1)
    assert_close(u, want, f"GEMM1 {tokens}x{hidden}x{ffn}")


# ------------------------------------------------- [out | down] GEMM + x --

@pytest.mark.parametrize("split", [False, True])
@pytest.mark.parametrize("tokens,hidden,ffn", GEMM_SHAPES)
def test_gemm_out_down_residual(ptb_lib, tokens, hidden, ffn, split):
    # ctx and g live as column blocks of one fused buffer, as in the layer.
    ld = 3 * hidden + ffn
    u = workloads.normal_bf16((tokens, ld), seed=6, std=0.5).cuda()
    ctx, g = u[:, :hidden], u[:, 3 * hidden:]
    w_o = workloads.normal_bf16((hidden, hidden), seed=7, std=1.0 / math.sqrt(hidden))
    w_down = workloads.normal_bf16((hidden, ffn), seed=8, std=1.0 / math.sqrt(ffn))
    x = workloads.normal_bf16((tokens, hidden), seed=9)
    y = ptb_lib.gemm_out_down(ctx, g, w_o.cuda(), w_down.cuda(), x.cuda(),
                              workspace=_gemm_ws(ptb_lib, split, tokens, hidden, ffn))
    want = to_np(x) + oracle.linear(ctx.cpu(), w_o) + oracle.linear(g.cpu(), w_down)
    assert_close(y, want, f"GEMM2 {tokens}x{hidden}x{ffn}")


# --------------------------------------------------------------------- SWA --

SWA_CASES = [  # batch, heads, seq, head_dim, window
    (1, 1, 1, 64, 1), (1, 2, 63, 64, 5), (2, 3, 64, 64, 64), (1, 2, 65, 32, 64),
    (2, 2, 200, 128, 17), (1, 4, 333, 96, 100), (1, 2, 257, 16, 1), (1, 2, 300, 64, 300),
    (1, 1, 500, 128, 2000), (2, 2, 1000, 128, 129), (1, 2, 700, 96, 511), (1, 1, 130, 32, 2),
    # Several items per CTA (256 items), up to 20 key tiles per query tile:
    # exercises the stage and score-buffer barrier phases across items.
    (2, 16, 2048, 96, 1000),
]


@pytest.mark.parametrize("b,h,s,d,w", SWA_CASES)
def test_swa_matches_oracle_and_counts(ptb_lib, b, h, s, d, w):
    q, k, v = workloads.swa_inputs(b, h, s, d, seed=s + w)
    o, counts = ptb_lib.swa_attention_counts(q.cuda(), k.cuda(), v.cuda(), w)
    assert_close(o, oracle.swa(q, k, v, w), f"SWA {b}x{h}x{s}x{d} w={w}")
    want_counts = np.broadcast_to(oracle.attended_counts(s, w), (b, h, s))
    assert np.array_equal(counts.cpu().numpy(), want_counts), "attended-key counts differ"
    o_plain = ptb_lib.swa_attention(q.cuda(), k.cuda(), v.cuda(), w)
    assert torch.equal(o_plain, o), "the counting kernel must compute the same output"


@pytest.mark.parametrize("s,d,w", [(128, 128, 32), (300, 64, 64), (260, 32, 7), (200, 128, 1000)])
def test_swa_mask_zero_pattern(ptb_lib, s, d, w):
    """Q = K = 0 makes every in-band weight 1/count; V row j is the one-hot of
    j mod d, so o[i, c] is nonzero exactly where a key j with j mod d = c is
    in row i's window.  The zero pattern is compared bit for bit."""
    z = torch.zeros(1, 1, s, d, dtype=torch.bfloat16)
    v = torch.zeros(1, 1, s, d, dtype=torch.bfloat16)
    v[0, 0, torch.arange(s), torch.arange(s) % d] = 1
    o = ptb_lib.swa_attention(z.cuda(), z.cuda(), v.cuda(), w).cpu()
    want = oracle.swa(z, z, v, w)
    got = to_np(o)
    assert np.array_equal(got == 0, want == 0), "mask zero pattern differs"
    nz = want != 0
    assert np.all(np.abs(got[nz] - want[nz]) <= 2.0 ** -8 * want[nz])


@pytest.mark.parametrize("w", [512, 2048, 1])
def test_swa_operator_config(ptb_lib, w):
    """The SWA operator at batch 4, 16 heads, head_dim 128, seq 2048."""
    cfg = workloads.SWA_CONFIGS["swa"]
    q, k, v = workloads.swa_inputs(cfg.batch, cfg.heads, cfg.seq, cfg.head_dim, cfg.seed)
    o, counts = ptb_lib.swa_attention_counts(q.cuda(), k.cuda(), v.cuda(), w)
    o = o.cpu()
    if w == 1:
        assert torch.equal(o, v), "window 1 must return V exactly"
    for bi in range(cfg.batch):
        assert_close(o[bi], oracle.swa(q[bi], k[bi], v[bi], w), f"SWA op w={w} batch {bi}")
    want_counts = np.broadcast_to(oracle.attended_counts(cfg.seq, w), counts.shape)
    assert np.array_equal(counts.cpu().numpy(), want_counts)


def test_swa_window_at_int32_max(ptb_lib):
    """Any window >= s is plain causal attention: w = 2^31 - 1 gives the same
    bits as w = s (no index arithmetic may overflow on the way)."""
    b, h, s, d = 1, 2, 300, 96
    q, k, v = (t.cuda() for t in workloads.swa_inputs(b, h, s, d, seed=31))
    o_big, counts = ptb_lib.swa_attention_counts(q, k, v, 2**31 - 1)
    o_s = ptb_lib.swa_attention(q, k, v, s)
    assert torch.equal(o_big, o_s)
    assert np.array_equal(counts.cpu().numpy(),
                          np.broadcast_to(oracle.attended_counts(s, s), (b, h, s)))
    assert_close(o_big, oracle.swa(q.cpu(), k.cpu(), v.cpu(), s), "SWA w = 2^31 - 1")


def test_swa_strided_in_place(ptb_lib):
    """Q, K, V as head-strided column blocks of one [T, 3H + F] buffer and the
    output written over Q, as the layer does."""
    b, s, nh, d, f, w = 2, 300, 4, 64, 128, 77
    hdim = nh * d
    ld = 3 * hdim + f
    u = workloads.normal_bf16((b, s, ld), seed=11).cuda()
    view = lambda off: u[:, :, off:off + hdim].unflatten(2, (nh, d)).transpose(1, 2)  # noqa: E731
    q, k, v = view(0), view(hdim), view(2 * hdim)
    want = oracle.swa(q.cpu(), k.cpu(), v.cpu(), w)
    untouched = u[:, :, hdim:].clone()
    ptb_lib.swa_attention_strided(q, k, v, q, w)
    assert_close(view(0), want, "strided in-place SWA")
    assert torch.equal(u[:, :, hdim:], untouched), "SWA wrote outside its output block"


@pytest.mark.parametrize("d,w", [(96, 77), (128, 300), (32, 50)])
def test_swa_output_layout_differs_from_inputs(ptb_lib, d, w):
    """Q, K, V as head-strided column blocks of a [B, s, 3H + 8] buffer and
    the output in its own [B, heads, s, d] buffer with a padded row stride:
    the output tensor map has the other dimension order and strides than
    the input maps, and ragged rows past the sequence must not be written."""
    b, s, nh = 2, 300, 3
    hdim = nh * d
    ld = 3 * hdim + 8
    u = workloads.normal_bf16((b, s, ld), seed=d + w).cuda()
    view = lambda off: u[:, :, off:off + hdim].unflatten(2, (nh, d)).transpose(1, 2)  # noqa: E731
    q, k, v = view(0), view(hdim), view(2 * hdim)
    pad = 8
    big = torch.full((b, nh, s + 1, d + pad), 7.0, dtype=torch.bfloat16, device="cuda")
    o = big[:, :, :s, :d]  # row stride d + pad, head stride (s + 1)(d + pad)
    ptb_lib.swa_attention_strided(q, k, v, o, w)
    assert_close(o, oracle.swa(q.cpu(), k.cpu(), v.cpu(), w), f"SWA d={d} w={w}, separate output")
    assert bool((big[:, :, s, :] == 7.0).all()), "a row past the sequence was written"
    assert bool((big[:, :, :, d:] == 7.0).all()), "columns past d were written"


# ---------------------------------------------------------------- PTB layer --

SMALL_LAYERS = [
    workloads.PTB_CONFIGS["tiny"],
    workloads.PTB_CONFIGS["tiny"].with_window(128),
    workloads.small_ptb(2, 300, 256, 4, 1024, 100, seed=21),
    workloads.small_ptb(1, 257, 384, 4, 1536, 65, seed=22),
    workloads.small_ptb(3, 130, 128, 8, 512, 1, seed=23),
    workloads.small_ptb(1, 200, 512, 4, 2048, 1000, seed=24),
    workloads.small_ptb(1, 1, 64, 2, 64, 5, seed=25),
]


@pytest.mark.parametrize("cfg", SMALL_LAYERS, ids=lambda c: c.name)
@pytest.mark.parametrize("own_workspace", [False, True])
def test_ptb_forward_small(ptb_lib, cfg, own_workspace):
    host = workloads.ptb_inputs(cfg)
    d = _cuda(host)
    ws = None
    if own_workspace:
        n = ptb_lib.workspace_size(cfg.batch, cfg.seq, cfg.hidden, cfg.ffn)
        ws = torch.full((n,), 0xFF, dtype=torch.uint8, device="cuda")  # NaN-pattern canary
    y = ptb_lib.ptb_forward(d["x"], d["ln_gamma"], d["ln_beta"], d["w_qkv"], d["w_o"], d["w_up"],
                            d["w_down"], cfg.heads, cfg.window, workspace=ws)
    want = oracle.ptb_forward(host["x"], host["ln_gamma"], host["ln_beta"], host["w_qkv"],
                              host["w_o"], host["w_up"], host["w_down"], cfg.heads, cfg.window)
    assert_close(y, want, cfg.name)


def test_ptb_forward_deterministic_and_events(ptb_lib):
    cfg = workloads.small_ptb(2, 300, 256, 4, 1024, 100, seed=21)
    d = _cuda(workloads.ptb_inputs(cfg))
    args = (d["x"], d["ln_gamma"], d["ln_beta"], d["w_qkv"], d["w_o"], d["w_up"], d["w_down"],
            cfg.heads, cfg.window)
    y0 = ptb_lib.ptb_forward(*args)
    events = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
    y1 = ptb_lib.ptb_forward_events(*args, events)
    torch.cuda.synchronize()
    assert torch.equal(y0, y1)
    for a, b in zip(events, events[1:]):
        assert a.elapsed_time(b) >= 0.0


def test_ptb_forward_fp8_deterministic_and_events(ptb_lib):
    cfg = workloads.small_ptb(2, 300, 256, 4, 1024, 100, seed=21)
    d = _cuda(workloads.ptb_inputs(cfg))
    w8 = ptb_lib.prepare_fp8_weights(d["w_qkv"], d["w_o"], d["w_up"], d["w_down"])
    args = (d["x"], d["ln_gamma"], d["ln_beta"], w8, cfg.heads, cfg.window)
    y0 = ptb_lib.ptb_forward_fp8(*args)
    events = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    y1 = ptb_lib.ptb_forward_fp8_events(*args, events)
    torch.cuda.synchronize()
    assert torch.equal(y0, y1)
    for a, b in zip(events, events[1:]):
        assert a.elapsed_time(b) >= 0.0


def test_gemm_split_repeatable(ptb_lib):
    """The split last wave gives the same bits call after call (the arrival
    order of the pieces does not change the summation order)."""
    tokens, hidden, ffn = 2048, 1024, 4096
    assert ptb_lib.gemm_workspace_size(tokens, hidden, ffn) > 0
    u = workloads.normal_bf16((tokens, 3 * hidden + ffn), seed=12, std=0.5).cuda()
    w_o = workloads.normal_bf16((hidden, hidden), seed=13, std=0.03).cuda()
    w_down = workloads.normal_bf16((hidden, ffn), seed=14, std=0.015).cuda()
    x = workloads.normal_bf16((tokens, hidden), seed=15).cuda()
    ws = _gemm_ws(ptb_lib, True, tokens, hidden, ffn)
    outs = [ptb_lib.gemm_out_down(u[:, :hidden], u[:, 3 * hidden:], w_o, w_down, x, workspace=ws)
            for _ in range(3)]
    assert all(torch.equal(outs[0], o) for o in outs[1:])


def test_fp8_rejects_shapes_off_the_128_grid(ptb_lib):
    cfg = workloads.PTB_CONFIGS["tiny"]  # hidden 64
    d = _cuda(workloads.ptb_inputs(cfg))
    with pytest.raises(ptb_lib.PTBError):
        ptb_lib.prepare_fp8_weights(d["w_qkv"], d["w_o"], d["w_up"], d["w_down"])


def test_ptb_special_case_attention_off(ptb_lib):
    """W_o = 0 leaves y = x + MLP(LN(x)); W_down = 0 leaves y = x + Attn(LN(x))."""
    cfg = workloads.small_ptb(1, 200, 256, 4, 512, 33, seed=26)
    host = workloads.ptb_inputs(cfg)
    for zero in ("w_o", "w_down"):
        h2 = dict(host)
        h2[zero] = torch.zeros_like(host[zero])
        d = _cuda(h2)
        y = ptb_lib.ptb_forward(d["x"], d["ln_gamma"], d["ln_beta"], d["w_qkv"], d["w_o"],
                                d["w_up"], d["w_down"], cfg.heads, cfg.window)
        want = oracle.ptb_forward(h2["x"], h2["ln_gamma"], h2["ln_beta"], h2["w_qkv"], h2["w_o"],
                                  h2["w_up"], h2["w_down"], cfg.heads, cfg.window)
        assert_close(y, want, f"{zero} = 0")


def _ln2(hidden, seed):
    g2 = workloads.normal_bf16((hidden,), seed=seed, std=0.1, mean=1.0)
    b2 = workloads.normal_bf16((hidden,), seed=seed + 1, std=0.1)
    return g2, b2


@pytest.mark.parametrize("cfg", SMALL_LAYERS, ids=lambda c: c.name)
def test_serial_forward_small(ptb_lib, cfg):
    host = workloads.ptb_inputs(cfg)
    g2, b2 = _ln2(cfg.hidden, 31)
    d = _cuda(host)
    y = ptb_lib.serial_forward(d["x"], d["ln_gamma"], d["ln_beta"], g2.cuda(), b2.cuda(),
                               d["w_qkv"], d["w_o"], d["w_up"], d["w_down"], cfg.heads, cfg.window)
    want = oracle.serial_block(host["x"], host["ln_gamma"], host["ln_beta"], g2, b2, host["w_qkv"],
                               host["w_o"], host["w_up"], host["w_down"], cfg.heads, cfg.window)
    assert_close(y, want, "serial " + cfg.name)


@pytest.mark.parametrize("name", ["13b", "175b"])
def test_serial_forward_full_size_sampled(ptb_lib, name):
    cfg = workloads.PTB_CONFIGS[name]
    d = workloads.ptb_inputs(cfg, device="cuda")
    g2, b2 = _ln2(cfg.hidden, 33)
    ws = torch.empty(ptb_lib.serial_workspace_size(cfg.batch, cfg.seq, cfg.hidden, cfg.ffn),
                     dtype=torch.uint8, device="cuda")
    y = ptb_lib.serial_forward(d["x"], d["ln_gamma"], d["ln_beta"], g2.cuda(), b2.cuda(),
                               d["w_qkv"], d["w_o"], d["w_up"], d["w_down"], cfg.heads, cfg.window,
                               workspace=ws)
    torch.cuda.synchronize()
    rows = workloads.sample_rows(cfg.seq, cfg.window)
    host = {k: v.cpu() for k, v in d.items()}
    del d, ws
    args = (host["x"], host["ln_gamma"], host["ln_beta"], g2, b2, host["w_qkv"], host["w_o"],
            host["w_up"], host["w_down"], cfg.heads, cfg.window)
    want = oracle.serial_block(*args, rows=rows)
    _, _, floor = errors(serial_bf16_storage(*args, rows), want[0])
    rel, mx, ex = errors(y[0, rows], want[0])
    bound = max(MAX_ABS, 1.25 * floor)
    print(f"serial {name}: rel-L2 {rel:.3e}, max-abs {mx:.3e}, beyond rounding {ex:.3e}, "
          f"bf16-storage floor {floor:.3e}, bound {bound:.3e}")
    assert rel <= REL_L2 and ex <= bound


def _fp8_check(ptb_lib, cfg, host, d, rows, what):
    """FP8 layer vs the fp64 oracle, bounded by 1.25x the error of an exact
    computation with the same e4m3/bf16 rounding points (rel-L2 and max-abs)."""
    w8 = ptb_lib.prepare_fp8_weights(d["w_qkv"], d["w_o"], d["w_up"], d["w_down"])
    y = ptb_lib.ptb_forward_fp8(d["x"], d["ln_gamma"], d["ln_beta"], w8, cfg.heads, cfg.window)
    torch.cuda.synchronize()
    args = (host["x"], host["ln_gamma"], host["ln_beta"], host["w_qkv"], host["w_o"],
            host["w_up"], host["w_down"], cfg.heads, cfg.window)
    want = oracle.ptb_forward(*args, rows=rows)[0]
    fl_rel, _, fl_ex = errors(ptb_forward_fp8_storage(*args, rows), want)
    rel, mx, ex = errors(y[0, rows], want)
    print(f"fp8 {what}: rel-L2 {rel:.3e} (floor {fl_rel:.3e}), max-abs beyond rounding {ex:.3e} "
          f"(floor {fl_ex:.3e}), plain max-abs {mx:.3e}")
    assert rel <= max(REL_L2, 1.25 * fl_rel), f"fp8 {what}: rel-L2 {rel:.3e}"
    assert ex <= max(MAX_ABS, 1.25 * fl_ex), f"fp8 {what}: max-abs {ex:.3e}"


@pytest.mark.parametrize("cfg", [c for c in SMALL_LAYERS if c.hidden % 128 == 0 and c.ffn % 128 == 0],
                         ids=lambda c: c.name)
def test_ptb_forward_fp8_small(ptb_lib, cfg):
    host = workloads.ptb_inputs(cfg)
    if cfg.batch != 1:
        host["x"] = host["x"][:1]
    d = _cuda(host)
    _fp8_check(ptb_lib, cfg, host, d, list(range(cfg.seq)), cfg.name)


@pytest.mark.parametrize("cfg", [workloads.small_ptb(1, 64, 384, 4, 1536, 16, seed=27),
                                 # [W_o | W_down] rows of 33536 elements (67 KB): the
                                 # quantizer's long-row CTA shape
                                 workloads.small_ptb(1, 64, 256, 2, 33280, 16, seed=28)],
                         ids=lambda c: c.name)
def test_fp8_weight_codes_bit_exact(ptb_lib, cfg):
    """The e4m3 weight codes and per-row scales are integer decisions taken in
    fp32; they must match an fp32 CPU computation bit for bit."""
    d = _cuda(workloads.ptb_inputs(cfg))
    w1, s1, w2, s2 = ptb_lib.prepare_fp8_weights(d["w_qkv"], d["w_o"], d["w_up"], d["w_down"])
    torch.cuda.synchronize()
    c1, r1 = e4m3_codes_fp32(torch.cat([d["w_qkv"], d["w_up"]], 0).cpu())
    c2, r2 = e4m3_codes_fp32(torch.cat([d["w_o"], d["w_down"]], 1).cpu())
    assert torch.equal(s1.cpu(), r1) and torch.equal(s2.cpu(), r2)
    assert torch.equal(w1.cpu(), c1) and torch.equal(w2.cpu(), c2)
    # An all-zero row takes scale 1 and zero codes.
    wz = d["w_up"].clone()
    wz[5].zero_()
    _, s1z, _, _ = ptb_lib.prepare_fp8_weights(d["w_qkv"], d["w_o"], wz, d["w_down"])
    assert float(s1z[3 * cfg.hidden + 5]) == 1.0
    # The same for a row of [W_o | W_down].
    woz, wdz = d["w_o"].clone(), d["w_down"].clone()
    woz[7].zero_()
    wdz[7].zero_()
    _, _, w2z, s2z = ptb_lib.prepare_fp8_weights(d["w_qkv"], woz, d["w_up"], wdz)
    assert float(s2z[7]) == 1.0 and int(w2z[7].abs().sum()) == 0


@pytest.mark.parametrize("name", ["13b", "175b", "530b"])
def test_ptb_forward_fp8_full_size_sampled(ptb_lib, name):
    """The FP8 layer at the shapes its throughput is reported on, launched as
    the benchmark launches it, on rows in every 128-row tile."""
    cfg = workloads.PTB_CONFIGS[name]
    d = workloads.ptb_inputs(cfg, device="cuda")
    host = {k: v.cpu() for k, v in d.items()}
    _fp8_check(ptb_lib, cfg, host, d, workloads.sample_rows(cfg.seq, cfg.window), name)


@pytest.mark.parametrize("name", ["13b", "175b", "530b"])
def test_ptb_forward_full_size_sampled(ptb_lib, name):
    """Full-size layers, launched exactly as the benchmark launches them
    (caller workspace, current stream), checked on sampled rows."""
    cfg = workloads.PTB_CONFIGS[name]
    d = workloads.ptb_inputs(cfg, device="cuda")
    ws = torch.empty(ptb_lib.workspace_size(cfg.batch, cfg.seq, cfg.hidden, cfg.ffn),
                     dtype=torch.uint8, device="cuda")
    y = ptb_lib.ptb_forward(d["x"], d["ln_gamma"], d["ln_beta"], d["w_qkv"], d["w_o"], d["w_up"],
                            d["w_down"], cfg.heads, cfg.window, workspace=ws)
    torch.cuda.synchronize()
    assert bool(torch.isfinite(y).all())
    rows = workloads.sample_rows(cfg.seq, cfg.window)
    host = {k: v.cpu() for k, v in d.items()}
    del d, ws
    want = oracle.ptb_forward(host["x"], host["ln_gamma"], host["ln_beta"], host["w_qkv"],
                              host["w_o"], host["w_up"], host["w_down"], cfg.heads, cfg.window,
                              rows=rows)
    # The bf16 storage floor: exact arithmetic between the bf16 storage points.
    model = ptb_forward_bf16_storage(host["x"], host["ln_gamma"], host["ln_beta"], host["w_qkv"],
                                     host["w_o"], host["w_up"], host["w_down"], cfg.heads,
                                     cfg.window, rows)
    _, _, floor = errors(model, want[0])
    rel, mx, ex = errors(y[0, rows], want[0])
    bound = max(MAX_ABS, 1.25 * floor)
    print(f"{name}: rel-L2 {rel:.3e}, max-abs {mx:.3e}, beyond rounding {ex:.3e}, "
          f"bf16-storage floor {floor:.3e}, bound {bound:.3e}")
    assert rel <= REL_L2, f"{name}: rel-L2 {rel:.3e}"
    assert ex <= bound, f"{name}: max-abs beyond rounding {ex:.3e} > {bound:.3e}"


# ------------------------------------------------ GEMM tile shapes --

@pytest.fixture
def gemm_pairs(ptb_lib, request):
    prev = ptb_lib.set_gemm_pairs(request.param)
    yield request.param
    ptb_lib.set_gemm_pairs(prev)


@pytest.mark.parametrize("gemm_pairs", [0, 1], indirect=True, ids=["single", "pairs"])
@pytest.mark.parametrize("cfg", [workloads.small_ptb(2, 300, 256, 4, 1024, 100, seed=41),
                                 workloads.small_ptb(1, 520, 512, 4, 2048, 300, seed=42)],
                         ids=lambda c: c.name)
def test_ptb_forward_both_gemm_tile_shapes(ptb_lib, gemm_pairs, cfg):
    """The layer with 128 x 256 single-CTA tiles and with 256 x 256 CTA-pair
    tiles (ragged last M tile included) against the oracle."""
    host = workloads.ptb_inputs(cfg)
    d = _cuda(host)
    y = ptb_lib.ptb_forward(d["x"], d["ln_gamma"], d["ln_beta"], d["w_qkv"], d["w_o"],
                            d["w_up"], d["w_down"], cfg.heads, cfg.window)
    torch.cuda.synchronize()
    want = oracle.ptb_forward(host["x"], host["ln_gamma"], host["ln_beta"], host["w_qkv"],
                              host["w_o"], host["w_up"], host["w_down"], cfg.heads, cfg.window)
    assert_close(y, want, f"{cfg.name} pairs={gemm_pairs}")


@pytest.mark.parametrize("gemm_pairs", [0], indirect=True, ids=["single"])
def test_ptb_forward_full_size_single_175b(ptb_lib, gemm_pairs):
    """Single-CTA tiles forced on the 175B-shaped layer (the automatic mode
    uses CTA pairs there, which the full-size sampled tests cover): 5376 and
    768 tiles of 128 x 256, the second GEMM's last wave of 8 tiles split along
    K into 19 pieces each."""
    cfg = workloads.PTB_CONFIGS["175b"]
    d = workloads.ptb_inputs(cfg, device="cuda")
    ws = torch.empty(ptb_lib.workspace_size(cfg.batch, cfg.seq, cfg.hidden, cfg.ffn),
                     dtype=torch.uint8, device="cuda")
    y = ptb_lib.ptb_forward(d["x"], d["ln_gamma"], d["ln_beta"], d["w_qkv"], d["w_o"], d["w_up"],
                            d["w_down"], cfg.heads, cfg.window, workspace=ws)
    torch.cuda.synchronize()
    rows = workloads.sample_rows(cfg.seq, cfg.window)
    host = {k: v.cpu() for k, v in d.items()}
    del d, ws
    want = oracle.ptb_forward(host["x"], host["ln_gamma"], host["ln_beta"], host["w_qkv"],
                              host["w_o"], host["w_up"], host["w_down"], cfg.heads, cfg.window,
                              rows=rows)
    model = ptb_forward_bf16_storage(host["x"], host["ln_gamma"], host["ln_beta"], host["w_qkv"],
                                     host["w_o"], host["w_up"], host["w_down"], cfg.heads,
                                     cfg.window, rows)
    _, _, floor = errors(model, want[0])
    rel, mx, ex = errors(y[0, rows], want[0])
    print(f"175b single: rel-L2 {rel:.3e}, max-abs {mx:.3e}, beyond rounding {ex:.3e}")
    assert rel <= REL_L2 and ex <= max(MAX_ABS, 1.25 * floor)


def test_forward_host_buffers_two_streams(ptb_lib):
    """ptb_forward_host on pinned host x / y, two calls in flight on two
    streams with their own workspaces: the same bits as ptb_forward."""
    cfg = workloads.small_ptb(2, 300, 256, 4, 1024, 100, seed=43)
    host = workloads.ptb_inputs(cfg)
    d = _cuda(host)
    w = (d["ln_gamma"], d["ln_beta"], d["w_qkv"], d["w_o"], d["w_up"], d["w_down"])
    want = ptb_lib.ptb_forward(d["x"], *w, cfg.heads, cfg.window).cpu()
    x2 = workloads.normal_bf16(tuple(host["x"].shape), seed=44)
    want2 = ptb_lib.ptb_forward(x2.cuda(), *w, cfg.heads, cfg.window).cpu()
    xs = [host["x"].pin_memory(), x2.pin_memory()]
    ys = [torch.empty_like(xs[0]).pin_memory() for _ in range(2)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    nbytes = ptb_lib.host_workspace_size(cfg.batch, cfg.seq, cfg.hidden, cfg.ffn)
    wss = [torch.empty(nbytes, dtype=torch.uint8, device="cuda") for _ in range(2)]
    for i in range(2):
        ptb_lib.ptb_forward_host(xs[i], *w, cfg.heads, cfg.window, ys[i], wss[i],
                                 stream=streams[i])
    torch.cuda.synchronize()
    assert torch.equal(ys[0], want) and torch.equal(ys[1], want2)


def test_forward_host_buffers_two_streams_serialised(ptb_lib):
    """The same for a layer whose first GEMM exceeds 2^39 multiply-adds,
    where each call's layer waits for the previous call's layer on the other
    stream (the path of the large layers): still the bits of ptb_forward."""
    cfg = workloads.small_ptb(1, 2048, 6144, 48, 32768, 512, seed=45)
    assert cfg.batch * cfg.seq * cfg.hidden * (3 * cfg.hidden + cfg.ffn) > 2 ** 39
    d = {k: v.cuda() for k, v in workloads.ptb_inputs(cfg).items()}
    w = (d["ln_gamma"], d["ln_beta"], d["w_qkv"], d["w_o"], d["w_up"], d["w_down"])
    x2 = workloads.normal_bf16(tuple(d["x"].shape), seed=46)
    want = ptb_lib.ptb_forward(d["x"], *w, cfg.heads, cfg.window).cpu()
    want2 = ptb_lib.ptb_forward(x2.cuda(), *w, cfg.heads, cfg.window).cpu()
    xs = [d["x"].cpu().pin_memory(), x2.pin_memory()]
    ys = [torch.full_like(xs[0], float("nan")).pin_memory() for _ in range(2)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    nbytes = ptb_lib.host_workspace_size(cfg.batch, cfg.seq, cfg.hidden, cfg.ffn)
    wss = [torch.empty(nbytes, dtype=torch.uint8, device="cuda") for _ in range(2)]
    for rep in range(2):  # the second round waits on the first round's layers
        for i in range(2):
            ptb_lib.ptb_forward_host(xs[i], *w, cfg.heads, cfg.window, ys[i], wss[i],
                                     stream=streams[i])
    torch.cuda.synchronize()
    assert torch.equal(ys[0], want) and torch.equal(ys[1], want2)
    assert ptb_lib.last_device_error() == 0
