"""CPU checks of the tolerance helper used by the parity tests."""
import numpy as np
import torch

from tests.parity import bf16_half_ulp, errors


def test_half_ulp_values():
    v = np.array([1.0, 1.5, 3.99, 4.0, 8.0, 9.27, 15.9, -8.5, 0.25])
    want = np.array([2.0 ** -8, 2.0 ** -8, 2.0 ** -7, 2.0 ** -6, 2.0 ** -5, 2.0 ** -5,
                     2.0 ** -5, 2.0 ** -5, 2.0 ** -10])
    assert np.array_equal(bf16_half_ulp(v), want)
    assert bf16_half_ulp(np.array([0.0]))[0] == 0.0


def test_rounding_to_bf16_stays_within_half_ulp():
    g = torch.Generator().manual_seed(0)
    v = (torch.randn(200000, generator=g, dtype=torch.float32) * 6).double()  # fp32 values: one rounding
    r = v.float().to(torch.bfloat16).double()
    assert bool(((r - v).abs().numpy() <= bf16_half_ulp(v.numpy())).all())
    rel, mx, ex = errors(r, v)
    assert ex == 0.0 and mx > 0.03  # plain max-abs exceeds 3e-2 from rounding alone


def test_bf16_storage_model_sane():
    import oracle
    from block_sliding_window_gb300 import workloads
    from tests.bf16_storage_model import ptb_forward_bf16_storage
    cfg = workloads.PTB_CONFIGS["tiny"]
    h = workloads.ptb_inputs(cfg)
    rows = workloads.sample_rows(cfg.seq, cfg.window)
    args = (h["x"], h["ln_gamma"], h["ln_beta"], h["w_qkv"], h["w_o"], h["w_up"], h["w_down"],
            cfg.heads, cfg.window)
    want = oracle.ptb_forward(*args, rows=rows)[0]
    model = ptb_forward_bf16_storage(*args, rows)
    rel, mx, ex = errors(model, want)
    assert 0 < rel < 1e-2 and ex < 1e-2
    # zero weights: y = x exactly, through every storage point
    z = {k: torch.zeros_like(h[k]) for k in ("w_qkv", "w_o", "w_up", "w_down")}
    model0 = ptb_forward_bf16_storage(h["x"], h["ln_gamma"], h["ln_beta"], z["w_qkv"], z["w_o"],
                                      z["w_up"], z["w_down"], cfg.heads, cfg.window, rows)
    assert np.array_equal(model0, h["x"][0, rows].double().numpy())


def test_e4m3_codes_known_values():
    """e4m3 (1-4-3, bias 7, no infinities): 448 = 0x7E, 1.0 = 0x38, 2^-9 (the
    smallest subnormal) = 0x01; an all-zero row takes scale 1."""
    from tests.bf16_storage_model import e4m3_codes_fp32
    codes, s = e4m3_codes_fp32(torch.tensor([[448.0, -448.0, 1.0, 2.0 ** -9, 0.0, -1.5],
                                             [0.0, 0.0, 0.0, 0.0, 0.0, 0.0]]))
    assert codes[0].tolist() == [0x7E, 0xFE, 0x38, 0x01, 0x00, 0xBC]
    assert codes[1].tolist() == [0] * 6 and s.tolist() == [1.0, 1.0]
    # amax maps to 448 and the scale is amax / 448; ties round to even:
    # 17 lies halfway between the e4m3 values 16 and 18 and goes to 16.
    codes, s = e4m3_codes_fp32(torch.tensor([[896.0, 34.0]]))
    assert s.tolist() == [2.0] and codes[0].tolist() == [0x7E, 0x58]


def test_e4m3_linear_slabs_equal_whole():
    """The FP8 storage model quantizes weights a slab of rows at a time; with
    per-row scales that is the same as quantizing the whole matrix."""
    from tests.bf16_storage_model import _e4m3_linear, e4m3_rows
    rng = np.random.default_rng(3)
    a = rng.standard_normal((5, 40))
    w = rng.standard_normal((23, 40)) * np.linspace(0.01, 3.0, 23)[:, None]
    whole = a @ e4m3_rows(w).T
    assert np.array_equal(_e4m3_linear(a, w, slab=4), whole)
    assert np.array_equal(_e4m3_linear(a, torch.from_numpy(w), slab=100), whole)
