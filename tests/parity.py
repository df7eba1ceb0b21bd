"""Shared helpers for the parity tests: error metrics and the tolerance.

Tolerance for floating-point parity against the fp64 oracle (bf16 inputs,
fp32 accumulation, bf16 outputs):
  * relative L2 error <= 1e-2, literally;
  * maximum absolute error <= 3e-2 beyond the output's own rounding: every
    output is stored in bf16, and for |value| >= 8 half a bf16 ulp (0.031) is
    already above 3e-2, so an exact result rounded once to bf16 would fail a
    literal bar.  The allowance is half an ulp of bf16 at the oracle's value
    (2**(floor(log2|want|) - 8)); below |want| = 4 it is <= 0.0078.
The plain max-abs error is reported alongside.
"""
import numpy as np
import torch

REL_L2 = 1e-2
MAX_ABS = 3e-2


def to_np(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        return t.detach().to("cpu", torch.float64).numpy()
    return np.asarray(t, dtype=np.float64)


def bf16_half_ulp(v: np.ndarray) -> np.ndarray:
    """Half the spacing of bf16 numbers at |v| (8 significant bits)."""
    a = np.abs(v)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.where(a > 0, 2.0 ** (e - 8), 0.0)


def errors(got, want):
    """(relative L2, plain max-abs, max-abs beyond the bf16 output rounding)."""
    g, w = to_np(got), to_np(want)
    assert g.shape == w.shape, (g.shape, w.shape)
    assert np.all(np.isfinite(g)), "non-finite output"
    if not g.size:
        return 0.0, 0.0, 0.0
    rel = float(np.linalg.norm(g - w) / max(np.linalg.norm(w), 1e-30))
    diff = np.abs(g - w)
    excess = np.maximum(diff - bf16_half_ulp(w), 0.0)
    return rel, float(diff.max()), float(excess.max())


def assert_close(got, want, what="", rel_l2=REL_L2, max_abs=MAX_ABS):
    rel, mx, ex = errors(got, want)
    assert rel <= rel_l2 and ex <= max_abs, (
        f"{what}: rel-L2 {rel:.3e} (<= {rel_l2}), max-abs beyond bf16 rounding {ex:.3e} "
        f"(<= {max_abs}), plain max-abs {mx:.3e}")
    return rel, mx
