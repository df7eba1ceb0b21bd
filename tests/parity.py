"""Shared helpers for the parity tests: error metrics and the tolerance.

Tolerance for floating-point parity against the fp64 oracle (bf16 inputs,
fp32 accumulation, bf16 outputs): relative L2 error <= 1e-2 and maximum
absolute error <= 3e-2.
"""
import numpy as np
import torch

REL_L2 = 1e-2
MAX_ABS = 3e-2


def to_np(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        return t.detach().to("cpu", torch.float64).numpy()
    return np.asarray(t, dtype=np.float64)


def errors(got, want):
    g, w = to_np(got), to_np(want)
    assert g.shape == w.shape, (g.shape, w.shape)
    assert np.all(np.isfinite(g)), "non-finite output"
    rel = float(np.linalg.norm(g - w) / max(np.linalg.norm(w), 1e-30))
    return rel, float(np.abs(g - w).max()) if g.size else 0.0


def assert_close(got, want, what="", rel_l2=REL_L2, max_abs=MAX_ABS):
    rel, mx = errors(got, want)
    assert rel <= rel_l2 and mx <= max_abs, f"{what}: rel-L2 {rel:.3e} (<= {rel_l2}), max-abs {mx:.3e} (<= {max_abs})"
    return rel, mx
