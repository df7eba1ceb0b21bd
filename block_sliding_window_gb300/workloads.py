"""Seeded synthetic workloads for the PTB + SWA forward pass.

This module holds the workload shapes and the seeded input generators, and
nothing of the method's arithmetic.  It is the one piece of code that feeds
both the CUDA path and the fp64 oracle (the tests pass the same bf16 tensors
to each side).

Shapes follow the pages' models (MegaScale study notes, §2.5 (paper §6.1),
Table 1: 175B = hidden 12288 with 128 heads, 530B = hidden 20480 with 160 heads,
sequence length 2048) plus a 13B-class layer, a tiny layer and the SWA
operator on its own.  Values are synthetic: x ~ N(0, 1), weights ~ N(0, std),
LayerNorm gamma = 1 and beta = 0, drawn in fp32 from a seeded torch generator
and rounded to bf16, so both sides see identical bf16 bits.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class PTBConfig:
    name: str
    batch: int
    seq: int
    hidden: int
    heads: int
    ffn: int
    window: int
    w_std: float
    seed: int

    @property
    def tokens(self) -> int:
        return self.batch * self.seq

    @property
    def head_dim(self) -> int:
        return self.hidden // self.heads

    def with_window(self, window: int) -> "PTBConfig":
        return replace(self, window=window, name=f"{self.name}_w{window}")


@dataclass(frozen=True)
class SWAConfig:
    name: str
    batch: int
    heads: int
    seq: int
    head_dim: int
    window: int
    seed: int


PTB_CONFIGS = {
    # MLP 64 -> 256 -> 64, 4 heads x 16, window 32 (and 128 = full causal).
    "tiny": PTBConfig("tiny", 1, 128, 64, 4, 256, 32, 0.02, 0),
    # 13B-class layer: 40 heads x 128, MLP 4H.
    "13b": PTBConfig("13b", 1, 2048, 5120, 40, 20480, 512, 0.02, 1),
    # 175B shape of Table 1: 128 heads x 96, MLP 4H.
    "175b": PTBConfig("175b", 1, 2048, 12288, 128, 49152, 1024, 0.006, 2),
    # 530B shape of Table 1: 160 heads x 128, MLP 4H (about 10 GB of bf16 weights).
    "530b": PTBConfig("530b", 1, 2048, 20480, 160, 81920, 512, 0.005, 3),
}

SWA_CONFIGS = {
    "swa": SWAConfig("swa", 4, 16, 2048, 128, 512, 0),
}


def _normal(gen: torch.Generator, shape, std: float, device) -> torch.Tensor:
    t = torch.randn(*shape, generator=gen, dtype=torch.float32, device=device)
    if std != 1.0:
        t.mul_(std)
    return t.to(torch.bfloat16)


def _generator(seed: int, device) -> torch.Generator:
    return torch.Generator(device=str(torch.device(device))).manual_seed(seed)


def ptb_inputs(cfg: PTBConfig, device="cpu") -> dict:
    """bf16 inputs of one PTB layer, drawn in a fixed order from `cfg.seed`.

    Returns x [B, s, H], ln_gamma [H] (ones), ln_beta [H] (zeros) and the
    nn.Linear-form weights w_qkv [3H, H], w_o [H, H], w_up [F, H],
    w_down [H, F].  The same seed gives the same bits for a given device
    type; the tests give the oracle a host copy of whatever was drawn."""
    g = _generator(cfg.seed, device)
    h, f = cfg.hidden, cfg.ffn
    x = _normal(g, (cfg.batch, cfg.seq, h), 1.0, device)
    w_qkv = _normal(g, (3 * h, h), cfg.w_std, device)
    w_o = _normal(g, (h, h), cfg.w_std, device)
    w_up = _normal(g, (f, h), cfg.w_std, device)
    w_down = _normal(g, (h, f), cfg.w_std, device)
    ones = torch.ones(h, dtype=torch.bfloat16, device=device)
    zeros = torch.zeros(h, dtype=torch.bfloat16, device=device)
    return {"x": x, "ln_gamma": ones, "ln_beta": zeros, "w_qkv": w_qkv,
            "w_o": w_o, "w_up": w_up, "w_down": w_down}


def swa_inputs(batch: int, heads: int, seq: int, head_dim: int, seed: int,
               device="cpu", std: float = 1.0):
    """q, k, v as bf16 [B, heads, s, d] tensors drawn from N(0, std^2)."""
    g = _generator(seed, device)
    shape = (batch, heads, seq, head_dim)
    return tuple(_normal(g, shape, std, device) for _ in range(3))


def normal_bf16(shape, seed: int, std: float = 1.0, mean: float = 0.0,
                device="cpu") -> torch.Tensor:
    """One seeded N(mean, std^2) tensor rounded to bf16."""
    t = torch.randn(*shape, generator=_generator(seed, device), dtype=torch.float32,
                    device=device)
    return (t * std + mean).to(torch.bfloat16)


def sample_rows(seq: int, window: int, tile: int = 128) -> list:
    """Sequence positions checked one by one on the full-size layers.

    The first rows, the edges around 64 and 128, the window edge and the last
    rows, plus one row inside every `tile`-row block of the sequence (the
    GEMMs' M tiles and the attention's query tiles are 128 rows).  The row
    inside block t sits at offset (37 t + 17) mod tile, so successive blocks
    probe different 32-row quarters (different TMEM lane groups)."""
    cand = {0, 1, 2, 63, 64, 127, 128, 129, window - 1, window, window + 1,
            seq // 2, seq - 2, seq - 1}
    for t in range((seq + tile - 1) // tile):
        cand.add(t * tile + (37 * t + 17) % tile)
    return sorted(r for r in cand if 0 <= r < seq)


def small_ptb(batch: int, seq: int, hidden: int, heads: int, ffn: int,
              window: int, seed: int, w_std: float = 0.02) -> PTBConfig:
    """An ad-hoc layer shape for the tile-edge parity cases.  Weights use the
    same N(0, 0.02^2) as the tiny and 13B-class workloads, which keeps |y|
    below 8, where one bf16 ulp of the output is 2^-5."""
    return PTBConfig(f"b{batch}s{seq}h{hidden}n{heads}f{ffn}w{window}", batch,
                     seq, hidden, heads, ffn, window, w_std, seed)
