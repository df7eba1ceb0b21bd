"""CPU checks that tie the measurement and the full-size parity sampling to
pinned definitions.

* The benchmark's FLOP accounting (bench.layer_flops / bench.backward_flops)
  must equal the oracle's pinned layer_flops / backward_flops (MegaScale
  study notes, §2.1, MFU definition: model FLOPs over peak) on every
  workload, so every TFLOP/s and roofline fraction the benchmark prints rests
  on the pinned arithmetic.
* The rows the full-size parity tests compare must fall in every 128-row
  tile of the sequence (every M tile of the GEMMs, every query tile of the
  attention), in all four 32-row quarters of a tile across the sample.
"""
import pytest

import bench
import oracle
from block_sliding_window_gb300 import workloads


@pytest.mark.parametrize("name", sorted(workloads.PTB_CONFIGS))
def test_bench_forward_flops_equal_the_oracle(name):
    cfg = workloads.PTB_CONFIGS[name]
    got = bench.layer_flops(cfg)
    want = oracle.layer_flops(cfg.batch, cfg.seq, cfg.hidden, cfg.ffn, cfg.window)
    assert got["gemm1"] + got["gemm2"] == want["gemm"]
    assert got["attn"] == want["attn"]
    assert got["total"] == want["total"]
    assert got["band_keys"] == cfg.batch * cfg.heads * want["band_keys"]


@pytest.mark.parametrize("name", sorted(workloads.PTB_CONFIGS))
def test_bench_backward_flops_equal_the_oracle(name):
    cfg = workloads.PTB_CONFIGS[name]
    got = bench.backward_flops(cfg)
    want = oracle.backward_flops(cfg.batch, cfg.seq, cfg.hidden, cfg.ffn, cfg.window)
    gemm = got["dgrad_out"] + got["wgrad_out"] + got["dgrad_in"] + got["wgrad_in"]
    assert gemm == want["gemm"]
    assert got["attn"] == want["attn"]
    assert got["total"] == want["total"]


def test_bench_swa_operator_flops_equal_the_oracle():
    """The SWA operator line counts 4 d FLOPs per in-band (query, key) pair."""
    cfg = workloads.SWA_CONFIGS["swa"]
    band = int(oracle.attended_counts(cfg.seq, cfg.window).sum())
    assert bench.swa_flops(cfg) == 4 * cfg.batch * cfg.heads * cfg.head_dim * band


@pytest.mark.parametrize("name", ["13b", "175b", "530b"])
def test_sampled_rows_cover_every_tile(name):
    cfg = workloads.PTB_CONFIGS[name]
    rows = workloads.sample_rows(cfg.seq, cfg.window)
    assert rows == sorted(set(rows)) and 0 <= rows[0] and rows[-1] < cfg.seq
    assert {r // 128 for r in rows} == set(range((cfg.seq + 127) // 128))
    assert {(r % 128) // 32 for r in rows} == {0, 1, 2, 3}
    for r in (0, cfg.seq - 1, cfg.window - 1, cfg.window):
        assert r in rows


def test_sampled_rows_ragged_sequence():
    rows = workloads.sample_rows(300, 100)
    assert {r // 128 for r in rows} == {0, 1, 2}
    assert max(rows) == 299
