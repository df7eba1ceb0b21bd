"""The allocation-free variant of the layer forward pass, through the C ABI.

ptb_forward_noalloc serves callers that cannot allocate device memory (their
framework or server owns all of it, or forbids cudaMalloc after start-up):
it runs the same kernels as ptb_forward with a fixed scratch array compiled
into the library.  Its output must be the same bits as ptb_forward's on the same inputs, call
after call (the shared array keeps the previous call's contents), a call must
leave the device's free memory unchanged, and layers that need more than the
array's 64 MiB must be refused up front.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test.
"""
import pytest
import torch

from block_sliding_window_gb300 import workloads

pytestmark = pytest.mark.gpu

LAYERS = [
    workloads.PTB_CONFIGS["tiny"],
    workloads.small_ptb(2, 300, 256, 4, 1024, 100, seed=21),
    workloads.small_ptb(1, 2048, 1024, 8, 4096, 512, seed=27),
]


def _noalloc(lib, d, cfg, y):
    return lib.ptb_forward_noalloc(
        d["x"].data_ptr(), d["ln_gamma"].data_ptr(), d["ln_beta"].data_ptr(),
        d["w_qkv"].data_ptr(), d["w_o"].data_ptr(), d["w_up"].data_ptr(), d["w_down"].data_ptr(),
        cfg.batch, cfg.seq, cfg.hidden, cfg.ffn, cfg.heads, cfg.window, y.data_ptr(),
        torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("cfg", LAYERS, ids=lambda c: c.name)
def test_noalloc_matches_ptb_forward_twice(ptb_lib, cfg):
    """Both entry points run the same kernels on the same inputs, so the
    outputs must be the same bits; two calls in a row also show that nothing
    depends on what the previous call left in the shared array."""
    lib = ptb_lib.load()
    d = {k: v.cuda() for k, v in workloads.ptb_inputs(cfg).items()}
    want = ptb_lib.ptb_forward(d["x"], d["ln_gamma"], d["ln_beta"], d["w_qkv"], d["w_o"],
                               d["w_up"], d["w_down"], cfg.heads, cfg.window)
    for call in range(2):
        y = torch.full_like(d["x"], float("nan"))
        assert _noalloc(lib, d, cfg, y) == 0
        torch.cuda.synchronize()
        assert torch.equal(y, want), f"{cfg.name}: no-alloc call {call} differs from ptb_forward"
    assert lib.ptb_last_device_error(torch.cuda.current_stream().cuda_stream) == 0


def test_noalloc_takes_no_device_memory(ptb_lib):
    """With the library's own arena released, calls of the entry point leave
    the device's free memory unchanged: it allocates nothing, not even
    through the arena."""
    lib = ptb_lib.load()
    cfg = LAYERS[-1]
    d = {k: v.cuda() for k, v in workloads.ptb_inputs(cfg).items()}
    ys = [torch.empty_like(d["x"]) for _ in range(3)]
    assert _noalloc(lib, d, cfg, ys[0]) == 0  # first call: the array's address is looked up
    torch.cuda.synchronize()
    ptb_lib.release_workspace()
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    for y in ys:
        assert _noalloc(lib, d, cfg, y) == 0
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after == free_before, f"free device memory moved by {free_before - free_after} B"
    assert torch.equal(ys[1], ys[0]) and torch.equal(ys[2], ys[0])


def test_noalloc_refuses_layers_beyond_its_scratch(ptb_lib):
    lib = ptb_lib.load()
    cfg = workloads.PTB_CONFIGS["13b"]  # needs about 168 MB of scratch
    assert ptb_lib.workspace_size(cfg.batch, cfg.seq, cfg.hidden, cfg.ffn) > 64 << 20
    t = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    p = t.data_ptr()
    st = lib.ptb_forward_noalloc(p, p, p, p, p, p, p, cfg.batch, cfg.seq, cfg.hidden, cfg.ffn,
                                 cfg.heads, cfg.window, p, torch.cuda.current_stream().cuda_stream)
    assert ptb_lib.STATUS_NAMES[st] == "PTB_ERR_WORKSPACE"
