"""fp64 CPU oracle for the PTB + causal SWA forward and backward passes.

TEST INFRASTRUCTURE ONLY: imported by the tests, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``; never by the product package.
"""
from .backward import (  # noqa: F401
    backward_flops, gelu_tanh_grad, layer_norm_backward, ptb_backward, swa_backward,
)
from .ptb_oracle import (  # noqa: F401
    LN_EPS, attended_counts, attention_branch, band_mask, gelu_tanh,
    layer_flops, layer_norm, linear, mfu, mlp_branch, needed_key_positions,
    ptb_forward, serial_block, swa, swa_weights,
)
