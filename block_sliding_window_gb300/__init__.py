"""GB300-native forward pass of MegaScale's parallel transformer block (PTB)
with causal sliding-window attention (SWA).

    y = x + MLP(LN(x)) + Attn(LN(x))       (MegaScale study notes, §2.2, PTB row)

Thin Python binding over the C ABI of libptb.so (include/ptb.h).  It only
marshals arguments: torch tensors provide device memory and the current
stream, and every step of the computation runs in the library's CUDA
kernels.  There is no fallback: if libptb.so is missing or cannot be
loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "PTBError", "load", "ptb_forward", "ptb_forward_events", "swa_attention",
    "swa_attention_strided", "swa_attention_counts", "layernorm", "gemm_qkv_up",
    "gemm_out_down", "gemm_workspace_size", "workspace_size", "release_workspace", "last_device_error",
    "wait_probe", "serial_forward", "serial_workspace_size", "prepare_fp8_weights",
    "fp8_workspace_size", "ptb_forward_fp8", "ptb_forward_fp8_events", "train_saved_size",
    "ptb_forward_train", "backward_workspace_size", "ptb_backward", "ptb_backward_events", "swa_attention_lse",
    "swa_attention_backward", "set_gemm_pairs", "host_workspace_size", "ptb_forward_host", "LIB_PATH", "SYMBOLS",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libptb.so")

_p = ctypes.c_void_p
_i64 = ctypes.c_int64
_i32 = ctypes.c_int32
_f32 = ctypes.c_float
_sz = ctypes.c_size_t
_st = ctypes.c_int

# Every entry point of include/ptb.h with its ctypes signature.
SYMBOLS = {
    "ptb_status_string": (ctypes.c_char_p, [_st]),
    "ptb_forward_workspace_size": (_sz, [_i64, _i64, _i64, _i64]),
    "ptb_forward": (_st, [_p] * 7 + [_i64] * 4 + [_i32, _i32, _p, _p, _sz, _p]),
    "ptb_forward_events": (_st, [_p] * 7 + [_i64] * 4 + [_i32, _i32, _p, _p, _sz, _p, _p, _i32]),
    "ptb_release_workspace": (_st, []),
    "ptb_serial_workspace_size": (_sz, [_i64, _i64, _i64, _i64]),
    "ptb_forward_fp8_workspace_size": (_sz, [_i64, _i64, _i64, _i64]),
    "ptb_prepare_fp8_weights": (_st, [_p] * 4 + [_i64, _i64] + [_p] * 4 + [_p]),
    "ptb_forward_fp8": (_st, [_p] * 7 + [_i64] * 4 + [_i32, _i32, _p, _p, _sz, _p]),
    "ptb_forward_fp8_events": (_st, [_p] * 7 + [_i64] * 4 + [_i32, _i32, _p, _p, _sz, _p, _p,
                                                             _i32]),
    "ptb_train_saved_size": (_sz, [_i64, _i64, _i64, _i64, _i32]),
    "ptb_forward_train": (_st, [_p] * 7 + [_i64] * 4 + [_i32, _i32, _p, _p, _sz, _p, _sz, _p]),
    "ptb_backward_workspace_size": (_sz, [_i64, _i64, _i64, _i64, _i32]),
    "ptb_backward": (_st, [_p] * 8 + [_sz] + [_i64] * 4 + [_i32, _i32] + [_p] * 8 + [_sz, _p]),
    "ptb_set_gemm_pairs": (_st, [_i32, _p]),
    "ptb_forward_host_workspace_size": (_sz, [_i64, _i64, _i64, _i64]),
    "ptb_forward_host": (_st, [_p] * 7 + [_i64] * 4 + [_i32, _i32, _p, _p, _sz, _p]),
    "ptb_backward_events": (_st, [_p] * 8 + [_sz] + [_i64] * 4 + [_i32, _i32] + [_p] * 8
                            + [_sz, _p, _p, _i32]),
    "swa_attention_lse": (_st, [_p, _p, _p, _i64, _i32, _i64, _i32, _i32, ctypes.c_float, _p, _p,
                                _p]),
    "swa_attention_backward": (_st, [_p] * 6 + [_i64, _i32, _i64, _i32, _i32, ctypes.c_float]
                               + [_p] * 5),
    "ptb_serial_forward": (_st, [_p] * 9 + [_i64] * 4 + [_i32, _i32, _p, _p, _sz, _p]),
    "ptb_forward_noalloc": (_st, [_p] * 7 + [_i64] * 4 + [_i32, _i32, _p, _p]),
    "swa_attention": (_st, [_p, _p, _p, _i64, _i32, _i64, _i32, _i32, _f32, _p, _p]),
    "swa_attention_strided": (_st, [_p, _i64, _i64, _i64] * 4 + [_i64, _i32, _i64, _i32, _i32, _f32, _p]),
    "swa_attention_counts": (_st, [_p, _p, _p, _i64, _i32, _i64, _i32, _i32, _f32, _p, _p, _p]),
    "ptb_layernorm": (_st, [_p, _p, _p, _i64, _i64, _f32, _p, _p]),
    "ptb_gemm_workspace_size": (_sz, [_i64, _i64, _i64]),
    "ptb_gemm_qkv_up": (_st, [_p, _p, _p, _i64, _i64, _i64, _p, _p, _sz, _p]),
    "ptb_gemm_out_down": (_st, [_p, _i64, _p, _i64, _p, _p, _p, _i64, _i64, _i64, _p, _p, _sz,
                                _p]),
    "ptb_last_device_error": (_st, [_p]),
    "ptb_wait_probe": (_st, [ctypes.c_uint64, _p]),
}

STATUS_NAMES = {0: "PTB_OK", 1: "PTB_ERR_ARG", 2: "PTB_ERR_SHAPE", 3: "PTB_ERR_ALIGN",
                4: "PTB_ERR_WORKSPACE", 5: "PTB_ERR_LAUNCH", 6: "PTB_ERR_TIMEOUT",
                7: "PTB_ERR_UNSUPPORTED", 8: "PTB_ERR_DEVICE"}

_lib = None


class PTBError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = _lib.ptb_status_string(status).decode() if _lib else STATUS_NAMES.get(status, "?")
        super().__init__(f"{where}: {msg}")


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libptb.so (once) and declares every entry point's signature."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SYMBOLS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(status: int, where: str) -> None:
    if status != 0:
        raise PTBError(status, where)


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _bf16_cuda(name: str, t: torch.Tensor, contiguous: bool = True) -> None:
    if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or not t.is_cuda:
        raise TypeError(f"{name} must be a bfloat16 CUDA tensor")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def workspace_size(batch: int, seq: int, hidden: int, ffn: int) -> int:
    return int(load().ptb_forward_workspace_size(batch, seq, hidden, ffn))


def _ptb_args(x, ln_gamma, ln_beta, w_qkv, w_o, w_up, w_down, heads, window, y, workspace):
    for n, t in (("x", x), ("ln_gamma", ln_gamma), ("ln_beta", ln_beta), ("w_qkv", w_qkv),
                 ("w_o", w_o), ("w_up", w_up), ("w_down", w_down)):
        _bf16_cuda(n, t)
    if x.dim() != 3:
        raise ValueError("x must be [batch, seq, hidden]")
    batch, seq, hidden = x.shape
    ffn = w_up.shape[0]
    if (tuple(w_qkv.shape) != (3 * hidden, hidden) or tuple(w_o.shape) != (hidden, hidden)
            or tuple(w_up.shape) != (ffn, hidden) or tuple(w_down.shape) != (hidden, ffn)
            or ln_gamma.numel() != hidden or ln_beta.numel() != hidden):
        raise ValueError("weight shapes do not match x")
    if y is None:
        y = torch.empty_like(x)
    _bf16_cuda("y", y)
    ws_bytes = 0
    if workspace is not None:
        if not workspace.is_cuda or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous CUDA tensor")
        ws_bytes = workspace.numel() * workspace.element_size()
    return (batch, seq, hidden, ffn), y, ws_bytes


def ptb_forward(x, ln_gamma, ln_beta, w_qkv, w_o, w_up, w_down, heads: int, window: int,
                y=None, workspace=None, stream=None) -> torch.Tensor:
    """y = x + Attn(LN(x)) + MLP(LN(x)) on the current device; returns y."""
    lib = load()
    (batch, seq, hidden, ffn), y, ws_bytes = _ptb_args(
        x, ln_gamma, ln_beta, w_qkv, w_o, w_up, w_down, heads, window, y, workspace)
    st = lib.ptb_forward(_ptr(x), _ptr(ln_gamma), _ptr(ln_beta), _ptr(w_qkv), _ptr(w_o),
                         _ptr(w_up), _ptr(w_down), batch, seq, hidden, ffn, heads, window,
                         _ptr(y), _ptr(workspace), ws_bytes, _stream(stream))
    _check(st, "ptb_forward")
    return y


def ptb_forward_events(x, ln_gamma, ln_beta, w_qkv, w_o, w_up, w_down, heads: int,
                       window: int, events, y=None, workspace=None, stream=None):
    """ptb_forward that also records 5 torch.cuda.Event objects at the kernel
    boundaries (before LN, GEMM1, SWA, GEMM2 and after GEMM2)."""
    lib = load()
    (batch, seq, hidden, ffn), y, ws_bytes = _ptb_args(
        x, ln_gamma, ln_beta, w_qkv, w_o, w_up, w_down, heads, window, y, workspace)
    if len(events) != 5:
        raise ValueError("need 5 events")
    st_obj = torch.cuda.current_stream() if stream is None else stream
    for ev in events:
        if not ev.cuda_event:  # torch creates the CUDA event on its first record
            ev.record(st_obj)
    handles = (ctypes.c_void_p * 5)(*[ev.cuda_event for ev in events])
    st = lib.ptb_forward_events(_ptr(x), _ptr(ln_gamma), _ptr(ln_beta), _ptr(w_qkv), _ptr(w_o),
                                _ptr(w_up), _ptr(w_down), batch, seq, hidden, ffn, heads, window,
                                _ptr(y), _ptr(workspace), ws_bytes, _stream(stream), handles, 5)
    _check(st, "ptb_forward_events")
    return y


def serial_workspace_size(batch: int, seq: int, hidden: int, ffn: int) -> int:
    return int(load().ptb_serial_workspace_size(batch, seq, hidden, ffn))


def serial_forward(x, ln1_gamma, ln1_beta, ln2_gamma, ln2_beta, w_qkv, w_o, w_up, w_down,
                   heads: int, window: int, y=None, workspace=None, stream=None):
    """The serial block h = x + Attn(LN1(x)), y = h + MLP(LN2(h)); returns y."""
    lib = load()
    (batch, seq, hidden, ffn), y, ws_bytes = _ptb_args(
        x, ln1_gamma, ln1_beta, w_qkv, w_o, w_up, w_down, heads, window, y, workspace)
    for n, t in (("ln2_gamma", ln2_gamma), ("ln2_beta", ln2_beta)):
        _bf16_cuda(n, t)
    st = lib.ptb_serial_forward(_ptr(x), _ptr(ln1_gamma), _ptr(ln1_beta), _ptr(ln2_gamma),
                                _ptr(ln2_beta), _ptr(w_qkv), _ptr(w_o), _ptr(w_up), _ptr(w_down),
                                batch, seq, hidden, ffn, heads, window, _ptr(y), _ptr(workspace),
                                ws_bytes, _stream(stream))
    _check(st, "ptb_serial_forward")
    return y


def prepare_fp8_weights(w_qkv, w_o, w_up, w_down, stream=None):
    """Quantizes the layer's weights to e4m3 with one scale per output row;
    returns (w1 [3H+F, H] uint8, s1 [3H+F] f32, w2 [H, H+F] uint8, s2 [H] f32)."""
    lib = load()
    for n, t in (("w_qkv", w_qkv), ("w_o", w_o), ("w_up", w_up), ("w_down", w_down)):
        _bf16_cuda(n, t)
    hidden, ffn = w_o.shape[0], w_up.shape[0]
    dev = w_o.device
    w1 = torch.empty(3 * hidden + ffn, hidden, dtype=torch.uint8, device=dev)
    s1 = torch.empty(3 * hidden + ffn, dtype=torch.float32, device=dev)
    w2 = torch.empty(hidden, hidden + ffn, dtype=torch.uint8, device=dev)
    s2 = torch.empty(hidden, dtype=torch.float32, device=dev)
    st = lib.ptb_prepare_fp8_weights(_ptr(w_qkv), _ptr(w_o), _ptr(w_up), _ptr(w_down), hidden,
                                     ffn, _ptr(w1), _ptr(s1), _ptr(w2), _ptr(s2), _stream(stream))
    _check(st, "ptb_prepare_fp8_weights")
    return w1, s1, w2, s2


def fp8_workspace_size(batch: int, seq: int, hidden: int, ffn: int) -> int:
    return int(load().ptb_forward_fp8_workspace_size(batch, seq, hidden, ffn))


def _fp8_layer(x, ln_gamma, ln_beta, fp8_weights, heads, window, y, workspace, stream, events):
    lib = load()
    w1, s1, w2, s2 = fp8_weights
    for n, t in (("x", x), ("ln_gamma", ln_gamma), ("ln_beta", ln_beta)):
        _bf16_cuda(n, t)
    batch, seq, hidden = x.shape
    ffn = w2.shape[1] - hidden
    for n, t, dt, shape in (("w1", w1, torch.uint8, (3 * hidden + ffn, hidden)),
                            ("s1", s1, torch.float32, (3 * hidden + ffn,)),
                            ("w2", w2, torch.uint8, (hidden, hidden + ffn)),
                            ("s2", s2, torch.float32, (hidden,))):
        if t.dtype != dt or tuple(t.shape) != shape or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous CUDA {dt} tensor of shape {shape}")
    if y is None:
        y = torch.empty_like(x)
    ws_bytes = 0
    if workspace is not None:
        ws_bytes = workspace.numel() * workspace.element_size()
    args = (_ptr(x), _ptr(ln_gamma), _ptr(ln_beta), _ptr(w1), _ptr(s1), _ptr(w2), _ptr(s2), batch,
            seq, hidden, ffn, heads, window, _ptr(y), _ptr(workspace), ws_bytes, _stream(stream))
    if events is None:
        _check(lib.ptb_forward_fp8(*args), "ptb_forward_fp8")
        return y
    if len(events) != 6:
        raise ValueError("need 6 events")
    st_obj = torch.cuda.current_stream() if stream is None else stream
    for ev in events:
        if not ev.cuda_event:  # torch creates the CUDA event on its first record
            ev.record(st_obj)
    handles = (ctypes.c_void_p * 6)(*[ev.cuda_event for ev in events])
    _check(lib.ptb_forward_fp8_events(*args, handles, 6), "ptb_forward_fp8_events")
    return y


def ptb_forward_fp8(x, ln_gamma, ln_beta, fp8_weights, heads: int, window: int, y=None,
                    workspace=None, stream=None):
    """The layer with e4m3 GEMM operands; fp8_weights from prepare_fp8_weights."""
    return _fp8_layer(x, ln_gamma, ln_beta, fp8_weights, heads, window, y, workspace, stream,
                      None)


def ptb_forward_fp8_events(x, ln_gamma, ln_beta, fp8_weights, heads: int, window: int, events,
                           y=None, workspace=None, stream=None):
    """ptb_forward_fp8 that also records 6 torch.cuda.Event objects at the
    kernel boundaries (before LN+quantize, GEMM1, SWA, quantize, GEMM2 and
    after GEMM2)."""
    return _fp8_layer(x, ln_gamma, ln_beta, fp8_weights, heads, window, y, workspace, stream,
                      events)


def swa_attention(q, k, v, window: int, scale: float = 0.0, o=None, stream=None):
    """Causal sliding-window attention over [B, heads, s, d] bf16 tensors."""
    lib = load()
    for n, t in (("q", q), ("k", k), ("v", v)):
        _bf16_cuda(n, t)
    if q.dim() != 4 or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must be [batch, heads, seq, head_dim] of one shape")
    if o is None:
        o = torch.empty_like(q)
    _bf16_cuda("o", o)
    b, h, s, d = q.shape
    st = lib.swa_attention(_ptr(q), _ptr(k), _ptr(v), b, h, s, d, window, scale, _ptr(o),
                           _stream(stream))
    _check(st, "swa_attention")
    return o


def swa_attention_strided(q, k, v, o, window: int, scale: float = 0.0, stream=None):
    """SWA on strided [B, heads, s, d] views (last dim contiguous)."""
    lib = load()
    args = []
    for n, t in (("q", q), ("k", k), ("v", v), ("o", o)):
        _bf16_cuda(n, t, contiguous=False)
        if t.dim() != 4 or t.stride(3) != 1:
            raise ValueError(f"{n} must be 4-D with a contiguous last dimension")
        args += [_ptr(t), t.stride(0), t.stride(1), t.stride(2)]
    b, h, s, d = q.shape
    st = lib.swa_attention_strided(*args, b, h, s, d, window, scale, _stream(stream))
    _check(st, "swa_attention_strided")
    return o


def swa_attention_counts(q, k, v, window: int, scale: float = 0.0, stream=None):
    """Runs the attention kernel with its per-row attended-key counter on;
    returns (o, counts[B, heads, s] int32)."""
    lib = load()
    for n, t in (("q", q), ("k", k), ("v", v)):
        _bf16_cuda(n, t)
    b, h, s, d = q.shape
    o = torch.empty_like(q)
    counts = torch.full((b, h, s), -1, dtype=torch.int32, device=q.device)
    st = lib.swa_attention_counts(_ptr(q), _ptr(k), _ptr(v), b, h, s, d, window, scale,
                                  _ptr(o), _ptr(counts), _stream(stream))
    _check(st, "swa_attention_counts")
    return o, counts


def host_workspace_size(batch: int, seq: int, hidden: int, ffn: int) -> int:
    return int(load().ptb_forward_host_workspace_size(batch, seq, hidden, ffn))


def ptb_forward_host(x_host, ln_gamma, ln_beta, w_qkv, w_o, w_up, w_down, heads: int,
                     window: int, y_host, workspace, stream=None):
    """The layer on host-memory x and y (pinned CPU bf16 tensors) with device
    parameters: enqueues H2D, the layer and D2H on the stream and returns
    without waiting."""
    lib = load()
    for n, t in (("x_host", x_host), ("y_host", y_host)):
        if t.dtype != torch.bfloat16 or t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous host bf16 tensor")
    if tuple(y_host.shape) != tuple(x_host.shape) or x_host.dim() != 3:
        raise ValueError("x_host and y_host must be [batch, seq, hidden] of one shape")
    for n, t in (("ln_gamma", ln_gamma), ("ln_beta", ln_beta), ("w_qkv", w_qkv), ("w_o", w_o),
                 ("w_up", w_up), ("w_down", w_down)):
        _bf16_cuda(n, t)
    batch, seq, hidden = x_host.shape
    ffn = w_up.shape[0]
    ws_bytes = workspace.numel() * workspace.element_size()
    st = lib.ptb_forward_host(_ptr(x_host), _ptr(ln_gamma), _ptr(ln_beta), _ptr(w_qkv), _ptr(w_o),
                              _ptr(w_up), _ptr(w_down), batch, seq, hidden, ffn, heads, window,
                              _ptr(y_host), _ptr(workspace), ws_bytes, _stream(stream))
    _check(st, "ptb_forward_host")
    return y_host


def set_gemm_pairs(mode: int) -> int:
    """GEMM tile mode on the current device: 1 CTA pairs (256 x 256 tiles), 0
    single CTAs, -1 automatic; returns the previous mode."""
    prev = ctypes.c_int32(0)
    _check(load().ptb_set_gemm_pairs(mode, ctypes.byref(prev)), "ptb_set_gemm_pairs")
    return prev.value


def train_saved_size(batch: int, seq: int, hidden: int, ffn: int, heads: int) -> int:
    return int(load().ptb_train_saved_size(batch, seq, hidden, ffn, heads))


def backward_workspace_size(batch: int, seq: int, hidden: int, ffn: int, heads: int) -> int:
    return int(load().ptb_backward_workspace_size(batch, seq, hidden, ffn, heads))


def ptb_forward_train(x, ln_gamma, ln_beta, w_qkv, w_o, w_up, w_down, heads: int, window: int,
                      y=None, saved=None, workspace=None, stream=None):
    """The layer forward that also keeps what ptb_backward needs; returns
    (y, saved) with saved a uint8 CUDA tensor owned by the caller."""
    lib = load()
    (batch, seq, hidden, ffn), y, ws_bytes = _ptb_args(
        x, ln_gamma, ln_beta, w_qkv, w_o, w_up, w_down, heads, window, y, workspace)
    need = train_saved_size(batch, seq, hidden, ffn, heads)
    if saved is None:
        saved = torch.empty(need, dtype=torch.uint8, device=x.device)
    st = lib.ptb_forward_train(_ptr(x), _ptr(ln_gamma), _ptr(ln_beta), _ptr(w_qkv), _ptr(w_o),
                               _ptr(w_up), _ptr(w_down), batch, seq, hidden, ffn, heads, window,
                               _ptr(y), _ptr(saved), saved.numel(), _ptr(workspace), ws_bytes,
                               _stream(stream))
    _check(st, "ptb_forward_train")
    return y, saved


def ptb_backward(dy, x, ln_gamma, w_qkv, w_o, w_up, w_down, saved, heads: int, window: int,
                 grads=None, workspace=None, stream=None) -> dict:
    """Gradients of the layer for upstream dy: dx (bf16) and fp32 dln_gamma,
    dln_beta, dw_qkv, dw_o, dw_up, dw_down, returned as a dict (or written
    into `grads`, a dict of preallocated tensors with those keys)."""
    return _backward(dy, x, ln_gamma, w_qkv, w_o, w_up, w_down, saved, heads, window, grads,
                     workspace, stream, None)


def ptb_backward_events(dy, x, ln_gamma, w_qkv, w_o, w_up, w_down, saved, heads: int,
                        window: int, events, grads=None, workspace=None, stream=None) -> dict:
    """ptb_backward that also records 7 torch.cuda.Event objects at its
    kernel boundaries (see the C declaration)."""
    return _backward(dy, x, ln_gamma, w_qkv, w_o, w_up, w_down, saved, heads, window, grads,
                     workspace, stream, events)


def _backward(dy, x, ln_gamma, w_qkv, w_o, w_up, w_down, saved, heads, window, grads, workspace,
              stream, events):
    lib = load()
    (batch, seq, hidden, ffn), _, ws_bytes = _ptb_args(
        x, ln_gamma, ln_gamma, w_qkv, w_o, w_up, w_down, heads, window, dy, workspace)
    if tuple(dy.shape) != tuple(x.shape):
        raise ValueError("dy must have the shape of x")
    if grads is None:
        dev, f32 = x.device, torch.float32
        grads = dict(dx=torch.empty_like(x),
                     dln_gamma=torch.empty(hidden, dtype=f32, device=dev),
                     dln_beta=torch.empty(hidden, dtype=f32, device=dev),
                     dw_qkv=torch.empty(3 * hidden, hidden, dtype=f32, device=dev),
                     dw_o=torch.empty(hidden, hidden, dtype=f32, device=dev),
                     dw_up=torch.empty(ffn, hidden, dtype=f32, device=dev),
                     dw_down=torch.empty(hidden, ffn, dtype=f32, device=dev))
    g = grads
    args = (_ptr(dy), _ptr(x), _ptr(ln_gamma), _ptr(w_qkv), _ptr(w_o), _ptr(w_up), _ptr(w_down),
            _ptr(saved), saved.numel(), batch, seq, hidden, ffn, heads, window, _ptr(g["dx"]),
            _ptr(g["dln_gamma"]), _ptr(g["dln_beta"]), _ptr(g["dw_qkv"]), _ptr(g["dw_o"]),
            _ptr(g["dw_up"]), _ptr(g["dw_down"]), _ptr(workspace), ws_bytes, _stream(stream))
    if events is None:
        _check(lib.ptb_backward(*args), "ptb_backward")
        return g
    if len(events) != 7:
        raise ValueError("need 7 events")
    st_obj = torch.cuda.current_stream() if stream is None else stream
    for ev in events:
        if not ev.cuda_event:  # torch creates the CUDA event on its first record
            ev.record(st_obj)
    handles = (ctypes.c_void_p * 7)(*[ev.cuda_event for ev in events])
    _check(lib.ptb_backward_events(*args, handles, 7), "ptb_backward_events")
    return g


def swa_attention_lse(q, k, v, window: int, scale: float = 0.0, stream=None):
    """swa_attention that also returns the per-row base-2 log-sum-exp:
    (o, lse[B, heads, s] fp32)."""
    lib = load()
    for n, t in (("q", q), ("k", k), ("v", v)):
        _bf16_cuda(n, t)
    b, h, s, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((b, h, s), dtype=torch.float32, device=q.device)
    st = lib.swa_attention_lse(_ptr(q), _ptr(k), _ptr(v), b, h, s, d, window, scale, _ptr(o),
                               _ptr(lse), _stream(stream))
    _check(st, "swa_attention_lse")
    return o, lse


def swa_attention_backward(q, k, v, o, dout, lse, window: int, scale: float = 0.0, stream=None):
    """Gradients (dq, dk, dv) of swa_attention for the upstream dout."""
    lib = load()
    for n, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout)):
        _bf16_cuda(n, t)
    b, h, s, d = q.shape
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    delta = torch.empty((b, h, s), dtype=torch.float32, device=q.device)
    st = lib.swa_attention_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), b,
                                    h, s, d, window, scale, _ptr(dq), _ptr(dk), _ptr(dv),
                                    _ptr(delta), _stream(stream))
    _check(st, "swa_attention_backward")
    return dq, dk, dv


def layernorm(x, gamma, beta, eps: float = 1e-5, out=None, stream=None):
    lib = load()
    _bf16_cuda("x", x)
    hidden = x.shape[-1]
    rows = x.numel() // hidden
    if out is None:
        out = torch.empty_like(x)
    st = lib.ptb_layernorm(_ptr(x), _ptr(gamma), _ptr(beta), rows, hidden, eps, _ptr(out),
                           _stream(stream))
    _check(st, "ptb_layernorm")
    return out


def gemm_workspace_size(tokens: int, hidden: int, ffn: int) -> int:
    return int(load().ptb_gemm_workspace_size(tokens, hidden, ffn))


def _ws(workspace):
    if workspace is None:
        return None, 0
    if not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    return workspace.data_ptr(), workspace.numel() * workspace.element_size()


def gemm_qkv_up(xn, w_qkv, w_up, u=None, workspace=None, stream=None):
    """u = [xn w_qkv^T | gelu_tanh(xn w_up^T)] for xn [T, H]."""
    lib = load()
    tokens, hidden = xn.shape
    ffn = w_up.shape[0]
    if u is None:
        u = torch.empty(tokens, 3 * hidden + ffn, dtype=torch.bfloat16, device=xn.device)
    ws, ws_bytes = _ws(workspace)
    st = lib.ptb_gemm_qkv_up(_ptr(xn), _ptr(w_qkv), _ptr(w_up), tokens, hidden, ffn, _ptr(u),
                             ws, ws_bytes, _stream(stream))
    _check(st, "ptb_gemm_qkv_up")
    return u


def gemm_out_down(ctx, g, w_o, w_down, x, y=None, workspace=None, stream=None):
    """y = x + ctx w_o^T + g w_down^T (ctx, g may be row-strided views)."""
    lib = load()
    tokens, hidden = x.shape
    ffn = w_down.shape[1]
    if y is None:
        y = torch.empty_like(x)
    ws, ws_bytes = _ws(workspace)
    st = lib.ptb_gemm_out_down(_ptr(ctx), ctx.stride(0), _ptr(g), g.stride(0), _ptr(w_o),
                               _ptr(w_down), _ptr(x), tokens, hidden, ffn, _ptr(y), ws, ws_bytes,
                               _stream(stream))
    _check(st, "ptb_gemm_out_down")
    return y


def release_workspace() -> None:
    _check(load().ptb_release_workspace(), "ptb_release_workspace")


def last_device_error(stream=None) -> int:
    """Waits for `stream` (default: the current stream) and returns (and
    clears) the kernels' device status word."""
    return int(load().ptb_last_device_error(_stream(stream)))


def wait_probe(limit_ns: int, stream=None) -> None:
    _check(load().ptb_wait_probe(limit_ns, _stream(stream)), "ptb_wait_probe")
