"""Thin Python binding over libnrc.so (include/nrc.h), same names as the C ABI.

Argument marshalling only: torch tensors become device pointers, the current
torch stream becomes the ``stream`` argument, outputs and workspaces are
allocated with torch.  Every step of every block runs in the library's CUDA
kernels; there is no CPU fallback -- if the library is not built, or no GPU
is present, the calls raise.

Host (CPU) input tensors are accepted for end-to-end use.  The pre-norm block
hands them to the library's host-buffer entry point, which pipelines the copies
with the GPU work (pinned memory lets them overlap); the other blocks copy them
to the current device before the call.  The result comes back in host memory,
ready when the call returns.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

NRC_OK, NRC_ERR_INVALID_ARG, NRC_ERR_UNSUPPORTED = 0, 1, 2
NRC_ERR_ALIGNMENT, NRC_ERR_WORKSPACE, NRC_ERR_CUDA, NRC_ERR_TIMEOUT = 3, 4, 5, 6
NRC_F32, NRC_BF16 = 0, 1

_lib = None


class NrcError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


def lib_path() -> str:
    return _build.LIB_PATH


def load() -> ctypes.CDLL:
    """Load libnrc.so (built by ``build.build()``); raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    path = lib_path()
    if not os.path.exists(path):
        raise RuntimeError(f"libnrc.so not built ({path}); run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    p, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    u64 = ctypes.c_uint64
    sig = {
        "nrc_status_string": ([i], ctypes.c_char_p),
        "nrc_version": ([], i),
        "nrc_prenorm_dilconv_residual_workspace_size": ([i, i], sz),
        "nrc_prenorm_dilconv_residual": ([p, p, i, i, i, i, i, i, i, p, p, p, p, f, p, p, p, sz,
                                          p], i),
        "nrc_prenorm_dilconv_residual_train_workspace_size": ([i, i, i, i], sz),
        "nrc_prenorm_dilconv_residual_train": ([p, p, i, i, i, i, i, i, i, p, p, p, p, p, f, f, p,
                                                p, p, sz, p], i),
        "nrc_prenorm_dilconv_residual_train_host_workspace_size": ([i, i, i, i, i], sz),
        "nrc_prenorm_dilconv_residual_train_host": ([p, p, i, i, i, i, i, i, i, p, p, p, p, p, f,
                                                     f, p, p, i, p, sz, p], i),
        "nrc_prenorm_dilconv_residual_host_workspace_size": ([i, i, i, i, i], sz),
        "nrc_prenorm_dilconv_residual_host": ([p, p, i, i, i, i, i, i, i, p, p, p, p, f, p, p, i,
                                               p, sz, p], i),
        "nrc_prenorm_dilconv_residual_noalloc_max_bytes": ([], sz),
        "nrc_prenorm_dilconv_residual_noalloc": ([p, p, i, i, i, i, i, i, i, p, p, p, p, f, p, p,
                                                  p], i),
        "nrc_conv1d_output_length": ([i, i, i, i, i], i),
        "nrc_conv1d_groupnorm_workspace_size": ([i, i, i, i, i, i, i, i, i], sz),
        "nrc_conv1d_groupnorm": ([p, p, i, i, i, i, i, i, i, i, p, p, i, p, p, f, p, sz, p], i),
        "nrc_conv1d_groupnorm_host_workspace_size": ([i, i, i, i, i, i, i, i, i, i], sz),
        "nrc_conv1d_groupnorm_host": ([p, p, i, i, i, i, i, i, i, i, p, p, i, p, p, f, i, p, sz,
                                       p], i),
        "nrc_linear_bn_swish_workspace_size": ([i, i, i], sz),
        "nrc_linear_bn_swish": ([p, p, i, i, i, p, p, p, p, p, p, p, f, f, i, p, f, p, sz, p], i),
        "nrc_linear_bn_swish_host_workspace_size": ([i, i, i, i], sz),
        "nrc_linear_bn_swish_host": ([p, p, i, i, i, p, p, p, p, p, p, p, f, f, i, p, f, i, p, sz,
                                      p], i),
        "nrc_query_status": ([p], i),
        "nrc_last_error_site": ([], i),
        "nrc_set_wait_timeout_ns": ([u64], None),
        "nrc_set_grid_barrier_timeout_ns": ([u64], None),
        "nrc_selftest_wait_timeout": ([u64, p], i),
        "nrc_trace_enable": ([i], None),
        "nrc_trace_count": ([], i),
        "nrc_trace_get": ([i, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(f)], i),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().nrc_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != NRC_OK:
        raise NrcError(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dev(t, device, dtype=None):
    """Device copy of an optional tensor (contiguous, given dtype)."""
    if t is None:
        return None
    t = t.to(device=device, dtype=dtype or t.dtype, non_blocking=True)
    return t.contiguous()


def _workspace(nbytes, device, workspace):
    if workspace is not None:
        if workspace.numel() * workspace.element_size() < nbytes:
            raise ValueError("workspace too small")
        return workspace
    return torch.empty(max(int(nbytes), 1), dtype=torch.uint8, device=device)


def _target_device(x):
    if x.is_cuda:
        return x.device
    if not torch.cuda.is_available():
        raise RuntimeError("nrc needs a CUDA device (no CPU fallback)")
    return torch.device("cuda", torch.cuda.current_device())


# ---------------------------------------------------------------------------
# Pre-norm residual block
# ---------------------------------------------------------------------------
def prenorm_dilconv_residual_workspace_size(C: int, dtype=torch.float32) -> int:
    dt = NRC_F32 if dtype == torch.float32 else NRC_BF16
    return int(load().nrc_prenorm_dilconv_residual_workspace_size(C, dt))


def prenorm_dilconv_residual(x, bn_running_mean, bn_running_var, bn_gamma, bn_beta, bn_eps,
                             conv_weight, conv_bias, dilation, padding=None, kernel_size=3,
                             out=None, workspace=None, stream=None, chunk_n=None):
    """out = x + Conv1d(ReLU(BatchNorm1d_eval(x))) with k=3, padding=dilation.

    x (N, C, L) fp32 or bf16; BN tensors (C) fp32; conv_weight (C, C, 3) and
    conv_bias (C) in x's dtype (bias may be None).  With x in host memory the
    result is a host tensor, computed in chunks of chunk_n samples (default
    N/8) whose copies overlap the GPU work."""
    lib = load()
    dev = _target_device(x)
    if x.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("x must be float32 or bfloat16")
    dt = NRC_F32 if x.dtype == torch.float32 else NRC_BF16
    if not x.is_cuda:
        return _prenorm_host(lib, dev, dt, x, bn_running_mean, bn_running_var, bn_gamma,
                             bn_beta, bn_eps, conv_weight, conv_bias, dilation, padding,
                             kernel_size, out, workspace, stream, chunk_n)
    xd = _dev(x, dev)
    N, C, L = xd.shape
    rm, rv, g, b = (_dev(t, dev, torch.float32) for t in (bn_running_mean, bn_running_var,
                                                           bn_gamma, bn_beta))
    w = _dev(conv_weight, dev, x.dtype)
    cb = _dev(conv_bias, dev, x.dtype)
    padding = dilation if padding is None else padding
    o = out if out is not None else torch.empty_like(xd)
    need = lib.nrc_prenorm_dilconv_residual_workspace_size(C, dt)
    ws = _workspace(need, dev, workspace)
    st = lib.nrc_prenorm_dilconv_residual(
        _ptr(xd), _ptr(o), dt, N, C, L, kernel_size, dilation, padding, _ptr(rm), _ptr(rv),
        _ptr(g), _ptr(b), float(bn_eps), _ptr(w), _ptr(cb), _ptr(ws), ws.numel(),
        _stream(stream))
    _check(st, "nrc_prenorm_dilconv_residual")
    _keep_alive(stream, xd, rm, rv, g, b, w, cb, ws)
    return o


def prenorm_dilconv_residual_train_workspace_size(N: int, C: int, L: int,
                                                  dtype=torch.float32) -> int:
    dt = NRC_F32 if dtype == torch.float32 else NRC_BF16
    return int(load().nrc_prenorm_dilconv_residual_train_workspace_size(N, C, L, dt))


def prenorm_dilconv_residual_train(x, bn_running_mean, bn_running_var, bn_gamma, bn_beta,
                                   bn_eps, bn_momentum, conv_weight, conv_bias, dilation,
                                   padding=None, kernel_size=3, num_batches_tracked=None,
                                   out=None, workspace=None, stream=None):
    """The block with BatchNorm1d in training mode: x is normalized with its
    own per-channel mean and biased variance over (N, L), and the running
    buffers (contiguous fp32 device tensors, or None) are updated in place
    with the unbiased variance; num_batches_tracked (an int64 device tensor
    or None) is incremented.  With x in host memory the call goes through
    nrc_prenorm_dilconv_residual_train_host (parameters taken to host memory,
    the result a pinned host tensor; the stream is synchronised before
    returning)."""
    lib = load()
    if x.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("x must be float32 or bfloat16")
    host = not x.is_cuda
    dev = _target_device(x)
    dt = NRC_F32 if x.dtype == torch.float32 else NRC_BF16
    for t in (bn_running_mean, bn_running_var):
        if t is not None and not (t.is_cuda and t.dtype == torch.float32 and t.is_contiguous()):
            raise TypeError("running statistics must be contiguous fp32 device tensors")
    if num_batches_tracked is not None and not (num_batches_tracked.is_cuda and
                                                num_batches_tracked.dtype == torch.int64):
        raise TypeError("num_batches_tracked must be an int64 device tensor")
    if host:
        return _train_host(lib, dev, dt, x, bn_running_mean, bn_running_var, bn_gamma, bn_beta,
                           bn_eps, bn_momentum, conv_weight, conv_bias, dilation, padding,
                           kernel_size, num_batches_tracked, out, workspace, stream)
    xd = _dev(x, dev)
    N, C, L = xd.shape
    g, b = (_dev(t, dev, torch.float32) for t in (bn_gamma, bn_beta))
    w = _dev(conv_weight, dev, x.dtype)
    cb = _dev(conv_bias, dev, x.dtype)
    padding = dilation if padding is None else padding
    o = out if (out is not None and not host) else torch.empty_like(xd)
    ws = _workspace(lib.nrc_prenorm_dilconv_residual_train_workspace_size(N, C, L, dt), dev,
                    workspace)
    st = lib.nrc_prenorm_dilconv_residual_train(
        _ptr(xd), _ptr(o), dt, N, C, L, kernel_size, dilation, padding, _ptr(bn_running_mean),
        _ptr(bn_running_var), _ptr(num_batches_tracked), _ptr(g), _ptr(b), float(bn_eps),
        float(bn_momentum), _ptr(w), _ptr(cb), _ptr(ws), ws.numel(), _stream(stream))
    _check(st, "nrc_prenorm_dilconv_residual_train")
    _keep_alive(stream, xd, g, b, w, cb, ws)
    if host:
        res = out if out is not None else torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
        res.copy_(o)
        return res
    return o


def _train_host(lib, dev, dt, x, rm, rv, g, b, eps, momentum, w, cb, dilation, padding,
                kernel_size, nbt, out, workspace, stream, chunk_n=None):
    """The training-mode block on host buffers through
    nrc_prenorm_dilconv_residual_train_host."""
    xh = x.contiguous()
    N, C, L = xh.shape
    gh, bh = (_host(t, torch.float32) for t in (g, b))
    wh, cbh = _host(w, x.dtype), _host(cb, x.dtype)
    padding = dilation if padding is None else padding
    chunk_n = chunk_n or _default_chunk(N)
    need = lib.nrc_prenorm_dilconv_residual_train_host_workspace_size(N, C, L, dt, chunk_n)
    if need == 0:
        raise ValueError("bad shape for the host-buffer training-mode block")
    ws = _workspace(need, dev, workspace)
    res = out if out is not None else torch.empty(xh.shape, dtype=xh.dtype, pin_memory=True)
    if res.is_cuda or res.shape != xh.shape or res.dtype != xh.dtype or not res.is_contiguous():
        raise ValueError("out must be a contiguous host tensor of x's shape and dtype")
    st = stream if stream is not None else torch.cuda.current_stream(dev)
    status = lib.nrc_prenorm_dilconv_residual_train_host(
        _ptr(xh), _ptr(res), dt, N, C, L, kernel_size, dilation, padding, _ptr(rm), _ptr(rv),
        _ptr(nbt), _ptr(gh), _ptr(bh), float(eps), float(momentum), _ptr(wh), _ptr(cbh),
        int(chunk_n), _ptr(ws), ws.numel(), ctypes.c_void_p(st.cuda_stream))
    _check(status, "nrc_prenorm_dilconv_residual_train_host")
    st.synchronize()                      # out is host memory: valid on return
    return res


def prenorm_dilconv_residual_train_host_workspace_size(N, C, L, dtype=torch.float32,
                                                       chunk_n=None) -> int:
    """Device workspace of the training-mode block on host buffers."""
    dt = NRC_F32 if dtype == torch.float32 else NRC_BF16
    return int(load().nrc_prenorm_dilconv_residual_train_host_workspace_size(
        N, C, L, dt, chunk_n or _default_chunk(N)))


def prenorm_dilconv_residual_host_workspace_size(N, C, L, dtype=torch.float32,
                                                 chunk_n=None) -> int:
    """Device workspace of the block on host buffers (x and out in host memory)."""
    dt = NRC_F32 if dtype == torch.float32 else NRC_BF16
    return int(load().nrc_prenorm_dilconv_residual_host_workspace_size(
        N, C, L, dt, chunk_n or _default_chunk(N)))


def _default_chunk(N):
    return max(1, N // 8)


def _host(t, dtype=None):
    """Contiguous host copy of an optional tensor."""
    if t is None:
        return None
    return t.to(device="cpu", dtype=dtype or t.dtype).contiguous()


def _prenorm_host(lib, dev, dt, x, rm, rv, g, b, eps, w, cb, dilation, padding, kernel_size,
                  out, workspace, stream, chunk_n=None):
    """The block on host buffers through nrc_prenorm_dilconv_residual_host."""
    xh = x.contiguous()
    N, C, L = xh.shape
    rm, rv, g, b = (_host(t, torch.float32) for t in (rm, rv, g, b))
    wh, cbh = _host(w, x.dtype), _host(cb, x.dtype)
    padding = dilation if padding is None else padding
    chunk_n = chunk_n or _default_chunk(N)
    need = lib.nrc_prenorm_dilconv_residual_host_workspace_size(N, C, L, dt, chunk_n)
    if need == 0:
        raise ValueError("bad shape for the host-buffer block")
    ws = _workspace(need, dev, workspace)
    res = out if out is not None else torch.empty(xh.shape, dtype=xh.dtype, pin_memory=True)
    st = stream if stream is not None else torch.cuda.current_stream(dev)
    status = lib.nrc_prenorm_dilconv_residual_host(
        _ptr(xh), _ptr(res), dt, N, C, L, kernel_size, dilation, padding, _ptr(rm), _ptr(rv),
        _ptr(g), _ptr(b), float(eps), _ptr(wh), _ptr(cbh), int(chunk_n), _ptr(ws),
        ws.numel(), ctypes.c_void_p(st.cuda_stream))
    _check(status, "nrc_prenorm_dilconv_residual_host")
    st.synchronize()                      # out is host memory: valid on return
    return res


def _keep_alive(stream, *tensors):
    """Temporaries used on a non-current stream must not be recycled early."""
    if stream is None:
        return
    for t in tensors:
        if t is not None and t.is_cuda:
            t.record_stream(stream)


# ---------------------------------------------------------------------------
# Conv1d + GroupNorm
# ---------------------------------------------------------------------------
def conv1d_output_length(T, kernel_size=3, stride=1, padding=1, dilation=1) -> int:
    """T_out of Conv1d(kernel_size, stride, padding, dilation) on T positions (0 if invalid)."""
    return int(load().nrc_conv1d_output_length(T, kernel_size, stride, padding, dilation))


def conv1d_groupnorm_workspace_size(N, C_in, C_out, T, num_groups, kernel_size=3, stride=1,
                                    padding=1, dilation=1) -> int:
    return int(load().nrc_conv1d_groupnorm_workspace_size(N, C_in, C_out, T, kernel_size, stride,
                                                          padding, dilation, num_groups))


def conv1d_groupnorm(x, conv_weight, conv_bias, num_groups, gn_gamma, gn_beta, eps=1e-5,
                     kernel_size=None, stride=1, padding=1, dilation=1, out=None, workspace=None,
                     stream=None):
    """GroupNorm(num_groups)(Conv1d(x)); x (N, C_in, T) fp32, conv_weight
    (C_out, C_in, kernel_size); the result is (N, C_out, T_out).  With x in
    host memory the call goes through nrc_conv1d_groupnorm_host (parameters
    taken to host memory, output in host memory; the stream is synchronised
    before returning)."""
    lib = load()
    host = not x.is_cuda
    dev = _target_device(x)
    if host:
        return _gn_host(lib, dev, x, conv_weight, conv_bias, num_groups, gn_gamma, gn_beta, eps,
                        kernel_size, stride, padding, dilation, out, workspace, stream)
    xd = _dev(x, dev, torch.float32)
    N, Cin, T = xd.shape
    w = _dev(conv_weight, dev, torch.float32)
    Cout = w.shape[0]
    if kernel_size is None:
        kernel_size = w.shape[2]
    if w.dim() != 3 or w.shape[1] != Cin or w.shape[2] != kernel_size:
        raise ValueError("conv_weight must be (C_out, C_in, kernel_size)")
    T_out = int(lib.nrc_conv1d_output_length(T, kernel_size, stride, padding, dilation))
    if T_out <= 0:
        raise ValueError("the conv's kernel does not fit the padded input")
    cb, g, b = (_dev(t, dev, torch.float32) for t in (conv_bias, gn_gamma, gn_beta))
    o = out if (out is not None and not host) else torch.empty((N, Cout, T_out), device=dev,
                                                                dtype=torch.float32)
    if o.shape != (N, Cout, T_out) or o.dtype != torch.float32 or not o.is_contiguous():
        raise ValueError("out must be a contiguous fp32 (N, C_out, T_out) tensor")
    ws = _workspace(lib.nrc_conv1d_groupnorm_workspace_size(N, Cin, Cout, T, kernel_size, stride,
                                                            padding, dilation, num_groups), dev,
                    workspace)
    st = lib.nrc_conv1d_groupnorm(_ptr(xd), _ptr(o), N, Cin, Cout, T, kernel_size, stride,
                                  padding, dilation, _ptr(w), _ptr(cb), num_groups, _ptr(g),
                                  _ptr(b), float(eps), _ptr(ws), ws.numel(), _stream(stream))
    _check(st, "nrc_conv1d_groupnorm")
    _keep_alive(stream, xd, w, cb, g, b, ws)
    if host:
        res = out if out is not None else torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
        res.copy_(o)
        return res
    return o


def _gn_host(lib, dev, x, w, cb, G, g, b, eps, kernel_size, stride, padding, dilation, out,
             workspace, stream, chunk_n=None):
    """Conv1d + GroupNorm on host buffers through nrc_conv1d_groupnorm_host."""
    if x.dtype != torch.float32:
        raise TypeError("x must be fp32")
    xh = x.contiguous()
    N, Cin, T = xh.shape
    wh = _host(w, torch.float32)
    Cout = wh.shape[0]
    if kernel_size is None:
        kernel_size = wh.shape[2]
    if wh.dim() != 3 or wh.shape[1] != Cin or wh.shape[2] != kernel_size:
        raise ValueError("conv_weight must be (C_out, C_in, kernel_size)")
    T_out = int(lib.nrc_conv1d_output_length(T, kernel_size, stride, padding, dilation))
    if T_out <= 0:
        raise ValueError("the conv's kernel does not fit the padded input")
    cbh, gh, bh = (_host(t, torch.float32) for t in (cb, g, b))
    chunk_n = chunk_n or (N + 1) // 2
    need = lib.nrc_conv1d_groupnorm_host_workspace_size(N, Cin, Cout, T, kernel_size, stride,
                                                        padding, dilation, G, chunk_n)
    if need == 0:
        raise ValueError("bad arguments for the host-buffer Conv1d + GroupNorm")
    ws = _workspace(need, dev, workspace)
    res = out if out is not None else torch.empty((N, Cout, T_out), dtype=torch.float32,
                                                  pin_memory=True)
    if res.is_cuda or res.shape != (N, Cout, T_out) or res.dtype != torch.float32 or \
            not res.is_contiguous():
        raise ValueError("out must be a contiguous fp32 (N, C_out, T_out) host tensor")
    st = stream if stream is not None else torch.cuda.current_stream(dev)
    status = lib.nrc_conv1d_groupnorm_host(
        _ptr(xh), _ptr(res), N, Cin, Cout, T, kernel_size, stride, padding, dilation, _ptr(wh),
        _ptr(cbh), G, _ptr(gh), _ptr(bh), float(eps), int(chunk_n), _ptr(ws), ws.numel(),
        ctypes.c_void_p(st.cuda_stream))
    _check(status, "nrc_conv1d_groupnorm_host")
    st.synchronize()                      # out is host memory: valid on return
    return res


def conv1d_groupnorm_host_workspace_size(N, C_in, C_out, T, num_groups, kernel_size=3, stride=1,
                                         padding=1, dilation=1, chunk_n=None) -> int:
    """Device workspace of Conv1d + GroupNorm on host buffers."""
    return int(load().nrc_conv1d_groupnorm_host_workspace_size(
        N, C_in, C_out, T, kernel_size, stride, padding, dilation, num_groups,
        chunk_n or (N + 1) // 2))


# ---------------------------------------------------------------------------
# Linear + BatchNorm1d + bias + divide + Swish
# ---------------------------------------------------------------------------
def linear_bn_swish_workspace_size(B, in_f, out_f) -> int:
    return int(load().nrc_linear_bn_swish_workspace_size(B, in_f, out_f))


def _default_chunk_f(out_f):
    return max(128, ((out_f + 3) // 4 + 127) // 128 * 128)


def linear_bn_swish_host_workspace_size(B, in_f, out_f, chunk_f=None) -> int:
    """Device workspace of the Linear on host buffers (x, weights and out in host memory)."""
    return int(load().nrc_linear_bn_swish_host_workspace_size(
        B, in_f, out_f, chunk_f or _default_chunk_f(out_f)))


def linear_bn_swish(x, lin_weight, lin_bias, bn_gamma, bn_beta, bn_running_mean,
                    bn_running_var, add_bias, divide_value=1.0, bn_eps=1e-5, bn_momentum=0.1,
                    training=True, num_batches_tracked=None, out=None, workspace=None,
                    stream=None):
    """Swish((BatchNorm1d(Linear(x)) + add_bias) / divide_value).

    In training mode bn_running_mean/var (device fp32 tensors) and
    num_batches_tracked (device int64 tensor or None) are updated in place.
    add_bias is a one-element tensor (read on the device).  With x in host
    memory the call goes through nrc_linear_bn_swish_host (weights and
    parameters taken to host memory, output in host memory; the stream is
    synchronised before returning)."""
    lib = load()
    host = not x.is_cuda
    dev = _target_device(x)
    if host:
        return _linear_host(lib, dev, x, lin_weight, lin_bias, bn_gamma, bn_beta,
                            bn_running_mean, bn_running_var, add_bias, divide_value, bn_eps,
                            bn_momentum, training, num_batches_tracked, out, workspace, stream)
    xd = _dev(x, dev, torch.float32)
    B, IN = xd.shape
    w = _dev(lin_weight, dev, torch.float32)
    OUT = w.shape[0]
    lb, g, b = (_dev(t, dev, torch.float32) for t in (lin_bias, bn_gamma, bn_beta))
    for t in (bn_running_mean, bn_running_var):
        if not (t.is_cuda and t.dtype == torch.float32 and t.is_contiguous()):
            raise TypeError("running statistics must be contiguous fp32 device tensors")
    if num_batches_tracked is not None and not (num_batches_tracked.is_cuda and
                                                num_batches_tracked.dtype == torch.int64):
        raise TypeError("num_batches_tracked must be an int64 device tensor")
    ab = _dev(torch.as_tensor(add_bias, dtype=torch.float32).reshape(1), dev, torch.float32)
    o = out if (out is not None and not host) else torch.empty((B, OUT), device=dev,
                                                                dtype=torch.float32)
    ws = _workspace(lib.nrc_linear_bn_swish_workspace_size(B, IN, OUT), dev, workspace)
    st = lib.nrc_linear_bn_swish(_ptr(xd), _ptr(o), B, IN, OUT, _ptr(w), _ptr(lb), _ptr(g),
                                 _ptr(b), _ptr(bn_running_mean), _ptr(bn_running_var),
                                 _ptr(num_batches_tracked), float(bn_eps), float(bn_momentum),
                                 int(bool(training)), _ptr(ab), float(divide_value), _ptr(ws),
                                 ws.numel(), _stream(stream))
    _check(st, "nrc_linear_bn_swish")
    _keep_alive(stream, xd, w, lb, g, b, ab, ws)
    if host:
        res = out if out is not None else torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
        res.copy_(o)
        return res
    return o


def _linear_host(lib, dev, x, w, lb, g, b, rm, rv, ab, divide_value, eps, momentum, training,
                 nbt, out, workspace, stream, chunk_f=None):
    """The Linear on host buffers through nrc_linear_bn_swish_host."""
    if x.dtype != torch.float32:
        raise TypeError("x must be fp32")
    xh = x.contiguous()
    B, IN = xh.shape
    wh = _host(w, torch.float32)
    OUT = wh.shape[0]
    if wh.shape != (OUT, IN):
        raise ValueError("lin_weight must be (out_features, in_features)")
    lbh, gh, bh = (_host(t, torch.float32) for t in (lb, g, b))
    abh = _host(torch.as_tensor(ab, dtype=torch.float32).reshape(1), torch.float32)
    for t in (rm, rv):
        if not (t.is_cuda and t.dtype == torch.float32 and t.is_contiguous() and
                t.numel() == OUT):
            raise TypeError("running statistics must be contiguous fp32 device tensors")
    if nbt is not None and not (nbt.is_cuda and nbt.dtype == torch.int64):
        raise TypeError("num_batches_tracked must be an int64 device tensor")
    chunk_f = chunk_f or _default_chunk_f(OUT)
    need = lib.nrc_linear_bn_swish_host_workspace_size(B, IN, OUT, chunk_f)
    if need == 0:
        raise ValueError("bad shape for the host-buffer Linear")
    ws = _workspace(need, dev, workspace)
    res = out if out is not None else torch.empty((B, OUT), dtype=torch.float32,
                                                  pin_memory=True)
    if res.is_cuda or res.shape != (B, OUT) or res.dtype != torch.float32 or \
            not res.is_contiguous():
        raise ValueError("out must be a contiguous fp32 (B, out_features) host tensor")
    st = stream if stream is not None else torch.cuda.current_stream(dev)
    status = lib.nrc_linear_bn_swish_host(
        _ptr(xh), _ptr(res), B, IN, OUT, _ptr(wh), _ptr(lbh), _ptr(gh), _ptr(bh), _ptr(rm),
        _ptr(rv), _ptr(nbt), float(eps), float(momentum), int(bool(training)), _ptr(abh),
        float(divide_value), int(chunk_f), _ptr(ws), ws.numel(), ctypes.c_void_p(st.cuda_stream))
    _check(status, "nrc_linear_bn_swish_host")
    st.synchronize()                      # out is host memory: valid on return
    return res


# ---------------------------------------------------------------------------
# Status
# ---------------------------------------------------------------------------
def query_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status code."""
    return int(load().nrc_query_status(_stream(stream)))


def last_error_site() -> int:
    return int(load().nrc_last_error_site())


def set_wait_timeout_ns(ns: int) -> None:
    load().nrc_set_wait_timeout_ns(int(ns))


def set_grid_barrier_timeout_ns(ns: int) -> None:
    """Limit of the one-wave GroupNorm kernel's grid barrier only (0: the general limit)."""
    load().nrc_set_grid_barrier_timeout_ns(int(ns))


def selftest_wait_timeout(limit_ns: int, stream=None) -> None:
    _check(load().nrc_selftest_wait_timeout(int(limit_ns), _stream(stream)),
           "nrc_selftest_wait_timeout")


# ---------------------------------------------------------------------------
# Launch trace
# ---------------------------------------------------------------------------
def trace_enable(on: bool = True) -> None:
    """Start (clearing earlier records) or stop recording an event pair around
    every kernel launch of the library."""
    load().nrc_trace_enable(int(bool(on)))


def trace_records():
    """[(kernel name, device ms), ...] for the launches recorded so far."""
    lib = load()
    out = []
    for i in range(lib.nrc_trace_count()):
        name = ctypes.c_char_p()
        ms = ctypes.c_float()
        _check(lib.nrc_trace_get(i, ctypes.byref(name), ctypes.byref(ms)), "nrc_trace_get")
        out.append((name.value.decode(), float(ms.value)))
    return out


# ---------------------------------------------------------------------------
# Allocation-free pre-norm block
# ---------------------------------------------------------------------------
def prenorm_dilconv_residual_noalloc(x, bn_running_mean, bn_running_var, bn_gamma, bn_beta,
                                     bn_eps, conv_weight, conv_bias, dilation, out,
                                     padding=None, kernel_size=3, stream=None):
    """The pre-norm block without a workspace, for callers that cannot hand the
    library scratch memory: its scratch is a fixed 4 MiB array inside the
    library (fp32 C <= 512, bf16 C <= 768).  All arguments must already be
    contiguous device tensors of the right dtypes and `out` must be given, so
    this binding allocates nothing either.  Calls that overlap on the GPU race
    on the shared scratch."""
    lib = load()
    if x.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("x must be float32 or bfloat16")
    if x.dim() != 3:
        raise ValueError("x must be (N, C, L)")
    if out is None or out.shape != x.shape or out.dtype != x.dtype:
        raise ValueError("out must be given with x's shape and dtype")
    dev = x.device
    for name, t, dtype in (("x", x, x.dtype), ("out", out, x.dtype),
                           ("bn_running_mean", bn_running_mean, torch.float32),
                           ("bn_running_var", bn_running_var, torch.float32),
                           ("bn_gamma", bn_gamma, torch.float32),
                           ("bn_beta", bn_beta, torch.float32),
                           ("conv_weight", conv_weight, x.dtype),
                           ("conv_bias", conv_bias, x.dtype)):
        if t is None:
            if name == "conv_bias":
                continue
            raise ValueError(f"{name} is required")
        if not t.is_cuda or t.device != dev:
            raise ValueError(f"{name} must be on x's device ({dev})")
        if t.dtype != dtype:
            raise TypeError(f"{name} must be {dtype}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    dt = NRC_F32 if x.dtype == torch.float32 else NRC_BF16
    N, C, L = x.shape
    padding = dilation if padding is None else padding
    st = lib.nrc_prenorm_dilconv_residual_noalloc(
        _ptr(x), _ptr(out), dt, N, C, L, kernel_size, dilation, padding, _ptr(bn_running_mean),
        _ptr(bn_running_var), _ptr(bn_gamma), _ptr(bn_beta), float(bn_eps), _ptr(conv_weight),
        _ptr(conv_bias), _stream(stream))
    _check(st, "nrc_prenorm_dilconv_residual_noalloc")
    return out
