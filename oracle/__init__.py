"""fp64 CPU oracle for the normalization-fused Conv1d blocks -- TEST INFRASTRUCTURE.

This package is the independent checker of the CUDA library.  Only the test
suite, ``__graft_entry__.smoke()`` and the benchmark's ``cpu_baseline`` /
``--impl reference`` legs may import it.  The product path never calls it and
shares no code with it: the arithmetic lives in ``oracle.c`` (plain C, fp64),
written from the problem definitions on the three PopcornBench pages:

* "Kimi-K2.6 l2_p12" -- pre-norm residual block (problem statement at the top
  of the page): out = x + Conv1d(ReLU(BatchNorm1d_eval(x))), k=3, pad=dil;
  its correctness discussion of batch against running statistics gives the
  training-mode variant.
* "FW-GLM-5-1 l2_p35" -- Conv1d(k=3, pad=1, no bias) + GroupNorm (problem
  analysis at the top of the page, and the normalisation kernel's formula).
* "Kimi-K2.6 l2_p97" -- Linear + BatchNorm1d (training) + bias + divide +
  Swish (the BatchNorm training-mode discussion at the top of the page).

This module only marshals numpy arrays (converted exactly to float64) into
the C functions.  Pins for every function live in ``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (-O2, OpenMP) into oracle/_build/liboracle.so."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-Wall",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # ORACLE_LIB_OVERRIDE lets the mutation test load a deliberately
            # broken copy of this oracle (built in a temporary directory).
            override = os.environ.get("ORACLE_LIB_OVERRIDE")
            lib = ctypes.CDLL(override if override else build())
            d, i, p = ctypes.c_double, ctypes.c_int, ctypes.c_void_p
            lib.oracle_prenorm_block.argtypes = [p, p, i, i, i, i, i, i, p, p, p, p, d,
                                                 p, p, i]
            lib.oracle_prenorm_block_rows.argtypes = [p, i, i, i, i, i, i, p, p, p, p,
                                                      d, p, p, p, p, i, p, i]
            lib.oracle_conv_groupnorm.argtypes = [p, p, i, i, i, i, i, i, i, i, p, p,
                                                  i, p, p, d, i]
            lib.oracle_conv_groupnorm_groups.argtypes = [p, i, i, i, i, i, i, i, i, p,
                                                         p, i, p, p, d, p, p, i, p, p, i]
            lib.oracle_linear_bn_swish_cols.argtypes = [p, i, i, i, p, p, p, p, p, p,
                                                        d, d, i, d, d, p, i, p, p, i]
            lib.oracle_conv1d_out_len.argtypes = [i, i, i, i, i]
            lib.oracle_prenorm_block_train.argtypes = [p, i, i, i, i, i, i, p, p, p, p, d,
                                                       d, p, p, p, p, i, p, p, p, i]
            for f in (lib.oracle_prenorm_block, lib.oracle_prenorm_block_rows,
                      lib.oracle_prenorm_block_train,
                      lib.oracle_conv_groupnorm, lib.oracle_conv_groupnorm_groups,
                      lib.oracle_linear_bn_swish_cols, lib.oracle_conv1d_out_len,
                      lib.oracle_max_threads):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def max_threads() -> int:
    return _load().oracle_max_threads()


def _f64(a):
    """Exact conversion to a C-contiguous float64 array (None stays None)."""
    if a is None:
        return None
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(rc, name):
    if rc != 0:
        raise ValueError(f"oracle {name}: invalid arguments (code {rc})")


def prenorm_block(x, rm, rv, gamma, beta, eps, w, bias, dilation, padding=None,
                  nthreads=0):
    """Pre-norm residual block out = x + Conv1d(relu(bn_eval(x))); x is (N, C, L),
    w is (C, C, K).  Returns a float64 (N, C, L) array."""
    x, rm, rv, gamma, beta, w, bias = map(_f64, (x, rm, rv, gamma, beta, w, bias))
    N, C, L = x.shape
    K = w.shape[2]
    padding = dilation if padding is None else padding
    out = np.empty_like(x)
    rc = _load().oracle_prenorm_block(_ptr(x), _ptr(out), N, C, L, K, dilation, padding,
                                      _ptr(rm), _ptr(rv), _ptr(gamma), _ptr(beta),
                                      float(eps), _ptr(w), _ptr(bias), nthreads)
    _check(rc, "prenorm_block")
    return out


def prenorm_block_rows(x, rm, rv, gamma, beta, eps, w, bias, dilation, rows_n, rows_o,
                       padding=None, nthreads=0):
    """Same block, only the output rows (rows_n[r], rows_o[r], :).  Returns (R, L)."""
    x, rm, rv, gamma, beta, w, bias = map(_f64, (x, rm, rv, gamma, beta, w, bias))
    N, C, L = x.shape
    K = w.shape[2]
    padding = dilation if padding is None else padding
    rn = np.ascontiguousarray(rows_n, dtype=np.int32)
    ro = np.ascontiguousarray(rows_o, dtype=np.int32)
    out = np.empty((len(rn), L), dtype=np.float64)
    rc = _load().oracle_prenorm_block_rows(_ptr(x), N, C, L, K, dilation, padding,
                                           _ptr(rm), _ptr(rv), _ptr(gamma), _ptr(beta),
                                           float(eps), _ptr(w), _ptr(bias), _ptr(rn),
                                           _ptr(ro), len(rn), _ptr(out), nthreads)
    _check(rc, "prenorm_block_rows")
    return out


def prenorm_block_train(x, running_mean, running_var, gamma, beta, eps, momentum, w, bias,
                        dilation, rows_n=None, rows_o=None, padding=None, nthreads=0):
    """The block with BatchNorm1d in training mode (batch mean and biased
    variance over (N, L) per channel; running buffers updated with the
    unbiased variance).

    Returns (out, running_mean', running_var', batch_mean, batch_var): out is
    (N, C, L), or (R, L) for the rows (rows_n[r], rows_o[r]); the running
    statistics come back as updated float64 copies (None stays None)."""
    x, gamma, beta, w, bias = map(_f64, (x, gamma, beta, w, bias))
    rm = _f64(running_mean).copy() if running_mean is not None else None
    rv = _f64(running_var).copy() if running_var is not None else None
    N, C, L = x.shape
    K = w.shape[2]
    padding = dilation if padding is None else padding
    if rows_n is None:
        rn = ro = None
        out = np.empty_like(x)
        nrows = 0
    else:
        rn = np.ascontiguousarray(rows_n, dtype=np.int32)
        ro = np.ascontiguousarray(rows_o, dtype=np.int32)
        nrows = len(rn)
        out = np.empty((nrows, L), dtype=np.float64)
    bm = np.empty(C, dtype=np.float64)
    bv = np.empty(C, dtype=np.float64)
    rc = _load().oracle_prenorm_block_train(
        _ptr(x), N, C, L, K, dilation, padding, _ptr(rm), _ptr(rv), _ptr(gamma), _ptr(beta),
        float(eps), float(momentum), _ptr(w), _ptr(bias), _ptr(rn), _ptr(ro), nrows, _ptr(out),
        _ptr(bm), _ptr(bv), nthreads)
    _check(rc, "prenorm_block_train")
    return out, rm, rv, bm, bv


def conv1d_out_len(T, K, stride=1, padding=1, dilation=1):
    """Conv1d output length (<= 0 when the kernel does not fit the padded input)."""
    return int(_load().oracle_conv1d_out_len(T, K, stride, padding, dilation))


def conv_groupnorm(x, w, bias, num_groups, gamma, beta, eps, stride=1, padding=1,
                   dilation=1, nthreads=0):
    """Conv1d (x (N, Cin, T), w (Cout, Cin, K)) followed by GroupNorm.  Returns
    float64 (N, Cout, T_out)."""
    x, w, bias, gamma, beta = map(_f64, (x, w, bias, gamma, beta))
    N, Cin, T = x.shape
    Cout, _, K = w.shape
    lib = _load()
    To = lib.oracle_conv1d_out_len(T, K, stride, padding, dilation)
    out = np.empty((N, Cout, max(To, 0)), dtype=np.float64)
    rc = lib.oracle_conv_groupnorm(_ptr(x), _ptr(out), N, Cin, Cout, T, K, stride,
                                   padding, dilation, _ptr(w), _ptr(bias), num_groups,
                                   _ptr(gamma), _ptr(beta), float(eps), nthreads)
    _check(rc, "conv_groupnorm")
    return out


def conv_groupnorm_groups(x, w, bias, num_groups, gamma, beta, eps, groups_n, groups_g,
                          stride=1, padding=1, dilation=1, nthreads=0):
    """Conv1d + GroupNorm for the chosen groups (groups_n[r], groups_g[r]).
    Returns (out (R, Cout/G, T_out), mean_var (R, 2))."""
    x, w, bias, gamma, beta = map(_f64, (x, w, bias, gamma, beta))
    N, Cin, T = x.shape
    Cout, _, K = w.shape
    lib = _load()
    To = lib.oracle_conv1d_out_len(T, K, stride, padding, dilation)
    gn = np.ascontiguousarray(groups_n, dtype=np.int32)
    gg = np.ascontiguousarray(groups_g, dtype=np.int32)
    cpg = Cout // num_groups if num_groups > 0 else 0
    out = np.empty((len(gn), cpg, max(To, 0)), dtype=np.float64)
    mv = np.empty((len(gn), 2), dtype=np.float64)
    rc = lib.oracle_conv_groupnorm_groups(_ptr(x), N, Cin, Cout, T, K, stride, padding,
                                          dilation, _ptr(w), _ptr(bias), num_groups,
                                          _ptr(gamma), _ptr(beta), float(eps), _ptr(gn),
                                          _ptr(gg), len(gn), _ptr(out), _ptr(mv),
                                          nthreads)
    _check(rc, "conv_groupnorm_groups")
    return out, mv


def linear_bn_swish(x, W, b_lin, gamma, beta, running_mean, running_var, eps, momentum,
                    training, add_bias, divide_value, cols=None, nthreads=0):
    """Linear + BatchNorm1d + scalar bias + divide + Swish.

    x (B, IN), W (OUT, IN).  ``cols`` selects output columns (default: all).
    Returns (out (B, ncols), running_mean', running_var', batch_mean_var (ncols, 2));
    the running stats are returned as updated float64 copies (full length OUT)."""
    x, W, b_lin, gamma, beta = map(_f64, (x, W, b_lin, gamma, beta))
    rm = _f64(running_mean).copy() if running_mean is not None else None
    rv = _f64(running_var).copy() if running_var is not None else None
    B, IN = x.shape
    OUT = W.shape[0]
    cols = np.arange(OUT, dtype=np.int32) if cols is None else np.ascontiguousarray(
        cols, dtype=np.int32)
    out = np.empty((B, len(cols)), dtype=np.float64)
    mv = np.empty((len(cols), 2), dtype=np.float64)
    rc = _load().oracle_linear_bn_swish_cols(
        _ptr(x), B, IN, OUT, _ptr(W), _ptr(b_lin), _ptr(gamma), _ptr(beta), _ptr(rm),
        _ptr(rv), float(eps), float(momentum), int(bool(training)), float(add_bias),
        float(divide_value), _ptr(cols), len(cols), _ptr(out), _ptr(mv), nthreads)
    _check(rc, "linear_bn_swish")
    return out, rm, rv, mv
