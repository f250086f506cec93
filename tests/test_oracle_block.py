"""Pins for the pre-norm residual block oracle (CPU only).

The oracle (``oracle.prenorm_block``) must agree with things other than itself:
hand-worked cases, PyTorch's own fp64 modules (the pages state the problem as
exactly that module composition), structural invariants of the conv, and an
independently written NumPy formulation on tiny shapes.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from normalization_convolution_blocks_gb300 import synthetic as syn

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _torch_modules_fp64(inp):
    """The problem statement as PyTorch modules, in float64."""
    C = inp.x.shape[1]
    bn = torch.nn.BatchNorm1d(C, eps=inp.eps).double().eval()
    conv = torch.nn.Conv1d(C, C, 3, padding=inp.dilation, dilation=inp.dilation).double()
    with torch.no_grad():
        bn.running_mean.copy_(inp.running_mean.double())
        bn.running_var.copy_(inp.running_var.double())
        bn.weight.copy_(inp.gamma.double())
        bn.bias.copy_(inp.beta.double())
        conv.weight.copy_(inp.weight.double())
        conv.bias.copy_(inp.bias.double())
        x = inp.x.double()
        return (x + conv(torch.relu(bn(x)))).numpy()


def _run(inp, **kw):
    return oracle.prenorm_block(inp.x, inp.running_mean, inp.running_var, inp.gamma,
                                inp.beta, inp.eps, kw.get("w", inp.weight),
                                kw.get("bias", inp.bias), inp.dilation)


def _rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


@pytest.mark.parametrize("case", json.load(open(os.path.join(GOLDEN, "prenorm_block_hand.json")))["cases"],
                         ids=lambda c: c["name"][:40])
def test_hand_worked_cases(case):
    out = oracle.prenorm_block(np.array(case["x"]), case["running_mean"], case["running_var"],
                               case["gamma"], case["beta"], case["eps"], np.array(case["weight"]),
                               case["bias"], case["dilation"])
    np.testing.assert_allclose(out, np.array(case["out"]), rtol=0, atol=1e-12)


@pytest.mark.parametrize("N,C,L,d", [(2, 32, 512, 128),      # tiny workload, full size
                                     (2, 64, 1024, 128),     # reduced full workload
                                     (1, 16, 300, 1), (1, 16, 300, 7), (2, 8, 64, 40),
                                     (1, 8, 100, 60)])       # d > L/2: side taps half padded
def test_matches_torch_fp64_modules(N, C, L, d):
    inp = syn.prenorm_block_inputs(N, C, L, d, seed=1)
    assert _rel(_run(inp), _torch_modules_fp64(inp)) < 1e-12


def test_matches_torch_bf16_storage():
    """bf16-stored inputs, upcast exactly: the oracle sees the same values."""
    inp = syn.prenorm_block_inputs(2, 32, 256, 8, seed=2, dtype=torch.bfloat16)
    ref = _torch_modules_fp64(inp)
    assert _rel(_run(inp), ref) < 1e-12


def test_zero_weights_give_identity():
    inp = syn.prenorm_block_inputs(2, 16, 200, 16, seed=3)
    out = _run(inp, w=torch.zeros_like(inp.weight), bias=torch.zeros_like(inp.bias))
    assert np.array_equal(out, inp.x.double().numpy())


def _bn_relu_torch(inp):
    return torch.relu(torch.nn.functional.batch_norm(
        inp.x.double(), inp.running_mean.double(), inp.running_var.double(),
        inp.gamma.double(), inp.beta.double(), training=False, eps=inp.eps)).numpy()


def _tap_identity(C, tap):
    w = torch.zeros(C, C, 3)
    w[torch.arange(C), torch.arange(C), tap] = 1.0
    return w


def test_center_tap_identity():
    inp = syn.prenorm_block_inputs(2, 16, 200, 16, seed=4)
    C = inp.x.shape[1]
    out = _run(inp, w=_tap_identity(C, 1), bias=torch.zeros(C))
    expect = inp.x.double().numpy() + _bn_relu_torch(inp)
    np.testing.assert_allclose(out, expect, rtol=0, atol=1e-12)


@pytest.mark.parametrize("d", [1, 5, 64])
def test_side_tap_identities_pin_direction_and_padding(d):
    inp = syn.prenorm_block_inputs(1, 8, 150, d, seed=5)
    C, L = inp.x.shape[1], inp.x.shape[2]
    x = inp.x.double().numpy()
    z = _bn_relu_torch(inp)
    left = _run(inp, w=_tap_identity(C, 0), bias=torch.zeros(C))
    expect = x.copy()
    expect[:, :, d:] += z[:, :, :L - d]            # tap 0 reads t - d; zeros for t < d
    np.testing.assert_allclose(left, expect, rtol=0, atol=1e-12)
    right = _run(inp, w=_tap_identity(C, 2), bias=torch.zeros(C))
    expect = x.copy()
    expect[:, :, :L - d] += z[:, :, d:]            # tap 2 reads t + d; zeros for t >= L-d
    np.testing.assert_allclose(right, expect, rtol=0, atol=1e-12)


def test_linear_in_weights():
    inp = syn.prenorm_block_inputs(1, 8, 128, 4, seed=6)
    x = inp.x.double().numpy()
    g = torch.Generator().manual_seed(7)
    w1, w2 = torch.randn(8, 8, 3, generator=g), torch.randn(8, 8, 3, generator=g)
    zero_b = torch.zeros(8)
    y1 = _run(inp, w=w1, bias=zero_b) - x
    y2 = _run(inp, w=w2, bias=zero_b) - x
    y12 = _run(inp, w=w1.double() + w2.double(), bias=zero_b) - x
    np.testing.assert_allclose(y12, y1 + y2, rtol=0, atol=1e-11)
    yb = _run(inp, w=torch.zeros(8, 8, 3), bias=inp.bias) - x
    np.testing.assert_allclose(yb, np.broadcast_to(inp.bias.double().numpy()[None, :, None],
                                                   yb.shape), rtol=0, atol=0)


def _numpy_shifted_matmuls(inp):
    """Independent formulation: pad z with d zeros each side, three shifted
    channel-mixing matmuls, bias, residual."""
    x = inp.x.double().numpy()
    rm, rv = inp.running_mean.double().numpy(), inp.running_var.double().numpy()
    g, b = inp.gamma.double().numpy(), inp.beta.double().numpy()
    w, bias, d = inp.weight.double().numpy(), inp.bias.double().numpy(), inp.dilation
    N, C, L = x.shape
    z = np.maximum((x - rm[None, :, None]) / np.sqrt(rv + inp.eps)[None, :, None]
                   * g[None, :, None] + b[None, :, None], 0.0)
    zp = np.pad(z, ((0, 0), (0, 0), (d, d)))
    out = np.empty_like(x)
    for n in range(N):
        y = bias[:, None] + sum(w[:, :, k] @ zp[n, :, k * d:k * d + L] for k in range(3))
        out[n] = x[n] + y
    return out


@pytest.mark.parametrize("N,C,L,d", [(1, 1, 8, 1), (2, 3, 16, 2), (2, 4, 16, 3), (1, 4, 16, 8),
                                     (2, 2, 9, 1), (1, 4, 12, 8)])
def test_brute_force_tiny(N, C, L, d):
    inp = syn.prenorm_block_inputs(N, C, L, d, seed=8)
    np.testing.assert_allclose(_run(inp), _numpy_shifted_matmuls(inp), rtol=1e-13, atol=1e-13)


def test_rows_match_full():
    inp = syn.prenorm_block_inputs(3, 16, 96, 16, seed=9)
    full = _run(inp)
    rn, ro = [0, 2, 1, 2], [0, 15, 7, 3]
    rows = oracle.prenorm_block_rows(inp.x, inp.running_mean, inp.running_var, inp.gamma,
                                     inp.beta, inp.eps, inp.weight, inp.bias, inp.dilation,
                                     rn, ro)
    assert np.array_equal(rows, full[rn, ro])


def test_rejects_length_changing_padding():
    inp = syn.prenorm_block_inputs(1, 4, 32, 2, seed=10)
    with pytest.raises(ValueError):
        oracle.prenorm_block(inp.x, inp.running_mean, inp.running_var, inp.gamma, inp.beta,
                             inp.eps, inp.weight, inp.bias, 2, padding=1)
