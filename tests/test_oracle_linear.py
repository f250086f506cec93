"""Pins for the Linear + BatchNorm1d + bias + divide + Swish oracle (CPU only)."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from normalization_convolution_blocks_gb300 import synthetic as syn

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _torch_fp64(inp, training=True):
    """The problem statement as PyTorch modules in float64: Linear, BatchNorm1d,
    + bias, / divide, x * sigmoid(x).  Returns (out, running_mean, running_var)."""
    B, IN = inp.x.shape
    OUT = inp.weight.shape[0]
    lin = torch.nn.Linear(IN, OUT).double()
    bn = torch.nn.BatchNorm1d(OUT, eps=inp.eps, momentum=inp.momentum).double()
    bn.train(training)
    with torch.no_grad():
        lin.weight.copy_(inp.weight.double())
        lin.bias.copy_(inp.lin_bias.double())
        bn.weight.copy_(inp.gamma.double())
        bn.bias.copy_(inp.beta.double())
        bn.running_mean.copy_(inp.running_mean.double())
        bn.running_var.copy_(inp.running_var.double())
        y = bn(lin(inp.x.double()))
        y = (y + inp.add_bias.double()) / inp.divide_value
        out = y * torch.sigmoid(y)
    return out.numpy(), bn.running_mean.numpy(), bn.running_var.numpy()


def _run(inp, training=True, cols=None, lin_bias=None):
    return oracle.linear_bn_swish(inp.x, inp.weight,
                                  inp.lin_bias if lin_bias is None else lin_bias,
                                  inp.gamma, inp.beta, inp.running_mean, inp.running_var,
                                  inp.eps, inp.momentum, training, float(inp.add_bias[0]),
                                  inp.divide_value, cols=cols)


def _rel(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


@pytest.mark.parametrize("case", json.load(open(os.path.join(GOLDEN, "linear_bn_swish_hand.json")))["cases"],
                         ids=lambda c: c["name"])
def test_hand_worked_case(case):
    out, rm, rv, _ = oracle.linear_bn_swish(
        np.array(case["x"]), np.array(case["weight"]), case["lin_bias"], case["gamma"],
        case["beta"], case["running_mean"], case["running_var"], case["eps"], case["momentum"],
        True, case["add_bias"], case["divide_value"])
    np.testing.assert_allclose(out, np.array(case["out"]), rtol=0, atol=1e-15)
    np.testing.assert_allclose(rm, case["running_mean_out"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(rv, case["running_var_out"], rtol=0, atol=1e-15)


@pytest.mark.parametrize("B,IN,OUT,affine", [(64, 256, 128, False), (64, 256, 128, True),
                                             (2, 16, 8, True), (3, 33, 17, True),
                                             (1024, 512, 64, True)])
@pytest.mark.parametrize("training", [True, False])
def test_matches_torch_fp64_modules(B, IN, OUT, affine, training):
    inp = syn.linear_bn_swish_inputs(B, IN, OUT, seed=21, random_affine=affine)
    if not training:      # eval mode with non-trivial running statistics
        g = torch.Generator().manual_seed(22)
        inp.running_mean = torch.randn(OUT, generator=g) * 0.1
        inp.running_var = torch.rand(OUT, generator=g) + 0.5
    out, rm, rv, _ = _run(inp, training)
    ref, rrm, rrv = _torch_fp64(inp, training)
    assert _rel(out, ref) < 1e-12
    np.testing.assert_allclose(rm, rrm, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(rv, rrv, rtol=1e-13, atol=1e-15)


def test_output_independent_of_linear_bias_and_running_mean_shift():
    inp = syn.linear_bn_swish_inputs(32, 64, 16, seed=23, random_affine=True)
    out_p, rm_p, rv_p, _ = _run(inp)
    out_m, rm_m, rv_m, _ = _run(inp, lin_bias=-inp.lin_bias)
    np.testing.assert_allclose(out_p, out_m, rtol=0, atol=1e-12)
    np.testing.assert_allclose(rm_p - rm_m, 2 * inp.momentum * inp.lin_bias.double().numpy(),
                               rtol=0, atol=1e-15)
    np.testing.assert_allclose(rv_p, rv_m, rtol=0, atol=1e-14)


def test_batch_of_two_closed_form():
    inp = syn.linear_bn_swish_inputs(2, 8, 5, seed=24, random_affine=True)
    out, _, _, mv = _run(inp)
    y = (inp.x.double() @ inp.weight.double().T + inp.lin_bias.double()).numpy()
    h = (y[0] - y[1]) / 2.0
    g, b = inp.gamma.double().numpy(), inp.beta.double().numpy()
    yhat0 = g * h / np.sqrt(h * h + inp.eps) + b
    yhat1 = -g * h / np.sqrt(h * h + inp.eps) + b
    for row, yh in ((0, yhat0), (1, yhat1)):
        u = (yh + float(inp.add_bias[0])) / inp.divide_value
        np.testing.assert_allclose(out[row], u / (1 + np.exp(-u)), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(mv[:, 1], h * h, rtol=1e-12)


def test_swish_special_values():
    inp = syn.linear_bn_swish_inputs(4, 8, 3, seed=25)
    zero, beta = torch.zeros(3), torch.tensor([0.0, 50.0, -50.0])
    out, _, _, _ = oracle.linear_bn_swish(inp.x, inp.weight, inp.lin_bias, zero, beta, None,
                                          None, 1e-5, 0.1, True, 0.0, 1.0)
    assert np.all(out[:, 0] == 0.0)                      # swish(0) = 0
    np.testing.assert_allclose(out[:, 1], 50.0 / (1 + math.exp(-50.0)), rtol=1e-15)
    np.testing.assert_allclose(out[:, 2], -50.0 * math.exp(-50.0) / (1 + math.exp(-50.0)),
                               rtol=1e-13)


def test_running_stats_on_hand_built_columns():
    # x = I, so column j of y is row j of W plus b_lin[j]: known mean and variance
    B = 4
    x = np.eye(B)
    W = np.array([[1.0, 2.0, 3.0, 4.0], [0.0, 0.0, 0.0, 8.0], [5.0, 5.0, 5.0, 5.0]])
    b_lin = np.array([0.0, 1.0, -2.0])
    rm0, rv0 = np.array([1.0, 0.0, 2.0]), np.array([1.0, 2.0, 0.5])
    m = 0.25
    _, rm, rv, mv = oracle.linear_bn_swish(x, W, b_lin, None, None, rm0, rv0, 1e-5, m, True,
                                           0.0, 1.0)
    mean = np.array([2.5, 3.0, 3.0])
    var_b = np.array([1.25, 12.0, 0.0])
    np.testing.assert_allclose(mv[:, 0], mean, rtol=0, atol=1e-15)
    np.testing.assert_allclose(mv[:, 1], var_b, rtol=0, atol=1e-14)
    np.testing.assert_allclose(rm, (1 - m) * rm0 + m * mean, rtol=0, atol=1e-15)
    np.testing.assert_allclose(rv, (1 - m) * rv0 + m * var_b * B / (B - 1), rtol=0, atol=1e-14)


def test_columns_match_full():
    inp = syn.linear_bn_swish_inputs(16, 32, 20, seed=26, random_affine=True)
    full, rm_f, _, _ = _run(inp)
    sub, rm_s, _, _ = _run(inp, cols=[19, 0, 7])
    assert np.array_equal(sub, full[:, [19, 0, 7]])
    assert np.array_equal(rm_s[[19, 0, 7]], rm_f[[19, 0, 7]])


def test_training_rejects_batch_of_one():
    inp = syn.linear_bn_swish_inputs(1, 8, 4, seed=27)
    with pytest.raises(ValueError):
        _run(inp)
