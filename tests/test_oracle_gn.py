"""Pins for the Conv1d + GroupNorm oracle (CPU only)."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from normalization_convolution_blocks_gb300 import synthetic as syn

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _torch_fp64(x, w, bias, G, gamma, beta, eps, stride=1, padding=1, dilation=1):
    Cout, Cin, K = w.shape
    conv = torch.nn.Conv1d(Cin, Cout, K, stride=stride, padding=padding, dilation=dilation,
                           bias=bias is not None).double()
    gn = torch.nn.GroupNorm(G, Cout, eps=eps, affine=gamma is not None).double()
    with torch.no_grad():
        conv.weight.copy_(torch.as_tensor(w).double())
        if bias is not None:
            conv.bias.copy_(torch.as_tensor(bias).double())
        if gamma is not None:
            gn.weight.copy_(torch.as_tensor(gamma).double())
            gn.bias.copy_(torch.as_tensor(beta).double())
        return gn(conv(torch.as_tensor(x).double())).numpy()


def _rel(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


@pytest.mark.parametrize("case", json.load(open(os.path.join(GOLDEN, "conv_groupnorm_hand.json")))["cases"],
                         ids=lambda c: c["name"][:40])
def test_hand_worked_case(case):
    out = oracle.conv_groupnorm(np.array(case["x"]), np.array(case["weight"]), None, case["G"],
                                case["gamma"], case["beta"], case["eps"])
    np.testing.assert_allclose(out, np.array(case["out"]), rtol=0, atol=1e-14)
    _, mv = oracle.conv_groupnorm_groups(np.array(case["x"]), np.array(case["weight"]), None,
                                         case["G"], case["gamma"], case["beta"], case["eps"],
                                         [0], [0])
    np.testing.assert_allclose(mv[0], [case["mean"], case["var"]], rtol=0, atol=1e-15)


def test_full_workload_matches_torch_fp64():
    inp = syn.conv_groupnorm_inputs(16, 128, 256, 1024, 32, seed=0)
    out = oracle.conv_groupnorm(inp.x, inp.weight, None, 32, inp.gamma, inp.beta, inp.eps)
    ref = _torch_fp64(inp.x, inp.weight, None, 32, inp.gamma, inp.beta, inp.eps)
    assert _rel(out, ref) < 1e-12


@pytest.mark.parametrize("stride,padding,dilation,K,bias,affine",
                         [(1, 1, 1, 3, False, True), (2, 1, 1, 3, True, True),
                          (1, 2, 2, 3, False, False), (1, 0, 1, 5, True, True),
                          (3, 4, 2, 5, False, True)])
def test_general_conv_parameters_match_torch(stride, padding, dilation, K, bias, affine):
    g = torch.Generator().manual_seed(11)
    x = torch.randn(2, 6, 37, generator=g)
    w = torch.randn(12, 6, K, generator=g) * 0.3
    b = torch.randn(12, generator=g) if bias else None
    gamma = torch.rand(12, generator=g) + 0.5 if affine else None
    beta = torch.rand(12, generator=g) - 0.5 if affine else None
    out = oracle.conv_groupnorm(x, w, b, 4, gamma, beta, 1e-5, stride, padding, dilation)
    ref = _torch_fp64(x, w, b, 4, gamma, beta, 1e-5, stride, padding, dilation)
    assert _rel(out, ref) < 1e-12


def test_groupwise_constant_affine_gives_beta_mean_and_scaled_variance():
    inp = syn.conv_groupnorm_inputs(2, 16, 32, 64, 4, seed=12)
    cpg = 8
    gam = torch.repeat_interleave(torch.tensor([0.5, 1.0, 2.0, 3.0]), cpg)
    bet = torch.repeat_interleave(torch.tensor([-1.0, 0.0, 0.25, 4.0]), cpg)
    out = oracle.conv_groupnorm(inp.x, inp.weight, None, 4, gam, bet, 1e-5)
    y = torch.nn.functional.conv1d(inp.x.double(), inp.weight.double(), padding=1).numpy()
    for n in range(2):
        for g in range(4):
            blk = out[n, g * cpg:(g + 1) * cpg]
            s2 = y[n, g * cpg:(g + 1) * cpg].var()           # biased, numpy default
            assert abs(blk.mean() - float(bet[g * cpg])) < 1e-12
            assert abs(blk.var() - float(gam[g * cpg]) ** 2 * s2 / (s2 + 1e-5)) < 1e-11


def test_no_affine_gives_zero_mean_groups():
    inp = syn.conv_groupnorm_inputs(2, 8, 16, 50, 2, seed=13)
    out = oracle.conv_groupnorm(inp.x, inp.weight, None, 2, None, None, 1e-5)
    means = out.reshape(2, 2, -1).mean(axis=2)
    assert np.abs(means).max() < 1e-14


def _numpy_brute(x, w, G, gamma, beta, eps):
    x, w = np.asarray(x, np.float64), np.asarray(w, np.float64)
    N, Cin, T = x.shape
    Cout = w.shape[0]
    xp = np.pad(x, ((0, 0), (0, 0), (1, 1)))
    y = np.stack([sum(w[:, :, k] @ xp[n, :, k:k + T] for k in range(3)) for n in range(N)])
    yg = y.reshape(N, G, -1)
    mu = yg.mean(axis=2, keepdims=True)
    var = ((yg - mu) ** 2).mean(axis=2, keepdims=True)
    yn = ((yg - mu) / np.sqrt(var + eps)).reshape(N, Cout, T)
    return yn * np.asarray(gamma, np.float64)[None, :, None] + np.asarray(beta, np.float64)[None, :, None]


@pytest.mark.parametrize("N,Cin,Cout,T,G", [(1, 1, 2, 4, 1), (2, 3, 4, 8, 2), (1, 2, 6, 5, 3)])
def test_brute_force_tiny(N, Cin, Cout, T, G):
    inp = syn.conv_groupnorm_inputs(N, Cin, Cout, T, G, seed=14)
    out = oracle.conv_groupnorm(inp.x, inp.weight, None, G, inp.gamma, inp.beta, inp.eps)
    np.testing.assert_allclose(out, _numpy_brute(inp.x, inp.weight, G, inp.gamma, inp.beta,
                                                 inp.eps), rtol=1e-12, atol=1e-12)


def test_groups_match_full():
    inp = syn.conv_groupnorm_inputs(3, 8, 16, 40, 4, seed=15)
    full = oracle.conv_groupnorm(inp.x, inp.weight, None, 4, inp.gamma, inp.beta, inp.eps)
    sel, mv = oracle.conv_groupnorm_groups(inp.x, inp.weight, None, 4, inp.gamma, inp.beta,
                                           inp.eps, [2, 0], [3, 1])
    assert np.array_equal(sel[0], full[2, 12:16])
    assert np.array_equal(sel[1], full[0, 4:8])
    assert mv.shape == (2, 2) and np.all(mv[:, 1] > 0)
