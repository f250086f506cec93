"""Property-based pins of the oracle (CPU only; skipped without hypothesis).

Random small problems -- shapes, dilations, strides, group counts, momenta,
affine on or off -- each compared with PyTorch's own fp64 modules, which the
pages state the problems as.  The fixed-shape pins elsewhere pick the edge
cases by hand; these sweep the space between them.
"""
import numpy as np
import pytest
import torch

import oracle

hyp = pytest.importorskip("hypothesis")
st = pytest.importorskip("hypothesis.strategies")
given, settings = hyp.given, hyp.settings

SETTINGS = dict(max_examples=40, deadline=None, derandomize=True)


def _rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def _draw(seed, *shapes):
    g = torch.Generator().manual_seed(seed)
    return [torch.randn(s, generator=g, dtype=torch.float64) for s in shapes]


@settings(**SETTINGS)
@given(N=st.integers(1, 3), C=st.integers(1, 6), L=st.integers(1, 40), d=st.integers(1, 45),
       train=st.booleans(), momentum=st.sampled_from([0.0, 0.1, 0.5, 1.0]),
       seed=st.integers(0, 2**31 - 1))
def test_block_matches_torch_modules(N, C, L, d, train, momentum, seed):
    if train and N * L < 2:
        return
    x, w, b, rm, gamma, beta = _draw(seed, (N, C, L), (C, C, 3), (C,), (C,), (C,), (C,))
    rv = torch.rand(C, generator=torch.Generator().manual_seed(seed + 1),
                    dtype=torch.float64) + 0.5
    bn = torch.nn.BatchNorm1d(C, eps=1e-5, momentum=momentum).double()
    conv = torch.nn.Conv1d(C, C, 3, padding=d, dilation=d).double()
    with torch.no_grad():
        bn.running_mean.copy_(rm)
        bn.running_var.copy_(rv)
        bn.weight.copy_(gamma)
        bn.bias.copy_(beta)
        conv.weight.copy_(w)
        conv.bias.copy_(b)
        bn.train(train)
        ref = (x + conv(torch.relu(bn(x)))).numpy()
    if train:
        out, o_rm, o_rv, _, _ = oracle.prenorm_block_train(x, rm, rv, gamma, beta, 1e-5, momentum,
                                                           w, b, d)
        np.testing.assert_allclose(o_rm, bn.running_mean.numpy(), rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(o_rv, bn.running_var.numpy(), rtol=1e-12, atol=1e-14)
    else:
        out = oracle.prenorm_block(x, rm, rv, gamma, beta, 1e-5, w, b, d)
    assert _rel(out, ref) < 1e-12


@settings(**SETTINGS)
@given(N=st.integers(1, 3), Cin=st.integers(1, 5), G=st.integers(1, 4), cpg=st.integers(1, 4),
       T=st.integers(3, 40), K=st.integers(1, 4), stride=st.integers(1, 3),
       padding=st.integers(0, 3), dilation=st.integers(1, 3), affine=st.booleans(),
       bias=st.booleans(), seed=st.integers(0, 2**31 - 1))
def test_conv_groupnorm_matches_torch_modules(N, Cin, G, cpg, T, K, stride, padding, dilation,
                                              affine, bias, seed):
    Cout = G * cpg
    if (T + 2 * padding - dilation * (K - 1) - 1) // stride + 1 < 1:
        return
    x, w, b, gamma, beta = _draw(seed, (N, Cin, T), (Cout, Cin, K), (Cout,), (Cout,), (Cout,))
    conv = torch.nn.Conv1d(Cin, Cout, K, stride=stride, padding=padding, dilation=dilation,
                           bias=bias).double()
    gn = torch.nn.GroupNorm(G, Cout, eps=1e-5, affine=affine).double()
    with torch.no_grad():
        conv.weight.copy_(w)
        if bias:
            conv.bias.copy_(b)
        if affine:
            gn.weight.copy_(gamma)
            gn.bias.copy_(beta)
        ref = gn(conv(x)).numpy()
    out = oracle.conv_groupnorm(x, w, b if bias else None, G, gamma if affine else None,
                                beta if affine else None, 1e-5, stride=stride, padding=padding,
                                dilation=dilation)
    # one output value per group makes the normalized group exactly zero: compare absolutely
    np.testing.assert_allclose(out, ref, rtol=1e-9, atol=1e-9)


@settings(**SETTINGS)
@given(B=st.integers(1, 12), IN=st.integers(1, 20), OUT=st.integers(1, 10),
       train=st.booleans(), momentum=st.sampled_from([0.0, 0.1, 0.7]),
       divide=st.sampled_from([1.0, 2.5, -0.5]), affine=st.booleans(),
       seed=st.integers(0, 2**31 - 1))
def test_linear_bn_swish_matches_torch_modules(B, IN, OUT, train, momentum, divide, affine, seed):
    if train and B < 2:
        return
    x, w, lb, gamma, beta, rm, add = _draw(seed, (B, IN), (OUT, IN), (OUT,), (OUT,), (OUT,),
                                           (OUT,), (1,))
    rv = torch.rand(OUT, generator=torch.Generator().manual_seed(seed + 2),
                    dtype=torch.float64) + 0.5
    lin = torch.nn.Linear(IN, OUT).double()
    bn = torch.nn.BatchNorm1d(OUT, eps=1e-5, momentum=momentum, affine=affine).double()
    with torch.no_grad():
        lin.weight.copy_(w)
        lin.bias.copy_(lb)
        bn.running_mean.copy_(rm)
        bn.running_var.copy_(rv)
        if affine:
            bn.weight.copy_(gamma)
            bn.bias.copy_(beta)
        bn.train(train)
        u = (bn(lin(x)) + add) / divide
        ref = (u * torch.sigmoid(u)).numpy()
    out, o_rm, o_rv, _ = oracle.linear_bn_swish(x, w, lb, gamma if affine else None,
                                                beta if affine else None, rm, rv, 1e-5, momentum,
                                                train, float(add[0]), divide)
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(o_rm, bn.running_mean.numpy(), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(o_rv, bn.running_var.numpy(), rtol=1e-12, atol=1e-14)
