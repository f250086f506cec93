"""GPU parity on adversarial inputs: wide dynamic range inside one K block.

The fp32-storage path splits every operand into two bf16 parts (hi + lo) and
sums three products per term.  Each part carries its own exponent, so the split
is exact to about 2^-16 relative whatever the operand's magnitude; these tests
pin that on inputs built to break a scheme with a shared or fixed scale:

* per-channel scales of x spanning 2^-8 .. 2^8, interleaved so that every
  32- and 64-channel K block mixes them;
* a sprinkling of large entries (|x| = 1e4) and exact zeros;
* per-channel BatchNorm affines and per-row weight scales spanning 2^-4 .. 2^4.

The comparison is scale-free: relative L2 over the whole output within the
fp32 bar (1e-4), the largest error within 1e-3 of the output's largest
magnitude (the max-abs bar of 1e-3 restated for data that is not of unit
scale), and every output channel's own relative L2 within 1e-3, so an error
confined to the small channels cannot hide behind the large ones.  Outputs that
a normalization brings back to unit scale (GroupNorm, training-mode BatchNorm)
are held to the plain fp32 bar.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import BF16_REL_L2, F32_MAX_ABS, F32_REL_L2, Guarded, assert_f32, errors, need_gpu, to
from normalization_convolution_blocks_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu


def _pow2(g, n, lo, hi):
    """n powers of two with exponents uniform in [lo, hi], in a shuffled order."""
    e = torch.randint(lo, hi + 1, (n,), generator=g)
    return torch.pow(2.0, e.float())


def _spiky(g, shape, frac=1e-3, big=1e4):
    """N(0,1) with a fraction of entries set to +-big and as many to zero."""
    x = torch.randn(shape, generator=g)
    u = torch.rand(shape, generator=g)
    sign = torch.where(torch.rand(shape, generator=g) < 0.5, -1.0, 1.0)
    x = torch.where(u < frac, sign * big, x)
    return torch.where((u >= frac) & (u < 2 * frac), torch.zeros_like(x), x)


def _scale_free_check(got, ref, what, axis_channels=1):
    rel, mx = errors(got, ref)
    scale = float(np.abs(ref).max())
    assert rel < F32_REL_L2, f"{what}: rel_l2={rel:.3e}"
    assert mx < F32_MAX_ABS * scale, f"{what}: max_abs={mx:.3e} against scale {scale:.3e}"
    moved = np.moveaxis(np.asarray(got, np.float64), axis_channels, 0)
    refm = np.moveaxis(np.asarray(ref, np.float64), axis_channels, 0)
    num = np.sqrt(((moved - refm) ** 2).reshape(moved.shape[0], -1).sum(axis=1))
    den = np.sqrt((refm ** 2).reshape(refm.shape[0], -1).sum(axis=1))
    worst = float((num / np.maximum(den, 1e-300)).max())
    assert worst < 1e-3, f"{what}: worst channel rel_l2={worst:.3e}"
    return rel, mx, worst


def _block_inputs(N, C, L, d, seed, dtype=torch.float32):
    g = torch.Generator("cpu").manual_seed(seed)
    x = _spiky(g, (N, C, L)) * _pow2(g, C, -8, 8).view(1, C, 1)
    rm = torch.zeros(C)
    rv = torch.ones(C)
    gamma = _pow2(g, C, -4, 4) * torch.where(torch.rand(C, generator=g) < 0.5, -1.0, 1.0)
    beta = torch.rand(C, generator=g) * 2 - 1
    bound = 1.0 / np.sqrt(3 * C)
    w = (torch.rand((C, C, 3), generator=g) * 2 - 1) * bound * _pow2(g, C, -4, 4).view(C, 1, 1)
    b = (torch.rand(C, generator=g) * 2 - 1) * bound
    if dtype != torch.float32:
        x, w, b = x.to(dtype), w.to(dtype), b.to(dtype)
    return syn.BlockInputs(x, rm, rv, gamma, beta, w, b, d)


def _block_gpu(dev, inp):
    from normalization_convolution_blocks_gb300 import api
    gd = Guarded(tuple(inp.x.shape), inp.x.dtype, dev)
    out = api.prenorm_dilconv_residual(to(dev, inp.x), to(dev, inp.running_mean),
                                       to(dev, inp.running_var), to(dev, inp.gamma),
                                       to(dev, inp.beta), inp.eps, to(dev, inp.weight),
                                       to(dev, inp.bias), inp.dilation, out=gd.view)
    assert api.query_status() == api.NRC_OK
    gd.check("adversarial block")
    return out.double().cpu().numpy()


def _block_ref(inp):
    return oracle.prenorm_block(inp.x, inp.running_mean, inp.running_var, inp.gamma, inp.beta,
                                inp.eps, inp.weight, inp.bias, inp.dilation)


@pytest.mark.parametrize("N,C,L,d", [
    (2, 256, 1024, 8),       # full-width output tile, 12 K stages
    (1, 320, 520, 128),      # two output tiles, ragged C and L
])
def test_block_fp32_wide_range(N, C, L, d):
    dev = need_gpu()
    inp = _block_inputs(N, C, L, d, seed=C + L + d)
    _scale_free_check(_block_gpu(dev, inp), _block_ref(inp), f"block N{N} C{C} L{L} d{d}")


def test_block_bf16_wide_range():
    dev = need_gpu()
    inp = _block_inputs(2, 256, 2048, 4, seed=17, dtype=torch.bfloat16)
    got, ref = _block_gpu(dev, inp), _block_ref(inp)
    rel, _ = errors(got, ref)
    assert rel < BF16_REL_L2, f"bf16 block: rel_l2={rel:.3e}"


def test_conv_groupnorm_wide_range():
    dev = need_gpu()
    from normalization_convolution_blocks_gb300 import api
    g = torch.Generator("cpu").manual_seed(5)
    N, Cin, Cout, T, G = 4, 128, 256, 512, 32
    x = _spiky(g, (N, Cin, T)) * _pow2(g, Cin, -8, 8).view(1, Cin, 1)
    bound = 1.0 / np.sqrt(3 * Cin)
    w = (torch.rand((Cout, Cin, 3), generator=g) * 2 - 1) * bound
    w = w * _pow2(g, Cout, -4, 4).view(Cout, 1, 1)
    gamma = torch.rand(Cout, generator=g) + 0.5
    beta = torch.rand(Cout, generator=g) - 0.5
    gd = Guarded((N, Cout, T), torch.float32, dev)
    out = api.conv1d_groupnorm(to(dev, x), to(dev, w), None, G, to(dev, gamma), to(dev, beta),
                               1e-5, out=gd.view)
    assert api.query_status() == api.NRC_OK
    gd.check("adversarial conv+GN")
    ref = oracle.conv_groupnorm(x, w, None, G, gamma, beta, 1e-5)
    assert_f32(out.double().cpu().numpy(), ref, "conv+GN wide range")


@pytest.mark.parametrize("training", [True, False])
def test_linear_wide_range(training):
    dev = need_gpu()
    from normalization_convolution_blocks_gb300 import api
    g = torch.Generator("cpu").manual_seed(9)
    B, IN, OUT = 256, 1024, 512
    x = _spiky(g, (B, IN)) * _pow2(g, IN, -8, 8).view(1, IN)
    bound = 1.0 / np.sqrt(IN)
    w = (torch.rand((OUT, IN), generator=g) * 2 - 1) * bound * _pow2(g, OUT, -4, 4).view(OUT, 1)
    b_lin = (torch.rand(OUT, generator=g) * 2 - 1) * bound
    gamma = torch.rand(OUT, generator=g) + 0.5
    beta = torch.rand(OUT, generator=g) - 0.5
    add_bias = torch.randn(1, generator=g)
    if training:
        rm, rv = torch.zeros(OUT), torch.ones(OUT)
    else:
        # running statistics of the right scale, so the output is of unit scale
        y = (x.double() @ w.double().t() + b_lin.double())
        rm = y.mean(0).float()
        rv = (y.var(0) * (1 + torch.rand(OUT, generator=g).double())).float()
    rm_d, rv_d = to(dev, rm).clone(), to(dev, rv).clone()
    gd = Guarded((B, OUT), torch.float32, dev)
    out = api.linear_bn_swish(to(dev, x), to(dev, w), to(dev, b_lin), to(dev, gamma),
                              to(dev, beta), rm_d, rv_d, to(dev, add_bias), 1.0, 1e-5, 0.1,
                              training, None, out=gd.view)
    assert api.query_status() == api.NRC_OK
    gd.check("adversarial linear")
    r_out, r_rm, r_rv, _ = oracle.linear_bn_swish(x, w, b_lin, gamma, beta, rm, rv, 1e-5, 0.1,
                                                  training, float(add_bias[0]), 1.0)
    assert_f32(out.double().cpu().numpy(), r_out, f"linear wide range training={training}")
    if training:
        # The running statistics carry the features' own scale (the variance
        # reaches ~1e12 here) and the batch mean is a cancelling sum, so each
        # is held against the scale of its own term: momentum * std(y) for the
        # mean, momentum * var(y) for the variance, y = x W^T + b_lin.
        y = x.double() @ w.double().t() + b_lin.double()
        std_y = y.std(0).numpy()
        for got, ref, unit, name in ((rm_d, r_rm, 0.1 * std_y, "running_mean"),
                                     (rv_d, r_rv, 0.1 * std_y ** 2, "running_var")):
            got = got.double().cpu().numpy()
            err = np.abs(got - ref) / unit
            assert float(err.max()) < 1e-4, f"{name}: {float(err.max()):.3e}"
