"""GPU parity of nrc_conv1d_groupnorm against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from normalization_convolution_blocks_gb300 import synthetic as syn
from gpu_util import Guarded, assert_f32, need_gpu, to

pytestmark = pytest.mark.gpu


def _gpu(dev, g, G, bias=None, affine=True, stride=1, padding=1, dilation=1):
    from normalization_convolution_blocks_gb300 import api
    N, _, T = g.x.shape
    Cout, _, k = g.weight.shape
    T_out = api.conv1d_output_length(T, k, stride, padding, dilation)
    gd = Guarded((N, Cout, T_out), torch.float32, dev)
    out = api.conv1d_groupnorm(to(dev, g.x), to(dev, g.weight), to(dev, bias), G,
                               to(dev, g.gamma) if affine else None,
                               to(dev, g.beta) if affine else None, g.eps, stride=stride,
                               padding=padding, dilation=dilation, out=gd.view)
    assert api.query_status() == api.NRC_OK
    gd.check(f"conv+GN N{N} {Cout} T_out{T_out}")
    return out.double().cpu().numpy()


def _ref(g, G, bias=None, affine=True, stride=1, padding=1, dilation=1):
    return oracle.conv_groupnorm(g.x, g.weight, bias, G, g.gamma if affine else None,
                                 g.beta if affine else None, g.eps, stride=stride,
                                 padding=padding, dilation=dilation)


def test_full_workload():
    """Every element, and each sample's groups on their own (an error in one
    sample's statistics cannot hide in the global norm)."""
    dev = need_gpu()
    g = syn.WORKLOADS["conv1d_groupnorm_f32"].make(seed=0)
    got, ref = _gpu(dev, g, 32), _ref(g, 32)
    assert_f32(got, ref, "N16 128->256 T1024 G32")
    cpg = got.shape[1] // 32
    for n in range(got.shape[0]):
        for grp in range(32):
            sl = slice(grp * cpg, (grp + 1) * cpg)
            assert_f32(got[n, sl], ref[n, sl], f"sample {n} group {grp}")


@pytest.mark.parametrize("N,Cin,Cout,T,G", [
    (1, 3, 16, 50, 2),        # tiny
    (2, 64, 40, 1000, 5),     # C_out not a multiple of 16 (tile 48), ragged T
    (1, 130, 96, 257, 12),    # C_in not a multiple of 64
    (2, 32, 512, 300, 32),    # two output tiles, 16 channels per group
    (1, 16, 256, 128, 1),     # one group spanning the whole tile
    (1, 16, 256, 130, 256),   # one channel per group
    (2, 24, 48, 136, 24),     # 2 channels per group
    (1, 40, 64, 200, 16),     # 4 channels per group
    (2, 70, 96, 264, 8),      # 12 channels per group: groups cross 16-channel chunks
])
def test_shapes(N, Cin, Cout, T, G):
    dev = need_gpu()
    g = syn.conv_groupnorm_inputs(N, Cin, Cout, T, G, seed=Cin + Cout + T)
    assert_f32(_gpu(dev, g, G), _ref(g, G), f"N{N} {Cin}->{Cout} T{T} G{G}")


# More tiles than SMs: the two-kernel path (per-row partials, then the
# finalize+normalize kernel).  The shapes above fit one wave of resident CTAs
# and take the fused path (statistics exchanged behind a grid-wide barrier,
# the normalization applied from tensor memory).
@pytest.mark.parametrize("N,Cin,Cout,T,G", [
    (4, 16, 64, 5000, 8),     # 160 tiles, ragged T
    (2, 16, 512, 5000, 32),   # 160 tiles over two output tiles
])
def test_shapes_more_tiles_than_sms(N, Cin, Cout, T, G):
    dev = need_gpu()
    n_tiles = N * -(-T // 128) * -(-Cout // 256)
    assert n_tiles > torch.cuda.get_device_properties(dev).multi_processor_count
    g = syn.conv_groupnorm_inputs(N, Cin, Cout, T, G, seed=Cin + Cout + T + 1)
    assert_f32(_gpu(dev, g, G), _ref(g, G), f"N{N} {Cin}->{Cout} T{T} G{G}")


def test_bias_and_no_affine():
    dev = need_gpu()
    g = syn.conv_groupnorm_inputs(2, 32, 64, 200, 8, seed=3)
    bias = torch.linspace(-1, 1, 64)
    assert_f32(_gpu(dev, g, 8, bias=bias), _ref(g, 8, bias=bias), "with bias")
    got = _gpu(dev, g, 8, affine=False)
    assert_f32(got, _ref(g, 8, affine=False), "affine off")
    assert np.abs(got.reshape(2, 8, -1).mean(axis=2)).max() < 1e-5


def test_full_workload_group_stats():
    """Group means and variances of the output match the oracle's (beta, gamma^2)
    relation on the full workload: the statistics path, checked on its own."""
    dev = need_gpu()
    g = syn.WORKLOADS["conv1d_groupnorm_f32"].make(seed=0)
    got = _gpu(dev, g, 32, affine=False)
    per = got.reshape(16, 32, -1)
    assert np.abs(per.mean(axis=2)).max() < 1e-5
    _, mv = oracle.conv_groupnorm_groups(g.x, g.weight, None, 32, None, None, g.eps,
                                         [0, 15], [0, 31])
    for r, (n, gg) in enumerate([(0, 0), (15, 31)]):
        s2 = mv[r, 1]
        assert abs(per[n, gg].var() - s2 / (s2 + g.eps)) < 1e-5


# General conv parameters (the module's kernel_size, stride, padding and
# dilation).  Stride 1 stages x by TMA boxes; stride > 1 loads it directly.
# Each case runs on one wave of resident CTAs (the fused kernel) and on more
# tiles than SMs (GEMM + finalize kernel), with the affine on and off.
GENERAL = [
    # (k, stride, padding, dilation)
    (3, 2, 1, 1),
    (3, 1, 2, 2),
    (5, 1, 2, 1),
    (5, 3, 4, 2),
    (1, 1, 0, 1),         # pointwise
    (7, 2, 0, 3),         # no padding: the output is shorter than the input
    (4, 1, 5, 1),         # even kernel, padding larger than half the span (T_out > T)
]


@pytest.mark.parametrize("k,s,pad,d", GENERAL)
@pytest.mark.parametrize("affine", [True, False])
@pytest.mark.parametrize("wave", ["one", "multi"])
def test_general_conv_parameters(k, s, pad, d, affine, wave):
    dev = need_gpu()
    from normalization_convolution_blocks_gb300 import api
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    if wave == "one":
        N, Cin, Cout, T, G = 2, 40, 96, 700, 12       # 8 ch/group, ragged Cin
    else:
        N, Cin, Cout, T, G = 3, 24, 64, 8000 * s, 8   # > SMs tiles
    T_out = api.conv1d_output_length(T, k, s, pad, d)
    assert T_out == oracle.conv1d_out_len(T, k, s, pad, d) > 0
    n_tiles = N * -(-T_out // 128) * -(-Cout // 256)
    assert (n_tiles <= sms) == (wave == "one"), n_tiles
    g = syn.conv_groupnorm_inputs(N, Cin, Cout, T, G, seed=k * 100 + s * 10 + pad + d,
                                  kernel_size=k)
    kw = dict(affine=affine, stride=s, padding=pad, dilation=d)
    got = _gpu(dev, g, G, **kw)
    assert got.shape == (N, Cout, T_out)
    assert_f32(got, _ref(g, G, **kw), f"k{k} s{s} p{pad} d{d} affine={affine} {wave} wave")


def test_general_conv_with_bias_and_unaligned_rows():
    """T not a multiple of 4 (rows not 16-byte aligned: no TMA boxes) with a
    dilated, padded kernel and a conv bias."""
    dev = need_gpu()
    g = syn.conv_groupnorm_inputs(2, 33, 48, 301, 6, seed=77, kernel_size=5)
    bias = torch.linspace(-0.5, 0.5, 48)
    kw = dict(bias=bias, stride=1, padding=3, dilation=2)
    assert_f32(_gpu(dev, g, 6, **kw), _ref(g, 6, **kw), "k5 d2 p3 T301 with bias")


@pytest.mark.parametrize("N,Cin,Cout,T,G,k,s,p,d,chunk_n,affine,bias", [
    (16, 128, 256, 1024, 32, 3, 1, 1, 1, 4, True, False),    # the workload, chunks of 4
    (7, 64, 40, 1000, 5, 3, 1, 1, 1, 2, True, True),         # ragged chunks, conv bias
    (5, 32, 64, 300, 8, 5, 3, 4, 2, 3, False, False),        # general conv, no affine
    (6, 64, 128, 4096, 16, 3, 1, 1, 1, 6, True, False),      # 192 tiles: the multi-wave path
])
def test_host_buffer_entry_matches_device_entry(N, Cin, Cout, T, G, k, s, p, d, chunk_n, affine,
                                                bias):
    """The host-buffer entry (chunks of samples) against the device entry:
    bitwise equal, and within the fp32 bar of the oracle."""
    dev = need_gpu()
    from normalization_convolution_blocks_gb300 import api
    g = syn.conv_groupnorm_inputs(N, Cin, Cout, T, G, seed=N + Cin + T, kernel_size=k)
    cb = torch.rand(Cout) - 0.5 if bias else None
    ref = api.conv1d_groupnorm(to(dev, g.x), to(dev, g.weight), to(dev, cb), G,
                               to(dev, g.gamma) if affine else None,
                               to(dev, g.beta) if affine else None, g.eps, stride=s, padding=p,
                               dilation=d)
    pin = lambda t: None if t is None else t.contiguous().pin_memory()  # noqa: E731
    T_out = api.conv1d_output_length(T, k, s, p, d)
    out = torch.full((N, Cout, T_out), float("nan")).pin_memory()
    got = api._gn_host(api.load(), dev, pin(g.x), pin(g.weight), pin(cb), G,
                       pin(g.gamma) if affine else None, pin(g.beta) if affine else None, g.eps,
                       None, s, p, d, out, None, None, chunk_n=chunk_n)
    assert api.query_status() == api.NRC_OK
    tiles = N * -(-api.conv1d_output_length(T, k, s, p, d) // 128) * -(-Cout // 256)
    if tiles <= torch.cuda.get_device_properties(dev).multi_processor_count:
        # the whole batch fits one wave, so every chunk does too: the same fused
        # kernel path, bitwise equal
        assert torch.equal(got, ref.cpu()), "host entry differs from the device entry"
    else:
        # the whole batch takes the multi-wave path, a chunk may take the fused
        # one: the group statistics are summed in another order
        assert (got - ref.cpu()).abs().max().item() < 1e-5, "host entry far from the device entry"
    want = oracle.conv_groupnorm(g.x, g.weight, cb, G, g.gamma if affine else None,
                                 g.beta if affine else None, g.eps, stride=s, padding=p,
                                 dilation=d)
    assert_f32(got.double().numpy(), want, f"host entry N{N} {Cin}->{Cout} T{T}")
