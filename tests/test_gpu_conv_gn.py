"""GPU parity of nrc_conv1d_groupnorm against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from normalization_convolution_blocks_gb300 import synthetic as syn
from gpu_util import assert_f32, need_gpu, to

pytestmark = pytest.mark.gpu


def _gpu(dev, g, G, bias=None, affine=True):
    from normalization_convolution_blocks_gb300 import api
    out = api.conv1d_groupnorm(to(dev, g.x), to(dev, g.weight), to(dev, bias), G,
                               to(dev, g.gamma) if affine else None,
                               to(dev, g.beta) if affine else None, g.eps)
    assert api.query_status() == api.NRC_OK
    return out.double().cpu().numpy()


def _ref(g, G, bias=None, affine=True):
    return oracle.conv_groupnorm(g.x, g.weight, bias, G, g.gamma if affine else None,
                                 g.beta if affine else None, g.eps)


def test_full_workload():
    dev = need_gpu()
    g = syn.WORKLOADS["conv1d_groupnorm_f32"].make(seed=0)
    assert_f32(_gpu(dev, g, 32), _ref(g, 32), "N16 128->256 T1024 G32")


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
