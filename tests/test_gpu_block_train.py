"""GPU parity of nrc_prenorm_dilconv_residual_train (BatchNorm1d in training
mode) against the fp64 oracle: the output, the updated running buffers and
num_batches_tracked."""
import numpy as np
import pytest
import torch

import oracle
from normalization_convolution_blocks_gb300 import synthetic as syn
from gpu_util import RUNNING_STAT_ABS, Guarded, assert_bf16, assert_f32, need_gpu, to

pytestmark = pytest.mark.gpu


def _gpu(dev, inp, momentum=0.1, x=None, buffers=True):
    """Runs the training-mode block; returns (out, running_mean, running_var, nbt)
    as float64 numpy arrays (None for absent buffers)."""
    from normalization_convolution_blocks_gb300 import api
    rm = to(dev, inp.running_mean).clone() if buffers else None
    rv = to(dev, inp.running_var).clone() if buffers else None
    nbt = torch.zeros(1, dtype=torch.int64, device=dev) if buffers else None
    xd = to(dev, inp.x) if x is None else x
    g = Guarded(tuple(xd.shape), xd.dtype, dev)
    out = api.prenorm_dilconv_residual_train(xd, rm, rv, to(dev, inp.gamma), to(dev, inp.beta),
                                             inp.eps, momentum, to(dev, inp.weight),
                                             to(dev, inp.bias), inp.dilation,
                                             num_batches_tracked=nbt, out=g.view)
    assert api.query_status() == api.NRC_OK
    g.check(f"training-mode block {tuple(xd.shape)}")
    cpu = (lambda t: None if t is None else t.double().cpu().numpy())
    return cpu(out), cpu(rm), cpu(rv), (None if nbt is None else int(nbt.item()))


def _oracle(inp, momentum=0.1, rows_n=None, rows_o=None):
    return oracle.prenorm_block_train(inp.x, inp.running_mean, inp.running_var, inp.gamma,
                                      inp.beta, inp.eps, momentum, inp.weight, inp.bias,
                                      inp.dilation, rows_n=rows_n, rows_o=rows_o)


def _check_buffers(rm, rv, ref_rm, ref_rv, what):
    drm, drv = np.abs(rm - ref_rm).max(), np.abs(rv - ref_rv).max()
    assert drm < RUNNING_STAT_ABS and drv < RUNNING_STAT_ABS, f"{what}: {drm:.2e} {drv:.2e}"


def test_tiny_workload_fp32():
    dev = need_gpu()
    inp = syn.WORKLOADS["prenorm_block_tiny_f32"].make(seed=0)
    out, rm, rv, nbt = _gpu(dev, inp)
    ref, ref_rm, ref_rv, _, _ = _oracle(inp)
    assert_f32(out, ref, "train N2 C32 L512 d128")
    _check_buffers(rm, rv, ref_rm, ref_rv, "train tiny")
    assert nbt == 1


@pytest.mark.parametrize("N,C,L,d", [
    (1, 16, 128, 1),        # one tile, one sample
    (2, 48, 300, 7),        # L % 4 != 0: scalar loads in the statistics kernel
    (3, 64, 5000, 64),      # two statistics chunks per row, ragged last chunk
    (1, 300, 260, 64),      # two output tiles
    (4, 8, 5, 2),           # L smaller than a tile
    (2, 256, 512, 128),     # full-width output tile
])
def test_shapes_fp32(N, C, L, d):
    dev = need_gpu()
    inp = syn.prenorm_block_inputs(N, C, L, d, seed=N * 1000 + C + d + 7)
    out, rm, rv, _ = _gpu(dev, inp, momentum=0.3)
    ref, ref_rm, ref_rv, _, _ = _oracle(inp, momentum=0.3)
    assert_f32(out, ref, f"train N{N} C{C} L{L} d{d}")
    _check_buffers(rm, rv, ref_rm, ref_rv, f"train N{N} C{C} L{L} d{d}")


@pytest.mark.parametrize("N,C,L,d", [
    (2, 128, 264, 2),       # L % 8 == 0: 16-byte loads
    (2, 64, 300, 5),        # L % 8 != 0: scalar loads
    (1, 32, 9000, 16),      # two statistics chunks per row
])
def test_shapes_bf16(N, C, L, d):
    dev = need_gpu()
    inp = syn.prenorm_block_inputs(N, C, L, d, seed=N * 13 + C + d, dtype=torch.bfloat16)
    out, rm, rv, _ = _gpu(dev, inp)
    ref, ref_rm, ref_rv, _, _ = _oracle(inp)
    assert_bf16(out, ref, f"train bf16 N{N} C{C} L{L} d{d}")
    _check_buffers(rm, rv, ref_rm, ref_rv, f"train bf16 N{N} C{C} L{L} d{d}")


def test_unaligned_view_takes_scalar_loads():
    """x starting one element past a 16-byte boundary."""
    dev = need_gpu()
    inp = syn.prenorm_block_inputs(2, 32, 256, 8, seed=21)
    flat = torch.empty(inp.x.numel() + 1, device=dev)
    xv = flat[1:].view(inp.x.shape)
    xv.copy_(inp.x.to(dev))
    out, rm, rv, _ = _gpu(dev, inp, x=xv)
    ref, ref_rm, ref_rv, _, _ = _oracle(inp)
    assert_f32(out, ref, "train unaligned x")
    _check_buffers(rm, rv, ref_rm, ref_rv, "train unaligned x")


def test_full_workload_fp32_every_element():
    """N=32 C=256 L=4096 d=128: every output element and every running
    statistic, and each 128-row tile of every sample on its own, so an error
    confined to a few tiles cannot hide in the global norm."""
    dev = need_gpu()
    inp = syn.WORKLOADS["prenorm_block_f32"].make(seed=0)
    out, rm, rv, nbt = _gpu(dev, inp)
    ref, ref_rm, ref_rv, _, _ = _oracle(inp)
    assert_f32(out, ref, "train full workload, every element")
    N, C, L = out.shape
    for n in range(N):
        for t0 in range(0, L, 128):
            assert_f32(out[n, :, t0:t0 + 128], ref[n, :, t0:t0 + 128], f"train tile n{n} t{t0}")
    _check_buffers(rm, rv, ref_rm, ref_rv, "train full workload")
    assert nbt == 1


def test_full_bf16_workload_every_element():
    dev = need_gpu()
    inp = syn.WORKLOADS["prenorm_block_bf16_C256_d128"].make(seed=0)
    out, rm, rv, _ = _gpu(dev, inp)
    ref, ref_rm, ref_rv, _, _ = _oracle(inp)
    assert_bf16(out, ref, "train bf16 full, every element")
    for n in range(out.shape[0]):
        assert_bf16(out[n], ref[n], f"train bf16 full, sample {n}")
    _check_buffers(rm, rv, ref_rm, ref_rv, "train bf16 full")


def test_without_buffers_same_output():
    dev = need_gpu()
    inp = syn.prenorm_block_inputs(2, 64, 384, 16, seed=22)
    a = _gpu(dev, inp)[0]
    b, rm, rv, nbt = _gpu(dev, inp, buffers=False)
    assert rm is None and rv is None and nbt is None
    assert np.array_equal(a, b)


def test_offset_input_statistics_stay_accurate():
    """x around 50: a one-pass sum of squares would lose the variance."""
    dev = need_gpu()
    inp = syn.prenorm_block_inputs(4, 32, 1024, 4, seed=23)
    inp.x = inp.x + 50.0
    out, rm, rv, _ = _gpu(dev, inp)
    ref, ref_rm, ref_rv, _, _ = _oracle(inp)
    assert_f32(out, ref, "train offset x")
    _check_buffers(rm, rv, ref_rm, ref_rv, "train offset x")


def test_three_steps_track_the_oracle():
    """Three calls on the same buffers: the running statistics follow three
    oracle updates and num_batches_tracked counts them."""
    dev = need_gpu()
    from normalization_convolution_blocks_gb300 import api
    inp = syn.prenorm_block_inputs(2, 32, 512, 8, seed=24)
    rm = inp.running_mean.to(dev).clone()
    rv = inp.running_var.to(dev).clone()
    nbt = torch.zeros(1, dtype=torch.int64, device=dev)
    ref_rm, ref_rv = inp.running_mean, inp.running_var
    for step in range(3):
        x = inp.x * (1.0 + 0.5 * step) + 0.25 * step          # a different batch each step
        api.prenorm_dilconv_residual_train(x.to(dev), rm, rv, inp.gamma.to(dev),
                                           inp.beta.to(dev), inp.eps, 0.1, inp.weight.to(dev),
                                           inp.bias.to(dev), inp.dilation,
                                           num_batches_tracked=nbt)
        _, ref_rm, ref_rv, _, _ = oracle.prenorm_block_train(
            x, ref_rm, ref_rv, inp.gamma, inp.beta, inp.eps, 0.1, inp.weight, inp.bias,
            inp.dilation, rows_n=[0], rows_o=[0])
    assert api.query_status() == api.NRC_OK
    _check_buffers(rm.double().cpu().numpy(), rv.double().cpu().numpy(), ref_rm, ref_rv,
                   "three steps")
    assert int(nbt.item()) == 3


@pytest.mark.parametrize("N,C,L,d,chunk_n,dtype", [
    (8, 64, 1000, 16, 2, torch.float32),      # ramped chunks 1,1,2,2,1,1 ... of a small batch
    (5, 96, 2048, 128, 2, torch.bfloat16),    # bf16, ragged chunking
    (3, 32, 300, 7, 1, torch.float32),        # L % 4 != 0: scalar statistics loads
    (32, 256, 4096, 128, 4, torch.float32),   # the full workload
])
def test_host_buffer_entry_matches_device_entry(N, C, L, d, chunk_n, dtype):
    """The host-buffer entry (statistics per chunk as x arrives, then the block
    per chunk) against the device entry on the whole batch: bitwise equal
    output, running buffers and num_batches_tracked."""
    dev = need_gpu()
    from normalization_convolution_blocks_gb300 import api
    inp = syn.prenorm_block_inputs(N, C, L, d, seed=N + C + L, dtype=dtype)
    rm_d, rv_d = to(dev, inp.running_mean).clone(), to(dev, inp.running_var).clone()
    nbt_d = torch.zeros(1, dtype=torch.int64, device=dev)
    ref = api.prenorm_dilconv_residual_train(to(dev, inp.x), rm_d, rv_d, to(dev, inp.gamma),
                                             to(dev, inp.beta), inp.eps, 0.1,
                                             to(dev, inp.weight), to(dev, inp.bias), d,
                                             num_batches_tracked=nbt_d)
    rm_h, rv_h = to(dev, inp.running_mean).clone(), to(dev, inp.running_var).clone()
    nbt_h = torch.zeros(1, dtype=torch.int64, device=dev)
    pin = lambda t: t.contiguous().pin_memory()  # noqa: E731
    out = torch.full(tuple(inp.x.shape), float("nan"), dtype=dtype).pin_memory()
    dt = api.NRC_F32 if dtype == torch.float32 else api.NRC_BF16
    got = api._train_host(api.load(), dev, dt, pin(inp.x), rm_h, rv_h, pin(inp.gamma),
                          pin(inp.beta), inp.eps, 0.1, pin(inp.weight), pin(inp.bias), d, None,
                          3, nbt_h, out, None, None, chunk_n=chunk_n)
    assert api.query_status() == api.NRC_OK
    assert torch.equal(got, ref.cpu()), "host entry differs from the device entry"
    assert torch.equal(rm_h, rm_d) and torch.equal(rv_h, rv_d), "running buffers differ"
    assert int(nbt_h.item()) == int(nbt_d.item()) == 1
