"""GPU parity of nrc_prenorm_dilconv_residual against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from normalization_convolution_blocks_gb300 import synthetic as syn
from gpu_util import Guarded, assert_bf16, assert_f32, need_gpu, to

pytestmark = pytest.mark.gpu


def _gpu(dev, inp, **kw):
    """One call into a guarded output buffer; the guards are checked after it."""
    from normalization_convolution_blocks_gb300 import api
    w = kw.get("w", inp.weight)
    b = kw.get("bias", inp.bias)
    g = Guarded(tuple(inp.x.shape), inp.x.dtype, dev)
    out = api.prenorm_dilconv_residual(to(dev, inp.x), to(dev, inp.running_mean),
                                       to(dev, inp.running_var), to(dev, inp.gamma),
                                       to(dev, inp.beta), inp.eps, to(dev, w), to(dev, b),
                                       inp.dilation, out=g.view)
    assert api.query_status() == api.NRC_OK
    g.check(f"block {tuple(inp.x.shape)} d{inp.dilation}")
    return out.double().cpu().numpy()


def _oracle(inp, **kw):
    return oracle.prenorm_block(inp.x, inp.running_mean, inp.running_var, inp.gamma, inp.beta,
                                inp.eps, kw.get("w", inp.weight), kw.get("bias", inp.bias),
                                inp.dilation)


def test_tiny_workload_fp32():
    dev = need_gpu()
    inp = syn.WORKLOADS["prenorm_block_tiny_f32"].make(seed=0)
    assert_f32(_gpu(dev, inp), _oracle(inp), "N2 C32 L512 d128")


@pytest.mark.parametrize("N,C,L,d", [
    (1, 16, 128, 1),        # one tile exactly
    (2, 48, 300, 7),        # C not a multiple of 32, ragged L tail
    (1, 64, 1000, 64),      # several tiles, ragged tail
    (2, 256, 512, 128),     # full-width o tile
    (1, 300, 260, 64),      # two o tiles, ragged channel count
    (1, 96, 200, 150),      # dilation > L/2: side taps mostly padding
    (1, 8, 5, 2),           # L smaller than a tile
    (1, 1, 64, 3),          # single channel
    (3, 80, 129, 128),      # tile + 1 row
])
def test_shapes_fp32(N, C, L, d):
    dev = need_gpu()
    inp = syn.prenorm_block_inputs(N, C, L, d, seed=N * 1000 + C + d)
    assert_f32(_gpu(dev, inp), _oracle(inp), f"N{N} C{C} L{L} d{d}")


@pytest.mark.parametrize("N,C,L,d", [
    (2, 128, 256, 4),       # 6 K stages: the column-half hand-over has no body stages
    (1, 2048, 64, 1),       # largest supported C: 96 K stages, 8 output tiles
])
def test_edge_shapes_fp32(N, C, L, d):
    dev = need_gpu()
    inp = syn.prenorm_block_inputs(N, C, L, d, seed=N * 7 + C + d)
    assert_f32(_gpu(dev, inp), _oracle(inp), f"N{N} C{C} L{L} d{d}")


@pytest.mark.parametrize("N,C,L,d", [
    (1, 128, 264, 2),       # 6 K stages, ragged tail
    (1, 768, 136, 3),       # three output tiles
])
def test_edge_shapes_bf16(N, C, L, d):
    dev = need_gpu()
    inp = syn.prenorm_block_inputs(N, C, L, d, seed=N * 11 + C + d, dtype=torch.bfloat16)
    assert_bf16(_gpu(dev, inp), _oracle(inp), f"bf16 N{N} C{C} L{L} d{d}")


def test_no_bias():
    dev = need_gpu()
    inp = syn.prenorm_block_inputs(2, 64, 256, 16, seed=5)
    assert_f32(_gpu(dev, inp, bias=None), _oracle(inp, bias=None), "no bias")


def test_zero_weights_reproduce_x_exactly():
    dev = need_gpu()
    inp = syn.prenorm_block_inputs(2, 64, 300, 8, seed=6)
    got = _gpu(dev, inp, w=torch.zeros_like(inp.weight), bias=torch.zeros_like(inp.bias))
    assert np.array_equal(got, inp.x.double().numpy())


def test_left_tap_identity_pins_padding_and_direction():
    dev = need_gpu()
    inp = syn.prenorm_block_inputs(1, 32, 400, 37, seed=7)
    C = 32
    w = torch.zeros(C, C, 3)
    w[torch.arange(C), torch.arange(C), 0] = 1.0
    assert_f32(_gpu(dev, inp, w=w, bias=torch.zeros(C)), _oracle(inp, w=w, bias=torch.zeros(C)),
               "left tap identity")


@pytest.mark.parametrize("C,d", [(256, 1), (256, 8), (256, 128), (256, 512), (512, 128)])
def test_bf16_storage(C, d):
    dev = need_gpu()
    inp = syn.prenorm_block_inputs(2, C, 2048, d, seed=C + d, dtype=torch.bfloat16)
    got = _gpu(dev, inp)
    assert_bf16(got, _oracle(inp), f"bf16 C{C} d{d}")


# bf16 rows are gathered by TMA boxes when L * 2 bytes is a multiple of 16 and
# loaded directly otherwise; both sides of that switch, with ragged tails,
# channel counts off the 32/64 grid and taps reaching past both ends.
@pytest.mark.parametrize("N,C,L,d", [
    (2, 96, 296, 5),        # boxes; ragged tail, odd dilation (unaligned tap offsets)
    (2, 96, 300, 5),        # direct loads (L*2 not a multiple of 16)
    (1, 40, 136, 200),      # boxes; dilation > L: side taps all padding
])
def test_bf16_shapes(N, C, L, d):
    dev = need_gpu()
    inp = syn.prenorm_block_inputs(N, C, L, d, seed=N * 100 + C + d, dtype=torch.bfloat16)
    assert_bf16(_gpu(dev, inp), _oracle(inp), f"bf16 N{N} C{C} L{L} d{d}")


def test_full_workload_fp32_every_element():
    """The full-size workload (N=32 C=256 L=4096 d=128) in the bench's launch
    configuration, compared with the oracle on every output element, and
    also per tile: each 128-row x 256-channel tile of every sample must meet
    the bar on its own, so an error confined to a few tiles cannot hide in
    the global norm."""
    dev = need_gpu()
    inp = syn.WORKLOADS["prenorm_block_f32"].make(seed=0)
    got = _gpu(dev, inp)
    ref = oracle.prenorm_block(inp.x, inp.running_mean, inp.running_var, inp.gamma, inp.beta,
                               inp.eps, inp.weight, inp.bias, inp.dilation)
    assert_f32(got, ref, "full workload, every element")
    N, C, L = got.shape
    for n in range(N):
        for t0 in range(0, L, 128):
            assert_f32(got[n, :, t0:t0 + 128], ref[n, :, t0:t0 + 128], f"tile n{n} t{t0}")


@pytest.mark.parametrize("C,d", [(C, d) for C in (256, 512) for d in (1, 8, 128, 512)])
def test_full_bf16_workload_every_element(C, d):
    dev = need_gpu()
    inp = syn.WORKLOADS[f"prenorm_block_bf16_C{C}_d{d}"].make(seed=0)
    got = _gpu(dev, inp)
    ref = oracle.prenorm_block(inp.x, inp.running_mean, inp.running_var, inp.gamma, inp.beta,
                               inp.eps, inp.weight, inp.bias, inp.dilation)
    assert_bf16(got, ref, f"bf16 full C{C} d{d}, every element")
    for n in range(got.shape[0]):
        assert_bf16(got[n], ref[n], f"bf16 full C{C} d{d}, sample {n}")


def test_repeat_calls_identical():
    dev = need_gpu()
    inp = syn.prenorm_block_inputs(2, 128, 640, 32, seed=8)
    a, b = _gpu(dev, inp), _gpu(dev, inp)
    assert np.array_equal(a, b)


def _host_call(inp, chunk_n, pinned=True):
    from normalization_convolution_blocks_gb300 import api
    x = inp.x.pin_memory() if pinned else inp.x
    g = Guarded(tuple(inp.x.shape), inp.x.dtype, pinned=True)
    out = api.prenorm_dilconv_residual(x, inp.running_mean, inp.running_var, inp.gamma,
                                       inp.beta, inp.eps, inp.weight, inp.bias, inp.dilation,
                                       chunk_n=chunk_n, out=g.view)
    assert not out.is_cuda and api.query_status() == api.NRC_OK
    g.check(f"host entry chunk {chunk_n}")
    return out.double().numpy()


@pytest.mark.parametrize("N,C,L,d,chunk_n,dtype", [
    (5, 64, 300, 8, 2, torch.float32),       # ragged last chunk, both buffers reused
    (4, 256, 512, 128, 1, torch.float32),    # one sample per chunk
    (3, 96, 296, 5, 8, torch.float32),       # chunk larger than the batch
    (6, 128, 264, 2, 4, torch.bfloat16),     # bf16, two chunks
])
def test_host_buffer_entry_matches_device_entry(N, C, L, d, chunk_n, dtype):
    """The host-buffer entry runs the same GEMM per chunk as the device entry:
    results must be bitwise equal, and within the parity bar of the oracle."""
    dev = need_gpu()
    inp = syn.prenorm_block_inputs(N, C, L, d, seed=N * 31 + C + d, dtype=dtype)
    got = _host_call(inp, chunk_n)
    assert np.array_equal(got, _gpu(dev, inp))
    check = assert_f32 if dtype == torch.float32 else assert_bf16
    check(got, _oracle(inp), f"host entry N{N} C{C} chunk {chunk_n}")


def test_host_buffer_entry_pageable_input():
    dev = need_gpu()
    inp = syn.prenorm_block_inputs(3, 48, 200, 3, seed=44)
    assert np.array_equal(_host_call(inp, 2, pinned=False), _gpu(dev, inp))


@pytest.mark.parametrize("dtype,which,offset", [
    (torch.bfloat16, "out", 1),     # out 2 bytes past a 16-byte boundary
    (torch.bfloat16, "out", 4),     # out 8-byte aligned, not 16
    (torch.bfloat16, "x", 1),
    (torch.float32, "out", 1),      # out 4 bytes past a 16-byte boundary
    (torch.float32, "x", 1),
])
def test_views_at_unaligned_offsets(dtype, which, offset):
    """x or out starting past a 16-byte boundary.  x there rules out the TMA
    boxes of the staged kernel (its rows load into registers instead).  bf16
    out off an 8-byte boundary rules out the staged kernel's 8-byte residual
    and output words (the register path runs); 8-byte aligned bf16 out and
    any fp32 out keep the staged kernel.  Every case must match the oracle
    and leave everything outside out unchanged."""
    dev = need_gpu()
    from normalization_convolution_blocks_gb300 import api
    inp = syn.prenorm_block_inputs(2, 64, 256, 4, seed=17, dtype=dtype)
    n = inp.x.numel()
    x = to(dev, inp.x)
    g = Guarded(tuple(inp.x.shape), dtype, dev, offset=offset if which == "out" else 0)
    out = g.view
    if which == "x":
        xb = torch.empty(n + offset, dtype=dtype, device=dev)
        xb[offset:].copy_(x.reshape(-1))
        x = xb[offset:].view(inp.x.shape)
    es = torch.tensor([], dtype=dtype).element_size()
    assert (x if which == "x" else out).data_ptr() % 16 == offset * es
    got = api.prenorm_dilconv_residual(x, to(dev, inp.running_mean), to(dev, inp.running_var),
                                       to(dev, inp.gamma), to(dev, inp.beta), inp.eps,
                                       to(dev, inp.weight), to(dev, inp.bias), inp.dilation,
                                       out=out)
    assert api.query_status() == api.NRC_OK
    g.check(f"{dtype} {which} at +{offset * es} bytes")
    check = assert_f32 if dtype == torch.float32 else assert_bf16
    check(got.double().cpu().numpy(), _oracle(inp), f"{dtype} {which} at +{offset * es} bytes")


@pytest.mark.parametrize("N,C,L,d", [
    (4, 256, 4096, 128),    # 128 tiles: one wave, the repack inside the GEMM kernel
    (8, 256, 4096, 128),    # 256 tiles: repack kernel, GEMM launched behind it
])
def test_back_to_back_calls_with_alternating_weights(N, C, L, d):
    """Calls queued back to back on one stream with different weights each time:
    a call's repack must not overwrite the image the previous GEMM still reads,
    and a GEMM must not read a half-written image.  Each result must equal the
    same call run on its own."""
    dev = need_gpu()
    from normalization_convolution_blocks_gb300 import api
    inp = syn.prenorm_block_inputs(N, C, L, d, seed=91)
    w2 = torch.flip(inp.weight, dims=[0]).contiguous()
    args = [to(dev, t) for t in (inp.x, inp.running_mean, inp.running_var, inp.gamma,
                                 inp.beta)]
    ws = [to(dev, inp.weight), to(dev, w2)]
    bias = to(dev, inp.bias)
    ref = []
    for w in ws:
        ref.append(api.prenorm_dilconv_residual(*args, inp.eps, w, bias, inp.dilation).clone())
        torch.cuda.synchronize()
    guards = [Guarded(tuple(args[0].shape), args[0].dtype, dev) for _ in range(6)]
    workspace = torch.empty(api.prenorm_dilconv_residual_workspace_size(C), dtype=torch.uint8,
                            device=dev)
    for i, g in enumerate(guards):         # one stream, shared workspace, no syncs
        api.prenorm_dilconv_residual(*args, inp.eps, ws[i % 2], bias, inp.dilation, out=g.view,
                                     workspace=workspace)
    torch.cuda.synchronize()
    assert api.query_status() == api.NRC_OK
    for i, g in enumerate(guards):
        g.check(f"call {i}")
        assert torch.equal(g.view, ref[i % 2]), f"call {i}"


def test_more_than_2_31_elements_sampled_rows():
    """N=128 C=256 L=65664 in bf16 storage: 2^31 + 4.2 M elements per tensor,
    so every element offset past 2^31 has to be formed in 64 bits.  Rows of the
    first, a middle and the last sample are compared with the oracle (run on
    one sample at a time); the 65,664 tiles also stress the persistent
    schedule."""
    dev = need_gpu()
    from normalization_convolution_blocks_gb300 import api
    N, C, L, d = 128, 256, 65664, 128
    assert N * C * L > 2 ** 31
    inp = syn.prenorm_block_inputs(N, C, L, d, seed=71, dtype=torch.bfloat16)
    x = to(dev, inp.x)
    out = torch.empty_like(x)
    api.prenorm_dilconv_residual(x, to(dev, inp.running_mean), to(dev, inp.running_var),
                                 to(dev, inp.gamma), to(dev, inp.beta), inp.eps,
                                 to(dev, inp.weight), to(dev, inp.bias), d, out=out)
    assert api.query_status() == api.NRC_OK
    rng = np.random.default_rng(5)
    for n in (0, 77, N - 1):
        ro = np.concatenate([[0, C - 1], rng.integers(0, C, 4)])
        ref = oracle.prenorm_block_rows(inp.x[n:n + 1], inp.running_mean, inp.running_var,
                                        inp.gamma, inp.beta, inp.eps, inp.weight, inp.bias, d,
                                        np.zeros(len(ro), dtype=np.int32), ro)
        got = out[n, torch.as_tensor(ro, device=dev)].double().cpu().numpy()
        assert_bf16(got, ref, f"sample {n} rows {list(ro)}")
