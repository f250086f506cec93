"""The allocation-free pre-norm block entry point.

nrc_prenorm_dilconv_residual_noalloc serves callers that cannot hand the
library scratch memory (their device memory belongs to a host framework's
allocator, or their loop must not call cudaMalloc/cudaFree): its scratch is a
fixed 4 MiB array inside the library.  The tests call it through the C ABI
several times in a row, with different shapes and dtypes so each call runs
over what the previous one left in the shared array, and check every result
twice: bitwise against the regular workspace entry point (both run the same
kernels on the same weight image), and against the fp64 oracle within the
fp32 / bf16 parity tolerances of the other GPU tests.  The cases cover both
of the entry point's paths: one wave of tiles (the GEMM kernel repacks the
weights into the array itself) and more tiles than SMs (a repack kernel
writes the array and the GEMM is launched behind it).  A C whose weight image
exceeds the array is refused.  The file name makes pytest collect it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from normalization_convolution_blocks_gb300 import synthetic as syn
from gpu_util import assert_bf16, assert_f32, need_gpu, to

pytestmark = pytest.mark.gpu


def _args(dev, inp):
    return [to(dev, t).contiguous() for t in (inp.x, inp.running_mean, inp.running_var,
                                              inp.gamma, inp.beta, inp.weight, inp.bias)]


def _noalloc_c_abi(lib, x, rm, rv, g, b, eps, w, bias, d, out):
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    dt = 0 if x.dtype == torch.float32 else 1
    N, C, L = x.shape
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.nrc_prenorm_dilconv_residual_noalloc(P(x), P(out), dt, N, C, L, 3, d, d, P(rm),
                                                    P(rv), P(g), P(b), float(eps), P(w), P(bias),
                                                    stream)


CASES = {
    # one wave (tiles <= SMs): the GEMM kernel repacks into the array
    "fp32_one_wave": dict(N=2, C=256, L=1000, d=64, dtype=torch.float32, seed=41),
    "bf16_one_wave": dict(N=1, C=96, L=700, d=5, dtype=torch.bfloat16, seed=42),
    # 256 tiles: repack kernel into the array, GEMM launched behind it
    "fp32_multi_wave": dict(N=2, C=256, L=16384, d=128, dtype=torch.float32, seed=44),
}


@pytest.mark.parametrize("order", [
    ("fp32_one_wave", "bf16_one_wave", "fp32_multi_wave"),
    ("fp32_multi_wave", "bf16_one_wave", "fp32_one_wave"),
])
def test_noalloc_matches_workspace_entry_point_and_oracle_on_consecutive_calls(order):
    dev = need_gpu()
    from normalization_convolution_blocks_gb300 import api
    lib = api.load()
    for name in order:
        case = CASES[name]
        inp = syn.prenorm_block_inputs(case["N"], case["C"], case["L"], case["d"],
                                       seed=case["seed"], dtype=case["dtype"])
        x, rm, rv, g, b, w, bias = _args(dev, inp)
        ref = api.prenorm_dilconv_residual(x, rm, rv, g, b, inp.eps, w, bias, inp.dilation)
        torch.cuda.synchronize()
        out = torch.full_like(x, float("nan"))
        st = _noalloc_c_abi(lib, x, rm, rv, g, b, inp.eps, w, bias, inp.dilation, out)
        assert st == api.NRC_OK, api.status_string(st)
        torch.cuda.synchronize()
        assert api.query_status() == api.NRC_OK
        assert torch.equal(out, ref), f"{name}: differs from the workspace entry point"
        want = oracle.prenorm_block(inp.x, inp.running_mean, inp.running_var, inp.gamma,
                                    inp.beta, inp.eps, inp.weight, inp.bias, inp.dilation)
        got = out.double().cpu().numpy()
        if case["dtype"] == torch.float32:
            assert_f32(got, want, name)
        else:
            assert_bf16(got, want, name)


def test_noalloc_refuses_channels_beyond_its_scratch():
    dev = need_gpu()
    from normalization_convolution_blocks_gb300 import api
    lib = api.load()
    assert lib.nrc_prenorm_dilconv_residual_noalloc_max_bytes() == 4 << 20
    inp = syn.prenorm_block_inputs(1, 640, 16, 1, seed=43)     # fp32 C=640 needs > 4 MiB
    x, rm, rv, g, b, w, bias = _args(dev, inp)
    out = torch.full_like(x, 7.0)
    assert _noalloc_c_abi(lib, x, rm, rv, g, b, inp.eps, w, bias, 1, out) == api.NRC_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((out == 7.0).all()), "a refused call wrote its output"
    assert np.isfinite(out.double().cpu().numpy()).all()
