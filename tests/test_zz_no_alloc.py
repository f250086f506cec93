"""The allocation-free pre-norm block entry point.

nrc_prenorm_dilconv_residual_noalloc serves callers that cannot hand the
library scratch memory (their device memory belongs to a host framework's
allocator, or their loop must not call cudaMalloc/cudaFree): its scratch is a
fixed 4 MiB array inside the library.  This test calls it through the C ABI
twice in a row, with different shapes and dtypes so the second call runs over
what the first left in the shared array, and compares each result with the
regular workspace entry point within the fp32 / bf16 parity tolerances used by
the other GPU tests.  It also checks that a C whose weight image exceeds the
array is refused.  The file name makes pytest collect it last.
"""
import ctypes

import numpy as np
import pytest
import torch

from normalization_convolution_blocks_gb300 import synthetic as syn
from gpu_util import BF16_REL_L2, F32_MAX_ABS, F32_REL_L2, errors, need_gpu, to

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


@pytest.mark.parametrize("order", ["fp32_then_bf16", "bf16_then_fp32"])
def test_noalloc_matches_workspace_entry_point_on_consecutive_calls(order):
    dev = need_gpu()
    from normalization_convolution_blocks_gb300 import api
    lib = api.load()
    cases = [dict(N=2, C=256, L=1000, d=64, dtype=torch.float32, seed=41),
             dict(N=1, C=96, L=700, d=5, dtype=torch.bfloat16, seed=42)]
    if order == "bf16_then_fp32":
        cases.reverse()
    for case in cases:
        inp = syn.prenorm_block_inputs(case["N"], case["C"], case["L"], case["d"],
                                       seed=case["seed"], dtype=case["dtype"])
        x, rm, rv, g, b, w, bias = _args(dev, inp)
        ref = api.prenorm_dilconv_residual(x, rm, rv, g, b, inp.eps, w, bias, inp.dilation)
        out = torch.full_like(x, float("nan"))
        st = _noalloc_c_abi(lib, x, rm, rv, g, b, inp.eps, w, bias, inp.dilation, out)
        assert st == api.NRC_OK, api.status_string(st)
        torch.cuda.synchronize()
        assert api.query_status() == api.NRC_OK
        rel, mx = errors(out.double().cpu().numpy(), ref.double().cpu().numpy())
        if case["dtype"] == torch.float32:
            assert rel < F32_REL_L2 and mx < F32_MAX_ABS, (rel, mx)
        else:
            assert rel < BF16_REL_L2, (rel, mx)


def test_noalloc_refuses_channels_beyond_its_scratch():
    dev = need_gpu()
    from normalization_convolution_blocks_gb300 import api
    lib = api.load()
    assert lib.nrc_prenorm_dilconv_residual_noalloc_max_bytes() == 4 << 20
    inp = syn.prenorm_block_inputs(1, 640, 16, 1, seed=43)     # fp32 C=640 needs > 4 MiB
    x, rm, rv, g, b, w, bias = _args(dev, inp)
    out = torch.empty_like(x)
    assert _noalloc_c_abi(lib, x, rm, rv, g, b, inp.eps, w, bias, 1, out) == api.NRC_ERR_WORKSPACE
