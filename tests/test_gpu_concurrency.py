"""Calls that overlap: device entries on several streams at once, and
host-buffer entries from several host threads (ctypes releases the GIL, so the
library's own locking is what keeps them apart).  Each result must equal the
same call made alone.  A cooperative one-wave launch may be refused while
another kernel occupies SMs; the call then takes its multi-launch path, whose
arithmetic for conv + GroupNorm differs in the last bits, so that block is
compared within 1e-5 rather than bitwise."""
import threading

import numpy as np
import pytest
import torch

from normalization_convolution_blocks_gb300 import synthetic as syn
from gpu_util import need_gpu, to


def _block_call(dev, seed, N=4, C=128, L=2048, d=16, dtype=torch.float32):
    from normalization_convolution_blocks_gb300 import api
    inp = syn.prenorm_block_inputs(N, C, L, d, seed=seed, dtype=dtype)
    x, rm, rv, g, b, w, bias = (to(dev, t) for t in (inp.x, inp.running_mean, inp.running_var,
                                                     inp.gamma, inp.beta, inp.weight, inp.bias))
    out = torch.empty_like(x)
    ws = torch.empty(api.prenorm_dilconv_residual_workspace_size(C, dtype), dtype=torch.uint8,
                     device=dev)
    return out, lambda st: api.prenorm_dilconv_residual(x, rm, rv, g, b, inp.eps, w, bias, d,
                                                        out=out, workspace=ws, stream=st)


def _gn_call(dev, seed, N=8, Cin=64, Cout=128, T=1024, G=16):
    from normalization_convolution_blocks_gb300 import api
    inp = syn.conv_groupnorm_inputs(N, Cin, Cout, T, G, seed=seed)
    x, w, g, b = (to(dev, t) for t in (inp.x, inp.weight, inp.gamma, inp.beta))
    out = torch.empty(N, Cout, T, device=dev)
    ws = torch.empty(api.conv1d_groupnorm_workspace_size(N, Cin, Cout, T, G), dtype=torch.uint8,
                     device=dev)
    return out, lambda st: api.conv1d_groupnorm(x, w, None, G, g, b, inp.eps, out=out,
                                                workspace=ws, stream=st)


def _linear_call(dev, seed, B=512, IN=1024, OUT=768):
    from normalization_convolution_blocks_gb300 import api
    inp = syn.linear_bn_swish_inputs(B, IN, OUT, seed=seed, random_affine=True)
    x, w, lb, g, b, ab = (to(dev, t) for t in (inp.x, inp.weight, inp.lin_bias, inp.gamma,
                                               inp.beta, inp.add_bias))
    rm = torch.zeros(OUT, device=dev)
    rv = torch.ones(OUT, device=dev)
    out = torch.empty(B, OUT, device=dev)
    ws = torch.empty(api.linear_bn_swish_workspace_size(B, IN, OUT), dtype=torch.uint8,
                     device=dev)
    return out, lambda st: api.linear_bn_swish(x, w, lb, g, b, rm, rv, ab, 1.0, inp.eps,
                                               inp.momentum, training=False, out=out,
                                               workspace=ws, stream=st)


@pytest.mark.gpu
def test_device_entries_on_three_streams_match_calls_made_alone():
    dev = need_gpu()
    from normalization_convolution_blocks_gb300 import api
    calls = [_block_call(dev, 41), _gn_call(dev, 42), _linear_call(dev, 43),
             _block_call(dev, 44, dtype=torch.bfloat16)]
    alone = []
    for out, call in calls:
        call(None)
        torch.cuda.synchronize()
        alone.append(out.clone())
    streams = [torch.cuda.Stream() for _ in calls]
    for _ in range(5):
        for out, _ in calls:
            out.fill_(float("nan"))
        torch.cuda.synchronize()
        for (out, call), st in zip(calls, streams):
            call(st)
        torch.cuda.synchronize()
        assert api.query_status() == api.NRC_OK
        for i, ((out, _), want) in enumerate(zip(calls, alone)):
            if i == 1:
                assert float((out - want).abs().max()) < 1e-5
            else:
                assert torch.equal(out, want), f"call {i} differs when run alongside the others"


@pytest.mark.gpu
def test_host_buffer_entries_from_two_threads_match_calls_made_alone():
    need_gpu()
    from normalization_convolution_blocks_gb300 import api
    inputs = [syn.prenorm_block_inputs(6, 64, 1024, 8, seed=51 + k) for k in range(2)]

    def run(inp):
        return api.prenorm_dilconv_residual(inp.x.pin_memory(), inp.running_mean,
                                            inp.running_var, inp.gamma, inp.beta, inp.eps,
                                            inp.weight, inp.bias, inp.dilation,
                                            chunk_n=2).double().numpy()

    alone = [run(inp) for inp in inputs]
    results = [[None] * 3 for _ in inputs]
    errors = []

    def worker(k):
        try:
            for r in range(3):
                results[k][r] = run(inputs[k])
        except Exception as e:          # reported by the main thread
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(k,)) for k in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not errors, errors
    assert not any(t.is_alive() for t in threads)
    for k in range(2):
        for r in range(3):
            assert np.array_equal(results[k][r], alone[k]), f"thread {k} call {r}"
    assert api.query_status() == api.NRC_OK
