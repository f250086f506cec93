"""Device-side fault path: a bounded wait that nothing satisfies gives up,
records NRC_ERR_TIMEOUT, and leaves the context usable.  The stall is a
barrier nobody arrives at -- no trap, no bad address, no endless loop."""
import pytest
import torch

import oracle
from normalization_convolution_blocks_gb300 import synthetic as syn
from gpu_util import assert_f32, need_gpu, to

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_context_survives():
    dev = need_gpu()
    from normalization_convolution_blocks_gb300 import api
    assert api.query_status() == api.NRC_OK
    api.selftest_wait_timeout(20_000_000)          # 20 ms limit
    assert api.query_status() == api.NRC_ERR_TIMEOUT
    assert api.last_error_site() == 99
    assert api.query_status() == api.NRC_OK        # cleared by the read
    inp = syn.prenorm_block_inputs(1, 32, 256, 4, seed=0)
    out = api.prenorm_dilconv_residual(to(dev, inp.x), to(dev, inp.running_mean),
                                       to(dev, inp.running_var), to(dev, inp.gamma),
                                       to(dev, inp.beta), inp.eps, to(dev, inp.weight),
                                       to(dev, inp.bias), inp.dilation)
    torch.cuda.synchronize()
    assert api.query_status() == api.NRC_OK
    assert torch.isfinite(out).all()


def test_fused_groupnorm_grid_barrier_gives_up_and_next_call_is_exact():
    """A real kernel's give-up path: the one-wave Conv1d + GroupNorm kernel
    (the conv+GN workload, 128 tiles on resident CTAs) with a 1 ns limit on
    its grid-wide barrier only.  By that barrier every CTA has finished its
    copies and MMAs, so a CTA that gives up just returns.  The call must report
    NRC_ERR_TIMEOUT at wait site 9 (the grid barrier); with the limit restored
    the next call must match the oracle.  No other wait is shortened."""
    dev = need_gpu()
    from normalization_convolution_blocks_gb300 import api
    g = syn.WORKLOADS["conv1d_groupnorm_f32"].make(seed=0)
    args = [to(dev, t) for t in (g.x, g.weight)]
    gamma, beta = to(dev, g.gamma), to(dev, g.beta)
    assert api.query_status() == api.NRC_OK

    def call():
        return api.conv1d_groupnorm(args[0], args[1], None, g.num_groups, gamma, beta, g.eps)

    status = api.NRC_OK
    api.set_grid_barrier_timeout_ns(1)
    try:
        # the last CTA to arrive never waits, so a give-up needs at least one
        # CTA to arrive early: certain in practice, retried to be safe
        for _ in range(5):
            call()
            status = api.query_status()
            if status != api.NRC_OK:
                break
    finally:
        api.set_grid_barrier_timeout_ns(0)
    assert status == api.NRC_ERR_TIMEOUT
    assert api.last_error_site() == 9
    assert api.query_status() == api.NRC_OK        # cleared by the read
    out = call()
    assert api.query_status() == api.NRC_OK
    ref = oracle.conv_groupnorm(g.x, g.weight, None, g.num_groups, g.gamma, g.beta, g.eps)
    assert_f32(out.double().cpu().numpy(), ref, "conv+GN after the give-up")
