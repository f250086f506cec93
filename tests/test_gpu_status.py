"""Device-side fault path: a bounded wait that nothing satisfies gives up,
records NRC_ERR_TIMEOUT, and leaves the context usable.  The stall is a
barrier nobody arrives at -- no trap, no bad address, no endless loop."""
import pytest
import torch

from normalization_convolution_blocks_gb300 import synthetic as syn
from gpu_util import need_gpu, to

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
