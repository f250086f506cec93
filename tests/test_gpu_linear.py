"""GPU parity of nrc_linear_bn_swish against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from normalization_convolution_blocks_gb300 import synthetic as syn
from gpu_util import RUNNING_STAT_ABS, Guarded, assert_f32, need_gpu, to

pytestmark = pytest.mark.gpu


def _gpu(dev, li, training=True, nbt=None):
    """One call into a guarded output buffer; the guards are checked after it."""
    from normalization_convolution_blocks_gb300 import api
    rm, rv = to(dev, li.running_mean).clone(), to(dev, li.running_var).clone()
    B, OUT = li.x.shape[0], li.weight.shape[0]
    g = Guarded((B, OUT), torch.float32, dev)
    out = api.linear_bn_swish(to(dev, li.x), to(dev, li.weight), to(dev, li.lin_bias),
                              to(dev, li.gamma), to(dev, li.beta), rm, rv, to(dev, li.add_bias),
                              li.divide_value, li.eps, li.momentum, training, nbt, out=g.view)
    assert api.query_status() == api.NRC_OK
    g.check(f"linear B{B} OUT{OUT} training={training}")
    return out.double().cpu().numpy(), rm.double().cpu().numpy(), rv.double().cpu().numpy()


def _ref(li, training=True, cols=None):
    return oracle.linear_bn_swish(li.x, li.weight, li.lin_bias, li.gamma, li.beta,
                                  li.running_mean, li.running_var, li.eps, li.momentum, training,
                                  float(li.add_bias[0]), li.divide_value, cols=cols)


def _check(got, ref, what):
    out, rm, rv = got
    r_out, r_rm, r_rv, _ = ref
    assert_f32(out, r_out, what)
    assert np.abs(rm - r_rm).max() < RUNNING_STAT_ABS, f"{what}: running_mean"
    assert np.abs(rv - r_rv).max() < RUNNING_STAT_ABS, f"{what}: running_var"


@pytest.mark.parametrize("B,IN,OUT,affine", [
    (64, 256, 128, True), (64, 256, 128, False),
    (100, 100, 70, True),     # ragged everywhere, in_features not a multiple of 4
    (2, 64, 32, True),        # smallest training batch
    (300, 520, 200, True),    # two batch tiles, ragged
    (1024, 1024, 256, True),
    (33, 37, 50, True),       # in_features % 4 != 0: W rows loaded directly, not by TMA
])
def test_training_shapes(B, IN, OUT, affine):
    dev = need_gpu()
    li = syn.linear_bn_swish_inputs(B, IN, OUT, seed=B + IN + OUT, random_affine=affine)
    _check(_gpu(dev, li), _ref(li), f"B{B} IN{IN} OUT{OUT}")


# More tiles (128 features x 256 batch rows) than SMs, not a whole number of
# waves: persistent CTAs take a second, partial round of tiles.  Checked on
# sampled columns (every batch row) and their running statistics.
@pytest.mark.parametrize("B,IN,OUT", [
    (256, 128, 20480),        # 160 tiles of 2 K stages
    (300, 1000, 10000),       # 79 x 2 tiles, ragged batch tile and K
])
def test_multi_wave_shapes_sampled_columns(B, IN, OUT):
    dev = need_gpu()
    n_tiles = -(-OUT // 128) * -(-B // 256)
    assert n_tiles > torch.cuda.get_device_properties(dev).multi_processor_count
    li = syn.linear_bn_swish_inputs(B, IN, OUT, seed=B + IN, random_affine=True)
    out, rm, rv = _gpu(dev, li)
    cols = np.unique(np.concatenate([[0, 127, 128, OUT - 1],
                                     np.random.default_rng(B).integers(0, OUT, 252)]))
    r_out, r_rm, r_rv, _ = _ref(li, cols=cols)
    assert_f32(out[:, cols], r_out, f"multi-wave B{B} IN{IN} OUT{OUT}")
    assert np.abs(rm[cols] - r_rm[cols]).max() < RUNNING_STAT_ABS
    assert np.abs(rv[cols] - r_rv[cols]).max() < RUNNING_STAT_ABS


def test_eval_mode_and_divide():
    dev = need_gpu()
    li = syn.linear_bn_swish_inputs(48, 160, 96, seed=4, random_affine=True)
    g = torch.Generator().manual_seed(5)
    li.running_mean = torch.randn(96, generator=g) * 0.1
    li.running_var = torch.rand(96, generator=g) + 0.5
    li.divide_value = 2.5
    _check(_gpu(dev, li, training=False), _ref(li, training=False), "eval, divide 2.5")


@pytest.mark.parametrize("B,IN,OUT,affine", [
    (1, 64, 32, True),        # one batch row: allowed in eval mode
    (100, 100, 70, True),     # ragged everywhere
    (33, 37, 50, True),       # W rows loaded directly, not by TMA
    (300, 520, 200, True),    # two batch tiles, ragged
    (64, 256, 128, False),    # affine off
])
def test_eval_shapes(B, IN, OUT, affine):
    """Eval mode runs as one GEMM whose epilogue applies BN with the running
    statistics, the scalar bias, the divide and Swish."""
    dev = need_gpu()
    li = syn.linear_bn_swish_inputs(B, IN, OUT, seed=B * 3 + IN + OUT, random_affine=affine)
    g = torch.Generator().manual_seed(B + OUT)
    li.running_mean = torch.randn(OUT, generator=g) * 0.1
    li.running_var = torch.rand(OUT, generator=g) + 0.5
    li.divide_value = 1.5
    _check(_gpu(dev, li, training=False), _ref(li, training=False), f"eval B{B} IN{IN} OUT{OUT}")


def test_eval_multi_wave_and_full_workload_sampled_columns():
    dev = need_gpu()
    for li, tag in ((syn.linear_bn_swish_inputs(256, 128, 20480, seed=9, random_affine=True),
                     "eval multi-wave"),
                    (syn.WORKLOADS["linear_bn_swish_f32"].make(seed=0), "eval full workload")):
        OUT = li.weight.shape[0]
        g = torch.Generator().manual_seed(OUT)
        li.running_mean = torch.randn(OUT, generator=g) * 0.05
        li.running_var = torch.rand(OUT, generator=g) * 0.1 + 0.05
        out, rm, rv = _gpu(dev, li, training=False)
        cols = np.unique(np.concatenate([[0, 127, 128, OUT - 1],
                                         np.random.default_rng(OUT).integers(0, OUT, 60)]))
        r_out, _, _, _ = _ref(li, training=False, cols=cols)
        assert_f32(out[:, cols], r_out, tag)
        assert np.array_equal(rm, li.running_mean.double().numpy())    # untouched
        assert np.array_equal(rv, li.running_var.double().numpy())


def test_num_batches_tracked_increments():
    dev = need_gpu()
    li = syn.linear_bn_swish_inputs(16, 32, 16, seed=6)
    nbt = torch.zeros(1, dtype=torch.int64, device=dev)
    _gpu(dev, li, nbt=nbt)
    _gpu(dev, li, nbt=nbt)
    assert int(nbt.item()) == 2
    _gpu(dev, li, training=False, nbt=nbt)
    assert int(nbt.item()) == 2


def test_full_workload_every_element():
    """Full-size workload (1024 x 8192 -> 8192) in the bench's launch
    configuration: every output element and all 8192 running statistics,
    plus the bar per 128-column block so a local error cannot hide."""
    dev = need_gpu()
    li = syn.WORKLOADS["linear_bn_swish_f32"].make(seed=0)
    out, rm, rv = _gpu(dev, li)
    r_out, r_rm, r_rv, _ = _ref(li)
    assert_f32(out, r_out, "full workload, every element")
    for j0 in range(0, out.shape[1], 128):
        assert_f32(out[:, j0:j0 + 128], r_out[:, j0:j0 + 128], f"columns {j0}..")
    assert np.abs(rm - r_rm).max() < RUNNING_STAT_ABS
    assert np.abs(rv - r_rv).max() < RUNNING_STAT_ABS


def test_full_workload_eval_every_element():
    dev = need_gpu()
    li = syn.WORKLOADS["linear_bn_swish_eval_f32"].make(seed=0)
    g = torch.Generator().manual_seed(8192)
    li.running_mean = torch.randn(8192, generator=g) * 0.05
    li.running_var = torch.rand(8192, generator=g) * 0.1 + 0.05
    out, _, _ = _gpu(dev, li, training=False)
    r_out, _, _, _ = _ref(li, training=False)
    assert_f32(out, r_out, "eval full workload, every element")


def test_back_to_back_calls_with_alternating_inputs():
    """Calls queued back to back on one stream with different x each time (the
    x repack, the GEMM launched behind it, then the chained finalize and
    normalize): each result must equal the same call run on its own."""
    dev = need_gpu()
    from normalization_convolution_blocks_gb300 import api
    li = syn.linear_bn_swish_inputs(512, 1024, 4096, seed=13, random_affine=True)
    xs = [to(dev, li.x), to(dev, torch.flip(li.x, dims=[0]).contiguous())]
    w, lb, g, b, ab = (to(dev, t) for t in (li.weight, li.lin_bias, li.gamma, li.beta,
                                            li.add_bias))

    def call(x, out=None):
        rm, rv = to(dev, li.running_mean).clone(), to(dev, li.running_var).clone()
        return api.linear_bn_swish(x, w, lb, g, b, rm, rv, ab, li.divide_value, li.eps,
                                   li.momentum, True, None, out=out)
    ref = []
    for x in xs:
        ref.append(call(x).clone())
        torch.cuda.synchronize()
    outs = [torch.empty_like(ref[0]) for _ in range(6)]
    for i, o in enumerate(outs):
        call(xs[i % 2], out=o)
    torch.cuda.synchronize()
    assert api.query_status() == api.NRC_OK
    for i, o in enumerate(outs):
        assert torch.equal(o, ref[i % 2]), f"call {i}"


def _host_vs_device(dev, li, training, chunk_f):
    """The host-buffer entry (chunked over output features) against the device
    entry on the same inputs: bitwise equal outputs and running statistics."""
    from normalization_convolution_blocks_gb300 import api
    B, OUT = li.x.shape[0], li.weight.shape[0]
    nbt_d = torch.zeros(1, dtype=torch.int64, device=dev)
    rm_d, rv_d = to(dev, li.running_mean).clone(), to(dev, li.running_var).clone()
    ref = api.linear_bn_swish(to(dev, li.x), to(dev, li.weight), to(dev, li.lin_bias),
                              to(dev, li.gamma), to(dev, li.beta), rm_d, rv_d,
                              to(dev, li.add_bias), li.divide_value, li.eps, li.momentum,
                              training, nbt_d)
    nbt_h = torch.zeros(1, dtype=torch.int64, device=dev)
    rm_h, rv_h = to(dev, li.running_mean).clone(), to(dev, li.running_var).clone()
    pin = lambda t: t.contiguous().pin_memory()  # noqa: E731
    out = torch.full((B, OUT), float("nan")).pin_memory()
    got = api._linear_host(api.load(), dev, pin(li.x), pin(li.weight), pin(li.lin_bias),
                           pin(li.gamma), pin(li.beta), rm_h, rv_h, pin(li.add_bias),
                           li.divide_value, li.eps, li.momentum, training, nbt_h, out, None,
                           None, chunk_f=chunk_f)
    assert api.query_status() == api.NRC_OK
    assert torch.equal(got, ref.cpu()), "host entry differs from the device entry"
    assert torch.equal(rm_h, rm_d) and torch.equal(rv_h, rv_d), "running statistics differ"
    assert int(nbt_h.item()) == int(nbt_d.item()) == (1 if training else 0)
    return got


@pytest.mark.parametrize("B,IN,OUT,chunk_f,training,affine", [
    (300, 520, 1000, 256, True, True),     # ragged last chunk, ramped chunk sizes
    (256, 1024, 2048, 512, False, True),   # eval mode
    (64, 128, 130, 128, True, False),      # two tiles, the last chunk of 2 features
    (33, 37, 50, 128, True, True),         # in_features % 4 != 0: W rows loaded directly
])
def test_host_buffer_entry_matches_device_entry(B, IN, OUT, chunk_f, training, affine):
    dev = need_gpu()
    li = syn.linear_bn_swish_inputs(B, IN, OUT, seed=B + OUT, random_affine=affine)
    got = _host_vs_device(dev, li, training, chunk_f)
    r_out = _ref(li, training)[0]
    assert_f32(got.double().numpy(), r_out, f"host entry B{B} IN{IN} OUT{OUT}")


def test_host_buffer_entry_full_workload():
    dev = need_gpu()
    li = syn.WORKLOADS["linear_bn_swish_f32"].make(seed=0)
    _host_vs_device(dev, li, True, 2048)
