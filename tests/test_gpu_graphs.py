"""Device entry points captured in a CUDA graph and replayed.

Every device-buffer entry only enqueues work on the caller's stream (memsets,
cooperative launches, launches behind the repack kernel with programmatic
dependent launch), so a caller can capture a call once and replay it without
the host-side planning and launch overhead.  Each replay must give exactly the
eager call's result, also after new input values are copied into the captured
buffers; training-mode calls must also update the running buffers exactly as
an eager call does."""
import pytest
import torch

from normalization_convolution_blocks_gb300 import synthetic as syn
from gpu_util import need_gpu, to


def _capture(call):
    """Warm up on a side stream, then capture one call; returns the graph."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    torch.cuda.synchronize()
    return g


def _status_ok():
    from normalization_convolution_blocks_gb300 import api
    assert api.query_status() == api.NRC_OK


def _replay_matches(call, out, inputs, fresh_inputs, state=()):
    """Eager result for each input set, then the graph's replay on the same
    values copied into the captured input buffers; `state` lists buffers the
    call updates in place (restored to the same start before each run)."""
    start = [t.clone() for t in state]

    def restore():
        for t, s0 in zip(state, start):
            t.copy_(s0)

    originals = [t.clone() for t in inputs]
    expected = []
    for values in (originals, fresh_inputs):
        for t, v in zip(inputs, values):
            t.copy_(v)
        restore()
        call()
        torch.cuda.synchronize()
        expected.append((out.clone(), [t.clone() for t in state]))
    for t, v in zip(inputs, originals):
        t.copy_(v)
    graph = _capture(call)
    for (want, want_state), values in zip(expected, (originals, fresh_inputs)):
        for t, v in zip(inputs, values):
            t.copy_(v)
        restore()
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, want)
        for t, w in zip(state, want_state):
            assert torch.equal(t, w)
    _status_ok()


@pytest.mark.gpu
@pytest.mark.parametrize("N,C,L,d,dtype", [
    (2, 64, 512, 8, torch.float32),        # one wave: cooperative launch, repack inside
    (8, 256, 4096, 128, torch.float32),    # repack kernel, GEMM behind it (PDL)
    (2, 128, 1024, 4, torch.bfloat16),
])
def test_block_graph_replay(N, C, L, d, dtype):
    dev = need_gpu()
    from normalization_convolution_blocks_gb300 import api
    inp = syn.prenorm_block_inputs(N, C, L, d, seed=N + C + d, dtype=dtype)
    x, rm, rv, g, b, w, bias = (to(dev, t) for t in (inp.x, inp.running_mean, inp.running_var,
                                                     inp.gamma, inp.beta, inp.weight, inp.bias))
    out = torch.empty_like(x)
    ws = torch.empty(api.prenorm_dilconv_residual_workspace_size(C, dtype), dtype=torch.uint8,
                     device=dev)
    call = lambda: api.prenorm_dilconv_residual(x, rm, rv, g, b, inp.eps, w, bias, d, out=out,
                                                workspace=ws)
    x2 = to(dev, syn.prenorm_block_inputs(N, C, L, d, seed=99, dtype=dtype).x)
    w2 = torch.flip(w, dims=[0])
    _replay_matches(call, out, [x, w], [x2, w2])


@pytest.mark.gpu
@pytest.mark.parametrize("N,Cin,Cout,T,G", [
    (4, 64, 128, 512, 16),       # one wave: the fused conv + GroupNorm kernel
    (16, 64, 64, 4096, 8),       # more tiles than SMs: conv with statistics, then normalize
])
def test_conv_groupnorm_graph_replay(N, Cin, Cout, T, G):
    dev = need_gpu()
    from normalization_convolution_blocks_gb300 import api
    inp = syn.conv_groupnorm_inputs(N, Cin, Cout, T, G, seed=T + G)
    x, w, g, b = (to(dev, t) for t in (inp.x, inp.weight, inp.gamma, inp.beta))
    cb = torch.linspace(-0.5, 0.5, Cout, device=dev)
    out = torch.empty(N, Cout, T, device=dev)
    ws = torch.empty(api.conv1d_groupnorm_workspace_size(N, Cin, Cout, T, G), dtype=torch.uint8,
                     device=dev)
    call = lambda: api.conv1d_groupnorm(x, w, cb, G, g, b, inp.eps, out=out, workspace=ws)
    x2 = to(dev, syn.conv_groupnorm_inputs(N, Cin, Cout, T, G, seed=7).x)
    _replay_matches(call, out, [x], [x2])


@pytest.mark.gpu
@pytest.mark.parametrize("training", [True, False])
def test_linear_graph_replay(training):
    dev = need_gpu()
    from normalization_convolution_blocks_gb300 import api
    B, IN, OUT = 256, 512, 384
    inp = syn.linear_bn_swish_inputs(B, IN, OUT, seed=5, random_affine=True)
    x, w, lb, g, b, ab = (to(dev, t) for t in (inp.x, inp.weight, inp.lin_bias, inp.gamma,
                                               inp.beta, inp.add_bias))
    rm = torch.linspace(-0.2, 0.2, OUT, device=dev)
    rv = torch.linspace(0.5, 1.5, OUT, device=dev)
    nbt = torch.zeros(1, dtype=torch.int64, device=dev)
    out = torch.empty(B, OUT, device=dev)
    ws = torch.empty(api.linear_bn_swish_workspace_size(B, IN, OUT), dtype=torch.uint8,
                     device=dev)
    call = lambda: api.linear_bn_swish(x, w, lb, g, b, rm, rv, ab, 1.5, inp.eps, inp.momentum,
                                       training=training, num_batches_tracked=nbt, out=out,
                                       workspace=ws)
    x2 = to(dev, syn.linear_bn_swish_inputs(B, IN, OUT, seed=6).x)
    _replay_matches(call, out, [x], [x2], state=(rm, rv, nbt) if training else ())


@pytest.mark.gpu
def test_block_train_graph_replay():
    dev = need_gpu()
    from normalization_convolution_blocks_gb300 import api
    N, C, L, d = 4, 64, 1024, 16
    inp = syn.prenorm_block_inputs(N, C, L, d, seed=3)
    x, g, b, w, bias = (to(dev, t) for t in (inp.x, inp.gamma, inp.beta, inp.weight, inp.bias))
    rm = to(dev, inp.running_mean).clone()
    rv = to(dev, inp.running_var).clone()
    nbt = torch.zeros(1, dtype=torch.int64, device=dev)
    out = torch.empty_like(x)
    ws = torch.empty(api.prenorm_dilconv_residual_train_workspace_size(N, C, L), dtype=torch.uint8,
                     device=dev)
    call = lambda: api.prenorm_dilconv_residual_train(x, rm, rv, g, b, inp.eps, 0.1, w, bias, d,
                                                      num_batches_tracked=nbt, out=out,
                                                      workspace=ws)
    x2 = to(dev, syn.prenorm_block_inputs(N, C, L, d, seed=4).x)
    _replay_matches(call, out, [x], [x2], state=(rm, rv, nbt))


@pytest.mark.gpu
def test_chained_entries_in_one_graph():
    """The block, then conv + GroupNorm on its output, then the Linear on a
    reshaped slice of that, captured as one graph: a replay equals the three
    calls run eagerly, also after new x values are copied in."""
    dev = need_gpu()
    from normalization_convolution_blocks_gb300 import api
    N, C, L, d, G, OUT = 4, 64, 512, 8, 8, 96
    inp = syn.prenorm_block_inputs(N, C, L, d, seed=21)
    x, rm, rv, g, b, w, bias = (to(dev, t) for t in (inp.x, inp.running_mean, inp.running_var,
                                                     inp.gamma, inp.beta, inp.weight, inp.bias))
    gn = syn.conv_groupnorm_inputs(N, C, C, L, G, seed=22)
    gw, gg, gb = (to(dev, t) for t in (gn.weight, gn.gamma, gn.beta))
    li = syn.linear_bn_swish_inputs(N * C, L, OUT, seed=23, random_affine=True)
    lw, lb, lg, lbe, lab = (to(dev, t) for t in (li.weight, li.lin_bias, li.gamma, li.beta,
                                                 li.add_bias))
    lrm = torch.zeros(OUT, device=dev)
    lrv = torch.ones(OUT, device=dev)
    y1 = torch.empty_like(x)
    y2 = torch.empty_like(x)
    y3 = torch.empty(N * C, OUT, device=dev)
    ws1 = torch.empty(api.prenorm_dilconv_residual_workspace_size(C), dtype=torch.uint8,
                      device=dev)
    ws2 = torch.empty(api.conv1d_groupnorm_workspace_size(N, C, C, L, G), dtype=torch.uint8,
                      device=dev)
    ws3 = torch.empty(api.linear_bn_swish_workspace_size(N * C, L, OUT), dtype=torch.uint8,
                      device=dev)

    def chain():
        api.prenorm_dilconv_residual(x, rm, rv, g, b, inp.eps, w, bias, d, out=y1, workspace=ws1)
        api.conv1d_groupnorm(y1, gw, None, G, gg, gb, gn.eps, out=y2, workspace=ws2)
        api.linear_bn_swish(y2.view(N * C, L), lw, lb, lg, lbe, lrm, lrv, lab, 2.0, li.eps,
                            li.momentum, training=False, out=y3, workspace=ws3)

    x2 = to(dev, syn.prenorm_block_inputs(N, C, L, d, seed=24).x)
    x1 = x.clone()
    want = []
    for xv in (x1, x2):
        x.copy_(xv)
        chain()
        torch.cuda.synchronize()
        want.append((y1.clone(), y2.clone(), y3.clone()))
    x.copy_(x1)
    graph = _capture(chain)
    for xv, (w1, w2, w3) in zip((x1, x2), want):
        x.copy_(xv)
        for t in (y1, y2, y3):
            t.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(y1, w1) and torch.equal(y2, w2) and torch.equal(y3, w3)
    _status_ok()
