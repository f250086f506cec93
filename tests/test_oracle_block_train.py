"""Pins for the training-mode pre-norm block oracle (CPU only).

``oracle.prenorm_block_train`` must agree with hand-worked cases and with
PyTorch's own fp64 modules in training mode (BatchNorm1d with batch
statistics and the running-buffer update, ReLU, Conv1d, residual), and keep
the invariants of the definition: the running buffers' old values do not
reach the output, momentum 0 leaves them alone, momentum 1 replaces them.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from normalization_convolution_blocks_gb300 import synthetic as syn

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _torch_train_fp64(inp, momentum):
    """The problem statement as PyTorch modules in training mode, float64.
    Returns (out, running_mean', running_var')."""
    C = inp.x.shape[1]
    bn = torch.nn.BatchNorm1d(C, eps=inp.eps, momentum=momentum).double().train()
    conv = torch.nn.Conv1d(C, C, 3, padding=inp.dilation, dilation=inp.dilation).double()
    with torch.no_grad():
        bn.running_mean.copy_(inp.running_mean.double())
        bn.running_var.copy_(inp.running_var.double())
        bn.weight.copy_(inp.gamma.double())
        bn.bias.copy_(inp.beta.double())
        conv.weight.copy_(inp.weight.double())
        conv.bias.copy_(inp.bias.double())
        x = inp.x.double()
        out = (x + conv(torch.relu(bn(x)))).numpy()
    return out, bn.running_mean.numpy(), bn.running_var.numpy()


def _run(inp, momentum, **kw):
    return oracle.prenorm_block_train(inp.x, kw.get("rm", inp.running_mean),
                                      kw.get("rv", inp.running_var), inp.gamma, inp.beta,
                                      inp.eps, momentum, kw.get("w", inp.weight),
                                      kw.get("bias", inp.bias), inp.dilation,
                                      rows_n=kw.get("rows_n"), rows_o=kw.get("rows_o"))


def _rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


@pytest.mark.parametrize("case", json.load(open(os.path.join(
    GOLDEN, "prenorm_block_train_hand.json")))["cases"], ids=lambda c: c["name"][:40])
def test_hand_worked_cases(case):
    out, rm, rv, bm, bv = oracle.prenorm_block_train(
        np.array(case["x"]), case["running_mean"], case["running_var"], case["gamma"],
        case["beta"], case["eps"], case["momentum"], np.array(case["weight"]), case["bias"],
        case["dilation"])
    np.testing.assert_allclose(out, np.array(case["out"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(bm, case["batch_mean"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(bv, case["batch_var"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(rm, case["running_mean_after"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(rv, case["running_var_after"], rtol=0, atol=1e-15)


@pytest.mark.parametrize("N,C,L,d,momentum", [(2, 32, 512, 128, 0.1),   # tiny workload
                                              (3, 16, 300, 7, 0.3),
                                              (1, 8, 100, 60, 0.1),     # one sample
                                              (4, 8, 64, 1, 0.9)])
def test_matches_torch_fp64_modules(N, C, L, d, momentum):
    inp = syn.prenorm_block_inputs(N, C, L, d, seed=11)
    out, rm, rv, _, _ = _run(inp, momentum)
    t_out, t_rm, t_rv = _torch_train_fp64(inp, momentum)
    assert _rel(out, t_out) < 1e-12
    np.testing.assert_allclose(rm, t_rm, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(rv, t_rv, rtol=1e-13, atol=1e-15)


def test_batch_statistics_are_numpy_mean_and_var():
    inp = syn.prenorm_block_inputs(3, 8, 200, 4, seed=12)
    _, rm, rv, bm, bv = _run(inp, 1.0)
    x = inp.x.double().numpy()
    np.testing.assert_allclose(bm, x.mean(axis=(0, 2)), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(bv, x.var(axis=(0, 2)), rtol=1e-13)
    np.testing.assert_allclose(rm, x.mean(axis=(0, 2)), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(rv, x.var(axis=(0, 2), ddof=1), rtol=1e-13)


def test_running_buffers_do_not_reach_the_output():
    inp = syn.prenorm_block_inputs(2, 8, 96, 8, seed=13)
    C = inp.x.shape[1]
    a = _run(inp, 0.1)[0]
    b = _run(inp, 0.1, rm=torch.full((C,), 3.0), rv=torch.full((C,), 7.0))[0]
    assert np.array_equal(a, b)
    _, rm, rv, _, _ = _run(inp, 0.0)
    assert np.array_equal(rm, inp.running_mean.double().numpy())
    assert np.array_equal(rv, inp.running_var.double().numpy())


def test_equals_eval_block_with_batch_statistics():
    """Training mode is the eval-mode block with the batch mean and biased
    variance in place of the running statistics."""
    inp = syn.prenorm_block_inputs(2, 16, 128, 16, seed=14)
    x = inp.x.double().numpy()
    out = _run(inp, 0.1)[0]
    ref = oracle.prenorm_block(x, x.mean(axis=(0, 2)), x.var(axis=(0, 2)), inp.gamma, inp.beta,
                               inp.eps, inp.weight, inp.bias, inp.dilation)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


def test_rows_match_full_and_null_buffers():
    inp = syn.prenorm_block_inputs(3, 16, 96, 16, seed=15)
    full = _run(inp, 0.1)[0]
    rn, ro = [0, 2, 1, 2], [0, 15, 7, 3]
    rows, rm, rv, _, _ = oracle.prenorm_block_train(
        inp.x, None, None, inp.gamma, inp.beta, inp.eps, 0.1, inp.weight, inp.bias,
        inp.dilation, rows_n=rn, rows_o=ro)
    assert rm is None and rv is None
    for r, (n, o) in enumerate(zip(rn, ro)):
        assert np.array_equal(rows[r], full[n, o])


def test_rejects_single_value_per_channel():
    inp = syn.prenorm_block_inputs(1, 4, 1, 1, seed=16)
    with pytest.raises(ValueError):
        _run(inp, 0.1)
