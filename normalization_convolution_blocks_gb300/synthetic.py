"""Seeded synthetic inputs for the three blocks.

This module only draws random tensors (CPU ``torch.Generator``, fixed draw
order); it holds none of the blocks' arithmetic, so the CUDA path and the CPU
oracle can both consume its output without sharing any computation.

Distributions follow the PopcornBench problem statements (PyTorch default
initialisation: weights and biases ~U(-1/sqrt(fan_in), 1/sqrt(fan_in)) with
fan_in = C_in * kernel_size; inputs ~N(0, 1)), with the BatchNorm buffers of
the pre-norm block drawn at random so that the eval-mode affine is not the
identity:

* pre-norm block: x ~N(0,1); running_mean ~U(-0.5,0.5); running_var
  ~U(0.5,2); gamma ~U(0.5,1.5); beta ~U(-0.5,0.5); conv weight and bias
  ~U(+-1/sqrt(3C)).  Draw order: x, rm, rv, gamma, beta, W, bias.  The
  training-mode workload draws the same tensors (rm, rv are then the running
  buffers' starting values; BatchNorm momentum 0.1).
* conv + GroupNorm: x ~N(0,1); W (C_out, C_in, k) ~U(+-1/sqrt(k*C_in)), k = 3
  unless another kernel size is asked for; gamma ~U(0.5,1.5);
  beta ~U(-0.5,0.5).  Draw order: x, W, gamma, beta.
* Linear + BN + bias + divide + Swish: x ~N(0,1); W, b_lin ~U(+-1/sqrt(IN));
  gamma = 1, beta = 0 (module defaults) unless ``random_affine``, then
  gamma ~U(0.5,1.5), beta ~U(-0.5,0.5); running stats 0 and 1; the added
  scalar bias ~N(0,1).  Draw order: x, W, b_lin, [gamma, beta], add_bias.
  The eval-mode workload draws the same tensors and normalizes with the
  running statistics (0 and 1).

bf16 storage: the fp32 draw is rounded to bf16 once (round to nearest even by
``Tensor.to``); both sides then read the same bf16 values.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


def _uniform(g, shape, lo, hi):
    return torch.rand(shape, generator=g, dtype=torch.float32) * (hi - lo) + lo


def _normal(g, shape):
    return torch.randn(shape, generator=g, dtype=torch.float32)


@dataclass
class BlockInputs:
    x: torch.Tensor
    running_mean: torch.Tensor
    running_var: torch.Tensor
    gamma: torch.Tensor
    beta: torch.Tensor
    weight: torch.Tensor
    bias: torch.Tensor
    dilation: int
    eps: float = 1e-5

    @property
    def shape(self):
        return tuple(self.x.shape)


def prenorm_block_inputs(N, C, L, dilation, seed=0, dtype=torch.float32, eps=1e-5):
    g = torch.Generator("cpu").manual_seed(seed)
    x = _normal(g, (N, C, L))
    rm = _uniform(g, (C,), -0.5, 0.5)
    rv = _uniform(g, (C,), 0.5, 2.0)
    gamma = _uniform(g, (C,), 0.5, 1.5)
    beta = _uniform(g, (C,), -0.5, 0.5)
    bound = 1.0 / math.sqrt(3 * C)
    w = _uniform(g, (C, C, 3), -bound, bound)
    b = _uniform(g, (C,), -bound, bound)
    if dtype != torch.float32:
        x, w, b = x.to(dtype), w.to(dtype), b.to(dtype)
    return BlockInputs(x, rm, rv, gamma, beta, w, b, int(dilation), eps)


@dataclass
class ConvGNInputs:
    x: torch.Tensor
    weight: torch.Tensor
    gamma: torch.Tensor
    beta: torch.Tensor
    num_groups: int
    eps: float = 1e-5
    bias: torch.Tensor | None = None


def conv_groupnorm_inputs(N, Cin, Cout, T, num_groups, seed=0, eps=1e-5, kernel_size=3):
    g = torch.Generator("cpu").manual_seed(seed)
    x = _normal(g, (N, Cin, T))
    bound = 1.0 / math.sqrt(kernel_size * Cin)
    w = _uniform(g, (Cout, Cin, kernel_size), -bound, bound)
    gamma = _uniform(g, (Cout,), 0.5, 1.5)
    beta = _uniform(g, (Cout,), -0.5, 0.5)
    return ConvGNInputs(x, w, gamma, beta, int(num_groups), eps)


@dataclass
class LinearInputs:
    x: torch.Tensor
    weight: torch.Tensor
    lin_bias: torch.Tensor
    gamma: torch.Tensor
    beta: torch.Tensor
    running_mean: torch.Tensor
    running_var: torch.Tensor
    add_bias: torch.Tensor          # shape (1,)
    eps: float = 1e-5
    momentum: float = 0.1
    divide_value: float = 1.0


def linear_bn_swish_inputs(B, IN, OUT, seed=0, random_affine=False, eps=1e-5,
                           momentum=0.1, divide_value=1.0):
    g = torch.Generator("cpu").manual_seed(seed)
    x = _normal(g, (B, IN))
    bound = 1.0 / math.sqrt(IN)
    w = _uniform(g, (OUT, IN), -bound, bound)
    b = _uniform(g, (OUT,), -bound, bound)
    if random_affine:
        gamma = _uniform(g, (OUT,), 0.5, 1.5)
        beta = _uniform(g, (OUT,), -0.5, 0.5)
    else:
        gamma = torch.ones(OUT)
        beta = torch.zeros(OUT)
    add_bias = _normal(g, (1,))
    return LinearInputs(x, w, b, gamma, beta, torch.zeros(OUT), torch.ones(OUT), add_bias,
                        eps, momentum, divide_value)


@dataclass(frozen=True)
class Workload:
    """A named workload: which block, and its sizes."""
    name: str
    kind: str                      # "block" | "block_train" | "conv_gn" | "linear"
    params: dict = field(default_factory=dict)

    def make(self, seed=0):
        p = dict(self.params)
        if self.kind in ("block", "block_train"):
            dt = torch.bfloat16 if p.pop("dtype", "f32") == "bf16" else torch.float32
            return prenorm_block_inputs(p["N"], p["C"], p["L"], p["dilation"], seed=seed,
                                        dtype=dt)
        if self.kind == "conv_gn":
            return conv_groupnorm_inputs(p["N"], p["Cin"], p["Cout"], p["T"], p["G"],
                                         seed=seed)
        if self.kind == "linear":
            return linear_bn_swish_inputs(p["B"], p["IN"], p["OUT"], seed=seed,
                                          random_affine=p.get("random_affine", False))
        raise ValueError(self.kind)


WORKLOADS = {
    "prenorm_block_tiny_f32": Workload("prenorm_block_tiny_f32", "block",
                                       dict(N=2, C=32, L=512, dilation=128)),
    "prenorm_block_f32": Workload("prenorm_block_f32", "block",
                                  dict(N=32, C=256, L=4096, dilation=128)),
    "prenorm_block_train_f32": Workload("prenorm_block_train_f32", "block_train",
                                        dict(N=32, C=256, L=4096, dilation=128)),
    "conv1d_groupnorm_f32": Workload("conv1d_groupnorm_f32", "conv_gn",
                                     dict(N=16, Cin=128, Cout=256, T=1024, G=32)),
    "linear_bn_swish_f32": Workload("linear_bn_swish_f32", "linear",
                                    dict(B=1024, IN=8192, OUT=8192)),
    "linear_bn_swish_eval_f32": Workload("linear_bn_swish_eval_f32", "linear",
                                         dict(B=1024, IN=8192, OUT=8192, training=False)),
}
for _C in (256, 512):
    for _d in (1, 8, 128, 512):
        _n = f"prenorm_block_bf16_C{_C}_d{_d}"
        WORKLOADS[_n] = Workload(_n, "block", dict(N=8, C=_C, L=16384, dilation=_d,
                                                   dtype="bf16"))
