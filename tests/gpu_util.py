"""Shared helpers of the GPU parity tests (tolerances, comparisons, device moves)."""
import numpy as np
import pytest
import torch

# Tolerances (parity bar): fp32 storage, compensated tensor-core math: relative
# L2 1e-4 and max-abs 1e-3 against the fp64 oracle; bf16 storage: relative L2
# 2e-2; BatchNorm running statistics: max-abs 1e-5.
F32_REL_L2, F32_MAX_ABS = 1e-4, 1e-3
BF16_REL_L2 = 2e-2
RUNNING_STAT_ABS = 1e-5


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from normalization_convolution_blocks_gb300 import api, build
    build.build()
    api.load()
    return torch.device("cuda", 0)


def to(dev, t):
    return None if t is None else t.to(dev)


def errors(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "non-finite output"
    rel = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))
    mx = float(np.abs(got - ref).max()) if got.size else 0.0
    return rel, mx


def assert_f32(got, ref, what=""):
    rel, mx = errors(got, ref)
    assert rel < F32_REL_L2 and mx < F32_MAX_ABS, f"{what}: rel_l2={rel:.3e} max_abs={mx:.3e}"
    return rel, mx


def assert_bf16(got, ref, what=""):
    rel, mx = errors(got, ref)
    assert rel < BF16_REL_L2, f"{what}: rel_l2={rel:.3e} max_abs={mx:.3e}"
    return rel, mx
