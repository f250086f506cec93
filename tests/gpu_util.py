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


# ---------------------------------------------------------------------------
# Out-of-bounds guards.  An output tensor is carved out of a larger buffer
# whose margins (before and after it, each at least one full 128 x 256 output
# tile) hold a NaN bit pattern no kernel writes.  After the call, every margin
# word must still hold that pattern, bit for bit: a write past a ragged tile's
# end, or before the tensor's start, changes it.
# ---------------------------------------------------------------------------
_PATTERN = {torch.float32: (torch.int32, 0x7FA5A5A5),
            torch.bfloat16: (torch.int16, 0x7FA5)}
GUARD_ELEMS = 128 * 256 + 4096


class Guarded:
    """`view` is a contiguous tensor of `shape` inside a guarded buffer.

    offset shifts the view by that many elements past the margin (odd-offset
    views); pinned=True puts the buffer in page-locked host memory (for the
    host-buffer entry points)."""

    def __init__(self, shape, dtype, device=None, offset=0, pinned=False):
        n = 1
        for s in shape:
            n *= int(s)
        self.dtype = dtype
        self.n, self.offset = n, offset
        total = n + 2 * GUARD_ELEMS + offset
        if pinned:
            self.buf = torch.empty(total, dtype=dtype, pin_memory=True)
        else:
            self.buf = torch.empty(total, dtype=dtype, device=device)
        itype, pat = _PATTERN[dtype]
        self.bits = self.buf.view(itype)
        self.bits.fill_(pat)
        self.pattern = pat
        start = GUARD_ELEMS + offset
        self.view = self.buf[start:start + n].view(tuple(shape))

    def check(self, what=""):
        """Asserts that both margins still hold the pattern."""
        if self.buf.is_cuda:
            torch.cuda.synchronize()
        start = GUARD_ELEMS + self.offset
        for name, part in (("before", self.bits[:start]), ("after", self.bits[start + self.n:])):
            bad = (part != self.pattern).nonzero()
            assert bad.numel() == 0, (
                f"{what}: {bad.numel()} guard word(s) {name} the output were overwritten "
                f"(first at margin index {int(bad[0])})")


def guarded_like(t, device=None, offset=0, pinned=False):
    return Guarded(tuple(t.shape), t.dtype, device if device is not None else t.device,
                   offset=offset, pinned=pinned)
