"""GB300-native (sm_103a) normalization-fused Conv1d blocks.

The compute path is the CUDA library ``libnrc.so`` (sources in ``csrc/``,
C ABI in ``include/nrc.h``); ``api`` is a thin ctypes binding over it that
only marshals arguments (torch tensors -> device pointers, stream handles).
There is no CPU fallback: calling ``api`` without the built library or a GPU
raises.
"""
__all__ = ["api", "synthetic", "build"]
