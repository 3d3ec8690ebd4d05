"""GB300-native selectively batched Transformer iteration (Orca-style).

liborca.so (C ABI, include/orca.h) holds the scheduler, the K/V slot pool and
the sm_103a kernels; `_orca` is its ctypes binding and `runtime` the PyTorch
plumbing (device memory, streams, serving loop).
"""
from . import _orca  # noqa: F401
from ._orca import OrcaError  # noqa: F401
