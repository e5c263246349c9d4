"""Batched W4A16 mixture-of-experts decode step on one GB300 (sm_103a).

The compute lives in the CUDA library ``_lib/libbitmoe.so`` behind the C ABI
of ``include/bitmoe.h``; ``binding`` is a ctypes layer with the same names.
PyTorch is used only for device memory and streams.
"""

from .binding import *  # noqa: F401,F403
from .binding import BitMoeError, lib, ptr, stream_handle, LIB_PATH  # noqa: F401
from . import build as _build


def build(force=False, verbose=False):
    """Compile libbitmoe.so for sm_103a in-tree; returns its path."""
    return _build.build(force=force, verbose=verbose)
