"""GB300-native (sm_103a) DFlash 2 drafter pass: context settle, block forward, head and selector.

The compute lives in ``_build/libdflash.so`` (hand-written CUDA behind the C ABI
of ``include/dflash.h``); ``_lib`` binds it with ctypes and ``drafter.Drafter``
holds the device memory with PyTorch. There is no host fallback: without the
built library every call raises.
"""
from . import _lib  # noqa: F401

__all__ = ["_lib"]
