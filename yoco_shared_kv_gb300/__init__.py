"""YOCO shared-KV cross-decoder hot path for GB300 (sm_103a).

The compute lives in ``libyoco_kv.so`` (C ABI declared in
``include/yoco_kv.h``); ``_native`` is its ctypes binding and ``pipeline``
strings the three calls into one step. Importing ``_native`` (or anything
that needs it) fails loudly when the library has not been built.
"""

__all__ = ["build", "native", "pipeline"]


def native():
    from . import _native
    return _native
