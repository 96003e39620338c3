"""B300-native WKV operator (RWKV time mixing): forward, backward and decode.

The compute lives in ``libwkv.so`` (hand-written CUDA for sm_103a behind a
C ABI declared in ``include/wkv.h``).  ``binding`` wraps that ABI for torch
tensors; importing it loads the library and raises if it is missing.  The
``inputs`` module (seeded synthetic inputs) needs no GPU and no library.
"""
from __future__ import annotations

__all__ = ["binding", "inputs"]


def __getattr__(name):
    if name == "binding":
        from . import binding as _b

        return _b
    if name == "inputs":
        from . import inputs as _i

        return _i
    raise AttributeError(name)
