"""B300-native WKV operator (RWKV time mixing): forward, backward and decode.

The compute lives in ``libwkv.so`` (hand-written CUDA for sm_103a behind a
C ABI declared in ``include/wkv.h``).  ``binding`` wraps that ABI for torch
tensors; importing it loads the library and raises if it is missing.  The
``inputs`` module (seeded synthetic inputs) needs no GPU and no library.
``tsplit`` runs the forward pass of one long sequence split over the ranks
of a process group along time.
"""
from __future__ import annotations

import importlib

__all__ = ["binding", "inputs", "build", "tsplit"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
