"""Float64 CPU oracle of the WKV operator (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library
and ``rwkv_linear_attention_backward_b300``) never does.

The arithmetic lives in ``wkv_oracle.c`` (plain C, float64, OpenMP over
independent channels); this module compiles it with gcc when needed and
wraps each entry point for numpy arrays.  Inputs of any float dtype are
widened to float64 before the call, so the oracle sees exactly the values
handed to the GPU (fp32, or bf16 rounded values).
"""
from __future__ import annotations

import ctypes
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
SOURCE = _HERE / "wkv_oracle.c"
LIBRARY = _HERE / "liboracle.so"

_DP = ctypes.POINTER(ctypes.c_double)


def build(source: Path = SOURCE, output: Path = LIBRARY, quiet: bool = True) -> Path:
    """Compile the oracle C source into a shared library with gcc."""
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-Wall", "-o", str(output), str(source), "-lm"]
    subprocess.run(cmd, check=True, capture_output=quiet)
    return output


def _stale(lib: Path, src: Path) -> bool:
    return (not lib.exists()) or lib.stat().st_mtime < src.stat().st_mtime


class Oracle:
    """ctypes handle on one compiled copy of the oracle library."""

    def __init__(self, library: Path | str):
        self.path = str(library)
        self._lib = ctypes.CDLL(self.path)
        i, p = ctypes.c_int, _DP
        sigs = {
            "wkv_oracle_forward_direct": [i, i, i, p, p, p, p, p],
            "wkv_oracle_forward_recurrent": [i, i, i, p, p, p, p, p],
            "wkv_oracle_forward_state": [i, i, i] + [p] * 11,
            "wkv_oracle_token_shift": [i, i, i] + [p] * 8,
            "wkv_oracle_token_shift_backward": [i, i, i] + [p] * 13,
            "wkv_oracle_backward_adjoint": [i, i, i, p, p, p, p, p, p, p, p, p],
            "wkv_oracle_backward_direct": [i, i, i, p, p, p, p, p, p, p, p, p],
            "wkv_oracle_backward_state": [i, i, i] + [p] * 16,
            "wkv_oracle_state": [i, i, i, p, p, p, i, p, p, p],
            "wkv_oracle_decode_step": [i, i, i] + [p] * 17,
            "wkv_oracle_forward_gated": [i, i, i] + [p] * 6,
            "wkv_oracle_forward_gated_recurrent": [i, i, i] + [p] * 6,
            "wkv_oracle_backward_gated": [i, i, i] + [p] * 11,
            "wkv_oracle_state_fold": [i, i, p, i, p, ctypes.POINTER(ctypes.c_longlong), p],
            "wkv_oracle_sqrelu": [ctypes.c_size_t] + [p] * 2,
            "wkv_oracle_sqrelu_backward": [ctypes.c_size_t] + [p] * 3,
            "wkv_oracle_cmix_gate": [ctypes.c_size_t] + [p] * 3,
            "wkv_oracle_cmix_gate_backward": [ctypes.c_size_t] + [p] * 5,
        }
        for name, args in sigs.items():
            fn = getattr(self._lib, name)
            fn.argtypes = args
            fn.restype = None
        self._lib.wkv_oracle_num_threads.restype = ctypes.c_int

    # ------------------------------------------------------------------ utils
    @staticmethod
    def _in(a) -> np.ndarray:
        if hasattr(a, "detach"):  # torch tensor (CPU); bf16 widened via float32
            import torch

            a = a.detach().to("cpu")
            if a.dtype == torch.bfloat16:
                a = a.float()
            a = a.numpy()
        return np.ascontiguousarray(np.asarray(a, dtype=np.float64))

    @staticmethod
    def _ptr(a: np.ndarray | None):
        if a is None:
            return ctypes.cast(None, _DP)
        return a.ctypes.data_as(_DP)

    def num_threads(self) -> int:
        return int(self._lib.wkv_oracle_num_threads())

    # -------------------------------------------------------------- forward
    def forward_direct(self, w, u, k, v) -> np.ndarray:
        w, u, k, v = map(self._in, (w, u, k, v))
        B, T, C = k.shape
        y = np.empty_like(k)
        self._lib.wkv_oracle_forward_direct(B, T, C, *map(self._ptr, (w, u, k, v, y)))
        return y

    def forward_recurrent(self, w, u, k, v) -> np.ndarray:
        w, u, k, v = map(self._in, (w, u, k, v))
        B, T, C = k.shape
        y = np.empty_like(k)
        self._lib.wkv_oracle_forward_recurrent(B, T, C, *map(self._ptr, (w, u, k, v, y)))
        return y

    def forward_state(self, w, u, k, v, state_in=None):
        """wkv over k, v [B, T, C] continuing from ``state_in`` = (num, den,
        pp), each [B, C] (None: the empty state).  Returns (y, (num, den, pp)),
        the state after the T tokens."""
        w, u, k, v = map(self._in, (w, u, k, v))
        B, T, C = k.shape
        y = np.empty_like(k)
        if state_in is None:
            sin = (None, None, None)
        else:
            sin = tuple(self._in(a).reshape(B, C).copy() for a in state_in)
        out = tuple(np.empty((B, C)) for _ in range(3))
        self._lib.wkv_oracle_forward_state(B, T, C, *map(self._ptr, (w, u, k, v) + sin + (y,) + out))
        return y, out

    # ------------------------------------------------------------ gated output
    def forward_gated(self, w, u, k, v, r) -> np.ndarray:
        """sigmoid(r) * wkv for k, v, r [B, T, C]."""
        w, u, k, v, r = map(self._in, (w, u, k, v, r))
        B, T, C = k.shape
        out = np.empty_like(k)
        self._lib.wkv_oracle_forward_gated(B, T, C, *map(self._ptr, (w, u, k, v, r, out)))
        return out

    def forward_gated_recurrent(self, w, u, k, v, r) -> np.ndarray:
        """sigmoid(r) * wkv through the recurrent form (the O(T) form timed
        as the CPU baseline)."""
        w, u, k, v, r = map(self._in, (w, u, k, v, r))
        B, T, C = k.shape
        out = np.empty_like(k)
        self._lib.wkv_oracle_forward_gated_recurrent(B, T, C, *map(self._ptr, (w, u, k, v, r, out)))
        return out

    def backward_gated(self, w, u, k, v, r, gout):
        """(gw, gu, gk, gv, gr): gradients of sum(gout * sigmoid(r) * wkv)."""
        w, u, k, v, r, gout = map(self._in, (w, u, k, v, r, gout))
        B, T, C = k.shape
        gw = np.empty(C)
        gu = np.empty(C)
        gk, gv, gr = (np.empty_like(k) for _ in range(3))
        self._lib.wkv_oracle_backward_gated(B, T, C, *map(self._ptr, (w, u, k, v, r, gout, gw, gu, gk, gv, gr)))
        return gw, gu, gk, gv, gr

    def state_fold(self, w, states, lengths):
        """(num, den, pp), each [B, C]: the state after consecutive segments
        given by their own states (a sequence of (num, den, pp) triples, or
        an array [n, 3, B, C]) and their lengths in tokens."""
        w = self._in(w)
        if not hasattr(states, "shape"):
            states = np.stack([np.stack([self._in(x) for x in st]) for st in states]) if len(states) else None
        else:
            states = self._in(states)
        n = 0 if states is None else states.shape[0]
        if n == 0:
            raise ValueError("give the shape through at least one segment")
        B, C = states.shape[2], states.shape[3]
        states = np.ascontiguousarray(states, dtype=np.float64)
        lens = (ctypes.c_longlong * n)(*[int(x) for x in lengths])
        out = np.empty((3, B, C))
        self._lib.wkv_oracle_state_fold(B, C, self._ptr(w), n, self._ptr(states), lens, self._ptr(out))
        return out[0], out[1], out[2]

    # --------------------------------------------------- channel mixing
    def _elementwise(self, fn, outs, *args):
        args = [self._in(a) for a in args]
        shape = args[0].shape
        for a in args[1:]:
            assert a.shape == shape, "elementwise inputs of different shapes"
        res = tuple(np.empty(shape) for _ in range(outs))
        fn(args[0].size, *map(self._ptr, tuple(args) + res))
        return res if outs > 1 else res[0]

    def sqrelu(self, k) -> np.ndarray:
        """max(k, 0)^2, elementwise."""
        return self._elementwise(self._lib.wkv_oracle_sqrelu, 1, k)

    def sqrelu_backward(self, k, ga) -> np.ndarray:
        """gk = 2 max(k, 0) ga."""
        return self._elementwise(self._lib.wkv_oracle_sqrelu_backward, 1, k, ga)

    def cmix_gate(self, r, vk) -> np.ndarray:
        """sigmoid(r) * vk, elementwise."""
        return self._elementwise(self._lib.wkv_oracle_cmix_gate, 1, r, vk)

    def cmix_gate_backward(self, r, vk, gout):
        """(gr, gvk) of sum(gout * sigmoid(r) * vk)."""
        return self._elementwise(self._lib.wkv_oracle_cmix_gate_backward, 2, r, vk, gout)

    # ---------------------------------------------------------- token shift
    def token_shift(self, x, x0, mu_k, mu_v, mu_r):
        """(xk, xv, xr) of x [B, T, C]; x0 [B, C] is the token before the
        sequence (None: zeros)."""
        x, mu_k, mu_v, mu_r = map(self._in, (x, mu_k, mu_v, mu_r))
        x0 = None if x0 is None else self._in(x0)
        B, T, C = x.shape
        outs = tuple(np.empty_like(x) for _ in range(3))
        self._lib.wkv_oracle_token_shift(B, T, C, *map(self._ptr, (x, x0, mu_k, mu_v, mu_r) + outs))
        return outs

    def token_shift_backward(self, x, x0, mu_k, mu_v, mu_r, gxk, gxv, gxr):
        """(gx, gx0, gmu_k, gmu_v, gmu_r); gx0 is None when x0 is None."""
        x, mu_k, mu_v, mu_r, gxk, gxv, gxr = map(self._in, (x, mu_k, mu_v, mu_r, gxk, gxv, gxr))
        x0 = None if x0 is None else self._in(x0)
        B, T, C = x.shape
        gx = np.empty_like(x)
        gx0 = None if x0 is None else np.empty((B, C))
        gm = tuple(np.empty(C) for _ in range(3))
        self._lib.wkv_oracle_token_shift_backward(
            B, T, C, *map(self._ptr, (x, x0, mu_k, mu_v, mu_r, gxk, gxv, gxr, gx, gx0) + gm))
        return (gx, gx0) + gm

    # ------------------------------------------------------------- backward
    def _backward(self, fn, w, u, k, v, gy):
        w, u, k, v, gy = map(self._in, (w, u, k, v, gy))
        B, T, C = k.shape
        gw = np.empty(C)
        gu = np.empty(C)
        gk = np.empty_like(k)
        gv = np.empty_like(k)
        fn(B, T, C, *map(self._ptr, (w, u, k, v, gy, gw, gu, gk, gv)))
        return gw, gu, gk, gv

    def backward_adjoint(self, w, u, k, v, gy):
        """Returns (gw, gu, gk, gv) by reverse-mode of the recurrence."""
        return self._backward(self._lib.wkv_oracle_backward_adjoint, w, u, k, v, gy)

    def backward_direct(self, w, u, k, v, gy):
        """Returns (gw, gu, gk, gv) by differentiating the O(T^2) sum."""
        return self._backward(self._lib.wkv_oracle_backward_direct, w, u, k, v, gy)

    def backward_state(self, w, u, k, v, gy, state_in=None, adj_end=None):
        """Gradients of sum(gy * wkv) + ga_end a_T + gb_end b_T for a segment
        starting from ``state_in`` = (num, den, pp) ([B, C] each; None:
        empty), ``adj_end`` = (ga_end, gb_end) the gradient of the unscaled
        end sums (None: zero).  Returns (gw, gu, gk, gv, (ga_start,
        gb_start)), the last the gradient of the unscaled start sums."""
        w, u, k, v, gy = map(self._in, (w, u, k, v, gy))
        B, T, C = k.shape
        sin = (None, None, None) if state_in is None else tuple(self._in(x).reshape(B, C).copy() for x in state_in)
        aend = (None, None) if adj_end is None else tuple(self._in(x).reshape(B, C).copy() for x in adj_end)
        gw, gu = np.empty(C), np.empty(C)
        gk, gv = np.empty_like(k), np.empty_like(k)
        ga, gb = np.empty((B, C)), np.empty((B, C))
        self._lib.wkv_oracle_backward_state(B, T, C, *map(self._ptr, (w, u, k, v, gy) + sin + aend +
                                                          (gw, gu, gk, gv, ga, gb)))
        return gw, gu, gk, gv, (ga, gb)

    # ---------------------------------------------------------------- state
    def state(self, w, k, v, t: int):
        """(num, den, pp), each [B, C], after the first t tokens."""
        w, k, v = map(self._in, (w, k, v))
        B, T, C = k.shape
        num = np.empty((B, C))
        den = np.empty((B, C))
        pp = np.empty((B, C))
        self._lib.wkv_oracle_state(B, T, C, *map(self._ptr, (w, k, v)), int(t), *map(self._ptr, (num, den, pp)))
        return num, den, pp

    # --------------------------------------------------------------- decode
    def decode_step(self, x, x_prev, mu_k, mu_v, mu_r, r, k, v, w, u, num, den, pp, mix: bool = True):
        """One RNN-mode step of L layers.  Returns (y, num, den, pp, xk, xv, xr)
        with the state arrays new (inputs are not modified); the mix outputs
        are None when ``mix`` is False."""
        x, x_prev, mu_k, mu_v, mu_r, r, k, v, w, u = map(self._in, (x, x_prev, mu_k, mu_v, mu_r, r, k, v, w, u))
        num, den, pp = (self._in(a).copy() for a in (num, den, pp))
        L, B, C = x.shape
        y = np.empty_like(x)
        xk = np.empty_like(x) if mix else None
        xv = np.empty_like(x) if mix else None
        xr = np.empty_like(x) if mix else None
        self._lib.wkv_oracle_decode_step(
            L, B, C,
            *map(self._ptr, (x, x_prev, mu_k, mu_v, mu_r, r, k, v, w, u, num, den, pp, y, xk, xv, xr)),
        )
        return y, num, den, pp, xk, xv, xr


_DEFAULT: Oracle | None = None


def load() -> Oracle:
    """The oracle built from ``wkv_oracle.c`` (compiled on first use)."""
    global _DEFAULT
    if _DEFAULT is None:
        if _stale(LIBRARY, SOURCE):
            build()
        _DEFAULT = Oracle(LIBRARY)
    return _DEFAULT


def __getattr__(name):  # convenience: oracle.forward_direct(...) etc.
    if name.startswith("_"):
        raise AttributeError(name)
    return getattr(load(), name)

