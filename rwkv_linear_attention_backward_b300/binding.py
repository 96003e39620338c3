"""Thin Python binding of libwkv.so (the C ABI in include/wkv.h) for torch tensors.

Argument marshalling only: every step of the computation runs in the
library's CUDA kernels.  torch provides device memory and streams.  Importing
this module loads ``libwkv.so`` from this package directory and raises
``ImportError`` if it is missing (build it with
``python -m rwkv_linear_attention_backward_b300.build``); there is no
fallback implementation.

Entry points mirror the ABI names: ``forward``, ``forward_with_state``,
``forward_gated``, ``backward``, ``backward_gated``, ``decode_step``,
``token_shift``, ``token_shift_backward``, the ``channel_mix_*`` pointwise
steps, ``workspace_check``, plus size queries and test hooks.  All tensors must be
contiguous CUDA tensors on the current device; calls are enqueued on the
current torch stream (or ``stream=``) and return without synchronising.
"""
from __future__ import annotations

import ctypes
from pathlib import Path

import torch

LIBRARY = Path(__file__).resolve().parent / "libwkv.so"

if not LIBRARY.exists():
    raise ImportError(f"{LIBRARY} is missing: build it with `python -m rwkv_linear_attention_backward_b300.build`")

_lib = ctypes.CDLL(str(LIBRARY))

_vp, _i, _sz, _ll = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_longlong

_SIGNATURES = {
    "wkv_status_string": ([_i], ctypes.c_char_p),
    "wkv_last_error_string": ([], ctypes.c_char_p),
    "wkv_version": ([], _i),
    "wkv_chunk_len": ([], _i),
    "wkv_checkpoint_floats": ([_i, _i, _i], _sz),
    "wkv_forward_workspace_bytes": ([_i, _i, _i], _sz),
    "wkv_backward_workspace_bytes": ([_i, _i, _i], _sz),
    "wkv_workspace_init": ([_vp, _sz, _vp], _i),
    "wkv_workspace_check": ([_vp, _vp], _i),
    "wkv_sync_status": ([_vp], _i),
    "wkv_forward": ([_i, _i, _i, _i] + [_vp] * 6 + [_vp, _sz, _vp], _i),
    "wkv_forward_with_state": ([_i, _i, _i, _i] + [_vp] * 8 + [_vp, _sz, _vp], _i),
    "wkv_backward": ([_i, _i, _i, _i] + [_vp] * 10 + [_vp, _sz, _vp], _i),
    "wkv_forward_gated": ([_i, _i, _i, _i] + [_vp] * 9 + [_vp, _sz, _vp], _i),
    "wkv_backward_gated": ([_i, _i, _i, _i] + [_vp] * 12 + [_vp, _sz, _vp], _i),
    "wkv_backward_with_state": ([_i, _i, _i, _i] + [_vp] * 13 + [_vp, _sz, _vp], _i),
    "wkv_decode_step": ([_i, _i, _i] + [_vp] * 17 + [_vp], _i),
    "wkv_decode_step_bf16": ([_i, _i, _i] + [_vp] * 17 + [_vp], _i),
    "wkv_forward_noalloc": ([_i, _i, _i, _i] + [_vp] * 6 + [_vp], _i),
    "wkv_debug_set_wait_budget_ns": ([_ll], _i),
    "wkv_debug_set_skip_chunk": ([_i], _i),
    "wkv_debug_set_scan_mode": ([_i], _i),
    "wkv_scan_strategy": ([_i, _i, _i], _i),
    "wkv_debug_set_max_runs": ([_i], _i),
    "wkv_debug_set_chain_len": ([_i], _i),
    "wkv_token_shift": ([_i, _i, _i] + [_vp] * 8 + [_vp], _i),
    "wkv_token_shift_backward_workspace_bytes": ([_i, _i, _i], _sz),
    "wkv_token_shift_backward": ([_i, _i, _i] + [_vp] * 13 + [_vp, _sz, _vp], _i),
    "wkv_state_fold": ([_i, _i, _vp, _i, _vp, ctypes.POINTER(_ll), _vp, _vp], _i),
    "wkv_adjoint_fold": ([_i, _i, _vp, _i, _vp, ctypes.POINTER(_ll), _vp, _vp, _vp], _i),
    "wkv_channel_mix_sqrelu": ([_ll] + [_vp] * 2 + [_vp], _i),
    "wkv_channel_mix_sqrelu_backward": ([_ll] + [_vp] * 3 + [_vp], _i),
    "wkv_channel_mix_gate": ([_ll] + [_vp] * 3 + [_vp], _i),
    "wkv_channel_mix_gate_backward": ([_ll] + [_vp] * 5 + [_vp], _i),
}
for _name, (_args, _res) in _SIGNATURES.items():
    _fn = getattr(_lib, _name)
    _fn.argtypes = _args
    _fn.restype = _res

WKV_OK, WKV_F32, WKV_BF16 = 0, 0, 1
EXPORTED = tuple(_SIGNATURES)


class WKVError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = _lib.wkv_status_string(status).decode()
        detail = _lib.wkv_last_error_string().decode()
        super().__init__(f"{where}: {msg}" + (f" ({detail})" if detail else ""))


def _check(status: int, where: str) -> None:
    if status != WKV_OK:
        raise WKVError(status, where)


def _p(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need(t: torch.Tensor, name: str, dtypes=(torch.float32,), shape=None) -> None:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} must have dtype in {dtypes}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


# ----------------------------------------------------------------- queries
def version() -> int:
    return int(_lib.wkv_version())


def chunk_len() -> int:
    return int(_lib.wkv_chunk_len())


def checkpoint_floats(B: int, T: int, C: int) -> int:
    return int(_lib.wkv_checkpoint_floats(B, T, C))


def forward_workspace_bytes(B: int, T: int, C: int) -> int:
    return int(_lib.wkv_forward_workspace_bytes(B, T, C))


def backward_workspace_bytes(B: int, T: int, C: int) -> int:
    return int(_lib.wkv_backward_workspace_bytes(B, T, C))


# -------------------------------------------------------------- workspace
class Workspace:
    """A zero-filled device buffer reused across calls in stream order."""

    def __init__(self, nbytes: int, device=None):
        self.tensor = torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device or "cuda")

    @property
    def nbytes(self) -> int:
        return self.tensor.numel()

    def ptr(self):
        return ctypes.c_void_p(self.tensor.data_ptr())


_WS_CACHE: dict = {}


def _workspace(kind: str, nbytes: int, device: torch.device) -> Workspace:
    key = (kind, device.index)
    ws = _WS_CACHE.get(key)
    if ws is None or ws.nbytes < nbytes:
        ws = Workspace(nbytes, device)
        _WS_CACHE[key] = ws
    return ws


def workspace_check(ws: Workspace, stream=None) -> None:
    """Synchronise and raise WKVError if a bounded device wait expired."""
    _check(_lib.wkv_workspace_check(ws.ptr(), _stream(stream)), "wkv_workspace_check")


def sync_status(stream=None) -> None:
    """Synchronise ``stream`` and raise WKVError if any call of the library
    on the current device gave up a bounded device wait since the last
    check (device-wide; the record is cleared)."""
    _check(_lib.wkv_sync_status(_stream(stream)), "wkv_sync_status")


# ---------------------------------------------------------------- forward
def forward(w, u, k, v, *, y=None, ckpt=None, want_ckpt: bool = False, workspace: Workspace | None = None,
            stream=None):
    """wkv for all t of k, v [B, T, C] (fp32 or bf16); w, u [C] fp32.

    Returns ``y`` (fp32 [B, T, C]), or ``(y, ckpt)`` when ``want_ckpt`` or a
    ``ckpt`` buffer is given (the chunk-boundary states for ``backward``).
    """
    if k.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("k must be float32 or bfloat16")
    B, T, C = k.shape
    _need(k, "k", (k.dtype,))
    _need(v, "v", (k.dtype,), k.shape)
    _need(w, "w", shape=(C,))
    _need(u, "u", shape=(C,))
    if y is None:
        y = torch.empty((B, T, C), dtype=torch.float32, device=k.device)
    _need(y, "y", shape=(B, T, C))
    if ckpt is None and want_ckpt:
        ckpt = torch.empty(checkpoint_floats(B, T, C), dtype=torch.float32, device=k.device)
    if ckpt is not None:
        _need(ckpt, "ckpt")
        if ckpt.numel() < checkpoint_floats(B, T, C):
            raise ValueError("ckpt is too small")
    need = forward_workspace_bytes(B, T, C)
    ws = workspace or _workspace("fwd", need, k.device)
    dt = WKV_BF16 if k.dtype == torch.bfloat16 else WKV_F32
    _check(_lib.wkv_forward(B, T, C, dt, _p(w), _p(u), _p(k), _p(v), _p(y), _p(ckpt), ws.ptr(), ws.nbytes,
                            _stream(stream)), "wkv_forward")
    return (y, ckpt) if ckpt is not None else y


def forward_with_state(w, u, k, v, state_in=None, *, y=None, state_out=None, ckpt=None, want_ckpt: bool = False,
                       want_y: bool = True, workspace: Workspace | None = None, stream=None):
    """wkv over k, v [B, T, C] continuing from ``state_in`` (fp32 [3, B, C]:
    the planes num, den, pp; None: the empty state).  Returns
    ``(y, state_out)``, or ``(y, state_out, ckpt)`` when ``want_ckpt`` or a
    ``ckpt`` buffer is given; ``state_out`` is [3, B, C] (the state after the
    last token, in the decode step's convention).  ``want_y=False`` (and no
    ``y``): a state-only pass, y is None."""
    if k.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("k must be float32 or bfloat16")
    B, T, C = k.shape
    _need(k, "k", (k.dtype,))
    _need(v, "v", (k.dtype,), k.shape)
    _need(w, "w", shape=(C,))
    _need(u, "u", shape=(C,))
    if state_in is not None:
        _need(state_in, "state_in", shape=(3, B, C))
    if y is None and want_y:
        y = torch.empty((B, T, C), dtype=torch.float32, device=k.device)
    if y is not None:
        _need(y, "y", shape=(B, T, C))
    if state_out is None:
        state_out = torch.empty((3, B, C), dtype=torch.float32, device=k.device)
    _need(state_out, "state_out", shape=(3, B, C))
    if ckpt is None and want_ckpt:
        ckpt = torch.empty(checkpoint_floats(B, T, C), dtype=torch.float32, device=k.device)
    if ckpt is not None:
        _need(ckpt, "ckpt")
        if ckpt.numel() < checkpoint_floats(B, T, C):
            raise ValueError("ckpt is too small")
    ws = workspace or _workspace("fwd", forward_workspace_bytes(B, T, C), k.device)
    dt = WKV_BF16 if k.dtype == torch.bfloat16 else WKV_F32
    _check(_lib.wkv_forward_with_state(B, T, C, dt, _p(w), _p(u), _p(k), _p(v), _p(state_in), _p(y), _p(state_out),
                                       _p(ckpt), ws.ptr(), ws.nbytes, _stream(stream)), "wkv_forward_with_state")
    return (y, state_out, ckpt) if ckpt is not None else (y, state_out)


def forward_gated(w, u, k, v, r, state_in=None, *, out=None, state_out=None, ckpt=None, want_ckpt: bool = False,
                  workspace: Workspace | None = None, stream=None):
    """sigmoid(r) * wkv for k, v, r [B, T, C] (all fp32 or all bf16); w, u [C]
    fp32.  Returns ``out`` (fp32 [B, T, C]), or ``(out, ckpt)`` when
    ``want_ckpt`` or a ``ckpt`` buffer is given.  ``state_in`` / ``state_out``
    ([3, B, C] fp32, optional) as for ``forward_with_state``."""
    if k.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("k must be float32 or bfloat16")
    B, T, C = k.shape
    _need(k, "k", (k.dtype,))
    _need(v, "v", (k.dtype,), k.shape)
    _need(r, "r", (k.dtype,), k.shape)
    _need(w, "w", shape=(C,))
    _need(u, "u", shape=(C,))
    if state_in is not None:
        _need(state_in, "state_in", shape=(3, B, C))
    if state_out is not None:
        _need(state_out, "state_out", shape=(3, B, C))
    if out is None:
        out = torch.empty((B, T, C), dtype=torch.float32, device=k.device)
    _need(out, "out", shape=(B, T, C))
    if ckpt is None and want_ckpt:
        ckpt = torch.empty(checkpoint_floats(B, T, C), dtype=torch.float32, device=k.device)
    if ckpt is not None:
        _need(ckpt, "ckpt")
        if ckpt.numel() < checkpoint_floats(B, T, C):
            raise ValueError("ckpt is too small")
    ws = workspace or _workspace("fwd", forward_workspace_bytes(B, T, C), k.device)
    dt = WKV_BF16 if k.dtype == torch.bfloat16 else WKV_F32
    _check(_lib.wkv_forward_gated(B, T, C, dt, _p(w), _p(u), _p(k), _p(v), _p(r), _p(state_in), _p(out),
                                  _p(state_out), _p(ckpt), ws.ptr(), ws.nbytes, _stream(stream)), "wkv_forward_gated")
    return (out, ckpt) if ckpt is not None else out


def state_fold(w, states, lengths, *, out=None, stream=None):
    """The state [3, B, C] after consecutive segments: ``states`` fp32
    [n, 3, B, C] (each segment's own state, from the empty state; n may be
    0 with any leading size), ``lengths`` the n segments' token counts."""
    C = w.shape[0]
    _need(w, "w", shape=(C,))
    _need(states, "states")
    if states.dim() != 4 or states.shape[1] != 3 or states.shape[3] != C:
        raise ValueError("states must be [n, 3, B, C]")
    n, B = states.shape[0], states.shape[2]
    lengths = [int(x) for x in lengths]
    if len(lengths) != n:
        raise ValueError("one length per segment")
    out = torch.empty((3, B, C), dtype=torch.float32, device=w.device) if out is None else out
    _need(out, "out", shape=(3, B, C))
    lens = (ctypes.c_longlong * max(n, 1))(*lengths)
    _check(_lib.wkv_state_fold(B, C, _p(w), n, _p(states) if n else None, lens, _p(out), _stream(stream)),
           "wkv_state_fold")
    return out


def adjoint_fold(w, adj, lengths, gstate_end=None, *, out=None, stream=None):
    """The start-state gradient [3, B, C] = (g_num, g_den, pp) of the first
    of n consecutive segments: ``adj`` fp32 [n, 3, B, C] is each segment's
    own start-state gradient (its summary pass with no end gradient),
    ``lengths`` their token counts, ``gstate_end`` [3, B, C] the gradient on
    the last segment's end state (None: none; required when n = 0)."""
    C = w.shape[0]
    _need(w, "w", shape=(C,))
    _need(adj, "adj")
    if adj.dim() != 4 or adj.shape[1] != 3 or adj.shape[3] != C:
        raise ValueError("adj must be [n, 3, B, C]")
    n, B = adj.shape[0], adj.shape[2]
    lengths = [int(x) for x in lengths]
    if len(lengths) != n:
        raise ValueError("one length per segment")
    if gstate_end is not None:
        _need(gstate_end, "gstate_end", shape=(3, B, C))
    out = torch.empty((3, B, C), dtype=torch.float32, device=w.device) if out is None else out
    _need(out, "out", shape=(3, B, C))
    lens = (ctypes.c_longlong * max(n, 1))(*lengths)
    _check(_lib.wkv_adjoint_fold(B, C, _p(w), n, _p(adj) if n else None, lens, _p(gstate_end), _p(out),
                                 _stream(stream)), "wkv_adjoint_fold")
    return out


def token_shift(x, x0, mu_k, mu_v, mu_r, *, xk=None, xv=None, xr=None, stream=None):
    """(xk, xv, xr) = mu x_t + (1 - mu) x_{t-1} for x [B, T, C] (fp32); x0
    [B, C] is the token before the sequence (None: zeros)."""
    B, T, C = x.shape
    _need(x, "x")
    if x0 is not None:
        _need(x0, "x0", shape=(B, C))
    for m, n in ((mu_k, "mu_k"), (mu_v, "mu_v"), (mu_r, "mu_r")):
        _need(m, n, shape=(C,))
    outs = []
    for t, n in ((xk, "xk"), (xv, "xv"), (xr, "xr")):
        t = torch.empty_like(x) if t is None else t
        _need(t, n, shape=(B, T, C))
        outs.append(t)
    _check(_lib.wkv_token_shift(B, T, C, _p(x), _p(x0), _p(mu_k), _p(mu_v), _p(mu_r), *map(_p, outs),
                                _stream(stream)), "wkv_token_shift")
    return tuple(outs)


def token_shift_backward(x, x0, mu_k, mu_v, mu_r, gxk, gxv, gxr, *, workspace: Workspace | None = None,
                         stream=None):
    """(gx, gx0, gmu_k, gmu_v, gmu_r) of token_shift; gx0 is None when x0 is."""
    B, T, C = x.shape
    _need(x, "x")
    if x0 is not None:
        _need(x0, "x0", shape=(B, C))
    for m, n in ((mu_k, "mu_k"), (mu_v, "mu_v"), (mu_r, "mu_r")):
        _need(m, n, shape=(C,))
    for g, n in ((gxk, "gxk"), (gxv, "gxv"), (gxr, "gxr")):
        _need(g, n, shape=(B, T, C))
    gx = torch.empty_like(x)
    gx0 = None if x0 is None else torch.empty_like(x0)
    gm = tuple(torch.empty(C, dtype=torch.float32, device=x.device) for _ in range(3))
    need = int(_lib.wkv_token_shift_backward_workspace_bytes(B, T, C))
    ws = workspace or _workspace("shift", need, x.device)
    _check(_lib.wkv_token_shift_backward(B, T, C, _p(x), _p(x0), _p(mu_k), _p(mu_v), _p(mu_r), _p(gxk), _p(gxv),
                                         _p(gxr), _p(gx), _p(gx0), *map(_p, gm), ws.ptr(), ws.nbytes,
                                         _stream(stream)), "wkv_token_shift_backward")
    return (gx, gx0) + gm


def forward_noalloc(w, u, k, v, *, y=None, ckpt=None, stream=None):
    """wkv_forward with the library's built-in scratch instead of a
    workspace, for callers that cannot allocate device memory (see
    wkv_forward_noalloc in include/wkv.h).  Shapes needing more than 32 MiB
    of scratch raise WKVError.  Returns ``y``, or ``(y, ckpt)`` when a
    ``ckpt`` buffer is given.  The call runs with the tensors' device
    current (the scratch array is chosen by the current device)."""
    if k.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("k must be float32 or bfloat16")
    B, T, C = k.shape
    _need(k, "k", (k.dtype,))
    _need(v, "v", (k.dtype,), k.shape)
    _need(w, "w", shape=(C,))
    _need(u, "u", shape=(C,))
    if y is None:
        y = torch.empty((B, T, C), dtype=torch.float32, device=k.device)
    _need(y, "y", shape=(B, T, C))
    if ckpt is not None:
        _need(ckpt, "ckpt")
        if ckpt.numel() < checkpoint_floats(B, T, C):
            raise ValueError("ckpt is too small")
    for name, t in (("v", v), ("w", w), ("u", u), ("y", y), ("ckpt", ckpt)):
        if t is not None and t.device != k.device:
            raise ValueError(f"{name} is on {t.device}, k on {k.device}")
    dt = WKV_BF16 if k.dtype == torch.bfloat16 else WKV_F32
    with torch.cuda.device(k.device):
        _check(_lib.wkv_forward_noalloc(B, T, C, dt, _p(w), _p(u), _p(k), _p(v), _p(y), _p(ckpt),
                                        _stream(stream)), "wkv_forward_noalloc")
    return (y, ckpt) if ckpt is not None else y


# --------------------------------------------------------------- backward
def backward(w, u, k, v, gy, *, ckpt=None, gw=None, gu=None, gk=None, gv=None, workspace: Workspace | None = None,
             stream=None):
    """Gradients (gw, gu, gk, gv) of sum(gy * wkv); k, v, gy all fp32 or all
    bf16 (fp32 arithmetic and fp32 gradients either way)."""
    if k.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("k must be float32 or bfloat16")
    B, T, C = k.shape
    _need(k, "k", (k.dtype,))
    _need(v, "v", (k.dtype,), k.shape)
    _need(gy, "gy", (k.dtype,), k.shape)
    _need(w, "w", shape=(C,))
    _need(u, "u", shape=(C,))
    if ckpt is not None:
        _need(ckpt, "ckpt")
        if ckpt.numel() < checkpoint_floats(B, T, C):
            raise ValueError("ckpt is too small")
    dev = k.device
    gw = torch.empty(C, dtype=torch.float32, device=dev) if gw is None else gw
    gu = torch.empty(C, dtype=torch.float32, device=dev) if gu is None else gu
    gk = torch.empty((B, T, C), dtype=torch.float32, device=dev) if gk is None else gk
    gv = torch.empty((B, T, C), dtype=torch.float32, device=dev) if gv is None else gv
    for t, n, s in ((gw, "gw", (C,)), (gu, "gu", (C,)), (gk, "gk", (B, T, C)), (gv, "gv", (B, T, C))):
        _need(t, n, shape=s)
    need = backward_workspace_bytes(B, T, C)
    ws = workspace or _workspace("bwd", need, dev)
    dt = WKV_BF16 if k.dtype == torch.bfloat16 else WKV_F32
    _check(_lib.wkv_backward(B, T, C, dt, _p(w), _p(u), _p(k), _p(v), _p(gy), _p(ckpt), _p(gw), _p(gu),
                             _p(gk), _p(gv), ws.ptr(), ws.nbytes, _stream(stream)), "wkv_backward")
    return gw, gu, gk, gv


def backward_with_state(w, u, k, v, gy, state_in=None, gstate_end=None, *, ckpt=None, gw=None, gu=None, gk=None,
                        gv=None, gstate_in=None, want_gstate_in: bool = True, summary: bool = False,
                        workspace: Workspace | None = None, stream=None):
    """``backward`` for a forward pass that started from ``state_in`` ([3, B,
    C] or None) and whose end state feeds later tokens: ``gstate_end`` [3, B,
    C] = (g_num, g_den, pp), the gradient with respect to the end state's
    num, den written at scale pp (None: none).  Returns (gw, gu, gk, gv,
    gstate_in), the last [3, B, C] = (g_num, g_den, pp) for state_in (None
    when not wanted).  ``summary``: the summary pass, which computes
    gstate_in alone (gw, gu, gk, gv are None)."""
    if k.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("k must be float32 or bfloat16")
    B, T, C = k.shape
    _need(k, "k", (k.dtype,))
    _need(v, "v", (k.dtype,), k.shape)
    _need(gy, "gy", (k.dtype,), k.shape)
    _need(w, "w", shape=(C,))
    _need(u, "u", shape=(C,))
    for t, n in ((state_in, "state_in"), (gstate_end, "gstate_end")):
        if t is not None:
            _need(t, n, shape=(3, B, C))
    if ckpt is not None:
        _need(ckpt, "ckpt")
        if ckpt.numel() < checkpoint_floats(B, T, C):
            raise ValueError("ckpt is too small")
    dev = k.device
    if summary:
        gw = gu = gk = gv = None
        want_gstate_in = True
    else:
        gw = torch.empty(C, dtype=torch.float32, device=dev) if gw is None else gw
        gu = torch.empty(C, dtype=torch.float32, device=dev) if gu is None else gu
        gk = torch.empty((B, T, C), dtype=torch.float32, device=dev) if gk is None else gk
        gv = torch.empty((B, T, C), dtype=torch.float32, device=dev) if gv is None else gv
        for t, n, s in ((gw, "gw", (C,)), (gu, "gu", (C,)), (gk, "gk", (B, T, C)), (gv, "gv", (B, T, C))):
            _need(t, n, shape=s)
    if gstate_in is None and want_gstate_in:
        gstate_in = torch.empty((3, B, C), dtype=torch.float32, device=dev)
    if gstate_in is not None:
        _need(gstate_in, "gstate_in", shape=(3, B, C))
    ws = workspace or _workspace("bwd", backward_workspace_bytes(B, T, C), dev)
    dt = WKV_BF16 if k.dtype == torch.bfloat16 else WKV_F32
    _check(_lib.wkv_backward_with_state(B, T, C, dt, _p(w), _p(u), _p(k), _p(v), _p(gy), _p(state_in),
                                        _p(gstate_end), _p(ckpt), _p(gw), _p(gu), _p(gk), _p(gv), _p(gstate_in),
                                        ws.ptr(), ws.nbytes, _stream(stream)), "wkv_backward_with_state")
    return gw, gu, gk, gv, gstate_in


def backward_gated(w, u, k, v, r, gout, *, ckpt=None, gw=None, gu=None, gk=None, gv=None, gr=None,
                   workspace: Workspace | None = None, stream=None):
    """Gradients (gw, gu, gk, gv, gr) of sum(gout * sigmoid(r) * wkv); k, v,
    r, gout all fp32 or all bf16 (fp32 arithmetic and gradients)."""
    if k.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("k must be float32 or bfloat16")
    B, T, C = k.shape
    for t, n in ((k, "k"), (v, "v"), (r, "r"), (gout, "gout")):
        _need(t, n, (k.dtype,), k.shape)
    _need(w, "w", shape=(C,))
    _need(u, "u", shape=(C,))
    if ckpt is not None:
        _need(ckpt, "ckpt")
        if ckpt.numel() < checkpoint_floats(B, T, C):
            raise ValueError("ckpt is too small")
    dev = k.device
    gw = torch.empty(C, dtype=torch.float32, device=dev) if gw is None else gw
    gu = torch.empty(C, dtype=torch.float32, device=dev) if gu is None else gu
    gk, gv, gr = (torch.empty((B, T, C), dtype=torch.float32, device=dev) if t is None else t for t in (gk, gv, gr))
    for t, n, s in ((gw, "gw", (C,)), (gu, "gu", (C,)), (gk, "gk", (B, T, C)), (gv, "gv", (B, T, C)),
                    (gr, "gr", (B, T, C))):
        _need(t, n, shape=s)
    ws = workspace or _workspace("bwd", backward_workspace_bytes(B, T, C), dev)
    dt = WKV_BF16 if k.dtype == torch.bfloat16 else WKV_F32
    _check(_lib.wkv_backward_gated(B, T, C, dt, _p(w), _p(u), _p(k), _p(v), _p(r), _p(gout), _p(ckpt), _p(gw),
                                   _p(gu), _p(gk), _p(gv), _p(gr), ws.ptr(), ws.nbytes, _stream(stream)),
           "wkv_backward_gated")
    return gw, gu, gk, gv, gr


# --------------------------------------------------------- channel mixing
def _same(name, t, like):
    _need(t, name, shape=tuple(like.shape))
    if t.device != like.device:
        raise ValueError(f"{name} must be on {like.device}")


def channel_mix_sqrelu(k, *, out=None, stream=None):
    """max(k, 0)^2 of an fp32 tensor of any shape (``out`` may be ``k``)."""
    _need(k, "k")
    out = torch.empty_like(k) if out is None else out
    _same("out", out, k)
    _check(_lib.wkv_channel_mix_sqrelu(k.numel(), _p(k), _p(out), _stream(stream)), "wkv_channel_mix_sqrelu")
    return out


def channel_mix_sqrelu_backward(k, ga, *, gk=None, stream=None):
    """gk = 2 max(k, 0) ga."""
    _need(k, "k")
    _same("ga", ga, k)
    gk = torch.empty_like(k) if gk is None else gk
    _same("gk", gk, k)
    _check(_lib.wkv_channel_mix_sqrelu_backward(k.numel(), _p(k), _p(ga), _p(gk), _stream(stream)),
           "wkv_channel_mix_sqrelu_backward")
    return gk


def channel_mix_gate(r, vk, *, out=None, stream=None):
    """sigmoid(r) * vk, fp32 tensors of one shape."""
    _need(r, "r")
    _same("vk", vk, r)
    out = torch.empty_like(r) if out is None else out
    _same("out", out, r)
    _check(_lib.wkv_channel_mix_gate(r.numel(), _p(r), _p(vk), _p(out), _stream(stream)), "wkv_channel_mix_gate")
    return out


def channel_mix_gate_backward(r, vk, gout, *, gr=None, gvk=None, stream=None):
    """(gr, gvk) of sum(gout * sigmoid(r) * vk)."""
    _need(r, "r")
    _same("vk", vk, r)
    _same("gout", gout, r)
    gr = torch.empty_like(r) if gr is None else gr
    gvk = torch.empty_like(r) if gvk is None else gvk
    _same("gr", gr, r)
    _same("gvk", gvk, r)
    _check(_lib.wkv_channel_mix_gate_backward(r.numel(), _p(r), _p(vk), _p(gout), _p(gr), _p(gvk), _stream(stream)),
           "wkv_channel_mix_gate_backward")
    return gr, gvk


# ----------------------------------------------------------------- decode
def decode_step(x, x_prev, mu_k, mu_v, mu_r, r, k, v, w, u, num, den, pp, *, y=None, xk=None, xv=None, xr=None,
                mix: bool = True, stream=None):
    """One fused RNN-mode step of L layers; num, den, pp [L, B, C] update in place.

    The token inputs x, x_prev, r, k, v are all fp32 or all bf16
    (wkv_decode_step_bf16); parameters, state and outputs are fp32.
    Returns (y, xk, xv, xr); the mix outputs are None when ``mix`` is False
    and no buffers are passed.
    """
    if x.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("x must be float32 or bfloat16")
    L, B, C = x.shape
    for t, n in ((x, "x"), (x_prev, "x_prev"), (r, "r"), (k, "k"), (v, "v")):
        _need(t, n, (x.dtype,), shape=(L, B, C))
    for t, n in ((num, "num"), (den, "den"), (pp, "pp")):
        _need(t, n, shape=(L, B, C))
    for t, n in ((mu_k, "mu_k"), (mu_v, "mu_v"), (mu_r, "mu_r"), (w, "w"), (u, "u")):
        _need(t, n, shape=(L, C))
    out = dict(dtype=torch.float32, device=x.device)
    if y is None:
        y = torch.empty((L, B, C), **out)
    if mix:
        xk = torch.empty((L, B, C), **out) if xk is None else xk
        xv = torch.empty((L, B, C), **out) if xv is None else xv
        xr = torch.empty((L, B, C), **out) if xr is None else xr
    for t, n in ((y, "y"), (xk, "xk"), (xv, "xv"), (xr, "xr")):
        if t is not None:
            _need(t, n, shape=(L, B, C))
    fn, name = ((_lib.wkv_decode_step_bf16, "wkv_decode_step_bf16") if x.dtype == torch.bfloat16 else
                (_lib.wkv_decode_step, "wkv_decode_step"))
    _check(fn(L, B, C, *map(_p, (x, x_prev, mu_k, mu_v, mu_r, r, k, v, w, u, num, den, pp, y, xk, xv, xr)),
              _stream(stream)), name)
    return y, xk, xv, xr


# ------------------------------------------------------------- test hooks
def set_wait_budget_ns(ns: int) -> None:
    _check(_lib.wkv_debug_set_wait_budget_ns(int(ns)), "wkv_debug_set_wait_budget_ns")


def set_skip_chunk(chunk: int) -> None:
    _check(_lib.wkv_debug_set_skip_chunk(int(chunk)), "wkv_debug_set_skip_chunk")


SCAN_MODES = {"auto": 0, "chunked": 1, "sequential": 2}


def scan_strategy(B: int, T: int, C: int) -> str:
    """"chunked" or "sequential": the kernels forward/backward run for a
    [B, T, C] call on the current device (under the current scan mode)."""
    r = int(_lib.wkv_scan_strategy(B, T, C))
    if r < 0:
        raise WKVError(1, "wkv_scan_strategy")  # WKV_ERR_INVALID_ARG
    return {1: "chunked", 2: "sequential"}[r]


def set_max_runs(runs: int) -> None:
    """Upper bound on the runs per column of the sequential kernels (0: the
    library's choice); process-wide, for tests and measurements."""
    _check(_lib.wkv_debug_set_max_runs(int(runs)), "wkv_debug_set_max_runs")


def set_chain_len(chunks: int) -> None:
    """> 0: the sequential forward walks chained runs of that many chunks;
    0: the library's choice (process-wide, for tests and measurements)."""
    _check(_lib.wkv_debug_set_chain_len(int(chunks)), "wkv_debug_set_chain_len")


def set_scan_mode(mode: str) -> None:
    """Which kernels forward/backward run: "auto" (by shape), "chunked" or
    "sequential" (process-wide, for tests and measurements)."""
    _check(_lib.wkv_debug_set_scan_mode(SCAN_MODES[mode]), "wkv_debug_set_scan_mode")


# -------------------------------------------------------------- autograd
class WKVFunction(torch.autograd.Function):
    """torch.autograd wrapper: forward saves the chunk checkpoints so the
    backward call skips its own pass over k and v."""

    @staticmethod
    def forward(ctx, w, u, k, v):
        y, ckpt = forward(w, u, k, v, want_ckpt=True)
        ctx.save_for_backward(w, u, k, v, ckpt)
        return y

    @staticmethod
    def backward(ctx, gy):
        w, u, k, v, ckpt = ctx.saved_tensors
        gw, gu, gk, gv = backward(w, u, k, v, gy.contiguous(), ckpt=ckpt)
        return gw, gu, gk, gv


def wkv(w, u, k, v):
    """Differentiable WKV (fp32 k, v for the backward)."""
    return WKVFunction.apply(w, u, k, v)


class GatedWKVFunction(torch.autograd.Function):
    """torch.autograd wrapper of the gated output sigmoid(r) * wkv."""

    @staticmethod
    def forward(ctx, w, u, k, v, r):
        out, ckpt = forward_gated(w, u, k, v, r, want_ckpt=True)
        ctx.save_for_backward(w, u, k, v, r, ckpt)
        return out

    @staticmethod
    def backward(ctx, gout):
        w, u, k, v, r, ckpt = ctx.saved_tensors
        return backward_gated(w, u, k, v, r, gout.contiguous(), ckpt=ckpt)


def wkv_gated(w, u, k, v, r):
    """Differentiable sigmoid(r) * wkv (fp32 k, v, r for the backward)."""
    return GatedWKVFunction.apply(w, u, k, v, r)
