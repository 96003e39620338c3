"""Host-side checks of the C ABI (no GPU): the library loads, exports every
function include/wkv.h declares, sizes its buffers as documented, and
rejects invalid arguments before launching anything."""
import ctypes
import re
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]
HEADER = ROOT / "include" / "wkv.h"


@pytest.fixture(scope="module")
def lib():
    from rwkv_linear_attention_backward_b300 import build

    path = build.build()
    lib = ctypes.CDLL(str(path))
    lib.wkv_status_string.restype = ctypes.c_char_p
    lib.wkv_last_error_string.restype = ctypes.c_char_p
    for n in ("wkv_checkpoint_floats", "wkv_forward_workspace_bytes", "wkv_backward_workspace_bytes",
              "wkv_token_shift_backward_workspace_bytes"):
        getattr(lib, n).restype = ctypes.c_size_t
    return lib


def declared_functions():
    text = re.sub(r"/\*.*?\*/", "", HEADER.read_text(), flags=re.S)
    return sorted(set(re.findall(r"\b(wkv_[a-z0-9_]+)\s*\(", text)))


# The boundary's calls: the forward and backward passes, the decode step, the
# workspace size queries, the status text and the expired-wait report; plus
# what this library adds around them.
BOUNDARY = ("wkv_status_string", "wkv_forward_workspace_bytes", "wkv_backward_workspace_bytes", "wkv_forward",
            "wkv_backward", "wkv_decode_step", "wkv_last_error_string", "wkv_sync_status")
ADDED = ("wkv_checkpoint_floats", "wkv_workspace_init", "wkv_workspace_check", "wkv_forward_with_state",
         "wkv_backward_with_state", "wkv_forward_gated", "wkv_backward_gated", "wkv_state_fold", "wkv_adjoint_fold",
         "wkv_decode_step_bf16", "wkv_token_shift",
         "wkv_token_shift_backward", "wkv_channel_mix_sqrelu", "wkv_channel_mix_gate", "wkv_forward_noalloc")


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in BOUNDARY + ADDED:
        assert n in names, n


def test_sync_status_without_work(lib):
    """No launch has recorded anything: wkv_sync_status of the default
    stream is WKV_OK (where no device exists it reports the CUDA error)."""
    import torch

    st = lib.wkv_sync_status(None)
    assert st == (0 if torch.cuda.is_available() else 5)


def test_every_declared_symbol_is_exported(lib):
    for n in declared_functions():
        assert hasattr(lib, n), f"{n} declared in wkv.h but not exported"


def test_binding_names_match_header():
    src = (ROOT / "rwkv_linear_attention_backward_b300" / "binding.py").read_text()
    for n in declared_functions():
        assert f'"{n}"' in src, f"binding does not wrap {n}"


def test_version_and_chunk(lib):
    assert lib.wkv_version() == 1
    assert lib.wkv_chunk_len() == 32


@pytest.mark.parametrize("B,T,C", [(1, 1, 1), (1, 64, 64), (8, 1024, 768), (3, 33, 129), (1, 131072, 2560)])
def test_sizes(lib, B, T, C):
    L = lib.wkv_chunk_len()
    nch = -(-T // L)
    assert lib.wkv_checkpoint_floats(B, T, C) == 3 * nch * B * C
    f = lib.wkv_forward_workspace_bytes(B, T, C)
    b = lib.wkv_backward_workspace_bytes(B, T, C)
    # header + flags + two [3, nchunks, B, C] fp32 arrays at least
    assert f >= 256 + 2 * 3 * nch * B * C * 4
    # + adjoint tree nodes (>= 3 planes) + gw, gu partials (2 planes)
    assert b >= f + 256 + 5 * nch * B * C * 4
    assert f % 256 == 0 and b % 256 == 0


def test_invalid_sizes_give_zero(lib):
    for B, T, C in ((0, 1, 1), (1, 0, 1), (1, 1, 0), (-1, 5, 5), (1 << 20, 1 << 20, 2)):
        assert lib.wkv_forward_workspace_bytes(B, T, C) == 0
        assert lib.wkv_checkpoint_floats(B, T, C) == 0


def test_status_strings(lib):
    for code, name in enumerate(["WKV_OK", "WKV_ERR_INVALID_ARG", "WKV_ERR_UNSUPPORTED", "WKV_ERR_MISALIGNED",
                                 "WKV_ERR_WORKSPACE", "WKV_ERR_CUDA", "WKV_ERR_TIMEOUT"]):
        assert lib.wkv_status_string(code).decode() == name
    assert lib.wkv_status_string(99).decode() == "WKV_ERR_UNKNOWN"


FAKE = ctypes.c_void_p(0x1000)  # never dereferenced: every call below fails validation first
NULL = ctypes.c_void_p(0)


def _fwd(lib, B=2, T=40, C=64, dtype=0, w=FAKE, u=FAKE, k=FAKE, v=FAKE, y=FAKE, ws=FAKE, wsb=None):
    if wsb is None:
        wsb = lib.wkv_forward_workspace_bytes(max(B, 1), max(T, 1), max(C, 1))
    return lib.wkv_forward(B, T, C, dtype, w, u, k, v, y, NULL, ws, ctypes.c_size_t(wsb), NULL)


def test_forward_rejects_before_launch(lib):
    assert _fwd(lib, B=0) == 1
    assert _fwd(lib, T=-3) == 1
    assert _fwd(lib, dtype=7) == 1
    for name in ("w", "u", "k", "v", "y"):
        assert _fwd(lib, **{name: NULL}) == 1
    assert _fwd(lib, ws=NULL) == 4
    assert _fwd(lib, wsb=100) == 4


def _bwd(lib, B=2, T=40, C=64, dtype=0, ws=FAKE, wsb=None, **nulls):
    p = {n: FAKE for n in ("w", "u", "k", "v", "gy", "gw", "gu", "gk", "gv")}
    p.update(nulls)
    if wsb is None:
        wsb = lib.wkv_backward_workspace_bytes(max(B, 1), max(T, 1), max(C, 1))
    return lib.wkv_backward(B, T, C, dtype, p["w"], p["u"], p["k"], p["v"], p["gy"], NULL, p["gw"], p["gu"],
                            p["gk"], p["gv"], ws, ctypes.c_size_t(wsb), NULL)


def test_backward_rejects_before_launch(lib):
    assert _bwd(lib, C=0) == 1
    assert _bwd(lib, dtype=5) == 1
    # bf16 inputs while the chunked scan (fp32 only) is forced: refused before
    # any launch (a bf16 call in the default mode is valid and would launch,
    # which this host test never does)
    lib.wkv_debug_set_scan_mode(1)
    try:
        assert _bwd(lib, dtype=1) == 2
    finally:
        lib.wkv_debug_set_scan_mode(0)
    for name in ("w", "u", "k", "v", "gy", "gw", "gu", "gk", "gv"):
        assert _bwd(lib, **{name: NULL}) == 1
    assert _bwd(lib, wsb=256) == 4


def test_gated_rejects_before_launch(lib):
    B, T, C = 2, 40, 64
    wsf = ctypes.c_size_t(lib.wkv_forward_workspace_bytes(B, T, C))
    wsb = ctypes.c_size_t(lib.wkv_backward_workspace_bytes(B, T, C))

    def fwd(r=FAKE, out=FAKE, ws=wsf):
        return lib.wkv_forward_gated(B, T, C, 0, FAKE, FAKE, FAKE, FAKE, r, NULL, out, NULL, NULL, FAKE, ws, NULL)

    def bwd(r=FAKE, gout=FAKE, gr=FAKE, ws=wsb):
        return lib.wkv_backward_gated(B, T, C, 0, FAKE, FAKE, FAKE, FAKE, r, gout, NULL, FAKE, FAKE, FAKE, FAKE, gr,
                                      FAKE, ws, NULL)

    assert fwd(r=NULL) == 1 and fwd(out=NULL) == 1
    assert fwd(ws=ctypes.c_size_t(64)) == 4
    assert bwd(r=NULL) == 1 and bwd(gout=NULL) == 1 and bwd(gr=NULL) == 1
    assert bwd(ws=ctypes.c_size_t(64)) == 4
    # the gate is fused into the sequential kernels only: refused before any
    # launch while the chunked scan is forced
    lib.wkv_debug_set_scan_mode(1)
    try:
        assert fwd() == 2 and bwd() == 2
        assert b"sequential" in lib.wkv_last_error_string()
    finally:
        lib.wkv_debug_set_scan_mode(0)


def test_channel_mix_rejects_before_launch(lib):
    n = ctypes.c_longlong
    assert lib.wkv_channel_mix_sqrelu(n(-1), FAKE, FAKE, NULL) == 1
    assert lib.wkv_channel_mix_sqrelu(n(0), NULL, NULL, NULL) == 0  # nothing to do, nothing launched
    assert lib.wkv_channel_mix_sqrelu(n(8), NULL, FAKE, NULL) == 1
    assert lib.wkv_channel_mix_sqrelu(n(8), FAKE, NULL, NULL) == 1
    assert lib.wkv_channel_mix_sqrelu_backward(n(8), FAKE, NULL, FAKE, NULL) == 1
    assert lib.wkv_channel_mix_gate(n(8), FAKE, NULL, FAKE, NULL) == 1
    assert lib.wkv_channel_mix_gate(n(-5), FAKE, FAKE, FAKE, NULL) == 1
    args = [FAKE] * 5  # r, vk, gout, gr, gvk
    for i in range(5):
        a = list(args)
        a[i] = NULL
        assert lib.wkv_channel_mix_gate_backward(n(8), *a, NULL) == 1
    assert lib.wkv_channel_mix_gate_backward(n(0), *([NULL] * 5), NULL) == 0


def test_state_fold_and_state_only_pass_reject_before_launch(lib):
    lens = (ctypes.c_longlong * 3)(5, 0, 7)
    bad = (ctypes.c_longlong * 3)(5, -1, 7)
    fold = lib.wkv_state_fold
    assert fold(0, 4, FAKE, 3, FAKE, lens, FAKE, NULL) == 1
    assert fold(2, 4, NULL, 3, FAKE, lens, FAKE, NULL) == 1
    assert fold(2, 4, FAKE, 3, FAKE, lens, NULL, NULL) == 1
    assert fold(2, 4, FAKE, -1, FAKE, lens, FAKE, NULL) == 1
    assert fold(2, 4, FAKE, 257, FAKE, lens, FAKE, NULL) == 1
    assert fold(2, 4, FAKE, 3, NULL, lens, FAKE, NULL) == 1
    assert fold(2, 4, FAKE, 3, FAKE, NULL, FAKE, NULL) == 1
    assert fold(2, 4, FAKE, 3, FAKE, bad, FAKE, NULL) == 1
    # a pass with no y must return the state or the checkpoints
    wsb = ctypes.c_size_t(lib.wkv_forward_workspace_bytes(2, 40, 64))
    assert lib.wkv_forward_with_state(2, 40, 64, 0, FAKE, FAKE, FAKE, FAKE, NULL, NULL, NULL, NULL, FAKE, wsb,
                                      NULL) == 1


def test_backward_with_state_rejects_before_launch(lib):
    B, T, C = 2, 40, 64
    wsb = ctypes.c_size_t(lib.wkv_backward_workspace_bytes(B, T, C))

    def call(**nulls):
        p = {n: FAKE for n in ("w", "u", "k", "v", "gy", "gw", "gu", "gk", "gv")}
        p.update(nulls)
        return lib.wkv_backward_with_state(B, T, C, 0, p["w"], p["u"], p["k"], p["v"], p["gy"], FAKE, FAKE, NULL,
                                           p["gw"], p["gu"], p["gk"], p["gv"], FAKE, FAKE, wsb, NULL)

    for name in ("w", "u", "k", "v", "gy", "gw", "gu", "gk", "gv"):
        assert call(**{name: NULL}) == 1
    # carried states are taken by the sequential kernels only
    lib.wkv_debug_set_scan_mode(1)
    try:
        assert call() == 2
        assert b"sequential" in lib.wkv_last_error_string()
    finally:
        lib.wkv_debug_set_scan_mode(0)


def test_summary_pass_and_adjoint_fold_reject_before_launch(lib):
    B, T, C = 2, 40, 64
    wsb = ctypes.c_size_t(lib.wkv_backward_workspace_bytes(B, T, C))
    # a summary pass (gk, gv NULL) must return the start state's gradient
    assert lib.wkv_backward_with_state(B, T, C, 0, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, NULL, NULL, NULL, NULL,
                                       NULL, NULL, FAKE, wsb, NULL) == 1
    lens = (ctypes.c_longlong * 3)(5, 0, 7)
    bad = (ctypes.c_longlong * 3)(5, -1, 7)
    fold = lib.wkv_adjoint_fold
    assert fold(0, 4, FAKE, 3, FAKE, lens, FAKE, FAKE, NULL) == 1
    assert fold(2, 4, NULL, 3, FAKE, lens, FAKE, FAKE, NULL) == 1
    assert fold(2, 4, FAKE, 3, FAKE, lens, FAKE, NULL, NULL) == 1
    assert fold(2, 4, FAKE, -1, FAKE, lens, FAKE, FAKE, NULL) == 1
    assert fold(2, 4, FAKE, 257, FAKE, lens, FAKE, FAKE, NULL) == 1
    assert fold(2, 4, FAKE, 3, NULL, lens, FAKE, FAKE, NULL) == 1
    assert fold(2, 4, FAKE, 3, FAKE, NULL, FAKE, FAKE, NULL) == 1
    assert fold(2, 4, FAKE, 3, FAKE, bad, FAKE, FAKE, NULL) == 1
    assert fold(2, 4, FAKE, 0, NULL, lens, NULL, FAKE, NULL) == 1  # nothing to fold and no end gradient


def test_decode_rejects_before_launch(lib):
    args = [FAKE] * 17
    assert lib.wkv_decode_step(0, 1, 1, *args, NULL) == 1
    for i in range(14):  # the 14 required pointers; the mix outputs may be NULL
        a = list(args)
        a[i] = NULL
        assert lib.wkv_decode_step(2, 3, 4, *a, NULL) == 1


def test_token_shift_rejects_before_launch(lib):
    args = [FAKE] * 8  # x, x0, mu_k, mu_v, mu_r, xk, xv, xr
    assert lib.wkv_token_shift(0, 4, 4, *args, NULL) == 1
    assert lib.wkv_token_shift(2, 4, -1, *args, NULL) == 1
    for i in (0, 2, 3, 4, 5, 6, 7):  # every pointer but x0 is required
        a = list(args)
        a[i] = NULL
        assert lib.wkv_token_shift(2, 4, 4, *a, NULL) == 1
    bargs = [FAKE] * 13  # x, x0, mu_k, mu_v, mu_r, gxk, gxv, gxr, gx, gx0, gmu_k, gmu_v, gmu_r
    need = lib.wkv_token_shift_backward_workspace_bytes(2, 4, 4)
    assert need > 0 and lib.wkv_token_shift_backward_workspace_bytes(0, 4, 4) == 0
    for i in (0, 2, 3, 4, 5, 6, 7, 8, 10, 11, 12):  # x0 and gx0 may be NULL
        a = list(bargs)
        a[i] = NULL
        assert lib.wkv_token_shift_backward(2, 4, 4, *a, FAKE, ctypes.c_size_t(need), NULL) == 1
    assert lib.wkv_token_shift_backward(2, 4, 4, *bargs, NULL, ctypes.c_size_t(need), NULL) == 4
    assert lib.wkv_token_shift_backward(2, 4, 4, *bargs, FAKE, ctypes.c_size_t(need - 1), NULL) == 4
