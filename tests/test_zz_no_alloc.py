"""The allocation-free forward entry point (wkv_forward_noalloc) against the
regular one (wkv_forward with a caller workspace) and the float64 oracle.

wkv_forward_noalloc serves callers that cannot call cudaMalloc, such as a
plugin host whose device memory belongs to another allocator, or a loop
that must never allocate; it takes its scratch from a fixed array inside
the library.  This file is collected last so that a run stopping at the
first failure has run every other test first, and it needs nothing from
earlier tests (it also passes alone in a fresh process)."""
import ctypes

import numpy as np
import pytest
import torch

import fp32_emulation as emu
from checks import check_y
from parity import TOL_Y, assert_close, assert_state_close, to_np
from rwkv_linear_attention_backward_b300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def wkv():
    from rwkv_linear_attention_backward_b300 import binding

    return binding


def _noalloc(wkv, w, u, k, v, y, ckpt):
    """The entry point through the C ABI itself."""
    B, T, C = k.shape
    p = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    dt = 1 if k.dtype == torch.bfloat16 else 0
    return wkv._lib.wkv_forward_noalloc(B, T, C, dt, p(w), p(u), p(k), p(v), p(y), p(ckpt), stream)


CASES = [((8, 1024, 768), 1002, "f32"), ((3, 333, 130), 5, "f32"), ((2, 777, 136), 9, "bf16")]


@pytest.mark.parametrize("shape,seed,dt", CASES, ids=["l169m", "ragged", "bf16"])
def test_noalloc_matches_workspace_forward(oracle, wkv, scan_mode, shape, seed, dt):
    """Two calls in a row (sharing, and reusing, the built-in scratch) give
    wkv_forward's outputs and checkpoints, under every scan strategy (the
    chunked scan's tile counters live in the shared array too); the
    outputs also match the oracle."""
    B, T, C = shape
    host = inputs.training_inputs(B, T, C, seed=seed, k_std=3.0, d_lo=-6.0, d_hi=2.0, kv_dtype=dt)
    w, u, k, v = (t.cuda() for t in host[:4])
    if dt == "bf16" and scan_mode == "chunked":
        return  # the chunked scan takes fp32 inputs only
    y_ref, ck_ref = wkv.forward(w, u, k, v, want_ckpt=True)
    torch.cuda.synchronize()
    for call in range(2):
        y = torch.full_like(y_ref, float("nan"))
        ck = torch.full_like(ck_ref, float("nan"))
        status = _noalloc(wkv, w, u, k, v, y, ck)
        assert status == 0, wkv._lib.wkv_last_error_string().decode()
        torch.cuda.synchronize()
        assert_close(y, y_ref, TOL_Y, f"noalloc call {call} y")
        assert_close(ck, ck_ref, TOL_Y, f"noalloc call {call} checkpoints")
    check_y(oracle, *host[:4], y, f"noalloc {dt}")
    if B * T * C <= 1 << 20:  # the checkpoints against the oracle's states
        L = wkv.chunk_len()
        nch = -(-T // L)
        cks = to_np(ck).reshape(3, nch, B, C)
        for j in (0, nch // 2, nch - 1):
            t = min((j + 1) * L, T)
            ea, eb = emu.sums_after(host[0], host[2], host[3], [t])[0]
            assert_state_close(cks[0, j], cks[1, j], cks[2, j], *oracle.state(host[0], host[2], host[3], t), TOL_Y,
                               f"noalloc checkpoint {j}", emu_sums=(ea, eb))


def test_noalloc_binding(oracle, wkv):
    """The Python wrapper: the same outputs as the C ABI call, and its
    argument checks (a checkpoint buffer that is too small is refused before
    anything runs)."""
    B, T, C = 2, 300, 96
    host = inputs.training_inputs(B, T, C, seed=11, k_std=2.0)
    w, u, k, v = (t.cuda() for t in host[:4])
    ck = torch.empty(wkv.checkpoint_floats(B, T, C), device="cuda")
    y, ck_out = wkv.forward_noalloc(w, u, k, v, ckpt=ck)
    y_ref, ck_ref = wkv.forward(w, u, k, v, want_ckpt=True)
    torch.cuda.synchronize()
    assert ck_out is ck
    assert torch.equal(y, y_ref) and torch.equal(ck, ck_ref)
    check_y(oracle, *host[:4], y, "noalloc binding")
    with pytest.raises(ValueError, match="ckpt is too small"):
        wkv.forward_noalloc(w, u, k, v, ckpt=torch.empty(ck.numel() - 1, device="cuda"))
    with pytest.raises(TypeError):
        wkv.forward_noalloc(w, u, k, v, ckpt=torch.empty(ck.numel(), device="cuda", dtype=torch.float64))


def test_noalloc_rejects_shapes_beyond_its_scratch(wkv):
    t = torch.zeros(8, device="cuda")
    B, T, C = 16, 4096, 2048  # needs ~150 MB of scratch; checked before any launch
    assert wkv.forward_workspace_bytes(B, T, C) > 32 << 20
    p = ctypes.c_void_p(t.data_ptr())
    status = wkv._lib.wkv_forward_noalloc(B, T, C, 0, p, p, p, p, p, None, None)
    assert status == 4
    assert "holds" in wkv._lib.wkv_last_error_string().decode()
    # a rejected argument leaves its own message, not the previous call's
    status = wkv._lib.wkv_forward_noalloc(0, T, C, 0, p, p, p, p, p, None, None)
    assert status == 1
    assert "holds" not in wkv._lib.wkv_last_error_string().decode()
    assert np.isfinite(to_np(t)).all()
