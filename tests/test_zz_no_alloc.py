"""The allocation-free forward entry point (wkv_forward_noalloc) against the
regular one (wkv_forward with a caller workspace).

wkv_forward_noalloc serves callers that cannot call cudaMalloc, such as a
plugin host whose device memory belongs to another allocator, or a loop
that must never allocate; it takes its scratch from a fixed array inside
the library.  This file is collected last so that a run stopping at the
first failure has run every other test first, and it needs nothing from
earlier tests (it also passes alone in a fresh process)."""
import ctypes

import pytest
import torch

from parity import TOL_Y, assert_close
from rwkv_linear_attention_backward_b300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def wkv():
    from rwkv_linear_attention_backward_b300 import binding

    return binding


def _noalloc(wkv, w, u, k, v, y, ckpt):
    B, T, C = k.shape
    p = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return wkv._lib.wkv_forward_noalloc(B, T, C, 0, p(w), p(u), p(k), p(v), p(y), p(ckpt), stream)


@pytest.mark.parametrize("shape,seed", [((8, 1024, 768), 1002), ((3, 333, 130), 5)])
def test_noalloc_matches_workspace_forward(wkv, shape, seed):
    B, T, C = shape
    w, u, k, v, _ = (t.cuda() for t in inputs.training_inputs(B, T, C, seed=seed, k_std=3.0, d_lo=-6.0, d_hi=2.0))
    y_ref, ck_ref = wkv.forward(w, u, k, v, want_ckpt=True)
    torch.cuda.synchronize()
    for call in range(2):  # two calls in a row share (and reuse) the built-in scratch
        y = torch.full_like(y_ref, float("nan"))
        ck = torch.full_like(ck_ref, float("nan"))
        status = _noalloc(wkv, w, u, k, v, y, ck)
        assert status == 0, wkv._lib.wkv_last_error_string().decode()
        torch.cuda.synchronize()
        assert_close(y, y_ref, TOL_Y, f"noalloc call {call} y")
        assert_close(ck, ck_ref, TOL_Y, f"noalloc call {call} checkpoints")


def test_noalloc_rejects_shapes_beyond_its_scratch(wkv):
    t = torch.zeros(8, device="cuda")
    B, T, C = 16, 4096, 2048  # needs ~150 MB of scratch; checked before any launch
    assert wkv.forward_workspace_bytes(B, T, C) > 32 << 20
    p = ctypes.c_void_p(t.data_ptr())
    status = wkv._lib.wkv_forward_noalloc(B, T, C, 0, p, p, p, p, p, None, None)
    assert status == 4
    assert "holds" in wkv._lib.wkv_last_error_string().decode()
