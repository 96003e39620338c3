"""GPU parity of the training-path token shift (wkv_token_shift and its
backward) through the C ABI, against the float64 oracle (pinned by
tests/oracle_pins.py::pin_token_shift)."""
import pytest
import torch

import fp32_emulation as emu
from parity import TOL_GRAD, TOL_Y, assert_close, cuda


def _close(got, want, em, tol, what):
    assert_close(got, want, tol, what, emu=em)
from rwkv_linear_attention_backward_b300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def wkv():
    from rwkv_linear_attention_backward_b300 import binding

    return binding


# C % 4 == 0 with aligned tensors takes the vectorised path; the others the
# scalar one
SHAPES = [(1, 1, 4), (2, 33, 128), (3, 200, 96), (1, 1000, 2048), (2, 77, 7), (4, 129, 130)]


@pytest.mark.parametrize("with_x0", [True, False])
@pytest.mark.parametrize("B,T,C", SHAPES, ids=[f"B{b}T{t}C{c}" for b, t, c in SHAPES])
def test_token_shift(oracle, wkv, B, T, C, with_x0):
    x, x0, mk, mv, mr, gk, gv, gr = inputs.shift_inputs(B, T, C, seed=500 + B + T + C)
    if not with_x0:
        x0 = None
    d = cuda(x, mk, mv, mr, gk, gv, gr)
    dx0 = None if x0 is None else cuda(x0)[0]
    xk, xv, xr = wkv.token_shift(d[0], dx0, d[1], d[2], d[3])
    gx, gx0, gmk, gmv, gmr = wkv.token_shift_backward(d[0], dx0, d[1], d[2], d[3], d[4], d[5], d[6])
    torch.cuda.synchronize()
    ok, ov, orr = oracle.token_shift(x, x0, mk, mv, mr)
    ek, ev, er = emu.token_shift(x, x0, mk, mv, mr)
    _close(xk, ok, ek, TOL_Y, "xk")
    _close(xv, ov, ev, TOL_Y, "xv")
    _close(xr, orr, er, TOL_Y, "xr")
    ogx, ogx0, ogk, ogv, ogr = oracle.token_shift_backward(x, x0, mk, mv, mr, gk, gv, gr)
    egx, egx0, egk, egv, egr = emu.token_shift_backward(x, x0, mk, mv, mr, gk, gv, gr)
    _close(gx, ogx, egx, TOL_GRAD, "gx")
    _close(gmk, ogk, egk, TOL_GRAD, "gmu_k")
    _close(gmv, ogv, egv, TOL_GRAD, "gmu_v")
    _close(gmr, ogr, egr, TOL_GRAD, "gmu_r")
    if with_x0:
        _close(gx0, ogx0, egx0, TOL_GRAD, "gx0")
    else:
        assert gx0 is None


def test_token_shift_unaligned_matches_aligned(oracle, wkv):
    """Tensors that start off a 16-byte boundary take the scalar path and
    give the vectorised path's results bit for bit (the same fmaf per
    element; the mu sums, per slice and in order, may group differently)."""
    B, T, C = 2, 300, 256
    host = inputs.shift_inputs(B, T, C, seed=520)
    x, x0, mk, mv, mr, gk, gv, gr = cuda(*host)
    a = wkv.token_shift(x, x0, mk, mv, mr)
    xs = torch.empty(x.numel() + 1, device="cuda")[1:].view(B, T, C)  # 4 bytes off alignment
    xs.copy_(x)
    b = wkv.token_shift(xs, x0, mk, mv, mr)
    torch.cuda.synchronize()
    for p, q, n in zip(a, b, ("xk", "xv", "xr")):
        assert torch.equal(p, q), n
    ga = wkv.token_shift_backward(x, x0, mk, mv, mr, gk, gv, gr)
    gb = wkv.token_shift_backward(xs, x0, mk, mv, mr, gk, gv, gr)
    torch.cuda.synchronize()
    assert torch.equal(ga[0], gb[0]) and torch.equal(ga[1], gb[1])
    og = oracle.token_shift_backward(*host)[2:]
    eg = emu.token_shift_backward(*host)[2:]
    for p, q, o, e, n in zip(ga[2:], gb[2:], og, eg, ("gmu_k", "gmu_v", "gmu_r")):
        assert_close(q, p, TOL_GRAD, n, emu=e, ref=o, pair=True)


def test_token_shift_backward_reproducible(wkv):
    x, x0, mk, mv, mr, gk, gv, gr = cuda(*inputs.shift_inputs(3, 700, 512, seed=530))
    a = wkv.token_shift_backward(x, x0, mk, mv, mr, gk, gv, gr)
    for _ in range(3):
        b = wkv.token_shift_backward(x, x0, mk, mv, mr, gk, gv, gr)
        for p, q in zip(a, b):
            assert torch.equal(p, q)


def test_token_shift_workload_sampled(oracle, wkv):
    """The shift workload (B=16, T=4096, C=2048) at full size, checked on
    sampled channels (channels are independent)."""
    from parity import sample_channels

    S = inputs.SHIFT
    host = inputs.shift_inputs(S.B, S.T, S.C, seed=S.seed)
    x, x0, mk, mv, mr, gk, gv, gr = cuda(*host)
    xk, xv, xr = wkv.token_shift(x, x0, mk, mv, mr)
    gx, gx0, gmk, gmv, gmr = wkv.token_shift_backward(x, x0, mk, mv, mr, gk, gv, gr)
    torch.cuda.synchronize()
    cs = sample_channels(S.C, 32, 14)
    cst = torch.as_tensor(cs, device="cuda")
    hx, hx0, hmk, hmv, hmr, hgk, hgv, hgr = host
    sl = lambda t: t[:, :, cs].contiguous()  # noqa: E731
    fwd_in = (sl(hx), hx0[:, cs].contiguous(), hmk[cs], hmv[cs], hmr[cs])
    ok, ov, orr = oracle.token_shift(*fwd_in)
    ek, ev, er = emu.token_shift(*fwd_in)
    _close(xk.index_select(2, cst), ok, ek, TOL_Y, "xk")
    _close(xr.index_select(2, cst), orr, er, TOL_Y, "xr")
    bwd_in = fwd_in + (sl(hgk), sl(hgv), sl(hgr))
    ogx, ogx0, ogk, ogv, ogr = oracle.token_shift_backward(*bwd_in)
    egx, egx0, egk, egv, egr = emu.token_shift_backward(*bwd_in)
    _close(gx.index_select(2, cst), ogx, egx, TOL_GRAD, "gx")
    _close(gmk.index_select(0, cst), ogk, egk, TOL_GRAD, "gmu_k")
    _close(gmr.index_select(0, cst), ogr, egr, TOL_GRAD, "gmu_r")
