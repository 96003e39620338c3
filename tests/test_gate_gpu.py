"""GPU parity of the gated time-mixing output sigmoid(r) * wkv and its
backward pass (the receptance gate, eq. (9) of "RWKV解读" section
"3、RWKV的网络架构", fused into the sequential kernels), through the C ABI,
against the float64 oracle (oracle.forward_gated / backward_gated, pinned by
tests/oracle_pins.py::pin_gate_special_values and
pin_gate_finite_differences).

Shapes span several chunks, ragged chunk and channel tails and T = 1; the
stress cases push lanes onto the per-token (running-maximum) path and the
gate into saturation; the l169m-sized workload runs at full size."""
import numpy as np
import pytest
import torch

import fp32_emulation as emu
from checks import check_pair_grads, grad_evaluations
from parity import TOL_BF16, TOL_GRAD, TOL_Y, assert_close, cuda, to_np
from rwkv_linear_attention_backward_b300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def wkv():
    from rwkv_linear_attention_backward_b300 import binding

    return binding


def _inputs(B, T, C, seed, kv_dtype="f32", k_std=2.0, r_std=2.0, **kw):
    w, u, k, v, gout = inputs.training_inputs(B, T, C, seed=seed, k_std=k_std, kv_dtype=kv_dtype, **kw)
    r = inputs.gate_inputs(B, T, C, seed=seed + 1, r_std=r_std, kv_dtype=kv_dtype)
    return w, u, k, v, r, gout


def _run(wkv, w, u, k, v, r, gout, use_ckpt=True):
    w, u, k, v, r, gout = cuda(w, u, k, v, r, gout)
    out, ckpt = wkv.forward_gated(w, u, k, v, r, want_ckpt=True)
    grads = wkv.backward_gated(w, u, k, v, r, gout, ckpt=ckpt if use_ckpt else None)
    torch.cuda.synchronize()
    return (out, ckpt) + grads


GATED = ("gw", "gu", "gk", "gv", "gr")


def _check_out(oracle, w, u, k, v, r, out, what, tol=TOL_Y):
    assert_close(out, oracle.forward_gated(w, u, k, v, r), tol, f"{what} out", emu=emu.forward_gated(w, u, k, v, r))


def _check_grads(oracle, w, u, k, v, r, gout, got, what):
    """``got``: the GPU's (gw, gu, gk, gv, gr)."""
    o = oracle.backward_gated(w, u, k, v, r, gout)
    e = grad_evaluations(emu.backward_gated, w, u, k, v, r, gout, names=GATED)
    for g, oo, n in zip(got, o, GATED):
        assert_close(g, oo, TOL_GRAD, f"{what} {n}", emu=e[n])


def _check(oracle, wkv, w, u, k, v, r, gout, what, tol_out=TOL_Y, use_ckpt=True):
    out, _, gw, gu, gk, gv, gr = _run(wkv, w, u, k, v, r, gout, use_ckpt)
    _check_out(oracle, w, u, k, v, r, out, what, tol_out)
    _check_grads(oracle, w, u, k, v, r, gout, (gw, gu, gk, gv, gr), what)


def _refused(wkv, w, u, k, v, r, gout):
    """The chunked scan has no gate: both calls refuse before launching."""
    w, u, k, v, r, gout = cuda(w, u, k, v, r, gout)
    for call in (lambda: wkv.forward_gated(w, u, k, v, r), lambda: wkv.backward_gated(w, u, k, v, r, gout)):
        with pytest.raises(wkv.WKVError) as exc:
            call()
        assert exc.value.status == 2


SHAPES = [(1, 1, 5), (1, 31, 33), (2, 33, 129), (3, 200, 100), (1, 1000, 32), (2, 513, 384)]


@pytest.mark.parametrize("B,T,C", SHAPES, ids=[f"B{b}T{t}C{c}" for b, t, c in SHAPES])
def test_gated_shapes(oracle, wkv, scan_mode, B, T, C):
    w, u, k, v, r, gout = _inputs(B, T, C, seed=500 + 3 * B + T + C)
    if scan_mode == "chunked":
        _refused(wkv, w, u, k, v, r, gout)
        return
    for use_ckpt in (True, False):
        _check(oracle, wkv, w, u, k, v, r, gout, f"B{B}T{T}C{C} ckpt={use_ckpt}", use_ckpt=use_ckpt)


@pytest.mark.parametrize("case", ["k_std_8", "r_std_30", "big_u"])
def test_gated_stress(oracle, wkv, scan_mode, case):
    """k_std_8 sends lanes onto the per-token path (gate there too);
    r_std_30 saturates the gate at 0 and 1 (e^{-r} overflowing for r below
    about -88); big_u makes the current token dominate."""
    if scan_mode == "chunked":
        return
    kw = dict(k_std=2.0, r_std=2.0)
    if case == "k_std_8":
        kw.update(k_std=8.0)
    if case == "r_std_30":
        kw.update(r_std=30.0)
    w, u, k, v, r, gout = _inputs(2, 400, 96, seed=520, **kw)
    if case == "big_u":
        u = u + 20.0
    _check(oracle, wkv, w, u, k, v, r, gout, case)


def test_gated_bf16(oracle, wkv, scan_mode):
    """bf16 k, v, r, gout (fp32 arithmetic and outputs): the oracle sees the
    same rounded values."""
    w, u, k, v, r, gout = _inputs(2, 777, 136, seed=530, kv_dtype="bf16", k_std=5.0)
    if scan_mode == "chunked":
        _refused(wkv, w, u, k, v, r, gout)
        return
    _check(oracle, wkv, w, u, k, v, r, gout, "bf16", tol_out=TOL_BF16)
    out = _run(wkv, w, u, k, v, r, gout)[0]
    _check_out(oracle, w, u, k, v, r, out, "bf16 (fp32-level)")


def test_gate_at_one_is_ungated(oracle, wkv):
    """r = 30: sigmoid(r) rounds to 1 in fp32, so the gated output is wkv bit
    for bit (one run per column, so both calls split the columns alike) and
    gr is exactly 0.  The gradients equal the ungated call's with gy = gout
    to rounding: the two backward kernels are separate compilations, free to
    fuse their multiply-adds differently."""
    w, u, k, v, gout = inputs.training_inputs(3, 300, 200, seed=540, k_std=3.0)
    r = torch.full_like(k, 30.0)
    try:
        wkv.set_max_runs(1)
        out, ckpt, gw, gu, gk, gv, gr = _run(wkv, w, u, k, v, r, gout)
        wc, uc, kc, vc, gc = cuda(w, u, k, v, gout)
        y, ckpt2 = wkv.forward(wc, uc, kc, vc, want_ckpt=True)
        ref = wkv.backward(wc, uc, kc, vc, gc, ckpt=ckpt2)
        torch.cuda.synchronize()
    finally:
        wkv.set_max_runs(0)
    assert torch.equal(out, y), "out vs y"
    assert torch.equal(ckpt, ckpt2), "ckpt"
    assert torch.count_nonzero(gr).item() == 0, "gr"
    names = ("gw", "gu", "gk", "gv")
    check_pair_grads(oracle, w, u, k, v, gout, dict(zip(names, (gw, gu, gk, gv))), dict(zip(names, ref)),
                     "r=30 vs ungated", tol=1e-6)


def test_gated_state_in_out(oracle, wkv):
    """The gated forward continues from a carried state like
    wkv_forward_with_state: out = sigmoid(r) * that call's y, and the same
    final state."""
    B, T, C = 2, 300, 160
    w, u, k, v, r, _ = _inputs(B, T, C, seed=550)
    wc, uc, kc, vc, rc = cuda(w, u, k, v, r)
    y1, s1 = wkv.forward_with_state(wc, uc, kc[:, :100].contiguous(), vc[:, :100].contiguous())
    y2, s2 = wkv.forward_with_state(wc, uc, kc[:, 100:].contiguous(), vc[:, 100:].contiguous(), state_in=s1)
    s3 = torch.empty_like(s2)
    out = wkv.forward_gated(wc, uc, kc[:, 100:].contiguous(), vc[:, 100:].contiguous(), rc[:, 100:].contiguous(),
                            state_in=s1, state_out=s3)
    torch.cuda.synchronize()
    assert torch.equal(s2, s3), "state out"
    want = oracle.forward_gated(w, u, k, v, r)[:, 100:]
    e = emu.forward_gated(w, u, k, v, r)[:, 100:]
    assert_close(out, want, TOL_Y, "gated continuation vs oracle", emu=e)
    sig = 1.0 / (1.0 + np.exp(-to_np(r[:, 100:])))
    assert_close(out, sig * to_np(y2), TOL_Y, "gated continuation vs ungated", emu=e, ref=want, pair=True)


def test_autograd_wrapper(oracle, wkv):
    B, T, C = 2, 120, 64
    w, u, k, v, r, gout = _inputs(B, T, C, seed=560)
    wc, uc, kc, vc, rc, gc = (t.clone().requires_grad_(True) for t in cuda(w, u, k, v, r, gout))
    out = wkv.wkv_gated(wc, uc, kc, vc, rc)
    out.backward(gc.detach())
    torch.cuda.synchronize()
    _check_grads(oracle, w, u, k, v, r, gout, tuple(t.grad for t in (wc, uc, kc, vc, rc)), "autograd")


def test_workload_l169m_gated_full(oracle, wkv):
    w, u, k, v, gout, r = inputs.workload_inputs("l169m_gated")
    _check(oracle, wkv, w, u, k, v, r, gout, "l169m_gated")
