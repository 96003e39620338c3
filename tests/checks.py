"""Parity checks shared by the GPU tests: a GPU result against the float64
oracle, with the float32 evaluation of the same inputs
(``fp32_emulation``) as the element-wise floor (``parity.assert_close``)."""
from __future__ import annotations

import fp32_emulation as emu
from parity import TOL_GRAD, TOL_Y, assert_close

GRADS = ("gw", "gu", "gk", "gv")


def check_y(oracle, w, u, k, v, y, what, tol=TOL_Y):
    """y (GPU) of the forward pass over k, v from the empty state."""
    assert_close(y, oracle.forward_recurrent(w, u, k, v), tol, f"{what} y", emu=emu.forward_recurrent(w, u, k, v))


def grad_evaluations(fn, *args, names=GRADS):
    """{name: [float32 evaluations]}: fn on the exact inputs and on two
    one-ulp perturbations of them (the gradients' floor)."""
    runs = emu.evaluations(fn, *args)
    return {n: [r[i] for r in runs] for i, n in enumerate(names)}


def check_grads(oracle, w, u, k, v, gy, got, what, tol=TOL_GRAD):
    """``got``: {name: GPU tensor} for any of gw, gu, gk, gv."""
    o = dict(zip(GRADS, oracle.backward_adjoint(w, u, k, v, gy)))
    e = grad_evaluations(emu.backward_adjoint, w, u, k, v, gy)
    for n, g in got.items():
        assert_close(g, o[n], tol, f"{what} {n}", emu=e[n])


def check_pair_y(oracle, w, u, k, v, a, b, what, tol=TOL_Y):
    """Two GPU evaluations of the same y against each other."""
    assert_close(a, b, tol, what, emu=emu.forward_recurrent(w, u, k, v), ref=oracle.forward_recurrent(w, u, k, v),
                 pair=True)


def check_pair_grads(oracle, w, u, k, v, gy, a, b, what, tol=TOL_GRAD):
    """Two GPU evaluations of the same gradients ({name: tensor} each)."""
    o = dict(zip(GRADS, oracle.backward_adjoint(w, u, k, v, gy)))
    e = grad_evaluations(emu.backward_adjoint, w, u, k, v, gy)
    for n in a:
        assert_close(a[n], b[n], tol, f"{what} {n}", emu=e[n], ref=o[n], pair=True)
