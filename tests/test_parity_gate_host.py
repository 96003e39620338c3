"""The parity gate itself (tests/parity.py), on the CPU: it accepts a
float32 evaluation of the operator, and it rejects a planted error on one
small-magnitude element, which the norm-wise reading alone lets through."""
import numpy as np
import pytest

import fp32_emulation as emu
from parity import K_EMU, TOL_GRAD, TOL_Y, assert_close
from rwkv_linear_attention_backward_b300 import inputs


@pytest.fixture(scope="module")
def case(oracle):
    w, u, k, v, gy = inputs.training_inputs(2, 300, 40, seed=77, k_std=3.0, d_lo=-7.0, d_hi=1.0)
    return dict(w=w, u=u, k=k, v=v, gy=gy, y=oracle.forward_recurrent(w, u, k, v),
                ye=emu.forward_recurrent(w, u, k, v), ge=emu.backward_adjoint(w, u, k, v, gy),
                go=oracle.backward_adjoint(w, u, k, v, gy))


def test_a_float32_evaluation_passes(case):
    """The float32 evaluation measured against its own floor passes (ratio
    1/K_EMU by construction), for [B, T, C] and [C] tensors."""
    assert_close(case["ye"], case["y"], TOL_Y, "y", emu=case["ye"])
    for g, o in zip(case["ge"], case["go"]):
        assert_close(g, o, TOL_GRAD, "grad", emu=g)


def test_a_planted_error_on_small_elements_fails(case):
    """Errors twice the float32 evaluation's pass; an error K_EMU times its
    worst planted on one near-zero output fails, though norm-wise it is far
    below the tolerance."""
    y, ye = case["y"], case["ye"]
    d = ye.astype(np.float64) - y
    assert_close(y + 2.0 * d, y, TOL_Y, "2x the fp32 error", emu=ye)
    scale = np.abs(y).max()
    floor = (np.abs(d) / np.maximum(np.abs(y), 1e-3 * scale)).max()
    i = np.unravel_index(np.argmin(np.where(np.abs(y) > 1e-3 * scale, np.abs(y), np.inf)), y.shape)
    bad = y.copy()
    bad[i] += 1.5 * K_EMU * max(floor, TOL_Y) * abs(y[i])
    assert np.abs(bad - y).max() / scale < TOL_Y  # invisible to the norm-wise gate
    with pytest.raises(AssertionError, match="element-wise"):
        assert_close(bad, y, TOL_Y, "planted", emu=ye)


def test_without_a_floor_the_gate_is_elementwise(case):
    y = case["y"]
    bad = y.copy()
    i = np.unravel_index(np.argmin(np.abs(y) + (np.abs(y) < 1e-3 * np.abs(y).max()) * 1e9), y.shape)
    bad[i] *= 1 + 3 * TOL_Y
    with pytest.raises(AssertionError, match="element-wise"):
        assert_close(bad, y, TOL_Y, "no floor")
