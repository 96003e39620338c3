"""Helpers of the GPU parity tests: error metric, tolerances, column sampling.

Error metric (per tensor), the gate: max relative error normalised by the
tensor's scale, max_i |g_i - r_i| / max_i |r_i|, with ``r`` the float64
oracle.  An fp32 evaluation of a weighted average of O(1) values carries an
absolute error of a few ulp of those values, so an element that is near
zero only by cancellation cannot be matched to 2e-5 of itself by any fp32
arithmetic; measured against the tensor's scale it can.  The element-wise
error with a small floor, max_i |g_i - r_i| / max(|r_i|, 1e-3 max|r|), is
computed too and recorded (``PARITY_LOG``, written to gpurun_out/ by
conftest.py) as a diagnostic.

Tolerances: 2e-5 for fp32 forward outputs and decode outputs/state, 1e-4 for
gradients, 1e-2 for workloads with bf16 inputs (the oracle is handed the
same bf16-rounded values, so this is loose).
"""
from __future__ import annotations

import numpy as np
import torch

TOL_Y = 2e-5
TOL_GRAD = 1e-4
TOL_BF16 = 1e-2


def to_np(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        t = t.detach().to("cpu")
        if t.dtype == torch.bfloat16:
            t = t.float()
        return t.numpy().astype(np.float64)
    return np.asarray(t, dtype=np.float64)


PARITY_LOG: list = []


def errors(got, want):
    """(norm-wise, element-wise floored) relative errors of got vs want."""
    g = to_np(got)
    r = to_np(want)
    assert g.shape == r.shape, f"shape {g.shape} vs {r.shape}"
    if r.size == 0:
        return 0.0, 0.0
    assert np.all(np.isfinite(g)), "non-finite GPU output"
    # a reference that is zero up to float64 rounding (e.g. gk at T = 1) is
    # measured against 1e-9, far below any value these workloads produce
    scale = max(float(np.max(np.abs(r))), 1e-9)
    d = np.abs(g - r)
    return float(d.max() / scale), float(np.max(d / np.maximum(np.abs(r), 1e-3 * scale)))


def rel_err(got, want) -> float:
    return errors(got, want)[0]


def assert_close(got, want, tol, what=""):
    e, el = errors(got, want)
    PARITY_LOG.append({"what": what, "norm": e, "elem": el, "tol": tol})
    assert e <= tol, f"{what}: rel err {e:.3e} > {tol:.1e} (element-wise {el:.3e})"
    return e


def assert_state_close(num, den, pp, onum, oden, opp, tol, what="", pp_atol=5e-3):
    """Compare a carried state (num, den, pp) with the oracle's.

    The state stands for the sums a = num e^{pp}, b = den e^{pp}; pp is only
    a scale (the oracle keeps it at the exact running maximum, fp32 pp moves
    by rounding), so what must match is the scale-free content
    num e^{pp - pp_ref}, den e^{pp - pp_ref}.  pp itself must stay a valid
    scale: within pp_atol of the running maximum, and den >= ~1.  Empty
    states (pp_ref = -1e38) must be empty on both sides."""
    g_num, g_den, g_pp = to_np(num), to_np(den), to_np(pp)
    r_num, r_den, r_pp = to_np(onum), to_np(oden), to_np(opp)
    empty = r_pp < -1e37
    assert np.all(g_pp[empty] < -1e37) and np.all(g_num[empty] == 0) and np.all(g_den[empty] == 0), \
        f"{what}: empty state not preserved"
    assert np.all(g_pp[~empty] > -1e37), f"{what}: state emptied"
    f = np.ones_like(g_pp)
    f[~empty] = np.exp(g_pp[~empty] - r_pp[~empty])
    assert_close(g_num * f, r_num, tol, f"{what} num e^pp")
    assert_close(g_den * f, r_den, tol, f"{what} den e^pp")
    dpp = float(np.max(np.abs(g_pp[~empty] - r_pp[~empty]))) if np.any(~empty) else 0.0
    assert dpp <= pp_atol, f"{what}: pp off the running maximum by {dpp:.2e}"
    assert np.all(g_den[~empty] >= 0.99), f"{what}: den < 1, pp is not the running maximum"


def cuda(*ts):
    return tuple(t.to("cuda").contiguous() for t in ts)


def sample_channels(C: int, n: int, seed: int) -> np.ndarray:
    """n distinct channels, always including the first and the last."""
    rng = np.random.default_rng(seed)
    pick = set(rng.choice(C, size=min(n, C), replace=False).tolist())
    pick.update({0, C - 1})
    return np.array(sorted(pick))
