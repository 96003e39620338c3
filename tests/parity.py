"""Helpers of the GPU parity tests: the two-part error gate, tolerances,
column sampling.

Tolerances (max relative error): 2e-5 for fp32 forward outputs and decode
outputs/state, 1e-4 for gradients, 1e-2 for workloads with bf16 inputs (the
oracle is handed the same bf16-rounded values, so this is loose).

Every comparison ``assert_close(got, want, tol, ...)`` passes two gates,
with r = want (the float64 oracle unless stated) and tau = 1e-3 max|r|:

1. norm-wise: max_i |g_i - r_i| / max_i |r_i| <= tol;
2. element-wise: e_i = |g_i - r_i| / max(|r_i|, tau) and
   max_i e_i <= max(tol, K_EMU * max_i f_i), where f_i is the same
   element-wise error of a float32 evaluation of the same quantity
   (``tests/fp32_emulation.py``: the plain recurrence, nothing rescaled or
   compensated) against the oracle, on the same inputs.

For gradients ``emu`` is a list of float32 evaluations: one on the
exact inputs and two on inputs moved by one ulp at random
(``fp32_emulation.evaluations``), and f_i is the worst of their errors.
One evaluation is a single sample of the fp32 rounding at an
ill-conditioned output: on the gated stress input, gw of one channel
(2.8e-3 of the largest) came out of two equally valid float32 evaluations
with errors 3.9e-5 and 1.1e-4, which differ only in the float32 sigmoid
that rounded the output gradient.

Gate 2 without a float32 evaluation (``emu`` not given) is plain
e_i <= tol.  Why the floor: an output that is near zero only by
cancellation (a weighted average of O(1) values that happens to be small)
cannot be matched to 2e-5 of itself by fp32 arithmetic; the absolute error
of the sums behind it is a few ulp of their size, amplified by the decay's
memory (about 1/w tokens).  The float32 evaluation measures that floor on
the very inputs of the test, so an error confined to small elements fails
gate 2 unless plain fp32 arithmetic makes one as large.  The floor is the
whole tensor's: per column, the few near-cancelling elements give the two
evaluations' rounding errors as independent draws, and their ratio ranged
up to 10 on the 169M-layer shape with both sides correct, while over the
whole tensor the GPU's maximum stayed at or below the float32 evaluation's.
The same ratio per magnitude bin of |r| / max|r| (below 1e-3, to 1e-2, to
1e-1, above) is computed and logged (``ratio_bins``) as a diagnostic.

``pair=True``: both sides are GPU results (a consistency check), so each
may sit K_EMU times the floor away from the oracle: the bound doubles, and
the floor is the float32 evaluation against ``ref`` (the oracle).

Set ``WKV_PARITY_LOG`` to a file path to have every comparison written
there as JSON at the end of the session (conftest.py).
"""
from __future__ import annotations

import numpy as np
import torch

TOL_Y = 2e-5
TOL_GRAD = 1e-4
TOL_BF16 = 1e-2
K_EMU = 4.0


def to_np(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        t = t.detach().to("cpu")
        if t.dtype == torch.bfloat16:
            t = t.float()
        return t.numpy().astype(np.float64)
    return np.asarray(t, dtype=np.float64)


PARITY_LOG: list = []


def _scale(r: np.ndarray) -> float:
    # a reference that is zero up to float64 rounding (e.g. gk at T = 1) is
    # measured against 1e-9, far below any value these workloads produce
    return max(float(np.max(np.abs(r))), 1e-9) if r.size else 1e-9


def _elem(g: np.ndarray, r: np.ndarray, scale: float) -> np.ndarray:
    return np.abs(g - r) / np.maximum(np.abs(r), 1e-3 * scale)


BIN_EDGES = (1e-3, 1e-2, 1e-1)  # of |r| / max|r|, for the logged per-bin ratios


def errors(got, want):
    """(norm-wise, element-wise floored) relative errors of got vs want."""
    g = to_np(got)
    r = to_np(want)
    assert g.shape == r.shape, f"shape {g.shape} vs {r.shape}"
    if r.size == 0:
        return 0.0, 0.0
    assert np.all(np.isfinite(g)), "non-finite GPU output"
    scale = _scale(r)
    d = np.abs(g - r)
    return float(d.max() / scale), float(_elem(g, r, scale).max())


def rel_err(got, want) -> float:
    return errors(got, want)[0]


def assert_close(got, want, tol, what="", emu=None, ref=None, pair=False):
    """Both gates (module docstring).  ``emu``: the float32 evaluation of
    ``want``'s quantity (or a list of such evaluations: the worst error
    counts); ``ref``: the float64 value it is measured against
    (default ``want``); ``pair``: got and want are both GPU results."""
    e, el = errors(got, want)
    g, r = to_np(got), to_np(want)
    entry = {"what": what, "norm": e, "elem": el, "tol": tol}
    if r.size == 0:
        PARITY_LOG.append(entry)
        return e
    eg = _elem(g, r, _scale(r))
    bound = tol
    if emu is not None:
        o = r if ref is None else to_np(ref)
        so = _scale(o)
        fe = None
        for m in (emu if isinstance(emu, list) else [emu]):  # several evaluations: the worst error
            m = to_np(m)
            assert m.shape == o.shape == r.shape, f"{what}: emulation shape {m.shape} vs {r.shape}"
            assert np.all(np.isfinite(m)), f"{what}: the float32 evaluation left float32's range"
            fe = _elem(m, o, so) if fe is None else np.maximum(fe, _elem(m, o, so))
        k = K_EMU * (2.0 if pair else 1.0)
        bound = max(tol, k * float(fe.max()))
        entry["emu_elem"] = float(fe.max())
        bins = np.digitize(np.abs(o) / so, BIN_EDGES)
        entry["ratio_bins"] = max(float(eg[bins == b].max()) / max(tol, k * float(fe[bins == b].max()))
                                  for b in np.unique(bins))
    entry["ratio"] = el / bound
    PARITY_LOG.append(entry)
    assert e <= tol, f"{what}: rel err {e:.3e} > {tol:.1e} (element-wise {el:.3e})"
    assert el <= bound, (f"{what}: element-wise err {el:.3e} > bound {bound:.3e}"
                         + ("" if emu is None else f" (the fp32 evaluation's {entry['emu_elem']:.3e})"))
    return e


def emu_state_content(emu_sums, r_pp):
    """The float32 evaluation's state (unscaled sums a, b) in the oracle's
    scale-free form: a e^{-pp_ref}, b e^{-pp_ref}; empty where pp_ref is."""
    r_pp = to_np(r_pp)
    a, b = (to_np(x).reshape(r_pp.shape) for x in emu_sums)
    s = np.where(r_pp < -1e37, 0.0, np.exp(-np.maximum(r_pp, -700.0)))
    return a * s, b * s


def assert_state_close(num, den, pp, onum, oden, opp, tol, what="", pp_atol=5e-3, emu_sums=None, oracle=None):
    """Compare a carried state (num, den, pp) with the oracle's.

    The state stands for the sums a = num e^{pp}, b = den e^{pp}; pp is only
    a scale (the oracle keeps it at the exact running maximum, fp32 pp moves
    by rounding), so what must match is the scale-free content
    num e^{pp - pp_ref}, den e^{pp - pp_ref}.  pp itself must stay a valid
    scale: within pp_atol of the running maximum, and den >= ~1.  Empty
    states (pp_ref = -1e38) must be empty on both sides.  ``emu_sums``: the
    float32 evaluation's unscaled sums (a, b), for the element-wise floor.
    ``oracle`` = (num, den, pp): (onum, oden, opp) is another GPU state and
    this the oracle's; both are measured at the oracle's scale and compared
    as a pair (``assert_close``)."""
    if oracle is not None:
        g_num, g_den, g_pp = to_np(num), to_np(den), to_np(pp)
        o_num, o_den, o_pp = (to_np(x) for x in oracle)
        b_num, b_den, b_pp = to_np(onum), to_np(oden), to_np(opp)
        empty = o_pp < -1e37
        assert np.all(g_pp[empty] < -1e37) and np.all(b_pp[empty] < -1e37), f"{what}: empty state not preserved"
        fg, fb = np.ones_like(g_pp), np.ones_like(b_pp)
        fg[~empty] = np.exp(g_pp[~empty] - o_pp[~empty])
        fb[~empty] = np.exp(b_pp[~empty] - o_pp[~empty])
        en, ed = emu_state_content(emu_sums, o_pp) if emu_sums is not None else (None, None)
        assert_close(g_num * fg, b_num * fb, tol, f"{what} num e^pp", emu=en, ref=o_num, pair=True)
        assert_close(g_den * fg, b_den * fb, tol, f"{what} den e^pp", emu=ed, ref=o_den, pair=True)
        return
    g_num, g_den, g_pp = to_np(num), to_np(den), to_np(pp)
    r_num, r_den, r_pp = to_np(onum), to_np(oden), to_np(opp)
    empty = r_pp < -1e37
    assert np.all(g_pp[empty] < -1e37) and np.all(g_num[empty] == 0) and np.all(g_den[empty] == 0), \
        f"{what}: empty state not preserved"
    assert np.all(g_pp[~empty] > -1e37), f"{what}: state emptied"
    f = np.ones_like(g_pp)
    f[~empty] = np.exp(g_pp[~empty] - r_pp[~empty])
    en = ed = None
    if emu_sums is not None:
        en, ed = emu_state_content(emu_sums, r_pp)
    assert_close(g_num * f, r_num, tol, f"{what} num e^pp", emu=en)
    assert_close(g_den * f, r_den, tol, f"{what} den e^pp", emu=ed)
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
