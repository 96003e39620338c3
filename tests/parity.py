"""Helpers of the GPU parity tests: error metric, tolerances, column sampling.

Error metric (per tensor): max_i |g_i - r_i| / max(|r_i|, tau) with
tau = 1e-3 * max_i |r_i|: a relative error that does not blow up at entries
that are near zero only by cancellation.  ``r`` is the float64 oracle.

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


def rel_err(got, want) -> float:
    g = to_np(got)
    r = to_np(want)
    assert g.shape == r.shape, f"shape {g.shape} vs {r.shape}"
    if r.size == 0:
        return 0.0
    assert np.all(np.isfinite(g)), "non-finite GPU output"
    scale = float(np.max(np.abs(r)))
    tau = 1e-3 * scale if scale > 0 else 1e-30
    return float(np.max(np.abs(g - r) / np.maximum(np.abs(r), tau)))


def assert_close(got, want, tol, what=""):
    e = rel_err(got, want)
    assert e <= tol, f"{what}: rel err {e:.3e} > {tol:.1e}"
    return e


def cuda(*ts):
    return tuple(t.to("cuda").contiguous() for t in ts)


def sample_channels(C: int, n: int, seed: int) -> np.ndarray:
    """n distinct channels, always including the first and the last."""
    rng = np.random.default_rng(seed)
    pick = set(rng.choice(C, size=min(n, C), replace=False).tolist())
    pick.update({0, C - 1})
    return np.array(sorted(pick))
