"""GPU parity of the fused decode step (token shift, wkv, sigmoid gate,
state update) against the float64 oracle, step after step."""
import numpy as np
import pytest
import torch

from parity import TOL_Y, assert_close, assert_state_close, cuda, to_np
from rwkv_linear_attention_backward_b300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def wkv():
    from rwkv_linear_attention_backward_b300 import binding

    return binding


def _run_steps(oracle, wkv, L, B, C, steps, seed, mix=True, offset=0):
    mu_k, mu_v, mu_r, w, u = inputs.decode_params(L, C, seed=seed)
    num, den, pp = inputs.initial_state(L, B, C)
    dev = [t.cuda() for t in (mu_k, mu_v, mu_r, w, u)]
    if offset:  # views that start one float past an aligned address: scalar path
        def shifted(t):
            buf = torch.empty(t.numel() + offset, device="cuda")
            view = buf[offset:].view(t.shape)
            view.copy_(t)
            return view
        gnum, gden, gpp = (shifted(t) for t in (num, den, pp))
    else:
        gnum, gden, gpp = cuda(num, den, pp)
    onum, oden, opp = num.numpy(), den.numpy(), pp.numpy()
    for s in range(steps):
        x, xp, r, k, v = inputs.decode_step_inputs(L, B, C, seed=seed, step=s)
        gx, gxp, gr, gk, gv = cuda(x, xp, r, k, v)
        y, xk, xv, xr = wkv.decode_step(gx, gxp, *dev[:3], gr, gk, gv, *dev[3:], gnum, gden, gpp, mix=mix)
        oy, onum, oden, opp, oxk, oxv, oxr = oracle.decode_step(x, xp, mu_k, mu_v, mu_r, r, k, v, w, u, onum, oden,
                                                                opp, mix=mix)
        torch.cuda.synchronize()
        assert_close(y, oy, TOL_Y, f"step {s} y")
        assert_state_close(gnum, gden, gpp, onum, oden, opp, TOL_Y, f"step {s}")
        if mix:
            for a_, b_, n in ((xk, oxk, "xk"), (xv, oxv, "xv"), (xr, oxr, "xr")):
                assert_close(a_, b_, TOL_Y, f"step {s} {n}")
        else:
            assert xk is None and xv is None and xr is None


@pytest.mark.parametrize("L,B,C", [(1, 1, 1), (2, 3, 8), (2, 3, 7), (3, 5, 64), (1, 2, 4097)])
def test_decode_small(oracle, wkv, L, B, C):
    _run_steps(oracle, wkv, L, B, C, steps=24, seed=31 + C)


def test_decode_without_mix(oracle, wkv):
    _run_steps(oracle, wkv, 2, 4, 16, steps=10, seed=32, mix=False)


def test_decode_unaligned_state(oracle, wkv):
    _run_steps(oracle, wkv, 2, 3, 16, steps=10, seed=33, offset=1)


def test_decode_workload(oracle, wkv):
    """Full-size decode (L=32, B=256, C=4096) for all 1024 steps in the launch
    configuration the benchmark uses (inputs from a device pool of 16 step
    sets).  The first 3 steps are compared at full width; all 1024 steps on a
    slice (layers 0 and 31, batch rows 0..7, every channel)."""
    D = inputs.DECODE
    L, B, C = D.L, D.B, D.C
    mu_k, mu_v, mu_r, w, u = inputs.decode_params(L, C, seed=D.seed, d_lo=D.d_lo, d_hi=D.d_hi)
    pool = inputs.decode_pool(L, B, C, seed=D.seed, n_sets=16, device="cuda")
    num, den, pp = cuda(*inputs.initial_state(L, B, C))
    dev = cuda(mu_k, mu_v, mu_r, w, u)
    y = torch.empty(L, B, C, device="cuda")
    xk, xv, xr = (torch.empty(L, B, C, device="cuda") for _ in range(3))
    lsel, bsel = [0, L - 1], list(range(8))
    osl = [np.zeros((2, 8, C)) for _ in range(2)] + [np.full((2, 8, C), -1e38)]
    slice_ = lambda t: to_np(t[lsel][:, bsel])  # noqa: E731
    psl = [to_np(t[lsel]) for t in (mu_k, mu_v, mu_r, w, u)]
    pool_sl = [[slice_(t) for t in st] for st in pool]
    ofull = None
    for s in range(D.steps):
        x, xp, r, k, v = pool[s % 16]
        wkv.decode_step(x, xp, *dev[:3], r, k, v, *dev[3:], num, den, pp, y=y, xk=xk, xv=xv, xr=xr)
        if s < 3:
            torch.cuda.synchronize()
            if ofull is None:
                ofull = [to_np(t) for t in inputs.initial_state(L, B, C)]
            oy, n1, d1, p1, oxk, oxv, oxr = oracle.decode_step(x, xp, mu_k, mu_v, mu_r, r, k, v, w, u, *ofull)
            ofull = [n1, d1, p1]
            assert_close(y, oy, TOL_Y, f"full step {s} y")
            assert_state_close(num, den, pp, n1, d1, p1, TOL_Y, f"full step {s}")
            assert_close(xk, oxk, TOL_Y, f"full step {s} xk")
        sx, sxp, sr, sk, sv = pool_sl[s % 16]
        oy, n2, d2, p2, _, _, _ = oracle.decode_step(sx, sxp, *psl[:3], sr, sk, sv, *psl[3:], *osl, mix=False)
        osl = [n2, d2, p2]
        if s % 128 == 127 or s == D.steps - 1:
            torch.cuda.synchronize()
            assert_close(slice_(y), oy, TOL_Y, f"slice step {s} y")
            assert_state_close(slice_(num), slice_(den), slice_(pp), *osl, TOL_Y, f"slice step {s}")
