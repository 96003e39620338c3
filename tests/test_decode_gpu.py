"""GPU parity of the fused decode step (token shift, wkv, sigmoid gate,
state update) against the float64 oracle, step after step."""
import numpy as np
import pytest
import torch

import fp32_emulation as emu
from parity import TOL_Y, assert_close, assert_state_close, cuda, to_np
from rwkv_linear_attention_backward_b300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def wkv():
    from rwkv_linear_attention_backward_b300 import binding

    return binding


def _run_steps(oracle, wkv, L, B, C, steps, seed, mix=True, offset=0, token_dtype="f32"):
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
    ea, eb = np.zeros((L, B, C), np.float32), np.zeros((L, B, C), np.float32)  # the empty state's sums
    for s in range(steps):
        x, xp, r, k, v = inputs.decode_step_inputs(L, B, C, seed=seed, step=s, token_dtype=token_dtype)
        gx, gxp, gr, gk, gv = cuda(x, xp, r, k, v)
        y, xk, xv, xr = wkv.decode_step(gx, gxp, *dev[:3], gr, gk, gv, *dev[3:], gnum, gden, gpp, mix=mix)
        oy, onum, oden, opp, oxk, oxv, oxr = oracle.decode_step(x, xp, mu_k, mu_v, mu_r, r, k, v, w, u, onum, oden,
                                                                opp, mix=mix)
        ey, ea, eb, exk, exv, exr = emu.decode_step(x, xp, mu_k, mu_v, mu_r, r, k, v, w, u, ea, eb)
        torch.cuda.synchronize()
        assert_close(y, oy, TOL_Y, f"step {s} y", emu=ey)
        assert_state_close(gnum, gden, gpp, onum, oden, opp, TOL_Y, f"step {s}", emu_sums=(ea, eb))
        if mix:
            for a_, b_, e_, n in ((xk, oxk, exk, "xk"), (xv, oxv, exv, "xv"), (xr, oxr, exr, "xr")):
                assert_close(a_, b_, TOL_Y, f"step {s} {n}", emu=e_)
        else:
            assert xk is None and xv is None and xr is None


@pytest.mark.parametrize("token_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("L,B,C", [(1, 1, 1), (2, 3, 8), (2, 3, 7), (3, 5, 64), (1, 2, 4097)])
def test_decode_small(oracle, wkv, L, B, C, token_dtype):
    """fp32 or bf16 token inputs (the oracle is handed the same rounded
    values, so the fp32 tolerance holds for both)."""
    _run_steps(oracle, wkv, L, B, C, steps=24, seed=31 + C, token_dtype=token_dtype)


def test_decode_without_mix(oracle, wkv):
    _run_steps(oracle, wkv, 2, 4, 16, steps=10, seed=32, mix=False)


@pytest.mark.parametrize("token_dtype", ["f32", "bf16"])
def test_decode_unaligned_state(oracle, wkv, token_dtype):
    _run_steps(oracle, wkv, 2, 3, 16, steps=10, seed=33, offset=1, token_dtype=token_dtype)


def test_decode_bf16_equals_fp32_of_rounded_inputs(wkv):
    """bf16 token inputs widen to fp32 exactly and the arithmetic is the
    same: the bf16 call equals the fp32 call on the widened values bit for
    bit (vectorised and scalar paths)."""
    for L, B, C in ((2, 5, 64), (2, 3, 7)):
        mu_k, mu_v, mu_r, w, u = cuda(*inputs.decode_params(L, C, seed=34))
        st_a = cuda(*inputs.initial_state(L, B, C))
        st_b = tuple(t.clone() for t in st_a)
        for s in range(6):
            tok = cuda(*inputs.decode_step_inputs(L, B, C, seed=34, step=s, token_dtype="bf16"))
            a = wkv.decode_step(*tok[:2], mu_k, mu_v, mu_r, *tok[2:], w, u, *st_a)
            wide = tuple(t.float() for t in tok)
            b = wkv.decode_step(*wide[:2], mu_k, mu_v, mu_r, *wide[2:], w, u, *st_b)
            torch.cuda.synchronize()
            for x, y_ in zip(a + st_a, b + st_b):
                assert torch.equal(x, y_)


@pytest.mark.parametrize("name", ["decode", "decode_bf16"])
def test_decode_workload(oracle, wkv, name):
    """Full-size decode (L=32, B=256, C=4096; fp32 or bf16 token inputs) for
    all 1024 steps in the launch configuration the benchmark uses (inputs
    from a device pool of 16 step sets).  The first 3 steps are compared at
    full width; all 1024 steps on a slice (layers 0 and 31, batch rows 0..7,
    every channel)."""
    D = inputs.DECODES[name]
    L, B, C = D.L, D.B, D.C
    mu_k, mu_v, mu_r, w, u = inputs.decode_params(L, C, seed=D.seed, d_lo=D.d_lo, d_hi=D.d_hi)
    pool = inputs.decode_pool(L, B, C, seed=D.seed, n_sets=16, device="cuda", token_dtype=D.token_dtype)
    num, den, pp = cuda(*inputs.initial_state(L, B, C))
    dev = cuda(mu_k, mu_v, mu_r, w, u)
    y = torch.empty(L, B, C, device="cuda")
    xk, xv, xr = (torch.empty(L, B, C, device="cuda") for _ in range(3))
    lsel, bsel = [0, L - 1], list(range(8))
    osl = [np.zeros((2, 8, C)) for _ in range(2)] + [np.full((2, 8, C), -1e38)]
    slice_ = lambda t: to_np(t[lsel][:, bsel])  # noqa: E731
    psl = [to_np(t[lsel]) for t in (mu_k, mu_v, mu_r, w, u)]
    pool_sl = [[slice_(t) for t in st] for st in pool]
    ofull = efull = None
    esl = [np.zeros((2, 8, C), np.float32) for _ in range(2)]
    for s in range(D.steps):
        x, xp, r, k, v = pool[s % 16]
        wkv.decode_step(x, xp, *dev[:3], r, k, v, *dev[3:], num, den, pp, y=y, xk=xk, xv=xv, xr=xr)
        if s < 3:
            torch.cuda.synchronize()
            if ofull is None:
                ofull = [to_np(t) for t in inputs.initial_state(L, B, C)]
                efull = [np.zeros((L, B, C), np.float32) for _ in range(2)]
            oy, n1, d1, p1, oxk, oxv, oxr = oracle.decode_step(x, xp, mu_k, mu_v, mu_r, r, k, v, w, u, *ofull)
            ey, ea, eb, exk, _, _ = emu.decode_step(x, xp, mu_k, mu_v, mu_r, r, k, v, w, u, *efull)
            ofull, efull = [n1, d1, p1], [ea, eb]
            assert_close(y, oy, TOL_Y, f"full step {s} y", emu=ey)
            assert_state_close(num, den, pp, n1, d1, p1, TOL_Y, f"full step {s}", emu_sums=(ea, eb))
            assert_close(xk, oxk, TOL_Y, f"full step {s} xk", emu=exk)
        sx, sxp, sr, sk, sv = pool_sl[s % 16]
        oy, n2, d2, p2, _, _, _ = oracle.decode_step(sx, sxp, *psl[:3], sr, sk, sv, *psl[3:], *osl, mix=False)
        ey, ea, eb, _, _, _ = emu.decode_step(sx, sxp, *psl[:3], sr, sk, sv, *psl[3:], *esl)
        osl, esl = [n2, d2, p2], [ea, eb]
        if s % 128 == 127 or s == D.steps - 1:
            torch.cuda.synchronize()
            assert_close(slice_(y), oy, TOL_Y, f"slice step {s} y", emu=ey)
            assert_state_close(slice_(num), slice_(den), slice_(pp), *osl, TOL_Y, f"slice step {s}", emu_sums=esl)
