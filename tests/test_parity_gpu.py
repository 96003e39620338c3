"""GPU parity: the CUDA path through the C ABI against the float64 oracle,
element by element, on seeded inputs (module rwkv_linear_attention_backward_b300.inputs).

Small shapes cover several chunks, ragged chunk and channel-block tails,
T = 1, deep look-back chains and stress values, each under both scan
strategies (chunked across CTAs, and sequential per column); the named
workloads run at full size in the strategy the library picks for them (the
oracle computes sampled channels exactly, since channels are
independent)."""
import numpy as np
import pytest
import torch

import fp32_emulation as emu
from checks import check_grads, check_pair_grads, check_pair_y, check_y
from parity import TOL_BF16, TOL_GRAD, TOL_Y, assert_close, assert_state_close, cuda, sample_channels, to_np
from rwkv_linear_attention_backward_b300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def wkv():
    from rwkv_linear_attention_backward_b300 import binding

    return binding


def run_fwd_bwd(wkv, w, u, k, v, gy, use_ckpt=True):
    w, u, k, v, gy = cuda(w, u, k, v, gy)
    y, ckpt = wkv.forward(w, u, k, v, want_ckpt=True)
    gw, gu, gk, gv = wkv.backward(w, u, k, v, gy, ckpt=ckpt if use_ckpt else None)
    torch.cuda.synchronize()
    return y, ckpt, gw, gu, gk, gv


def check_all(oracle, wkv, w, u, k, v, gy, use_ckpt=True, what=""):
    y, ckpt, gw, gu, gk, gv = run_fwd_bwd(wkv, w, u, k, v, gy, use_ckpt)
    check_y(oracle, w, u, k, v, y, what)
    check_grads(oracle, w, u, k, v, gy, dict(gk=gk, gv=gv, gw=gw, gu=gu), what)
    return y, ckpt


SHAPES = [
    (1, 1, 1), (1, 1, 64), (1, 31, 5), (1, 32, 33), (2, 33, 129), (3, 65, 100), (1, 64, 64),
    (2, 200, 256), (1, 257, 130), (4, 96, 7), (1, 1000, 32), (2, 513, 384),
]


@pytest.mark.parametrize("B,T,C", SHAPES, ids=[f"B{b}T{t}C{c}" for b, t, c in SHAPES])
def test_small_shapes(oracle, wkv, scan_mode, B, T, C):
    w, u, k, v, gy = inputs.training_inputs(B, T, C, seed=100 + B * 7 + T + C, k_std=2.0, d_lo=-5.0, d_hi=1.5)
    check_all(oracle, wkv, w, u, k, v, gy, what=f"B{B}T{T}C{C}")


def test_without_checkpoint_matches(oracle, wkv, scan_mode):
    w, u, k, v, gy = inputs.training_inputs(2, 300, 160, seed=5, k_std=2.0)
    check_all(oracle, wkv, w, u, k, v, gy, use_ckpt=False, what="no ckpt")


def test_checkpoint_is_the_carried_state(oracle, wkv, scan_mode):
    B, T, C = 2, 150, 70
    w, u, k, v, gy = inputs.training_inputs(B, T, C, seed=6, k_std=3.0)
    y, ckpt = wkv.forward(*cuda(w, u, k, v), want_ckpt=True)
    L = wkv.chunk_len()
    nch = -(-T // L)
    ck = to_np(ckpt).reshape(3, nch, B, C)
    ends = [min((j + 1) * L, T) for j in range(nch)]
    sums = emu.sums_after(w, k, v, ends)
    for j in range(nch):
        num, den, pp = oracle.state(w, k, v, ends[j])
        assert_state_close(ck[0, j], ck[1, j], ck[2, j], num, den, pp, TOL_Y, f"after chunk {j}", emu_sums=sums[j])


@pytest.mark.parametrize("case", ["k_shift_64", "tiny_w", "huge_w", "big_u", "k_std_8"])
def test_stress_values(oracle, wkv, scan_mode, case):
    B, T, C = 2, 400, 96
    kw = dict(k_std=2.0, d_lo=-5.0, d_hi=1.0)
    if case == "tiny_w":
        kw.update(d_lo=-12.0, d_hi=-9.0)
    if case == "huge_w":
        kw.update(d_lo=2.0, d_hi=3.5)
    if case == "k_std_8":
        kw.update(k_std=8.0)
    w, u, k, v, gy = inputs.training_inputs(B, T, C, seed=7, **kw)
    if case == "k_shift_64":
        k = k + 64.0
    if case == "big_u":
        u = u + 20.0
    check_all(oracle, wkv, w, u, k, v, gy, what=case)


def test_deep_lookback_chain(oracle, wkv, scan_mode):
    """One 32-channel group and 2048 chunks: every tile of a row waits on a
    long chain of predecessors in both directions."""
    B, T, C = 1, 65536, 32
    w, u, k, v, gy = inputs.training_inputs(B, T, C, seed=8, k_std=3.0, d_lo=-9.0, d_hi=0.0)
    check_all(oracle, wkv, w, u, k, v, gy, what="deep chain")


def test_bf16_forward(oracle, wkv, scan_mode):
    B, T, C = 2, 777, 136
    w, u, k, v, _ = inputs.training_inputs(B, T, C, seed=9, k_std=5.0, d_lo=-8.0, d_hi=1.0, kv_dtype="bf16")
    y = wkv.forward(*cuda(w, u, k, v))
    torch.cuda.synchronize()
    check_y(oracle, w, u, k, v, y, "bf16", tol=TOL_BF16)
    # far inside the loose bf16 tolerance: the oracle sees the same rounded inputs
    check_y(oracle, w, u, k, v, y, "bf16 (fp32-level)")


BF16_SHAPES = [(1, 1, 8), (2, 33, 136), (3, 200, 96), (1, 1000, 40), (2, 513, 384)]


@pytest.mark.parametrize("B,T,C", BF16_SHAPES, ids=[f"B{b}T{t}C{c}" for b, t, c in BF16_SHAPES])
def test_bf16_backward(oracle, wkv, scan_mode, B, T, C):
    """bf16 k, v, gy with fp32 arithmetic and fp32 gradients: the oracle sees
    the same rounded inputs, so the gradients meet the fp32 tolerance.  The
    chunked scan takes fp32 inputs only and refuses before launching."""
    w, u, k, v, gy = inputs.training_inputs(B, T, C, seed=400 + B + T + C, k_std=3.0, kv_dtype="bf16")
    if scan_mode == "chunked":
        with pytest.raises(wkv.WKVError) as exc:
            wkv.backward(*cuda(w, u, k, v, gy))
        assert exc.value.status == 2
        return
    for use_ckpt in (True, False):
        check_all(oracle, wkv, w, u, k, v, gy, use_ckpt=use_ckpt, what=f"bf16 ckpt={use_ckpt}")


def test_bf16_backward_agrees_with_fp32_of_rounded_inputs(wkv):
    """The bf16 call equals the fp32 call on the same rounded values bit for
    bit: the only difference is the staged type, and widening bf16 to fp32
    is exact (one run per column, so both calls split the columns alike)."""
    w, u, k, v, gy = inputs.training_inputs(4, 600, 256, seed=410, k_std=3.0, kv_dtype="bf16")
    try:
        wkv.set_max_runs(1)
        a = run_fwd_bwd(wkv, w, u, k, v, gy)
        b = run_fwd_bwd(wkv, w, u, k.float(), v.float(), gy.float())
    finally:
        wkv.set_max_runs(0)
    for x, y_, n in zip(a, b, ("y", "ckpt", "gw", "gu", "gk", "gv")):
        assert torch.equal(x, y_), n


def _both_modes(wkv, w, u, k, v, gy, max_runs=0):
    res = {}
    try:
        wkv.set_max_runs(max_runs)
        for mode in ("chunked", "sequential"):
            wkv.set_scan_mode(mode)
            res[mode] = run_fwd_bwd(wkv, w, u, k, v, gy)
    finally:
        wkv.set_scan_mode("auto")
        wkv.set_max_runs(0)
    return res["chunked"], res["sequential"]


def test_scan_modes_agree_bitwise(oracle, wkv):
    """With one run per column, the sequential walk carries the state across
    chunk boundaries with the chunked scan's combine, in the same order, and
    computes a chunk's outputs with the same fixed-scale arithmetic: on
    inputs where every chunk stays on the fixed scale, y and the checkpoints
    agree bit for bit.  The gradients add a chunk's carried adjoint in
    another order: equal to rounding."""
    w, u, k, v, gy = inputs.training_inputs(8, 1000, 768, seed=42, k_std=2.0, d_lo=-6.0, d_hi=2.0)
    a, b = _both_modes(wkv, w, u, k, v, gy, max_runs=1)
    assert torch.equal(a[0], b[0]), "y"
    assert torch.equal(a[1], b[1]), "ckpt"
    _pairs(oracle, w, u, k, v, gy, a, b)


def _pairs(oracle, w, u, k, v, gy, a, b):
    """The two strategies' results against each other (both fp32
    evaluations: the floor is twice the float32 evaluation's error)."""
    check_pair_y(oracle, w, u, k, v, b[0], a[0], "y sequential vs chunked")
    check_pair_grads(oracle, w, u, k, v, gy, dict(zip(("gw", "gu", "gk", "gv"), b[2:])),
                     dict(zip(("gw", "gu", "gk", "gv"), a[2:])), "sequential vs chunked")


def test_scan_modes_agree_runs(oracle, wkv):
    """At the 169M layer shape each column's walk is split into several runs
    (one-warp CTAs exchanging their summaries through the workspace): both
    strategies match the oracle and each other."""
    B, T, C = 8, 1000, 768
    w, u, k, v, gy = inputs.training_inputs(B, T, C, seed=41, k_std=3.0, d_lo=-6.0, d_hi=2.0)
    a, b = _both_modes(wkv, w, u, k, v, gy)
    _pairs(oracle, w, u, k, v, gy, a, b)
    cs = sample_channels(C, 24, 41)
    ws, us, ks, vs, gs = w[cs], u[cs], k[:, :, cs].contiguous(), v[:, :, cs].contiguous(), gy[:, :, cs].contiguous()
    cst = torch.as_tensor(cs, device="cuda")
    check_y(oracle, ws, us, ks, vs, b[0].index_select(2, cst), "sequential")
    check_grads(oracle, ws, us, ks, vs, gs, dict(gk=b[4].index_select(2, cst), gv=b[5].index_select(2, cst),
                                                 gw=b[2].index_select(0, cst), gu=b[3].index_select(0, cst)),
                "sequential")


# ------------------------------------------------------------ named workloads
def test_workload_tiny(oracle, wkv):
    w, u, k, v, gy = inputs.workload_inputs("tiny")
    y, _ = check_all(oracle, wkv, w, u, k, v, gy, what="tiny")
    assert_close(y, oracle.forward_direct(w, u, k, v), TOL_Y, "tiny y vs direct form",
                 emu=emu.forward_recurrent(w, u, k, v))


def test_workload_l169m_full(oracle, wkv):
    w, u, k, v, gy = inputs.workload_inputs("l169m")
    check_all(oracle, wkv, w, u, k, v, gy, what="l169m")


def _sampled(oracle, wkv, name, nchan, seed):
    w, u, k, v, gy = inputs.workload_inputs(name)
    wl = inputs.WORKLOADS[name]
    cs = sample_channels(wl.C, nchan, seed)
    ws, us, ks, vs = w[cs], u[cs], k[:, :, cs].contiguous(), v[:, :, cs].contiguous()
    cst = torch.as_tensor(cs, device="cuda")
    if wl.backward:
        y, _, gw, gu, gk, gv = run_fwd_bwd(wkv, w, u, k, v, gy)
        check_grads(oracle, ws, us, ks, vs, gy[:, :, cs].contiguous(),
                    dict(gk=gk.index_select(2, cst), gv=gv.index_select(2, cst), gw=gw.index_select(0, cst),
                         gu=gu.index_select(0, cst)), name)
    else:
        y = wkv.forward(*cuda(w, u, k, v))
        torch.cuda.synchronize()
    check_y(oracle, ws, us, ks, vs, y.index_select(2, cst), name, tol=TOL_BF16 if wl.kv_dtype == "bf16" else TOL_Y)


def test_workload_l1b5_sampled(oracle, wkv):
    _sampled(oracle, wkv, "l1b5", 48, 11)


def test_workload_long_sampled(oracle, wkv):
    _sampled(oracle, wkv, "long", 48, 12)


def test_workload_l169m_bf16_sampled(oracle, wkv):
    _sampled(oracle, wkv, "l169m_bf16", 48, 13)
