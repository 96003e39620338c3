"""Properties of the CUDA path that hold at any size: bitwise run-to-run
reproducibility, causality, agreement of the checkpoint and recompute paths,
workspace reuse, streams, and the bounded-wait error report."""
import pytest
import torch

import fp32_emulation as emu
from checks import check_grads, check_pair_grads, check_pair_y, check_y
from parity import TOL_Y, assert_close, assert_state_close, cuda, to_np
from rwkv_linear_attention_backward_b300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def wkv():
    from rwkv_linear_attention_backward_b300 import binding

    return binding


def _run(wkv, w, u, k, v, gy, ckpt_to_bwd=True):
    y, ckpt = wkv.forward(w, u, k, v, want_ckpt=True)
    g = wkv.backward(w, u, k, v, gy, ckpt=ckpt if ckpt_to_bwd else None)
    torch.cuda.synchronize()
    return (y, ckpt) + tuple(g)


def test_bitwise_reproducible(wkv, scan_mode):
    t = cuda(*inputs.training_inputs(3, 3000, 200, seed=21, k_std=3.0))
    a = _run(wkv, *t)
    for _ in range(3):
        b = _run(wkv, *t)
        for x, y_ in zip(a, b):
            assert torch.equal(x, y_)


def test_checkpoint_and_recompute_agree_bitwise(wkv, scan_mode):
    t = cuda(*inputs.training_inputs(2, 1500, 130, seed=22, k_std=3.0))
    a = _run(wkv, *t, ckpt_to_bwd=True)
    b = _run(wkv, *t, ckpt_to_bwd=False)
    for x, y_ in zip(a[2:], b[2:]):
        assert torch.equal(x, y_)


@pytest.mark.parametrize("t0", [333, 320])
def test_forward_causal(oracle, wkv, scan_mode, t0):
    """y_t depends on tokens <= t only.  Whole chunks before the change are
    bitwise unchanged.  Inside the chunk holding the change, earlier outputs
    share the chunk's exponent reference (its largest k) with the changed
    tokens, so they may move by rounding only."""
    host = inputs.training_inputs(2, 777, 96, seed=23, k_std=2.0)
    w, u, k, v, gy = cuda(*host)
    y = wkv.forward(w, u, k, v)
    k2, v2 = k.clone(), v.clone()
    k2[:, t0:] += 3.0
    v2[:, t0:] -= 1.0
    y2 = wkv.forward(w, u, k2, v2)
    torch.cuda.synchronize()
    L = wkv.chunk_len()
    c0 = (t0 // L) * L  # first token of the chunk holding t0
    assert torch.equal(y[:, :c0], y2[:, :c0])
    if c0 < t0:
        hw, hu, hk, hv = host[:4]
        assert_close(y2[:, c0:t0], y[:, c0:t0], 1e-6, "same-chunk outputs before the change",
                     emu=emu.forward_recurrent(hw, hu, hk, hv)[:, c0:t0],
                     ref=oracle.forward_recurrent(hw, hu, hk, hv)[:, c0:t0], pair=True)
    assert not torch.equal(y[:, t0:], y2[:, t0:])


def test_backward_anticausal(wkv, scan_mode):
    """gk_t, gv_t depend on gy_s for s >= t only."""
    w, u, k, v, gy = cuda(*inputs.training_inputs(2, 777, 96, seed=24, k_std=2.0))
    _, _, _, _, gk, gv = _run(wkv, w, u, k, v, gy)
    t0 = 400
    gy2 = gy.clone()
    gy2[:, :t0] *= -2.0
    _, _, _, _, gk2, gv2 = _run(wkv, w, u, k, v, gy2)
    assert torch.equal(gk[:, t0:], gk2[:, t0:]) and torch.equal(gv[:, t0:], gv2[:, t0:])


def test_k_shift_invariance(oracle, wkv, scan_mode):
    host = inputs.training_inputs(2, 600, 64, seed=25, k_std=2.0)
    w, u, k, v, gy = cuda(*host)
    a = _run(wkv, w, u, k, v, gy)
    b = _run(wkv, w, u, k + 30.0, v, gy)
    check_pair_y(oracle, *host[:4], b[0], a[0], "y(k+30)")
    names = ("gw", "gu", "gk", "gv")
    check_pair_grads(oracle, *host, dict(zip(names, b[2:])), dict(zip(names, a[2:])), "k+30")
    s = a[4].double().sum(dim=1).abs().max().item()  # sum_t gk_t = 0 per (b, c)
    assert s <= 1e-4 * a[4].abs().max().item() * 600 ** 0.5


def test_workspace_reused_across_shapes(oracle, wkv, scan_mode):
    ws = wkv.Workspace(wkv.backward_workspace_bytes(4, 2000, 300))
    for (B, T, C), seed in (((4, 2000, 300), 1), ((1, 50, 7), 2), ((3, 999, 129), 3), ((4, 2000, 300), 4)):
        w, u, k, v, gy = inputs.training_inputs(B, T, C, seed=seed, k_std=2.0)
        wc, uc, kc, vc, gyc = cuda(w, u, k, v, gy)
        y = wkv.forward(wc, uc, kc, vc, workspace=ws)
        gw, gu, gk, gv = wkv.backward(wc, uc, kc, vc, gyc, workspace=ws)
        torch.cuda.synchronize()
        check_y(oracle, w, u, k, v, y, "reused workspace")
        check_grads(oracle, w, u, k, v, gy, dict(gk=gk, gw=gw), "reused workspace")
        wkv.workspace_check(ws)


def test_side_stream(oracle, wkv, scan_mode):
    w, u, k, v, gy = inputs.training_inputs(2, 400, 80, seed=26)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        tw = cuda(w, u, k, v, gy)
        y = wkv.forward(*tw[:4], stream=s)
        gw, gu, gk, gv = wkv.backward(*tw, stream=s)
    s.synchronize()
    check_y(oracle, w, u, k, v, y, "side stream")
    check_grads(oracle, w, u, k, v, gy, dict(gv=gv), "side stream")


@pytest.mark.parametrize("mode", ["chunked", "sequential", "sequential-chain3"])
@pytest.mark.parametrize("which", ["forward", "backward"])
def test_expired_wait_is_reported(oracle, wkv, which, mode):
    """A chunk whose results are never published (the chunked scan: its
    tiles; the sequential kernels: the summary of the run holding it) makes
    the bounded waits of the CTAs that need them expire: the call reports
    WKV_ERR_TIMEOUT through wkv_workspace_check and the device stays
    usable."""
    B, T, C = 1, 32 * 40, 64
    w, u, k, v, gy = inputs.training_inputs(B, T, C, seed=27)
    tw = cuda(w, u, k, v, gy)
    ws = wkv.Workspace(wkv.backward_workspace_bytes(B, T, C))
    try:
        wkv.set_scan_mode(mode.split("-")[0])
        wkv.set_chain_len(3 if mode.endswith("chain3") else 0)
        wkv.set_wait_budget_ns(2_000_000)  # 2 ms
        wkv.set_skip_chunk(0 if which == "forward" else T // 32 - 1)
        if which == "forward":
            wkv.forward(*tw[:4], workspace=ws)
        else:
            y, ckpt = wkv.forward(*tw[:4], want_ckpt=True)
            wkv.backward(*tw, ckpt=ckpt, workspace=ws)
        with pytest.raises(wkv.WKVError) as exc:
            wkv.workspace_check(ws)
        assert exc.value.status == 6
        # the device-wide record reports it too, once
        with pytest.raises(wkv.WKVError) as exc:
            wkv.sync_status()
        assert exc.value.status == 6
    finally:
        wkv.set_skip_chunk(-1)
        wkv.set_wait_budget_ns(0)
    wkv.workspace_check(ws)  # the records were cleared
    wkv.sync_status()
    try:
        y = wkv.forward(*tw[:4], workspace=ws)
        gw, gu, gk, gv = wkv.backward(*tw, workspace=ws)
        wkv.workspace_check(ws)
        wkv.sync_status()
    finally:
        wkv.set_scan_mode("auto")
        wkv.set_chain_len(0)
    check_y(oracle, w, u, k, v, y, "after timeout")
    check_grads(oracle, w, u, k, v, gy, dict(gk=gk), "after timeout")


@pytest.mark.parametrize("kv_dtype", ["f32", "bf16"])
def test_chained_runs_do_not_depend_on_the_warps(oracle, wkv, kv_dtype):
    """Chained runs: the state before run r is the start state with the
    summaries of runs 0..r-1 folded in left to right, whichever warp walks
    which run, so one warp walking all 67 runs of a column and many warps
    sharing them give the same bits; both match the oracle."""
    B, T, C = 2, 32 * 200, 64
    w, u, k, v, _ = inputs.training_inputs(B, T, C, seed=29, k_std=3.0, d_lo=-7.0, d_hi=1.0, kv_dtype=kv_dtype)
    tw = cuda(w, u, k, v)
    outs = []
    try:
        wkv.set_scan_mode("sequential")
        wkv.set_chain_len(3)
        for runs in (1, 5, 0):
            wkv.set_max_runs(runs)
            outs.append(wkv.forward(*tw, want_ckpt=True))
            torch.cuda.synchronize()
    finally:
        wkv.set_scan_mode("auto")
        wkv.set_chain_len(0)
        wkv.set_max_runs(0)
    for (y, ck), runs in zip(outs[1:], (5, 0)):
        assert torch.equal(y, outs[0][0]), f"y, max runs {runs}"
        assert torch.equal(ck, outs[0][1]), f"checkpoints, max runs {runs}"
    check_y(oracle, w, u, k, v, outs[0][0], f"chained {kv_dtype}")


CHAIN_LENS = [1, 2, 4, 7]


@pytest.mark.parametrize("kv_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("chain", CHAIN_LENS, ids=[f"len{n}" for n in CHAIN_LENS])
def test_chained_run_lengths(oracle, wkv, kv_dtype, chain):
    """Chained runs of 1, 2, 4 and 7 chunks over a ragged sequence (T not a
    multiple of the chunk), with the column's warps each walking several
    runs.  With bf16 inputs the walk moves two chunks per item: runs of one
    chunk make every item a lone chunk, even lengths only full items, odd
    ones a lone last item per phase.  The outputs, the checkpoints at the
    first, a middle and the last chunk boundary, and the state after the
    last token match the oracle."""
    B, T, C = 2, 32 * 37 + 11, 96
    w, u, k, v, _ = inputs.training_inputs(B, T, C, seed=31 + chain, k_std=3.0, d_lo=-7.0, d_hi=1.0,
                                           kv_dtype=kv_dtype)
    tw = cuda(w, u, k, v)
    try:
        wkv.set_scan_mode("sequential")
        wkv.set_chain_len(chain)
        wkv.set_max_runs(4)
        y, ck = wkv.forward(*tw, want_ckpt=True)
        _, state = wkv.forward_with_state(*tw)
        torch.cuda.synchronize()
    finally:
        wkv.set_scan_mode("auto")
        wkv.set_chain_len(0)
        wkv.set_max_runs(0)
    what = f"chained len {chain} {kv_dtype}"
    check_y(oracle, w, u, k, v, y, what)
    nch = -(-T // 32)
    cks = to_np(ck).reshape(3, nch, B, C)
    for j in (0, nch // 2, nch - 1):
        t = min((j + 1) * 32, T)
        ea, eb = emu.sums_after(w, k, v, [t])[0]
        assert_state_close(cks[0, j], cks[1, j], cks[2, j], *oracle.state(w, k, v, t), TOL_Y,
                           f"{what} checkpoint {j}", emu_sums=(ea, eb))
    st = to_np(state)
    ea, eb = emu.sums_after(w, k, v, [T])[0]
    assert_state_close(st[0], st[1], st[2], *oracle.state(w, k, v, T), TOL_Y, f"{what} final state",
                       emu_sums=(ea, eb))


def test_graph_replay_with_new_inputs(wkv, scan_mode):
    """Forward + backward captured once in a CUDA graph and replayed after the
    inputs change in place give the results of direct calls on the new
    inputs (every launch takes a fresh tag on the device, so results carried
    between CTAs by an earlier replay are never taken for the current one)."""
    B, T, C = 2, 700, 160
    a = cuda(*inputs.training_inputs(B, T, C, seed=31, k_std=3.0))
    b = cuda(*inputs.training_inputs(B, T, C, seed=32, k_std=3.0))
    w, u, k, v, gy = (t.clone() for t in a)
    y = torch.empty(B, T, C, device="cuda")
    ck = torch.empty(wkv.checkpoint_floats(B, T, C), device="cuda")
    gw, gu = torch.empty(C, device="cuda"), torch.empty(C, device="cuda")
    gk, gv = torch.empty(B, T, C, device="cuda"), torch.empty(B, T, C, device="cuda")
    wsf = wkv.Workspace(wkv.forward_workspace_bytes(B, T, C))
    wsb = wkv.Workspace(wkv.backward_workspace_bytes(B, T, C))

    def step():
        wkv.forward(w, u, k, v, y=y, ckpt=ck, workspace=wsf)
        wkv.backward(w, u, k, v, gy, ckpt=ck, gw=gw, gu=gu, gk=gk, gv=gv, workspace=wsb)

    step()  # first calls: per-device set-up happens outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for src in (a, b, a, b):
        for dst, s in zip((w, u, k, v, gy), src):
            dst.copy_(s)
        g.replay()
        torch.cuda.synchronize()
        got = [t.clone() for t in (y, ck, gw, gu, gk, gv)]
        ref = _run(wkv, *src)
        for x, r_, n in zip(got, ref, ("y", "ckpt", "gw", "gu", "gk", "gv")):
            assert torch.equal(x, r_), n
    wkv.workspace_check(wsf)
    wkv.workspace_check(wsb)


def test_scan_strategy_by_shape(wkv):
    """The automatic choice is the sequential kernels for every shape; the
    test hook overrides it."""
    for shape in ((8, 1024, 768), (1, 131072, 2560), (1, 64, 64), (16, 4096, 2048)):
        assert wkv.scan_strategy(*shape) == "sequential"
    try:
        wkv.set_scan_mode("chunked")
        assert wkv.scan_strategy(1, 64, 64) == "chunked"
        wkv.set_scan_mode("sequential")
        assert wkv.scan_strategy(16, 4096, 2048) == "sequential"
    finally:
        wkv.set_scan_mode("auto")
    with pytest.raises(wkv.WKVError):
        wkv.scan_strategy(0, 1, 1)
