"""GPU parity of the backward pass from a carried state with a gradient on
the end state (wkv_backward_with_state), through the C ABI, against the
float64 oracle (oracle.backward_state, pinned by
tests/oracle_pins.py::pin_backward_state), and of a sequence's backward cut
into segments chained through those gradients (the time split's backward,
its ranks run in turn on one device) against one call over the whole
sequence."""
import numpy as np
import pytest
import torch

import fp32_emulation as emu
from checks import check_grads, check_pair_grads
from parity import TOL_GRAD, assert_close, cuda, to_np
from rwkv_linear_attention_backward_b300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def wkv():
    from rwkv_linear_attention_backward_b300 import binding

    return binding


@pytest.fixture(scope="module")
def tsplit():
    from rwkv_linear_attention_backward_b300 import tsplit

    return tsplit


@pytest.mark.parametrize("B,P,T,C", [(2, 40, 333, 96), (1, 7, 1000, 32), (3, 64, 64, 129)])
def test_backward_with_state_vs_oracle(oracle, wkv, scan_mode, B, P, T, C):
    """A segment after a P-token prefix (its state given) with a gradient on
    its end state from later tokens: gk, gv, gw, gu and the gradient of the
    start state against the oracle handed the same fp32 state."""
    w, u, k, v, gy = inputs.training_inputs(B, P + T, C, seed=800 + T, k_std=1.0)
    sin = torch.tensor(np.stack(oracle.state(w, k[:, :P], v[:, :P], P)), dtype=torch.float32)
    ks, vs, gs = (x[:, P:].contiguous() for x in (k, v, gy))
    wc, uc, kc, vc, gc, sc = cuda(w, u, ks, vs, gs, sin)
    if scan_mode == "chunked":
        with pytest.raises(wkv.WKVError) as exc:
            wkv.backward_with_state(wc, uc, kc, vc, gc, sc)
        assert exc.value.status == 2
        return
    _, s_out, ckpt = wkv.forward_with_state(wc, uc, kc, vc, state_in=sc, want_ckpt=True)
    torch.cuda.synchronize()
    g = torch.Generator().manual_seed(801)
    gend = torch.stack([torch.randn(B, C, generator=g) * 0.3, torch.randn(B, C, generator=g) * 0.3,
                        s_out[2].cpu()])  # written at the end state's own scale
    sin64 = tuple(sin.double().numpy())
    ge = gend.double().numpy()
    aend = (ge[0] * np.exp(-ge[2]), ge[1] * np.exp(-ge[2]))
    ow, ou, ok, ov, (ga, gb) = oracle.backward_state(w, u, ks, vs, gs, sin64, aend)
    evs = emu.evaluations(lambda *x: emu.backward(*x[:5], state_in=x[5], adj_end=x[6]), w, u, ks, vs, gs, sin64,
                          aend)
    eo = {n: [e[n] for e in evs] for n in evs[0]}
    for use_ckpt in (True, False):
        gw, gu, gk, gv, gin = wkv.backward_with_state(wc, uc, kc, vc, gc, sc, gend.cuda(),
                                                      ckpt=ckpt if use_ckpt else None)
        torch.cuda.synchronize()
        what = f"B{B}P{P}T{T}C{C} ckpt={use_ckpt}"
        for g, o, n in ((gk, ok, "gk"), (gv, ov, "gv"), (gw, ow, "gw"), (gu, ou, "gu")):
            assert_close(g, o, TOL_GRAD, f"{what} {n}", emu=eo[n])
        gi = to_np(gin)
        assert np.array_equal(gi[2], sin64[2]), f"{what}: pp plane of the start-state gradient"
        sp = np.exp(sin64[2])
        assert_close(gi[0], ga * sp, TOL_GRAD, f"{what} g_num of the start state", emu=[x * sp for x in eo["ga"]])
        assert_close(gi[1], gb * sp, TOL_GRAD, f"{what} g_den of the start state", emu=[x * sp for x in eo["gb"]])


def test_without_states_is_plain_backward(wkv, scan_mode):
    if scan_mode == "chunked":
        return
    w, u, k, v, gy = cuda(*inputs.training_inputs(2, 500, 160, seed=810, k_std=2.0))
    _, ckpt = wkv.forward(w, u, k, v, want_ckpt=True)
    a = wkv.backward(w, u, k, v, gy, ckpt=ckpt)
    b = wkv.backward_with_state(w, u, k, v, gy, ckpt=ckpt, want_gstate_in=False)
    torch.cuda.synchronize()
    assert b[4] is None
    for x, y, n in zip(a, b[:4], ("gw", "gu", "gk", "gv")):
        assert torch.equal(x, y), n


def test_summary_pass_is_the_start_gradient(oracle, wkv, scan_mode):
    """The summary pass (gk, gv not computed) gives the start state's
    gradient of the full pass, with and without an end gradient."""
    if scan_mode == "chunked":
        return
    B, P, T, C = 2, 40, 700, 96
    w, u, k, v, gy = inputs.training_inputs(B, P + T, C, seed=830, k_std=2.0)
    sin = torch.tensor(np.stack(oracle.state(w, k[:, :P], v[:, :P], P)), dtype=torch.float32)
    ks, vs, gs = (x[:, P:].contiguous() for x in (k, v, gy))
    wc, uc, kc, vc, gc, sc = cuda(w, u, ks, vs, gs, sin)
    _, s_out, ckpt = wkv.forward_with_state(wc, uc, kc, vc, state_in=sc, want_ckpt=True)
    g = torch.Generator().manual_seed(831)
    gend = torch.stack([torch.randn(B, C, generator=g) * 0.3, torch.randn(B, C, generator=g) * 0.3,
                        s_out[2].cpu()]).cuda()
    sin64 = tuple(sin.double().numpy())
    sp = np.exp(sin64[2])
    for ge in (None, gend):
        full = wkv.backward_with_state(wc, uc, kc, vc, gc, sc, ge, ckpt=ckpt)[4]
        for ck in (ckpt, None):
            summ = wkv.backward_with_state(wc, uc, kc, vc, gc, sc, ge, ckpt=ck, summary=True)
            torch.cuda.synchronize()
            assert summ[0] is None and summ[2] is None
            gi = to_np(summ[4])
            assert np.array_equal(gi[2], sin64[2])
            aend = None
            if ge is not None:
                gn = ge.double().cpu().numpy()
                aend = (gn[0] * np.exp(-gn[2]), gn[1] * np.exp(-gn[2]))
            _, _, _, _, (ga, gb) = oracle.backward_state(w, u, ks, vs, gs, sin64, aend)
            evs = emu.evaluations(lambda *x: emu.backward(*x[:5], state_in=x[5], adj_end=x[6]), w, u, ks, vs, gs,
                                  sin64, aend)
            what = f"summary end={ge is not None} ckpt={ck is not None}"
            assert_close(gi[0], ga * sp, TOL_GRAD, f"{what} g_num", emu=[e["ga"] * sp for e in evs])
            assert_close(gi[1], gb * sp, TOL_GRAD, f"{what} g_den", emu=[e["gb"] * sp for e in evs])
            assert_close(gi[0], to_np(full)[0], TOL_GRAD, f"{what} g_num vs the full pass",
                         emu=[e["ga"] * sp for e in evs], ref=ga * sp, pair=True)


def test_adjoint_fold_kernel(oracle, wkv):
    """Segments' own start-state gradients (the oracle's, with no end
    gradient, rounded to fp32) folded on the device after a gradient on the
    last end state give the oracle's start-state gradient of the first
    segment with everything after it; n = 0 returns the end gradient."""
    B, C, T = 3, 70, 400
    w, u, k, v, gy = inputs.training_inputs(B, T, C, seed=840, k_std=2.0, d_lo=-6.0, d_hi=1.0)
    cuts = [0, 10, 10, 150, 399, 400]
    segs = list(zip(cuts[:-1], cuts[1:]))
    lengths = [b - a for a, b in segs]
    starts = [oracle.state(w, k, v, a) if a > 0 else None for a, _ in segs]
    pp_end = oracle.state(w, k, v, T)[2]
    g = np.random.default_rng(841)
    ga_end, gb_end = g.normal(0, 0.3, (B, C)), g.normal(0, 0.3, (B, C))
    adj = []
    for (a, b), st in zip(segs, starts):
        if st is None:  # the first segment starts empty: its pp plane is the empty state's
            st = (np.zeros((B, C)), np.zeros((B, C)), np.full((B, C), -1e38))
        _, _, _, _, (sa, sb) = oracle.backward_state(w, u, k[:, a:b], v[:, a:b], gy[:, a:b],
                                                     None if a == 0 else st, None)
        adj.append(np.stack([sa * np.exp(st[2]), sb * np.exp(st[2]), st[2]]))
    gend = np.stack([ga_end * np.exp(pp_end), gb_end * np.exp(pp_end), pp_end])
    dev = lambda x: torch.tensor(np.asarray(x), dtype=torch.float32).cuda()  # noqa: E731
    # the start gradient of segment 1 (tokens 10..) with everything after it
    recs = dev(np.stack(adj[1:]))
    out = wkv.adjoint_fold(w.cuda(), recs, lengths[1:], dev(gend))
    none = wkv.adjoint_fold(w.cuda(), torch.empty((0, 3, B, C), device="cuda"), [], dev(gend))
    torch.cuda.synchronize()
    _, _, _, _, (ra, rb) = oracle.backward_state(w, u, k[:, 10:], v[:, 10:], gy[:, 10:], starts[1],
                                                 (ga_end, gb_end))
    o = to_np(out)
    sp = np.exp(starts[1][2])
    assert np.array_equal(o[2], to_np(dev(starts[1][2])))
    fe = emu.adjoint_fold(w, recs.cpu(), lengths[1:], dev(gend).cpu())
    assert_close(o[0], ra * sp, TOL_GRAD, "fold g_num", emu=fe[0])
    assert_close(o[1], rb * sp, TOL_GRAD, "fold g_den", emu=fe[1])
    assert torch.equal(none, dev(gend))


CUTS = [[0, 200, 533], [0, 100, 101, 300, 533], [0, 32, 64, 533]]


@pytest.mark.parametrize("cuts", CUTS, ids=["2seg", "4seg_ragged", "3seg_aligned"])
def test_segments_backward_give_the_whole(oracle, wkv, tsplit, scan_mode, cuts):
    """The time split's steps on one device: forward start states by the
    fold; each segment's summary pass (its own start-state gradient); each
    segment's end gradient by the fold of the later ones; then the full
    backward passes, which on several devices run at the same time: the
    whole sequence's gradients."""
    if scan_mode == "chunked":
        return
    B, T, C = 2, cuts[-1], 96
    w, u, k, v, gy = inputs.training_inputs(B, T, C, seed=820 + len(cuts), k_std=2.0)
    wc, uc, kc, vc, gc = cuda(w, u, k, v, gy)
    segs = list(zip(cuts[:-1], cuts[1:]))
    part = [tuple(x[:, a:b].contiguous() for x in (kc, vc, gc)) for a, b in segs]
    states = torch.stack([tsplit.segment_state(wc, uc, kk, vv) for kk, vv, _ in part])
    lengths = [b - a for a, b in segs]
    starts = [tsplit.start_state(wc, states, lengths, r) for r in range(len(segs))]
    own = torch.stack([wkv.backward_with_state(wc, uc, kk, vv, gg, starts[r], summary=True)[4]
                       for r, (kk, vv, gg) in enumerate(part)])
    gw = torch.zeros(C, device="cuda", dtype=torch.float64)
    gu = torch.zeros_like(gw)
    gks, gvs = [None] * len(segs), [None] * len(segs)
    for r, (kk, vv, gg) in enumerate(part):
        g_end = tsplit.end_gradient(wc, own, lengths, r)
        w_r, u_r, gks[r], gvs[r], _ = wkv.backward_with_state(wc, uc, kk, vv, gg, starts[r], g_end)
        gw += w_r.double()
        gu += u_r.double()
    torch.cuda.synchronize()
    split = dict(gk=torch.cat(gks, dim=1), gv=torch.cat(gvs, dim=1), gw=gw, gu=gu)
    check_grads(oracle, w, u, k, v, gy, split, f"{cuts}")
    whole = wkv.backward(wc, uc, kc, vc, gc)
    torch.cuda.synchronize()
    check_pair_grads(oracle, w, u, k, v, gy, dict(gk=split["gk"]), dict(gk=whole[2]), f"{cuts} vs one call")
