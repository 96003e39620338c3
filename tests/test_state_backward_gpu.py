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


CUTS = [[0, 200, 533], [0, 100, 101, 300, 533], [0, 32, 64, 533]]


@pytest.mark.parametrize("cuts", CUTS, ids=["2seg", "4seg_ragged", "3seg_aligned"])
def test_segments_backward_give_the_whole(oracle, wkv, tsplit, scan_mode, cuts):
    """The time split's steps on one device: forward start states by the
    fold, then the segments' backward passes last first, each fed the next
    segment's start-state gradient: the whole sequence's gradients."""
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
    g_end = None
    gw = torch.zeros(C, device="cuda", dtype=torch.float64)
    gu = torch.zeros_like(gw)
    gks, gvs = [None] * len(segs), [None] * len(segs)
    for r in reversed(range(len(segs))):
        kk, vv, gg = part[r]
        w_r, u_r, gks[r], gvs[r], g_end = wkv.backward_with_state(wc, uc, kk, vv, gg, starts[r], g_end)
        gw += w_r.double()
        gu += u_r.double()
    torch.cuda.synchronize()
    split = dict(gk=torch.cat(gks, dim=1), gv=torch.cat(gvs, dim=1), gw=gw, gu=gu)
    check_grads(oracle, w, u, k, v, gy, split, f"{cuts}")
    whole = wkv.backward(wc, uc, kc, vc, gc)
    torch.cuda.synchronize()
    check_pair_grads(oracle, w, u, k, v, gy, dict(gk=split["gk"]), dict(gk=whole[2]), f"{cuts} vs one call")
