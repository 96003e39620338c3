"""GPU parity of the time split of one sequence (tsplit.py): the state-only
pass, wkv_state_fold and the forward pass from the folded state, through
the C ABI, against the float64 oracle (oracle.state_fold, pinned by
tests/oracle_pins.py::pin_state_fold) and against one call over the whole
sequence.  The ranks' steps run one after another on one device (the
all-gather, host logic only, is tests/test_tsplit_host.py)."""
import numpy as np
import pytest
import torch

import fp32_emulation as emu
from parity import TOL_BF16, TOL_Y, assert_close, assert_state_close, cuda, to_np
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


def _segments(tsplit, wkv, w, u, k, v, cuts, state_in=None):
    """Every rank's outputs and end state, the ranks run in turn."""
    segs = list(zip(cuts[:-1], cuts[1:]))
    parts = [(k[:, a:b].contiguous(), v[:, a:b].contiguous()) for a, b in segs]
    states = torch.stack([tsplit.segment_state(w, u, kk, vv) for kk, vv in parts])
    lengths = [b - a for a, b in segs]
    ys, ends = [], []
    for r, (kk, vv) in enumerate(parts):
        start = tsplit.start_state(w, states, lengths, r, state_in)
        y, end = wkv.forward_with_state(w, u, kk, vv, state_in=start)
        ys.append(y)
        ends.append(end)
    torch.cuda.synchronize()
    return torch.cat(ys, dim=1), ends


CUTS = [[0, 1100], [0, 300, 1100], [0, 300, 301, 700, 733, 1100], [0, 32, 64, 96, 1100]]


@pytest.mark.parametrize("cuts", CUTS, ids=["1seg", "2seg", "5seg_ragged", "4seg_aligned"])
def test_segments_give_the_whole_sequence(oracle, wkv, tsplit, scan_mode, cuts):
    B, T, C = 2, 1100, 160
    w, u, k, v, _ = inputs.training_inputs(B, T, C, seed=700 + len(cuts), k_std=2.5)
    wc, uc, kc, vc = cuda(w, u, k, v)
    y, ends = _segments(tsplit, wkv, wc, uc, kc, vc, cuts)
    y_whole, s_whole = wkv.forward_with_state(wc, uc, kc, vc)
    torch.cuda.synchronize()
    fe = emu.forward(w, u, k, v)
    yo = oracle.forward_recurrent(w, u, k, v)
    assert_close(y, yo, TOL_Y, f"{cuts} y vs oracle", emu=fe["y"])
    assert_close(y, y_whole, TOL_Y, f"{cuts} y vs one call", emu=fe["y"], ref=yo, pair=True)
    n, d, p = oracle.state(w, k, v, T)
    e = to_np(ends[-1])
    assert_state_close(e[0], e[1], e[2], n, d, p, TOL_Y, f"{cuts} end state", emu_sums=(fe["a"], fe["b"]))


def test_segments_after_a_given_state(oracle, wkv, tsplit):
    """The sequence continues a prefix whose state is given: it enters the
    fold as a leading segment of length 0."""
    B, P, T, C = 2, 57, 900, 96
    w, u, k, v, _ = inputs.training_inputs(B, P + T, C, seed=720, k_std=2.5)
    sin = torch.tensor(np.stack(oracle.state(w, k[:, :P], v[:, :P], P)), dtype=torch.float32)
    wc, uc, kc, vc, sc = cuda(w, u, k[:, P:].contiguous(), v[:, P:].contiguous(), sin)
    y, ends = _segments(tsplit, wkv, wc, uc, kc, vc, [0, 250, 251, 900], state_in=sc)
    fe = emu.forward(w, u, k[:, P:], v[:, P:], state_in=sin)
    assert_close(y, oracle.forward_recurrent(w, u, k, v)[:, P:], TOL_Y, "y after a given state", emu=fe["y"])
    n, d, p = oracle.state(w, k, v, P + T)
    e = to_np(ends[-1])
    assert_state_close(e[0], e[1], e[2], n, d, p, TOL_Y, "end state after a given state",
                       emu_sums=(fe["a"], fe["b"]))


def test_segments_bf16(oracle, wkv, tsplit, scan_mode):
    B, T, C = 2, 777, 136
    w, u, k, v, _ = inputs.training_inputs(B, T, C, seed=730, k_std=4.0, kv_dtype="bf16")
    wc, uc, kc, vc = cuda(w, u, k, v)
    y, _ = _segments(tsplit, wkv, wc, uc, kc, vc, [0, 100, 400, 777])
    yo, ye = oracle.forward_recurrent(w, u, k, v), emu.forward_recurrent(w, u, k, v)
    assert_close(y, yo, TOL_BF16, "bf16 segments y", emu=ye)
    assert_close(y, yo, TOL_Y, "bf16 segments y (fp32-level)", emu=ye)


def test_state_only_pass_matches_full_pass(oracle, wkv, scan_mode):
    B, T, C = 3, 500, 200
    w, u, k, v, _ = inputs.training_inputs(B, T, C, seed=740, k_std=3.0)
    wc, uc, kc, vc = cuda(w, u, k, v)
    y0, s_none, ck_none = wkv.forward_with_state(wc, uc, kc, vc, want_y=False, want_ckpt=True)
    y1, s_full, ck_full = wkv.forward_with_state(wc, uc, kc, vc, want_ckpt=True)
    torch.cuda.synchronize()
    assert y0 is None
    a, b = to_np(s_none), to_np(s_full)
    assert_state_close(a[0], a[1], a[2], b[0], b[1], b[2], TOL_Y, "state-only vs full pass")
    n, d, p = oracle.state(w, k, v, T)
    fe = emu.forward(w, u, k, v)
    assert_state_close(a[0], a[1], a[2], n, d, p, TOL_Y, "state-only vs oracle", emu_sums=(fe["a"], fe["b"]))
    assert_close(ck_none, ck_full, TOL_Y, "checkpoints")


def test_state_fold_kernel(oracle, wkv):
    """Segments' own states (the oracle's, rounded to fp32) folded on the
    device against the oracle's fold, including an empty segment; n = 0 is
    the empty state."""
    B, C = 3, 70
    T = 300
    w, u, k, v, _ = inputs.training_inputs(B, T, C, seed=750, k_std=3.0, d_lo=-7.0, d_hi=1.5)
    cuts = [0, 10, 10, 150, 299, 300]
    segs = list(zip(cuts[:-1], cuts[1:]))
    states = np.stack([np.stack(oracle.state(w, k[:, a:b], v[:, a:b], b - a)) for a, b in segs])
    lengths = [b - a for a, b in segs]
    st = torch.tensor(states, dtype=torch.float32)
    out = wkv.state_fold(w.cuda(), st.cuda(), lengths)
    empty = wkv.state_fold(w.cuda(), st[:0].cuda(), [])
    torch.cuda.synchronize()
    n, d, p = oracle.state_fold(w, st.double().numpy(), lengths)
    g = to_np(out)
    assert_state_close(g[0], g[1], g[2], n, d, p, TOL_Y, "fold vs oracle")
    n2, d2, p2 = oracle.state(w, k, v, T)
    fe = emu.forward(w, u, k, v)
    assert_state_close(g[0], g[1], g[2], n2, d2, p2, TOL_Y, "fold vs whole", emu_sums=(fe["a"], fe["b"]))
    e = to_np(empty)
    assert np.all(e[0] == 0) and np.all(e[1] == 0) and np.all(e[2] < -1e37)
