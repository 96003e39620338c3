"""GPU parity of the forward pass that continues from a carried state and
returns the state after its last token (the prefill -> decode handoff),
through the C ABI, against the float64 oracle (oracle.forward_state, pinned
by tests/oracle_pins.py::pin_forward_state_split)."""
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


def _split(B, P, T, C, seed, kv_dtype="f32", k_std=2.0):
    """Inputs of P + T tokens, cut after P: (w, u, k, v of the first P, k, v of the last T)."""
    w, u, k, v, _ = inputs.training_inputs(B, P + T, C, seed=seed, k_std=k_std, kv_dtype=kv_dtype)
    return w, u, k[:, :P].contiguous(), v[:, :P].contiguous(), k[:, P:].contiguous(), v[:, P:].contiguous()


def _planes(state):
    return torch.tensor(np.stack(state), dtype=torch.float32)


SHAPES = [(1, 1, 5), (2, 33, 129), (3, 200, 100), (1, 1000, 32), (2, 513, 384)]


@pytest.mark.parametrize("B,T,C", SHAPES, ids=[f"B{b}T{t}C{c}" for b, t, c in SHAPES])
def test_forward_from_state(oracle, wkv, scan_mode, B, T, C):
    """Continuing from the exact state of a 57-token prefix (the oracle's
    direct-sum state) gives the oracle's outputs and final state."""
    w, u, kp, vp, k, v = _split(B, 57, T, C, seed=300 + B + T + C)
    sin = oracle.state(w, kp, vp, 57)
    y, sout = wkv.forward_with_state(*cuda(w, u, k, v), state_in=cuda(_planes(sin))[0])
    torch.cuda.synchronize()
    yo, (no, do, po) = oracle.forward_state(w, u, k, v, sin)
    fe = emu.forward(w, u, k, v, state_in=sin)
    assert_close(y, yo, TOL_Y, "y", emu=fe["y"])
    s = to_np(sout)
    assert_state_close(s[0], s[1], s[2], no, do, po, TOL_Y, "state out", emu_sums=(fe["a"], fe["b"]))


def test_forward_from_state_bf16(oracle, wkv, scan_mode):
    w, u, kp, vp, k, v = _split(2, 100, 777, 136, seed=310, kv_dtype="bf16", k_std=5.0)
    sin = oracle.state(w, kp, vp, 100)
    y, sout = wkv.forward_with_state(*cuda(w, u, k, v), state_in=cuda(_planes(sin))[0])
    torch.cuda.synchronize()
    yo, (no, do, po) = oracle.forward_state(w, u, k, v, sin)
    fe = emu.forward(w, u, k, v, state_in=sin)
    assert_close(y, yo, TOL_BF16, "bf16 y", emu=fe["y"])
    s = to_np(sout)
    assert_state_close(s[0], s[1], s[2], no, do, po, TOL_Y, "bf16 state out", emu_sums=(fe["a"], fe["b"]))


@pytest.mark.parametrize("t0", [1, 32, 100, 699])
def test_split_matches_whole(oracle, wkv, scan_mode, t0):
    """A sequence run in two calls, the second continuing from the first's
    state, gives the outputs of one call over the whole sequence and ends in
    the whole sequence's last checkpoint state."""
    B, T, C = 2, 700, 160
    w, u, k, v, _ = inputs.training_inputs(B, T, C, seed=320 + t0, k_std=3.0)
    wc, uc, kc, vc = cuda(w, u, k, v)
    y, ckpt = wkv.forward(wc, uc, kc, vc, want_ckpt=True)
    y1, s1 = wkv.forward_with_state(wc, uc, kc[:, :t0].contiguous(), vc[:, :t0].contiguous())
    y2, s2 = wkv.forward_with_state(wc, uc, kc[:, t0:].contiguous(), vc[:, t0:].contiguous(), state_in=s1)
    torch.cuda.synchronize()
    fe = emu.forward(w, u, k, v)
    assert_close(torch.cat([y1, y2], dim=1), y, TOL_Y, "split vs whole", emu=fe["y"],
                 ref=oracle.forward_recurrent(w, u, k, v), pair=True)
    nch = -(-T // wkv.chunk_len())
    last = to_np(ckpt).reshape(3, nch, B, C)[:, nch - 1]
    s = to_np(s2)
    n, d, p = oracle.state(w, k, v, T)
    assert_state_close(s[0], s[1], s[2], last[0], last[1], last[2], TOL_Y, "state after both calls",
                       emu_sums=(fe["a"], fe["b"]), oracle=(n, d, p))
    assert_state_close(s[0], s[1], s[2], n, d, p, TOL_Y, "state after both calls vs oracle",
                       emu_sums=(fe["a"], fe["b"]))


def test_empty_state_is_forward(wkv, scan_mode):
    """No state in is wkv_forward, bit for bit; the state out is the last
    checkpoint entry, bit for bit."""
    B, T, C = 3, 333, 96
    w, u, k, v = cuda(*inputs.training_inputs(B, T, C, seed=330, k_std=2.0)[:4])
    y, ckpt = wkv.forward(w, u, k, v, want_ckpt=True)
    y2, s2, ckpt2 = wkv.forward_with_state(w, u, k, v, want_ckpt=True)
    torch.cuda.synchronize()
    assert torch.equal(y, y2) and torch.equal(ckpt, ckpt2)
    nch = -(-T // wkv.chunk_len())
    assert torch.equal(s2, ckpt.reshape(3, nch, B, C)[:, nch - 1])


def test_prefill_then_decode(oracle, wkv):
    """Prefill T tokens with the parallel form, then decode 20 more tokens
    one by one with wkv_decode_step from the returned state: the decode
    outputs match the oracle's decode steps from the oracle's state after
    the same T tokens."""
    B, T, C, n = 4, 300, 256, 20
    w, u, k, v, _ = inputs.training_inputs(B, T + n, C, seed=340, k_std=2.0)
    wc, uc = cuda(w, u)
    _, sout = wkv.forward_with_state(wc, uc, *cuda(k[:, :T].contiguous(), v[:, :T].contiguous()))
    num, den, pp = (sout[i].clone().unsqueeze(0) for i in range(3))  # one layer: [1, B, C]
    g = torch.Generator().manual_seed(341)
    on, od, op = (a[None] for a in oracle.state(w, k, v, T))
    ea, eb = (x[None] for x in emu.sums_after(w, k, v, [T])[0])
    for t in range(T, T + n):
        x, xp, r = (torch.randn(1, B, C, generator=g) for _ in range(3))
        mu = [torch.rand(1, C, generator=g) for _ in range(3)]
        kt, vt = k[:, t][None].contiguous(), v[:, t][None].contiguous()
        y, _, _, _ = wkv.decode_step(*cuda(x, xp, mu[0], mu[1], mu[2], r, kt, vt, w[None], u[None]), num, den, pp)
        yo, on, od, op, _, _, _ = oracle.decode_step(x, xp, mu[0], mu[1], mu[2], r, kt, vt, w[None], u[None],
                                                     on, od, op)
        ye, ea, eb, _, _, _ = emu.decode_step(x, xp, mu[0], mu[1], mu[2], r, kt, vt, w[None], u[None], ea, eb)
        torch.cuda.synchronize()
        assert_close(y, yo, TOL_Y, f"decode step {t - T}", emu=ye)
    assert_state_close(to_np(num)[0], to_np(den)[0], to_np(pp)[0], on[0], od[0], op[0], TOL_Y, "final state",
                       emu_sums=(ea[0], eb[0]))
