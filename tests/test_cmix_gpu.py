"""GPU parity of channel mixing's pointwise steps (squared ReLU between the
key and value projections, the sigmoid gate after the value projection, and
both backward passes), through the C ABI, against the float64 oracle
(oracle.sqrelu / sqrelu_backward / cmix_gate / cmix_gate_backward, pinned by
tests/oracle_pins.py::pin_channel_mix).

Sizes cover n < 4, ragged tails of the 16-byte path, misaligned pointers
(the one-per-thread path, which must agree bit for bit), in-place calls and
the full 169M-layer shapes."""
import pytest
import torch

import fp32_emulation as emu
from parity import TOL_Y, assert_close, cuda
from rwkv_linear_attention_backward_b300 import inputs

pytestmark = pytest.mark.gpu

TOL = 1e-6  # one or two fp32 roundings per element (sigmoid within a few ulp)


@pytest.fixture(scope="module")
def wkv():
    from rwkv_linear_attention_backward_b300 import binding

    return binding


def _all(wkv, k, ga, r, vk, gout):
    a = wkv.channel_mix_sqrelu(k)
    gk = wkv.channel_mix_sqrelu_backward(k, ga)
    out = wkv.channel_mix_gate(r, vk)
    gr, gvk = wkv.channel_mix_gate_backward(r, vk, gout)
    torch.cuda.synchronize()
    return a, gk, out, gr, gvk


def _close(got, want, em, what, tol=TOL):
    assert_close(got, want, tol, what, emu=em)


def _check(oracle, got, k, ga, r, vk, gout, what):
    a, gk, out, gr, gvk = got
    _close(a, oracle.sqrelu(k), emu.sqrelu(k), f"{what} a")
    _close(gk, oracle.sqrelu_backward(k, ga), emu.sqrelu_backward(k, ga), f"{what} gk")
    _close(out, oracle.cmix_gate(r, vk), emu.cmix_gate(r, vk), f"{what} out")
    ogr, ogvk = oracle.cmix_gate_backward(r, vk, gout)
    egr, egvk = emu.cmix_gate_backward(r, vk, gout)
    _close(gr, ogr, egr, f"{what} gr")
    _close(gvk, ogvk, egvk, f"{what} gvk")


SIZES = [1, 3, 4, 5, 7, 1000, 4097, (1 << 20) + 3]


@pytest.mark.parametrize("n", SIZES)
def test_sizes(oracle, wkv, n):
    g = torch.Generator().manual_seed(600 + n % 997)
    k, ga, r, vk, gout = (torch.randn(n, generator=g) * 2.0 for _ in range(5))
    got = _all(wkv, *cuda(k, ga, r, vk, gout))
    _check(oracle, got, k, ga, r, vk, gout, f"n={n}")


def test_misaligned_matches_aligned_bitwise(wkv):
    """One element off the 16-byte boundary takes the one-per-thread path;
    the arithmetic per element is the same, so the results are the same."""
    n = 10_001
    g = torch.Generator().manual_seed(610)
    host = [torch.randn(n, generator=g) * 3.0 for _ in range(5)]
    aligned = _all(wkv, *cuda(*host))
    bufs = [torch.empty(n + 1, device="cuda") for _ in range(5)]
    for b, h in zip(bufs, host):
        b[1:].copy_(h)
    shifted = _all(wkv, *(b[1:] for b in bufs))
    for x, y, name in zip(aligned, shifted, ("a", "gk", "out", "gr", "gvk")):
        assert torch.equal(x, y), name


def test_in_place(wkv):
    g = torch.Generator().manual_seed(620)
    k, ga, r, vk, gout = cuda(*(torch.randn(4099, generator=g) for _ in range(5)))
    want = _all(wkv, k, ga, r, vk, gout)
    kk = k.clone()
    wkv.channel_mix_sqrelu(kk, out=kk)
    vv = vk.clone()
    wkv.channel_mix_gate(r, vv, out=vv)
    rr, vv2 = r.clone(), vk.clone()
    wkv.channel_mix_gate_backward(rr, vv2, gout, gr=rr, gvk=vv2)
    torch.cuda.synchronize()
    assert torch.equal(kk, want[0]) and torch.equal(vv, want[2])
    assert torch.equal(rr, want[3]) and torch.equal(vv2, want[4])


def test_saturation_and_signs(oracle, wkv):
    """k at and around 0 (the ReLU kink: zero value and gradient at k <= 0),
    r far in both tails (sigmoid 0 and 1, e^{-r} overflowing)."""
    k = torch.tensor([-5.0, -1e-30, -0.0, 0.0, 1e-30, 2.0, 1e4] * 3)
    r = torch.tensor([-200.0, -90.0, -30.0, 0.0, 30.0, 90.0, 200.0] * 3)
    ones = torch.ones_like(k)
    got = _all(wkv, *cuda(k, ones, r, ones * 3.0, ones))
    a, gk, out, gr, gvk = (t.cpu() for t in got)
    assert torch.equal(a[k <= 0], torch.zeros_like(a[k <= 0])) and torch.equal(gk[k <= 0], torch.zeros_like(gk[k <= 0]))
    _check(oracle, got, k, ones, r, ones * 3.0, ones, "saturation")
    assert torch.all(torch.isfinite(gr)) and torch.all(torch.isfinite(out))


def test_workload_cmix_full(oracle, wkv):
    M = inputs.CMIX
    k, ga, r, vk, gout = inputs.cmix_inputs(M.B, M.T, M.C, M.H, seed=M.seed)
    got = _all(wkv, *cuda(k, ga, r, vk, gout))
    _check(oracle, got, k, ga, r, vk, gout, "cmix")
    _close(got[0].view(M.B, M.T, M.H), oracle.sqrelu(k), emu.sqrelu(k), "cmix a shape", tol=TOL_Y)
