"""The seeded synthetic inputs (rwkv_linear_attention_backward_b300/inputs.py)
that both the CUDA path and the oracle are handed: deterministic per seed,
in the documented shapes and types, bf16 inputs the round-to-nearest-even
of their fp32 draws, and the gate's r drawn apart from the WKV inputs."""
import torch

from rwkv_linear_attention_backward_b300 import inputs


def test_training_inputs_are_seeded():
    a = inputs.training_inputs(2, 33, 17, seed=5, k_std=2.0)
    b = inputs.training_inputs(2, 33, 17, seed=5, k_std=2.0)
    c = inputs.training_inputs(2, 33, 17, seed=6, k_std=2.0)
    assert all(torch.equal(x, y) for x, y in zip(a, b))
    assert not torch.equal(a[2], c[2])
    w, u, k, v, gy = a
    assert w.shape == (17,) and u.shape == (17,) and k.shape == v.shape == gy.shape == (2, 33, 17)
    assert all(t.dtype == torch.float32 for t in a)
    assert torch.all(w > 0) and torch.all(u.abs() <= 1)


def test_bf16_inputs_are_the_rounded_fp32_draws():
    f = inputs.training_inputs(3, 40, 9, seed=11, k_std=3.0)
    h = inputs.training_inputs(3, 40, 9, seed=11, k_std=3.0, kv_dtype="bf16")
    for x, y in zip(f[2:], h[2:]):
        assert y.dtype == torch.bfloat16 and torch.equal(x.to(torch.bfloat16), y)
    assert torch.equal(f[0], h[0]) and torch.equal(f[1], h[1])  # w, u stay fp32


def test_named_workloads():
    for name, wl in inputs.WORKLOADS.items():
        assert wl.elements == wl.B * wl.T * wl.C and wl.kv_dtype in ("f32", "bf16")
    assert inputs.WORKLOADS["l169m_gated"].gated and not inputs.WORKLOADS["l169m"].gated
    assert len(inputs.workload_inputs("tiny")) == 5


def test_gate_and_channel_mix_inputs():
    r1 = inputs.gate_inputs(2, 10, 6, seed=4)
    r2 = inputs.gate_inputs(2, 10, 6, seed=4)
    assert torch.equal(r1, r2) and r1.shape == (2, 10, 6)
    assert inputs.gate_inputs(2, 10, 6, seed=4, kv_dtype="bf16").dtype == torch.bfloat16
    k, ga, r, vk, gout = inputs.cmix_inputs(2, 5, 3, 12, seed=8)
    assert k.shape == ga.shape == (2, 5, 12) and r.shape == vk.shape == gout.shape == (2, 5, 3)
    x, x0, mk, mv, mr, gk, gv, gr = inputs.shift_inputs(2, 5, 3, seed=9)
    assert x.shape == (2, 5, 3) and x0.shape == (2, 3) and mk.shape == (3,)
    assert torch.all((mk >= 0) & (mk <= 1))


def test_decode_inputs():
    mk, mv, mr, w, u = inputs.decode_params(2, 8, seed=3)
    assert mk.shape == w.shape == (2, 8) and torch.all(w > 0)
    a = inputs.decode_step_inputs(2, 3, 8, seed=3, step=0)
    b = inputs.decode_step_inputs(2, 3, 8, seed=3, step=1)
    assert all(t.shape == (2, 3, 8) for t in a) and not torch.equal(a[0], b[0])
    num, den, pp = inputs.initial_state(2, 3, 8)
    assert torch.all(num == 0) and torch.all(den == 0) and torch.all(pp == -1e38)
