"""Seeded synthetic inputs shared by the tests, the oracle checks and bench.py.

This module draws random numbers and nothing else: it holds none of the WKV
arithmetic.  Tensors are drawn with a seeded ``torch.Generator`` in a fixed
draw order (documented per function): on the CPU, so the same seed gives the
same values on any machine, except the large decode input pools, which are
drawn on the device that uses them (``decode_pool``).  bf16 tensors are drawn in fp32 and then
rounded to nearest-even by ``Tensor.to(torch.bfloat16)``; the oracle is
handed the rounded values.

Named workloads (sizes and distributions of the training / inference
shapes this library targets):

=========  ==========================================================
name       shape and distributions
=========  ==========================================================
tiny       fwd+bwd fp32, B=1 T=64 C=64; k,v ~ N(0,1); w=exp(d),
           d ~ U(-5,1); u ~ U(-1,1); gy ~ N(0,1)
l169m      fwd+bwd fp32, B=8 T=1024 C=768 (one layer of a 169M RWKV-4);
           k ~ N(0,3^2), v ~ N(0,1); d ~ U(-6,2); u ~ U(-1,1); gy ~ N(0,1)
l1b5       fwd+bwd fp32, B=16 T=4096 C=2048 (1.5B-class layer); as l169m
long       fwd only, bf16 k,v, fp32 state and output, B=1 T=131072
           C=2560; k ~ N(0,5^2), v ~ N(0,1); d ~ U(-8,1); u ~ U(-1,1)
l169m_bf16 fwd+bwd with bf16 k, v, gy (fp32 arithmetic and outputs), the
           l169m shape and distributions
l169m_gated fwd+bwd of the gated output sigmoid(r) * wkv, the l169m shape
           and distributions, r ~ N(0,2^2) (gy is the gated output's
           gradient)
shift      token shift of the training path, fwd+bwd, B=16 T=4096 C=2048;
           x, gxk, gxv, gxr ~ N(0,1); x0 ~ N(0,1); mu_k, mu_v, mu_r ~ U(0,1)
cmix       channel mixing's pointwise steps (squared ReLU, sigmoid gate)
           fwd+bwd at the 169M layer: B=8 T=1024 C=768, hidden H=3072;
           k, ga [B,T,H] ~ N(0,1); r, vk, gout [B,T,C] ~ N(0,1)
decode     RNN decode, L=32 layers, B=256, C=4096, 1024 steps; x, x_prev,
           r, k, v ~ N(0,1); mu_k, mu_v, mu_r ~ U(0,1); d ~ U(-6,2),
           u ~ U(-1,1) per layer; state starts at (0, 0, -1e38)
decode_bf16 as decode, with x, x_prev, r, k, v rounded to bf16 (state,
           parameters and outputs fp32)
=========  ==========================================================
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class TrainingWorkload:
    name: str
    B: int
    T: int
    C: int
    k_std: float
    d_lo: float
    d_hi: float
    kv_dtype: str  # "f32" or "bf16"
    backward: bool
    seed: int
    gated: bool = False  # the output gate sigmoid(r) * wkv (r from gate_inputs, seed + 1)

    @property
    def elements(self) -> int:
        return self.B * self.T * self.C


@dataclass(frozen=True)
class DecodeWorkload:
    name: str
    L: int
    B: int
    C: int
    steps: int
    d_lo: float
    d_hi: float
    seed: int
    token_dtype: str = "f32"  # x, x_prev, r, k, v: "f32" or "bf16" (state and outputs fp32)

    @property
    def elements_per_step(self) -> int:
        return self.L * self.B * self.C


WORKLOADS = {
    "tiny": TrainingWorkload("tiny", 1, 64, 64, 1.0, -5.0, 1.0, "f32", True, 1001),
    "l169m": TrainingWorkload("l169m", 8, 1024, 768, 3.0, -6.0, 2.0, "f32", True, 1002),
    "l1b5": TrainingWorkload("l1b5", 16, 4096, 2048, 3.0, -6.0, 2.0, "f32", True, 1003),
    "long": TrainingWorkload("long", 1, 131072, 2560, 5.0, -8.0, 1.0, "bf16", False, 1004),
    "l169m_bf16": TrainingWorkload("l169m_bf16", 8, 1024, 768, 3.0, -6.0, 2.0, "bf16", True, 1006),
    "l169m_gated": TrainingWorkload("l169m_gated", 8, 1024, 768, 3.0, -6.0, 2.0, "f32", True, 1008, gated=True),
}
DECODE = DecodeWorkload("decode", 32, 256, 4096, 1024, -6.0, 2.0, 1005)
DECODE_BF16 = DecodeWorkload("decode_bf16", 32, 256, 4096, 1024, -6.0, 2.0, 1011, token_dtype="bf16")
DECODES = {"decode": DECODE, "decode_bf16": DECODE_BF16}


@dataclass(frozen=True)
class ShiftWorkload:
    name: str
    B: int
    T: int
    C: int
    seed: int

    @property
    def elements(self) -> int:
        return self.B * self.T * self.C


SHIFT = ShiftWorkload("shift", 16, 4096, 2048, 1007)


@dataclass(frozen=True)
class ChannelMixWorkload:
    name: str
    B: int
    T: int
    C: int
    H: int  # hidden width of the channel mix (the key projection's outputs)
    seed: int

    @property
    def elements(self) -> int:
        return self.B * self.T * self.C


CMIX = ChannelMixWorkload("cmix", 8, 1024, 768, 3072, 1010)


def cmix_inputs(B: int, T: int, C: int, H: int, *, seed: int):
    """Draw (k, ga) [B,T,H] and (r, vk, gout) [B,T,C] ~ N(0,1) on the CPU,
    fp32, in that order."""
    g = _gen(seed)
    k, ga = (torch.randn(B, T, H, generator=g, dtype=torch.float32) for _ in range(2))
    r, vk, gout = (torch.randn(B, T, C, generator=g, dtype=torch.float32) for _ in range(3))
    return k, ga, r, vk, gout


def shift_inputs(B: int, T: int, C: int, *, seed: int):
    """Draw (x, x0, mu_k, mu_v, mu_r, gxk, gxv, gxr) on the CPU, fp32.

    Draw order: x [B,T,C] ~ N(0,1), x0 [B,C] ~ N(0,1), mu_k, mu_v, mu_r [C]
    ~ U(0,1), gxk, gxv, gxr [B,T,C] ~ N(0,1).
    """
    g = _gen(seed)
    x = torch.randn(B, T, C, generator=g, dtype=torch.float32)
    x0 = torch.randn(B, C, generator=g, dtype=torch.float32)
    mus = [torch.rand(C, generator=g, dtype=torch.float32) for _ in range(3)]
    gs = [torch.randn(B, T, C, generator=g, dtype=torch.float32) for _ in range(3)]
    return (x, x0, *mus, *gs)


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def training_inputs(B: int, T: int, C: int, *, seed: int, k_std: float = 1.0, d_lo: float = -5.0,
                    d_hi: float = 1.0, kv_dtype: str = "f32", k_shift: float = 0.0):
    """Draw (w, u, k, v, gy) on the CPU.

    Draw order: d [C], u [C], k [B,T,C], v [B,T,C], gy [B,T,C].
    w = exp(d) in fp32 (the decay is handed to the operator directly).
    ``k_shift`` adds a constant to every k after drawing (used by the
    shift-invariance checks).  k, v and gy are rounded to bf16 when
    ``kv_dtype == "bf16"``; w and u stay fp32.
    """
    g = _gen(seed)
    d = torch.rand(C, generator=g, dtype=torch.float32) * (d_hi - d_lo) + d_lo
    u = torch.rand(C, generator=g, dtype=torch.float32) * 2.0 - 1.0
    k = torch.randn(B, T, C, generator=g, dtype=torch.float32) * k_std
    v = torch.randn(B, T, C, generator=g, dtype=torch.float32)
    gy = torch.randn(B, T, C, generator=g, dtype=torch.float32)
    if k_shift:
        k = k + k_shift
    w = torch.exp(d)
    if kv_dtype == "bf16":
        k = k.to(torch.bfloat16)
        v = v.to(torch.bfloat16)
        gy = gy.to(torch.bfloat16)
    elif kv_dtype != "f32":
        raise ValueError(f"kv_dtype must be 'f32' or 'bf16', got {kv_dtype!r}")
    return w, u, k, v, gy


def workload_inputs(name: str):
    """(w, u, k, v, gy) of a named workload, and r (gate_inputs, seed + 1)
    after them when the workload is gated."""
    wl = WORKLOADS[name]
    base = training_inputs(wl.B, wl.T, wl.C, seed=wl.seed, k_std=wl.k_std, d_lo=wl.d_lo, d_hi=wl.d_hi,
                           kv_dtype=wl.kv_dtype)
    if wl.gated:
        return base + (gate_inputs(wl.B, wl.T, wl.C, seed=wl.seed + 1, kv_dtype=wl.kv_dtype),)
    return base


def gate_inputs(B: int, T: int, C: int, *, seed: int, r_std: float = 2.0, kv_dtype: str = "f32"):
    """Draw the receptance r [B,T,C] ~ N(0, r_std^2) of the output gate on the
    CPU, from its own generator (so the WKV inputs drawn with another seed
    keep their values); rounded to bf16 when ``kv_dtype == "bf16"``."""
    g = _gen(seed)
    r = torch.randn(B, T, C, generator=g, dtype=torch.float32) * r_std
    if kv_dtype == "bf16":
        r = r.to(torch.bfloat16)
    elif kv_dtype != "f32":
        raise ValueError(f"kv_dtype must be 'f32' or 'bf16', got {kv_dtype!r}")
    return r


def decode_params(L: int, C: int, *, seed: int, d_lo: float = -6.0, d_hi: float = 2.0):
    """Per-layer decode parameters, each [L, C]: (mu_k, mu_v, mu_r, w, u).

    Draw order: d, u, mu_k, mu_v, mu_r.  w = exp(d).
    """
    g = _gen(seed)
    d = torch.rand(L, C, generator=g, dtype=torch.float32) * (d_hi - d_lo) + d_lo
    u = torch.rand(L, C, generator=g, dtype=torch.float32) * 2.0 - 1.0
    mu_k = torch.rand(L, C, generator=g, dtype=torch.float32)
    mu_v = torch.rand(L, C, generator=g, dtype=torch.float32)
    mu_r = torch.rand(L, C, generator=g, dtype=torch.float32)
    return mu_k, mu_v, mu_r, torch.exp(d), u


def _token_dtype(ts, token_dtype: str):
    if token_dtype == "bf16":
        return tuple(t.to(torch.bfloat16) for t in ts)
    if token_dtype != "f32":
        raise ValueError(f"token_dtype must be 'f32' or 'bf16', got {token_dtype!r}")
    return tuple(ts)


def decode_step_inputs(L: int, B: int, C: int, *, seed: int, step: int, token_dtype: str = "f32"):
    """Per-step decode inputs, each [L, B, C]: (x, x_prev, r, k, v) ~ N(0,1).

    Each step index has its own generator (seed * 1_000_003 + step), so any
    step can be drawn without drawing the ones before it.  Draw order: x,
    x_prev, r, k, v.  ``token_dtype="bf16"``: drawn in fp32, then rounded.
    """
    g = _gen(int(seed) * 1_000_003 + int(step))
    shape = (L, B, C)
    return _token_dtype([torch.randn(shape, generator=g, dtype=torch.float32) for _ in range(5)], token_dtype)


def initial_state(L: int, B: int, C: int):
    """Decode state before any token: num = den = 0, pp = -1e38."""
    z = torch.zeros(L, B, C, dtype=torch.float32)
    return z.clone(), z.clone(), torch.full((L, B, C), -1e38, dtype=torch.float32)


def decode_pool(L: int, B: int, C: int, *, seed: int, n_sets: int, device="cpu", token_dtype: str = "f32"):
    """A pool of ``n_sets`` per-step decode input sets (x, x_prev, r, k, v),
    each [L, B, C] ~ N(0,1), drawn directly on ``device`` from one generator
    seeded with ``seed`` (set after set, in that order within a set; bf16:
    each set drawn in fp32, then rounded).  A run of more steps than sets
    uses set ``step % n_sets`` at each step."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    shape = (L, B, C)
    return [_token_dtype([torch.randn(shape, generator=g, dtype=torch.float32, device=device) for _ in range(5)],
                         token_dtype) for _ in range(n_sets)]
