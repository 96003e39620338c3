"""A float32 evaluation of the WKV recurrence and its adjoint, for the parity
gate's element-wise floor (test code; shares nothing with the CUDA sources
or the float64 oracle).

What it is for.  The GPU path computes in fp32.  Where an output is near
zero only by cancellation (a weighted average of O(1) values that happens to
be small, a gradient whose terms cancel), no fp32 arithmetic can match it to
2e-5 of itself: the absolute error of the sums it comes from is a few ulp of
their size, amplified by the length of the decay's memory (about 1/w
tokens).  This module measures that floor directly: the same inputs pushed
through the plain recurrence in float32, step by step, with nothing
rescaled and nothing compensated, i.e. what a straightforward fp32 kernel
computes.  Its element-wise error against the oracle is the error an honest
fp32 evaluation carries at each element; the parity gate requires the GPU's
element-wise error to stay within a small multiple of it (or within the
stated tolerance, whichever is larger).

The recurrence (RWKV time mixing, "RWKV解读：在Transformer的时代的新RNN",
section "3、RWKV的网络架构", eq. (8) and its recursive form), per batch row
and channel, with a_0 = b_0 = 0 (or a given state's sums):

    y_t     = (a_t + e^{u+k_t} v_t) / (b_t + e^{u+k_t})
    a_{t+1} = e^{-w} a_t + e^{k_t} v_t
    b_{t+1} = e^{-w} b_t + e^{k_t}

and its reverse mode, with lambda_a, lambda_b the adjoints of a, b
(zero after the last token unless an end gradient is given):

    D = b_t + e^{u+k_t},  gN = gy_t / D,  gD = -gy_t y_t / D
    gu     += (gN v_t + gD) e^{u+k_t}
    gk_t    = (gN v_t + gD) e^{u+k_t} + (lambda_a v_t + lambda_b) e^{k_t}
    gv_t    = gN e^{u+k_t} + lambda_a e^{k_t}
    gw     += -e^{-w} (lambda_a a_t + lambda_b b_t)
    lambda_a <- gN + e^{-w} lambda_a,   lambda_b <- gD + e^{-w} lambda_b

Every operation is a float32 operation (numpy float32 arrays, vectorised over
the independent (batch row, channel) columns, one numpy step per token).
gw and gu are summed in float32 along t per column, then over the batch
rows, in that order.

Limits: the sums are unscaled, so e^{k} must stay below float32's range
(k < 88) and so must the sums; every input the parity tests draw does (the
largest is k + 64 with |k| < 8 over a memory of under 150 tokens).  Callers
that shift k far beyond that pass ``shift_k=True``: k is taken relative to
its largest value per column, which leaves every output unchanged in exact
arithmetic (y is invariant under adding a constant to a column's k).
"""
from __future__ import annotations

import numpy as np

F32 = np.float32


def _f32(a) -> np.ndarray:
    if hasattr(a, "detach"):
        import torch

        a = a.detach().to("cpu")
        if a.dtype == torch.bfloat16:
            a = a.float()
        a = a.numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=F32))


def _sigmoid(r: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        return (F32(1) / (F32(1) + np.exp(-r))).astype(F32)


def _columns(w, u, k, v):
    """Inputs as float32 with k, v laid out [T, B, C] (one row per token)."""
    w, u = _f32(w), _f32(u)
    k = np.moveaxis(_f32(k), 1, 0).copy()
    v = np.moveaxis(_f32(v), 1, 0).copy()
    return w, u, k, v


def start_sums(state, B: int, C: int, shift=None):
    """The unscaled sums (a, b) of a state (num, den, pp) as float32 [B, C]
    (None: the empty state).  With ``shift`` (the per-column k offset in
    use), the sums are those of the shifted problem."""
    if state is None:
        return np.zeros((B, C), F32), np.zeros((B, C), F32)
    num, den, pp = (np.asarray(_f32(x), dtype=np.float64).reshape(B, C) for x in state)
    s = np.exp(pp - (0.0 if shift is None else shift))
    return (num * s).astype(F32), (den * s).astype(F32)


def forward(w, u, k, v, state_in=None, keep_sums: bool = False, shift_k: bool = False):
    """y [B, T, C] (float32) of the plain fp32 recurrence, and the sums
    (a, b) after the last token ([B, C], unscaled; with ``shift_k`` they
    belong to the shifted problem and ``shift`` is returned as well).  With
    ``keep_sums`` also the sums before every token, [T + 1, B, C] each."""
    w, u, k, v = _columns(w, u, k, v)
    T, B, C = k.shape
    shift = None
    if shift_k and T > 0:
        shift = k.max(axis=0)
        k = (k - shift).astype(F32)
    a, b = start_sums(state_in, B, C, None if shift is None else shift.astype(np.float64))
    ew = np.exp(-w).astype(F32)
    eu = np.exp(u).astype(F32)
    y = np.empty((T, B, C), F32)
    if keep_sums:
        As = np.empty((T + 1, B, C), F32)
        Bs = np.empty((T + 1, B, C), F32)
    for t in range(T):
        ek = np.exp(k[t])
        ec = ek * eu
        if keep_sums:
            As[t], Bs[t] = a, b
        y[t] = (a + ec * v[t]) / (b + ec)
        a = ew * a + ek * v[t]
        b = ew * b + ek
    out = {"y": np.moveaxis(y, 0, 1), "a": a, "b": b, "shift": shift}
    if keep_sums:
        As[T], Bs[T] = a, b
        out["A"], out["B"] = As, Bs
    return out


def forward_recurrent(w, u, k, v, shift_k: bool = False) -> np.ndarray:
    return forward(w, u, k, v, shift_k=shift_k)["y"]


def forward_gated(w, u, k, v, r, shift_k: bool = False) -> np.ndarray:
    """sigmoid(r) * wkv in float32."""
    return (_sigmoid(_f32(r)) * forward_recurrent(w, u, k, v, shift_k=shift_k)).astype(F32)


def backward(w, u, k, v, gy, state_in=None, adj_end=None, r=None, shift_k: bool = False):
    """Gradients of sum(gy * wkv) (+ ga_end a_T + gb_end b_T) by the float32
    adjoint recurrence.  ``r``: the output is the gated sigmoid(r) * wkv and
    gy its gradient.  Returns a dict with gw, gu [C], gk, gv [B, T, C], the
    unscaled start-sum gradients ga, gb [B, C], and gr with the gate."""
    fw = forward(w, u, k, v, state_in=state_in, keep_sums=True, shift_k=shift_k)
    w, u, k, v = _columns(w, u, k, v)
    if fw["shift"] is not None:
        k = (k - fw["shift"]).astype(F32)
    gy = np.moveaxis(_f32(gy), 1, 0).copy()
    T, B, C = k.shape
    gr = None
    if r is not None:
        sg = np.moveaxis(_sigmoid(_f32(r)), 1, 0)
        gr_t = np.empty((T, B, C), F32)
    ew = np.exp(-w).astype(F32)
    eu = np.exp(u).astype(F32)
    la = np.zeros((B, C), F32)
    lb = np.zeros((B, C), F32)
    if adj_end is not None:
        ga_end, gb_end = (_f32(x).reshape(B, C) for x in adj_end)
        if fw["shift"] is not None:  # gradients of the shifted problem's sums
            s = np.exp(fw["shift"].astype(np.float64))
            ga_end, gb_end = (ga_end * s).astype(F32), (gb_end * s).astype(F32)
        la, lb = ga_end.copy(), gb_end.copy()
    gk = np.empty((T, B, C), F32)
    gv = np.empty((T, B, C), F32)
    gw = np.zeros((B, C), F32)
    gu = np.zeros((B, C), F32)
    As, Bs = fw["A"], fw["B"]
    for t in range(T - 1, -1, -1):
        ek = np.exp(k[t])
        ec = ek * eu
        D = Bs[t] + ec
        yt = (As[t] + ec * v[t]) / D
        g = gy[t]
        if r is not None:
            gr_t[t] = g * yt * sg[t] * (F32(1) - sg[t])
            g = g * sg[t]
        gN = g / D
        gD = -g * yt / D
        cur = (gN * v[t] + gD) * ec
        gu = gu + cur
        gk[t] = cur + (la * v[t] + lb) * ek
        gv[t] = gN * ec + la * ek
        gw = gw - ew * (la * As[t] + lb * Bs[t])
        la = gN + ew * la
        lb = gD + ew * lb
    gw_c = np.zeros(C, F32)
    gu_c = np.zeros(C, F32)
    for bi in range(B):
        gw_c = gw_c + gw[bi]
        gu_c = gu_c + gu[bi]
    if fw["shift"] is not None:  # back to the start sums of the unshifted problem
        s = np.exp(-fw["shift"].astype(np.float64))
        la, lb = (la * s).astype(F32), (lb * s).astype(F32)
    out = {"gw": gw_c, "gu": gu_c, "gk": np.moveaxis(gk, 0, 1), "gv": np.moveaxis(gv, 0, 1), "ga": la, "gb": lb}
    if r is not None:
        out["gr"] = np.moveaxis(gr_t, 0, 1)
    return out


def backward_adjoint(w, u, k, v, gy, shift_k: bool = False):
    """(gw, gu, gk, gv) like the oracle's adjoint backward, in float32."""
    o = backward(w, u, k, v, gy, shift_k=shift_k)
    return o["gw"], o["gu"], o["gk"], o["gv"]


def backward_gated(w, u, k, v, r, gout, shift_k: bool = False):
    """(gw, gu, gk, gv, gr) of sum(gout * sigmoid(r) * wkv), in float32."""
    o = backward(w, u, k, v, gout, r=r, shift_k=shift_k)
    return o["gw"], o["gu"], o["gk"], o["gv"], o["gr"]


def sums_after(w, k, v, ts, state_in=None):
    """The unscaled sums (a, b) after each token count in ``ts`` ([B, C] each),
    from the plain float32 recurrence (u does not enter the sums)."""
    w = _f32(w)
    fw = forward(w, np.zeros_like(w), k, v, state_in=state_in, keep_sums=True)
    return [(fw["A"][t], fw["B"][t]) for t in ts]


def decode_step(x, x_prev, mu_k, mu_v, mu_r, r, k, v, w, u, a, b):
    """One RNN-mode step of L layers in float32 on the unscaled sums (a, b)
    [L, B, C]: the token-shift mixes, wkv of the given k, v from (a, b),
    the sigmoid(r) gate, and the sums after the token.  Returns
    (y, a', b', xk, xv, xr)."""
    x, x_prev, r, k, v, a, b = map(_f32, (x, x_prev, r, k, v, a, b))
    mk, mv, mr, w, u = (_f32(p)[:, None, :] for p in (mu_k, mu_v, mu_r, w, u))
    one = F32(1)
    xk = mk * x + (one - mk) * x_prev
    xv = mv * x + (one - mv) * x_prev
    xr = mr * x + (one - mr) * x_prev
    ek = np.exp(k)
    ec = ek * np.exp(u)
    y = _sigmoid(r) * ((a + ec * v) / (b + ec))
    ew = np.exp(-w)
    return y, ew * a + ek * v, ew * b + ek, xk, xv, xr


# ------------------------------------------------------------- token shift
def token_shift(x, x0, mu_k, mu_v, mu_r):
    """(xk, xv, xr) = mu x_t + (1 - mu) x_{t-1} in float32, x [B, T, C];
    x0 [B, C] the token before the sequence (None: zeros)."""
    x = _f32(x)
    prev = np.empty_like(x)
    prev[:, 1:] = x[:, :-1]
    prev[:, 0] = 0 if x0 is None else _f32(x0)
    one = F32(1)
    return tuple((m * x + (one - m) * prev).astype(F32) for m in map(_f32, (mu_k, mu_v, mu_r)))


def token_shift_backward(x, x0, mu_k, mu_v, mu_r, gxk, gxv, gxr):
    """(gx, gx0, gmu_k, gmu_v, gmu_r) in float32: gx_t sums mu g_t and
    (1 - mu) g_{t+1} over the three mixes; gmu sums g_t (x_t - x_{t-1}) over
    t, then over the batch rows."""
    x = _f32(x)
    B, T, C = x.shape
    prev = np.empty_like(x)
    prev[:, 1:] = x[:, :-1]
    prev[:, 0] = 0 if x0 is None else _f32(x0)
    dx = (x - prev).astype(F32)
    one = F32(1)
    gx = np.zeros_like(x)
    gx0 = np.zeros((B, C), F32)
    gmus = []
    for m, g in zip(map(_f32, (mu_k, mu_v, mu_r)), map(_f32, (gxk, gxv, gxr))):
        gx += m * g
        gx[:, :-1] += (one - m) * g[:, 1:]
        gx0 += (one - m) * g[:, 0]
        per_row = np.zeros((B, C), F32)
        for t in range(T):
            per_row += g[:, t] * dx[:, t]
        gm = np.zeros(C, F32)
        for bi in range(B):
            gm += per_row[bi]
        gmus.append(gm)
    return (gx, None if x0 is None else gx0, *gmus)


# ----------------------------------------------------------- channel mixing
def sqrelu(k):
    k = _f32(k)
    r = np.maximum(k, F32(0))
    return (r * r).astype(F32)


def sqrelu_backward(k, ga):
    k, ga = _f32(k), _f32(ga)
    return (F32(2) * np.maximum(k, F32(0)) * ga).astype(F32)


def cmix_gate(r, vk):
    return (_sigmoid(_f32(r)) * _f32(vk)).astype(F32)


def cmix_gate_backward(r, vk, gout):
    """(gr, gvk) of sum(gout * sigmoid(r) * vk) in float32."""
    s = _sigmoid(_f32(r))
    g = _f32(gout)
    return (g * _f32(vk) * s * (F32(1) - s)).astype(F32), (g * s).astype(F32)


# --------------------------------------------------------- adjoint fold
def adjoint_fold(w, adj, lengths, gstate_end=None):
    """The start-state gradient of the first of n segments in float32, from
    their own start gradients ``adj`` [n, 3, B, C] planes (g_num, g_den, pp)
    and the gradient on the last end state: in unscaled form (g e^{-pp}),
    each segment's own plus e^{-n w} times the next one's, last to first;
    returned as planes at the first segment's pp."""
    w = _f32(w)
    a = _f32(adj)
    X = None
    if gstate_end is not None:
        g = _f32(gstate_end)
        s = np.exp(-g[2])
        X = (g[0] * s, g[1] * s)
    for i in range(a.shape[0] - 1, -1, -1):
        s = np.exp(-a[i, 2])
        own = (a[i, 0] * s, a[i, 1] * s)
        dec = np.exp(-(F32(lengths[i]) * w))
        X = own if X is None else (own[0] + dec * X[0], own[1] + dec * X[1])
    pp = a[0, 2]
    e = np.exp(pp)
    return np.stack([X[0] * e, X[1] * e, pp]).astype(F32)


# ----------------------------------------------------------- perturbations
def perturbed(arrays, seed: int):
    """The float inputs moved by one unit in the last place of float32, up or
    down at random per element (other arguments unchanged).  A float32
    evaluation on these is as valid as one on the exact inputs: the inputs of
    an fp32 pipeline carry that much rounding from upstream, and a kernel
    rounds its intermediates as much.  The spread of the results measures how
    sensitive each output is to fp32 rounding (see ``evaluations``)."""
    rng = np.random.default_rng(seed)
    out = []
    for a in arrays:
        if a is None or isinstance(a, (int, float, str)):
            out.append(a)
            continue
        if isinstance(a, tuple):
            out.append(tuple(perturbed(list(a), int(rng.integers(1 << 30)))))
            continue
        x = _f32(a)
        up = rng.random(x.shape) < 0.5
        out.append(np.where(up, np.nextafter(x, np.float32(np.inf)), np.nextafter(x, np.float32(-np.inf))))
    return out


def evaluations(fn, *args, n: int = 2):
    """fn(*args) and fn on ``n`` one-ulp perturbations of the float inputs:
    float32 evaluations of the same quantity, whose worst error against the
    oracle is the floor the parity gate uses for gradients."""
    return [fn(*args)] + [fn(*perturbed(list(args), 1000 + i)) for i in range(n)]

