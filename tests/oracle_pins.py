"""Pins of the float64 oracle against facts that do not come from the oracle.

Each ``pin_*`` function takes an oracle handle (``oracle.Oracle``) and raises
``AssertionError`` when the oracle disagrees with what the definition of the
operator fixes: hand-derived values (``golden/hand_cases.json``), closed
forms of special cases, limits, invariants and brute-force finite
differences.  ``test_oracle_pins.py`` runs them on the real oracle;
``test_oracle_mutants.py`` runs them on deliberately broken copies and
checks that every broken copy fails at least one pin.

Sources (page title, section):
  * "RWKV についての調査記録" (qiita), "wkvとは": wkv is a weighted average of
    v with weights from k, a bonus u for the current token, a decay that
    grows with distance through one channel-wise vector w, and independent
    channels.
  * "RWKV解读：在Transformer的时代的新RNN" (segmentfault),
    "3、RWKV的网络架构": eq. (8) and its recursive form, token shift eq. (7),
    sigmoid(r) gate eq. (9).
  * qiita "Trainingについて": gradients for every parameter.
"""
from __future__ import annotations

import json
from pathlib import Path

import numpy as np
from scipy.special import expit

GOLDEN = json.loads((Path(__file__).parent / "golden" / "hand_cases.json").read_text())


def _rng(seed):
    return np.random.default_rng(seed)


def _rand_inputs(seed, B=2, T=37, C=5, k_std=1.0, w_lo=-3.0, w_hi=1.0):
    r = _rng(seed)
    w = np.exp(r.uniform(w_lo, w_hi, C))
    u = r.uniform(-1, 1, C)
    k = r.normal(0, k_std, (B, T, C))
    v = r.normal(0, 1, (B, T, C))
    gy = r.normal(0, 1, (B, T, C))
    return w, u, k, v, gy


def _close(a, b, rtol, atol=0.0, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    err = np.abs(a - b)
    bound = atol + rtol * np.abs(b)
    assert np.all(err <= bound), f"{what}: max err {err.max():.3e} (rtol {rtol}, atol {atol})"


def _col(vals, T):
    return np.asarray(vals, dtype=np.float64).reshape(1, T, 1)


# --------------------------------------------------------------------------
# forward
# --------------------------------------------------------------------------
def pin_forward_hand_values(o):
    """Hand-derived values of small cases, both forms."""
    for case in GOLDEN["forward"]:
        T = len(case["k"])
        w, u = np.array(case["w"]), np.array(case["u"])
        k, v = _col(case["k"], T), _col(case["v"], T)
        want = _col(case["y"], T)
        for fn in (o.forward_direct, o.forward_recurrent):
            _close(fn(w, u, k, v), want, 1e-13, 1e-13, f"{case['name']}/{fn.__name__}")


def pin_forward_forms_agree(o):
    """The direct sum and the recurrence are two independent formulations."""
    for seed, kstd in ((1, 1.0), (2, 3.0), (3, 0.1)):
        w, u, k, v, _ = _rand_inputs(seed, k_std=kstd)
        yd = o.forward_direct(w, u, k, v)
        yr = o.forward_recurrent(w, u, k, v)
        _close(yr, yd, 1e-12, 1e-13, f"direct vs recurrent seed {seed}")


def pin_forward_t1_is_v(o):
    """T = 1: only the current token, wkv_0 = v_0."""
    w, u, k, v, _ = _rand_inputs(4, T=1, C=7)
    for fn in (o.forward_direct, o.forward_recurrent):
        _close(fn(w, u, k, v), v, 1e-15, 0.0, f"T=1 {fn.__name__}")


def pin_forward_constant_v(o):
    """A weighted average of a constant is that constant."""
    w, u, k, _, _ = _rand_inputs(5)
    v = np.full(k.shape, -1.75)
    for fn in (o.forward_direct, o.forward_recurrent):
        _close(fn(w, u, k, v), v, 1e-14, 0.0, f"constant v {fn.__name__}")


def pin_forward_convex(o):
    """wkv_t lies between min and max of v_0..v_t (weighted average)."""
    w, u, k, v, _ = _rand_inputs(6, k_std=2.0)
    for fn in (o.forward_direct, o.forward_recurrent):
        y = fn(w, u, k, v)
        lo = np.minimum.accumulate(v, axis=1)
        hi = np.maximum.accumulate(v, axis=1)
        assert np.all(y >= lo - 1e-12) and np.all(y <= hi + 1e-12), f"convexity {fn.__name__}"


def pin_forward_affine(o):
    """wkv(alpha v + beta) = alpha wkv(v) + beta (weights do not depend on v)."""
    w, u, k, v, _ = _rand_inputs(7)
    for fn in (o.forward_direct, o.forward_recurrent):
        y = fn(w, u, k, v)
        _close(fn(w, u, k, -2.5 * v + 0.75), -2.5 * y + 0.75, 1e-12, 1e-12, f"affine {fn.__name__}")


def pin_forward_k_shift(o):
    """Adding one constant to every k of a channel scales all weights alike."""
    w, u, k, v, _ = _rand_inputs(8, T=24)
    for fn in (o.forward_direct, o.forward_recurrent):
        y = fn(w, u, k, v)
        for s in (-300.0, -40.0, 40.0, 300.0):
            _close(fn(w, u, k + s, v), y, 1e-11, 1e-12, f"k shift {s} {fn.__name__}")


def pin_forward_causal_and_independent(o):
    """Future tokens do not change the past; channels and rows do not mix."""
    w, u, k, v, _ = _rand_inputs(9, B=3, T=20, C=6)
    for fn in (o.forward_direct, o.forward_recurrent):
        y = fn(w, u, k, v)
        k2, v2 = k.copy(), v.copy()
        k2[:, 11:, :] += 5.0
        v2[:, 11:, :] -= 3.0
        y2 = fn(w, u, k2, v2)
        assert np.array_equal(y2[:, :11], y[:, :11]), "causality"
        pc = _rng(10).permutation(6)
        pb = _rng(11).permutation(3)
        yp = fn(w[pc], u[pc], k[pb][:, :, pc], v[pb][:, :, pc])
        _close(yp, y[pb][:, :, pc], 1e-15, 0.0, "permutation")


def pin_forward_limits(o):
    """Closed forms of limits of w and u."""
    w, u, k, v, _ = _rand_inputs(12, T=30, C=4)
    ew = np.exp(k)
    for fn in (o.forward_direct, o.forward_recurrent):
        # w = 0: no decay -> a cumulative e^k-weighted mean with the bonus on t
        zero = np.zeros_like(w)
        past_n = np.concatenate([np.zeros_like(k[:, :1]), np.cumsum(ew * v, axis=1)[:, :-1]], axis=1)
        past_d = np.concatenate([np.zeros_like(k[:, :1]), np.cumsum(ew, axis=1)[:, :-1]], axis=1)
        cur = np.exp(u[None, None, :] + k)
        _close(fn(zero, u, k, v), (past_n + cur * v) / (past_d + cur), 1e-12, 1e-13, "w=0")
        # u -> +inf: the current token dominates, wkv_t -> v_t
        _close(fn(w, np.full_like(u, 60.0), k, v), v, 1e-12, 1e-13, "u=+60")
        # w -> inf: only token t-1 (undecayed) and token t survive, for t >= 1
        big = np.full_like(w, 80.0)
        y = fn(big, u, k, v)
        e1 = np.exp(k[:, :-1])
        e2 = np.exp(u[None, None, :] + k[:, 1:])
        _close(y[:, 1:], (e1 * v[:, :-1] + e2 * v[:, 1:]) / (e1 + e2), 1e-12, 1e-13, "w=80")
        _close(y[:, 0], v[:, 0], 1e-15, 0.0, "w=80 t=0")
        # u -> -inf, w = 0, t >= 1: e^k-weighted mean of the past only
        y = fn(zero, np.full_like(u, -80.0), k, v)
        for t in (1, 7, 29):
            want = np.stack([np.average(v[b, :t], axis=0, weights=ew[b, :t]) for b in range(v.shape[0])])
            _close(y[:, t], want, 1e-12, 1e-13, f"u=-80 w=0 t={t}")


# --------------------------------------------------------------------------
# backward
# --------------------------------------------------------------------------
def _loss(o, w, u, k, v, gy):
    return float(np.sum(gy * o.forward_direct(w, u, k, v)))


def pin_backward_hand_values(o):
    for case in GOLDEN["backward"]:
        T = len(case["k"])
        args = (np.array(case["w"]), np.array(case["u"]), _col(case["k"], T), _col(case["v"], T), _col(case["gy"], T))
        for fn in (o.backward_adjoint, o.backward_direct):
            gw, gu, gk, gv = fn(*args)
            _close(gw, case["gw"], 1e-12, 1e-14, f"{case['name']} gw {fn.__name__}")
            _close(gu, case["gu"], 1e-12, 1e-14, f"{case['name']} gu {fn.__name__}")
            _close(gk, _col(case["gk"], T), 1e-12, 1e-14, f"{case['name']} gk {fn.__name__}")
            _close(gv, _col(case["gv"], T), 1e-12, 1e-14, f"{case['name']} gv {fn.__name__}")


def pin_backward_finite_differences(o):
    """Central differences of sum(gy * wkv) in float64 on tiny inputs."""
    for seed in (20, 21):
        w, u, k, v, gy = _rand_inputs(seed, B=2, T=6, C=3, k_std=1.5)
        grads = {fn.__name__: fn(w, u, k, v, gy) for fn in (o.backward_adjoint, o.backward_direct)}
        fd = {"w": np.zeros_like(w), "u": np.zeros_like(u), "k": np.zeros_like(k), "v": np.zeros_like(v)}
        params = {"w": w, "u": u, "k": k, "v": v}
        for name, arr in params.items():
            it = np.nditer(arr, flags=["multi_index"])
            for _ in it:
                idx = it.multi_index
                h = 1e-6 * max(1.0, abs(arr[idx]))
                plus = {n: a.copy() for n, a in params.items()}
                minus = {n: a.copy() for n, a in params.items()}
                plus[name][idx] += h
                minus[name][idx] -= h
                fd[name][idx] = (_loss(o, plus["w"], plus["u"], plus["k"], plus["v"], gy)
                                 - _loss(o, minus["w"], minus["u"], minus["k"], minus["v"], gy)) / (2 * h)
        for fname, (gw, gu, gk, gv) in grads.items():
            for got, want, what in ((gw, fd["w"], "gw"), (gu, fd["u"], "gu"), (gk, fd["k"], "gk"), (gv, fd["v"], "gv")):
                scale = max(1.0, float(np.max(np.abs(want))))
                _close(got, want, 0.0, 1e-7 * scale, f"FD {what} {fname} seed {seed}")


def pin_backward_forms_agree(o):
    for seed, kstd in ((30, 1.0), (31, 3.0)):
        w, u, k, v, gy = _rand_inputs(seed, B=2, T=48, C=4, k_std=kstd)
        a = o.backward_adjoint(w, u, k, v, gy)
        d = o.backward_direct(w, u, k, v, gy)
        for x, y_, n in zip(a, d, ("gw", "gu", "gk", "gv")):
            scale = float(np.max(np.abs(y_)))
            _close(x, y_, 0.0, 1e-12 * max(scale, 1.0), f"adjoint vs direct {n} seed {seed}")


def pin_backward_identities(o):
    """Identities that follow from invariances of the forward pass:
    k-shift invariance => sum_t gk_t = 0 per (b, c); v -> v + beta shifts
    wkv by beta => sum_t gv_t = sum_t gy_t per (b, c); w never enters for
    T <= 2 => gw = 0; T = 1 => wkv = v so gv = gy and gk = gu = gw = 0."""
    w, u, k, v, gy = _rand_inputs(40, B=2, T=33, C=5, k_std=2.0)
    for fn in (o.backward_adjoint, o.backward_direct):
        gw, gu, gk, gv = fn(w, u, k, v, gy)
        _close(gk.sum(axis=1), np.zeros_like(gk[:, 0]), 0.0, 1e-12 * max(1.0, np.abs(gk).max()), "sum gk")
        _close(gv.sum(axis=1), gy.sum(axis=1), 1e-12, 1e-12, "sum gv")
        for T in (1, 2):
            gw2, gu2, gk2, gv2 = fn(w, u, k[:, :T], v[:, :T], gy[:, :T])
            assert np.all(np.abs(gw2) < 1e-14), f"gw != 0 at T={T}"
            if T == 1:
                _close(gv2, gy[:, :1], 1e-15, 0.0, "T=1 gv")
                assert np.all(np.abs(gk2) < 1e-15) and np.all(np.abs(gu2) < 1e-15), "T=1 gk/gu"


def pin_backward_state(o):
    """The backward pass of a segment with a carried start state and a
    gradient on its end sums: with neither it is the plain adjoint backward;
    central finite differences of sum(gy * wkv) + ga_end a_T + gb_end b_T
    give gw, gu, gk, gv and the gradient of the start sums; and a sequence's
    backward cut in two (the later half from the state at the cut, the
    earlier half fed the later half's start gradient) gives the whole
    sequence's gradients."""
    names = ("gw", "gu", "gk", "gv")
    w, u, k, v, gy = _rand_inputs(95, B=2, T=12, C=3, k_std=1.0)
    for g, r, n in zip(o.backward_state(w, u, k, v, gy)[:4], o.backward_adjoint(w, u, k, v, gy), names):
        _close(g, r, 1e-14, 1e-15, f"no state, no end gradient: {n}")
    rng = _rng(96)
    B, T, C = k.shape
    pp_in = np.full((B, C), 0.3)
    num_in, den_in = rng.normal(0, 1, (B, C)), rng.uniform(0.5, 2.0, (B, C))
    ga_end, gb_end = rng.normal(0, 0.2, (B, C)), rng.normal(0, 0.2, (B, C))

    def loss(p):
        y, (n, d, pe) = o.forward_state(p["w"], p["u"], p["k"], p["v"], (p["num"], p["den"], pp_in))
        return float(np.sum(gy * y) + np.sum(ga_end * n * np.exp(pe)) + np.sum(gb_end * d * np.exp(pe)))

    params = {"w": w, "u": u, "k": k, "v": v, "num": num_in, "den": den_in}
    gw, gu, gk, gv, (ga, gb) = o.backward_state(w, u, k, v, gy, (num_in, den_in, pp_in), (ga_end, gb_end))
    got = {"w": gw, "u": gu, "k": gk, "v": gv, "num": ga * np.exp(pp_in), "den": gb * np.exp(pp_in)}
    for name, arr in params.items():
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            h = 1e-6 * max(1.0, abs(arr[idx]))
            plus = {n: a.copy() for n, a in params.items()}
            minus = {n: a.copy() for n, a in params.items()}
            plus[name][idx] += h
            minus[name][idx] -= h
            fd[idx] = (loss(plus) - loss(minus)) / (2 * h)
        _close(got[name], fd, 0.0, 1e-7 * max(1.0, float(np.max(np.abs(fd)))), f"FD with state: d{name}")
    whole = o.backward_adjoint(w, u, k, v, gy)
    t0 = 5
    late = o.backward_state(w, u, k[:, t0:], v[:, t0:], gy[:, t0:], o.state(w, k, v, t0))
    early = o.backward_state(w, u, k[:, :t0], v[:, :t0], gy[:, :t0], None, late[4])
    _close(np.concatenate([early[2], late[2]], axis=1), whole[2], 1e-12, 1e-14, "cut in two: gk")
    _close(np.concatenate([early[3], late[3]], axis=1), whole[3], 1e-12, 1e-14, "cut in two: gv")
    _close(early[0] + late[0], whole[0], 1e-12, 1e-14, "cut in two: gw")
    _close(early[1] + late[1], whole[1], 1e-12, 1e-14, "cut in two: gu")


# --------------------------------------------------------------------------
# state and decode
# --------------------------------------------------------------------------
def pin_state_definition(o):
    """state(t) combined with token t through the definition gives wkv_t,
    and pp is the running maximum max_{i<t}(k_i - (t-1-i) w)."""
    w, u, k, v, _ = _rand_inputs(50, B=2, T=25, C=3, k_std=2.0)
    y = o.forward_direct(w, u, k, v)
    for t in (0, 1, 5, 24):
        num, den, pp = o.state(w, k, v, t)
        if t == 0:
            assert np.all(num == 0) and np.all(den == 0) and np.all(pp == -1e38), "empty state"
            continue
        ex = k[:, :t] - (t - 1 - np.arange(t))[None, :, None] * w[None, None, :]
        _close(pp, ex.max(axis=1), 1e-15, 1e-15, f"pp t={t}")
        cur = np.exp(u + k[:, t])
        got = (num * np.exp(pp) + cur * v[:, t]) / (den * np.exp(pp) + cur)
        _close(got, y[:, t], 1e-12, 1e-13, f"state -> wkv t={t}")
        assert np.all(den >= 1.0 - 1e-12), "den >= 1 (the max term is exactly 1)"


def pin_forward_state_split(o):
    """A sequence cut at t0 and continued from the state of its first t0
    tokens (the direct-sum state) gives the parallel form's outputs for the
    remaining tokens, and ends in the direct-sum state of all tokens; the
    empty state is the plain forward; two cuts chained through the returned
    state agree with one."""
    w, u, k, v, _ = _rand_inputs(70, B=2, T=30, C=4, k_std=2.5)
    y = o.forward_direct(w, u, k, v)
    T = k.shape[1]
    y0, _ = o.forward_state(w, u, k, v, None)
    _close(y0, y, 1e-12, 1e-13, "empty state in")
    n_all, d_all, p_all = o.state(w, k, v, T)
    for t0 in (0, 1, 7, 29, 30):
        sin = o.state(w, k, v, t0)
        y2, (n2, d2, p2) = o.forward_state(w, u, k[:, t0:], v[:, t0:], sin)
        _close(y2, y[:, t0:], 1e-12, 1e-13, f"continued outputs t0={t0}")
        _close(p2, p_all, 1e-13, 1e-13, f"state out pp t0={t0}")
        _close(n2, n_all, 1e-12, 1e-13, f"state out num t0={t0}")
        _close(d2, d_all, 1e-12, 1e-13, f"state out den t0={t0}")
    ya, sa = o.forward_state(w, u, k[:, :11], v[:, :11], None)
    yb, sb = o.forward_state(w, u, k[:, 11:], v[:, 11:], sa)
    _close(np.concatenate([ya, yb], axis=1), y, 1e-12, 1e-13, "two chained cuts")
    _close(sb[2], p_all, 1e-13, 1e-13, "chained state pp")


def pin_state_fold(o):
    """Segments' own states folded in order give the direct-sum state of the
    whole sequence (oracle.state over all tokens), for uneven cuts, a
    zero-length segment and a single segment; a state given before the
    first segment (a leading segment of length 0) continues the same way."""
    w, u, k, v, _ = _rand_inputs(75, B=2, T=40, C=3, k_std=2.5, w_lo=-4.0, w_hi=1.5)
    whole = o.state(w, k, v, 40)
    for cuts in ((0, 40), (0, 13, 40), (0, 1, 2, 17, 17, 39, 40), (0, 25, 40)):
        segs = [o.state(w, k[:, a:b], v[:, a:b], b - a) for a, b in zip(cuts[:-1], cuts[1:])]
        lens = [b - a for a, b in zip(cuts[:-1], cuts[1:])]
        got = o.state_fold(w, segs, lens)
        for g, r, name in zip(got, whole, ("num", "den", "pp")):
            _close(g, r, 1e-12, 1e-13, f"fold {cuts} {name}")
    head = o.state(w, k[:, :9], v[:, :9], 9)
    tail = [o.state(w, k[:, 9:30], v[:, 9:30], 21), o.state(w, k[:, 30:], v[:, 30:], 10)]
    got = o.state_fold(w, [head] + tail, [0, 21, 10])
    for g, r, name in zip(got, whole, ("num", "den", "pp")):
        _close(g, r, 1e-12, 1e-13, f"fold after a given state {name}")


def pin_token_shift(o):
    """mu = 1 keeps the current token, mu = 0 takes the previous one (the
    given x0 before the first), and the mix is the decode step's (which its
    own pins tie to the definition); the backward matches central finite
    differences of sum(g * mix) in x, x0 and every mu."""
    r = _rng(80)
    B, T, C = 2, 9, 3
    x = r.normal(0, 1, (B, T, C))
    x0 = r.normal(0, 1, (B, C))
    one, zero = np.ones(C), np.zeros(C)
    xk, xv, xr = o.token_shift(x, x0, one, zero, one)
    _close(xk, x, 0, 0, "mu=1 keeps x_t")
    prev = np.concatenate([x0[:, None], x[:, :-1]], axis=1)
    _close(xv, prev, 0, 0, "mu=0 takes x_{t-1}")
    _close(o.token_shift(x, None, zero, zero, zero)[0][:, 0], np.zeros((B, C)), 0, 0, "no x0: zeros")
    mk, mv, mr = (r.uniform(0, 1, C) for _ in range(3))
    xk, xv, xr = o.token_shift(x, x0, mk, mv, mr)
    for t in range(T):  # the decode step's mix of (x_t, x_{t-1}) for one layer
        p = prev[:, t]
        y, _, _, _, dk, dv, dr = o.decode_step(x[None, :, t], p[None], mk[None], mv[None], mr[None],
                                               np.zeros((1, B, C)), np.zeros((1, B, C)), np.zeros((1, B, C)),
                                               np.ones((1, C)), np.zeros((1, C)), np.zeros((1, B, C)),
                                               np.zeros((1, B, C)), np.full((1, B, C), -1e38))
        _close(dk[0], xk[:, t], 1e-15, 1e-15, "shift vs decode mix k")
        _close(dv[0], xv[:, t], 1e-15, 1e-15, "shift vs decode mix v")
        _close(dr[0], xr[:, t], 1e-15, 1e-15, "shift vs decode mix r")
    g = [r.normal(0, 1, (B, T, C)) for _ in range(3)]
    gx, gx0, gmk, gmv, gmr = o.token_shift_backward(x, x0, mk, mv, mr, *g)

    def loss(x_, x0_, mk_, mv_, mr_):
        outs = o.token_shift(x_, x0_, mk_, mv_, mr_)
        return sum(float(np.sum(gi * oi)) for gi, oi in zip(g, outs))

    h = 1e-6
    for arr, grad, name in ((x, gx, "x"), (x0, gx0, "x0"), (mk, gmk, "mu_k"), (mv, gmv, "mu_v"), (mr, gmr, "mu_r")):
        flat = arr.reshape(-1)
        num = np.empty_like(flat)
        for i in range(flat.size):
            keep = flat[i]
            flat[i] = keep + h
            lp = loss(x, x0, mk, mv, mr)
            flat[i] = keep - h
            lm = loss(x, x0, mk, mv, mr)
            flat[i] = keep
            num[i] = (lp - lm) / (2 * h)
        _close(grad.reshape(-1), num, 1e-6, 1e-7, f"token shift d/d{name}")


def pin_decode_hand_values(o):
    for case in GOLDEN["decode"]:
        for s in case["steps"]:
            f = lambda x: np.array([[[x]]], dtype=np.float64)  # noqa: E731
            p = lambda x: np.array([[x]], dtype=np.float64)  # noqa: E731
            num, den, pp = (f(x) for x in s["state_in"])
            y, num2, den2, pp2, xk, xv, xr = o.decode_step(
                f(s["x"]), f(s["x_prev"]), p(s["mu_k"]), p(s["mu_v"]), p(s["mu_r"]), f(s["r"]), f(s["k"]),
                f(s["v"]), p(s["w"]), p(s["u"]), num, den, pp)
            _close(y, f(s["y"]), 1e-13, 1e-15, "decode y")
            _close(np.concatenate([num2, den2, pp2]).ravel(), s["state_out"], 1e-13, 1e-15, "decode state")
            _close(np.concatenate([xk, xv, xr]).ravel(), [s["xk"], s["xv"], s["xr"]], 1e-15, 0.0, "decode mix")


def pin_decode_matches_forward(o):
    """Running the decode step token by token from the empty state gives
    sigmoid(r) * wkv of the parallel form, and ends in state(T)."""
    r_ = _rng(60)
    L, B, C, T = 2, 3, 4, 17
    w = np.exp(r_.uniform(-3, 1, (L, C)))
    u = r_.uniform(-1, 1, (L, C))
    mu = [r_.uniform(0, 1, (L, C)) for _ in range(3)]
    k = r_.normal(0, 2, (L, B, T, C))
    v = r_.normal(0, 1, (L, B, T, C))
    rr = r_.normal(0, 1, (L, B, T, C))
    x = r_.normal(0, 1, (L, B, T + 1, C))
    num = np.zeros((L, B, C))
    den = np.zeros((L, B, C))
    pp = np.full((L, B, C), -1e38)
    ys = []
    for t in range(T):
        y, num, den, pp, xk, xv, xr = o.decode_step(x[:, :, t + 1], x[:, :, t], mu[0], mu[1], mu[2], rr[:, :, t],
                                                    k[:, :, t], v[:, :, t], w, u, num, den, pp)
        for m, got in zip(mu, (xk, xv, xr)):
            # mu = 1 keeps the current token, mu = 0 the previous one
            want = x[:, :, t] + m[:, None, :] * (x[:, :, t + 1] - x[:, :, t])
            _close(got, want, 1e-14, 1e-14, "mix")
        ys.append(y)
    ys = np.stack(ys, axis=2)
    for l in range(L):
        yf = o.forward_direct(w[l], u[l], k[l], v[l])
        _close(ys[l], yf * expit(rr[l]), 1e-12, 1e-13, f"decode vs forward layer {l}")
        n2, d2, p2 = o.state(w[l], k[l], v[l], T)
        _close(pp[l], p2, 1e-13, 1e-13, "decode pp vs state")
        _close(num[l], n2, 1e-12, 1e-13, "decode num vs state")
        _close(den[l], d2, 1e-12, 1e-13, "decode den vs state")


# --------------------------------------------------------------------------
# the receptance gate on the output (eq. (9))
# --------------------------------------------------------------------------
def pin_gate_special_values(o):
    """The gate at points where sigmoid is exact: 3/4 at ln 3, 1/2 at 0, 1/4
    at -ln 3, and 1 to within e^{-40} at 40, applied to the ungated wkv
    (pinned above).  At r = 40 the gradients are the ungated ones with
    gy = gout, and gr vanishes with sigmoid'(40) < 5e-18."""
    w, u, k, v, g = _rand_inputs(50, B=2, T=21, C=4, k_std=1.5)
    y = o.forward_direct(w, u, k, v)
    for rv, s in ((np.log(3.0), 0.75), (0.0, 0.5), (-np.log(3.0), 0.25), (40.0, 1.0)):
        _close(o.forward_gated(w, u, k, v, np.full_like(k, rv)), s * y, 1e-14, 1e-15, f"gate at r={rv:.3f}")
    gw, gu, gk, gv, gr = o.backward_gated(w, u, k, v, np.full_like(k, 40.0), g)
    for got, want, n in zip((gw, gu, gk, gv), o.backward_adjoint(w, u, k, v, g), ("gw", "gu", "gk", "gv")):
        _close(got, want, 1e-14, 1e-15, f"r=40 {n}")
    assert np.all(np.abs(gr) <= 5e-18 * np.abs(g * y) + 1e-300), "r=40 gr"


def pin_gate_recurrent_form(o):
    """The gated output through the recurrent form (the form the CPU baseline
    times) equals the gated direct sums, and at the exact sigmoid points the
    pinned direct wkv times 3/4, 1/2, 1/4."""
    for seed in (55, 56):
        w, u, k, v, _ = _rand_inputs(seed, B=2, T=40, C=4, k_std=2.0)
        r = _rng(seed + 7).normal(0, 2.0, k.shape)
        _close(o.forward_gated_recurrent(w, u, k, v, r), o.forward_gated(w, u, k, v, r), 1e-12, 1e-13,
               f"gated recurrent vs direct seed {seed}")
    y = o.forward_direct(w, u, k, v)
    for rv, s in ((np.log(3.0), 0.75), (0.0, 0.5), (-np.log(3.0), 0.25)):
        _close(o.forward_gated_recurrent(w, u, k, v, np.full_like(k, rv)), s * y, 1e-12, 1e-13,
               f"gated recurrent at r={rv:.3f}")


def pin_gate_finite_differences(o):
    """Central differences of sum(gout * sigmoid(r) * wkv) in float64 on tiny
    inputs give all five gradients of the gated backward pass."""
    names = ("w", "u", "k", "v", "r")
    for seed in (60, 61):
        w, u, k, v, gout = _rand_inputs(seed, B=2, T=5, C=3, k_std=1.5)
        r = _rng(seed + 100).normal(0, 1.5, k.shape)
        params = dict(zip(names, (w, u, k, v, r)))

        def loss(p):
            return float(np.sum(gout * o.forward_gated(*(p[n] for n in names))))

        got = dict(zip(names, o.backward_gated(w, u, k, v, r, gout)))
        for name, arr in params.items():
            fd = np.zeros_like(arr)
            for idx in np.ndindex(arr.shape):
                h = 1e-6 * max(1.0, abs(arr[idx]))
                plus = {n: a.copy() for n, a in params.items()}
                minus = {n: a.copy() for n, a in params.items()}
                plus[name][idx] += h
                minus[name][idx] -= h
                fd[idx] = (loss(plus) - loss(minus)) / (2 * h)
            scale = max(1.0, float(np.max(np.abs(fd))))
            _close(got[name], fd, 0.0, 1e-7 * scale, f"gated FD g{name} seed {seed}")


def pin_channel_mix(o):
    """Squared ReLU: zero for k <= 0 and k^2 above (hand values); the channel
    mix's gate at the exact sigmoid points; the gate equals the time-mixing
    output's gate applied to the pinned wkv; central finite differences of
    sum(ga * a) and sum(gout * sigmoid(r) * vk) give both backward passes."""
    k = np.array([-3.0, -0.5, 0.0, 0.25, 1.0, 7.0])
    _close(o.sqrelu(k), [0.0, 0.0, 0.0, 0.0625, 1.0, 49.0], 0.0, 0.0, "sqrelu hand values")
    rng = _rng(90)
    vk = rng.normal(0, 1, (3, 7, 5))
    for rv, s in ((np.log(3.0), 0.75), (0.0, 0.5), (-np.log(3.0), 0.25), (40.0, 1.0)):
        _close(o.cmix_gate(np.full_like(vk, rv), vk), s * vk, 1e-15, 0.0, f"cmix gate at r={rv:.3f}")
    w, u, kk, v, _ = _rand_inputs(91, B=2, T=9, C=3)
    r = rng.normal(0, 2, kk.shape)
    _close(o.cmix_gate(r, o.forward_direct(w, u, kk, v)), o.forward_gated(w, u, kk, v, r), 1e-15, 1e-16,
           "cmix gate vs time-mixing gate")
    x = rng.normal(0, 1.5, (4, 6))
    x[np.abs(x) < 1e-3] = 0.5  # keep central differences off the kink at 0
    g = rng.normal(0, 1, x.shape)
    h = 1e-6
    fd = np.zeros_like(x)
    for idx in np.ndindex(x.shape):
        xp, xm = x.copy(), x.copy()
        xp[idx] += h
        xm[idx] -= h
        fd[idx] = (np.sum(g * o.sqrelu(xp)) - np.sum(g * o.sqrelu(xm))) / (2 * h)
    _close(o.sqrelu_backward(x, g), fd, 0.0, 1e-7 * max(1.0, np.abs(fd).max()), "FD sqrelu")
    r = rng.normal(0, 1.5, x.shape)
    gr, gvk = o.cmix_gate_backward(r, x, g)
    for name, arr, got in (("r", r, gr), ("vk", x, gvk)):
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            ap, am = arr.copy(), arr.copy()
            ap[idx] += h
            am[idx] -= h
            args_p = (ap, x) if name == "r" else (r, ap)
            args_m = (am, x) if name == "r" else (r, am)
            fd[idx] = (np.sum(g * o.cmix_gate(*args_p)) - np.sum(g * o.cmix_gate(*args_m))) / (2 * h)
        _close(got, fd, 0.0, 1e-7 * max(1.0, np.abs(fd).max()), f"FD cmix gate g{name}")


ALL_PINS = [
    pin_forward_hand_values,
    pin_forward_forms_agree,
    pin_forward_t1_is_v,
    pin_forward_constant_v,
    pin_forward_convex,
    pin_forward_affine,
    pin_forward_k_shift,
    pin_forward_causal_and_independent,
    pin_forward_limits,
    pin_backward_hand_values,
    pin_backward_finite_differences,
    pin_backward_forms_agree,
    pin_backward_identities,
    pin_backward_state,
    pin_forward_state_split,
    pin_state_fold,
    pin_token_shift,
    pin_state_definition,
    pin_decode_hand_values,
    pin_decode_matches_forward,
    pin_gate_special_values,
    pin_gate_recurrent_form,
    pin_gate_finite_differences,
    pin_channel_mix,
]


def failing_pins(o):
    """Names of the pins that fail on oracle handle ``o``."""
    bad = []
    for pin in ALL_PINS:
        try:
            pin(o)
        except AssertionError:
            bad.append(pin.__name__)
        except (FloatingPointError, ValueError, ZeroDivisionError, OverflowError):
            bad.append(pin.__name__)
    return bad

