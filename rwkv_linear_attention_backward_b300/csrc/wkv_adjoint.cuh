// wkv_adjoint.cuh -- pieces of the WKV backward pass shared by its kernels:
// the per-token terms of the reverse-mode recurrence, adjoint records and
// their fold across chunks, and the per-token (running-maximum) form used
// by lanes whose values leave the fixed scale's fp32 range.  The reverse
// mode of the recurrence is derived in wkv_bwd.cu.  Token stride S: the
// distance in floats between consecutive tokens of a lane's column in the
// shared-memory tile.
#pragma once

#include "wkv_common.cuh"

namespace wkv {

// Everything the per-token reverse pass needs at one token, from the state
// before it (running-maximum form).
struct Local {
  float gb;  // gy e^{pp-q} / Dhat : scaled gN
  float gc;  // gy e^{u+k-q} / Dhat : gN e^{u+k}
  float y;   // wkv_t
  float vmy; // v_t - wkv_t, formed without subtracting the two
  Decay t;   // carry factors of the forward step (same as the forward pass)
};

__device__ __forceinline__ Local local_terms(const State& s, float k, float v, float g, float w, float u) {
  Local o;
  const float d1 = s.pp - (u + k);
  const float e1 = exp_neg_abs(d1);
  const bool past = d1 >= 0.f;
  const float cp = past ? 1.f : e1;
  const float cc = past ? e1 : 1.f;
  const float inv = rcp(fmaf(cp, s.den, cc));
  o.y = fmaf(cp, s.num, cc * v) * inv;
  // v - wkv = cp (den v - num) / Dhat: exact cancellation of the current
  // token's own share, so no rounding noise when the bonus dominates
  o.vmy = cp * fmaf(s.den, v, -s.num) * inv;
  const float gi = g * inv;
  o.gb = gi * cp;
  o.gc = gi * cc;
  o.t = decay_terms(s.pp, k, w);
  return o;
}

// An adjoint record: la_true = la e^{-f}, lb_true = lb e^{-f}.
struct Adj {
  float la, lb, f;
};

// The adjoint at the start of a chunk from its own zero-carry record `A` and
// the adjoint at the start of the next chunk `X`: A + e^{-Lw} X.  The scale
// of X never exceeds A's decayed by the chunk ((A.f - Lw) - X.f <= 0: the
// forward states are running maxima), so one exponential of a non-positive
// number.
__device__ __forceinline__ Adj fold_adj(const Adj& A, float Lw, const Adj& X) {
  // __fsub_rn: never fused with the multiply that formed Lw (same roundings
  // in every kernel; see combine)
  const float e = exp_nat(__fsub_rn(A.f, Lw) - X.f);
  return Adj{fmaf(e, X.la, A.la), fmaf(e, X.lb, A.lb), A.f};
}

// The per-token (running-maximum) form for lanes outside the fixed scale's
// bounds.  Rare, so its loops stay rolled with the per-token states (num,
// den, pp before each token) in local memory, leaving the fast form's
// registers alone.  The states from P; returns pp after the chunk.  E: the
// element type of the staged k, v, gy (float or bf16).
template <int S, typename E = float>
__device__ __forceinline__ float exact_states(const E* sk, const E* sv, int len, State s, float w, float* xa,
                                              float* xb, float* xp) {
#pragma unroll 1
  for (int i = 0; i < len; ++i) {
    xa[i] = s.num;
    xb[i] = s.den;
    xp[i] = s.pp;
    step(s, to_f32<E>(sk[i * S]), to_f32<E>(sv[i * S]), w);
  }
  return s.pp;
}

// The gradient reaching wkv_t from the staged plane sg at offset o: gy
// itself (RP = 0), or, for the gated output out_t = sigmoid(r_t) wkv_t, the
// output's gradient times sigmoid(r_t), with the r plane staged RP elements
// after sg.  gq receives the factor that turns wkv_t into gr_t: gout
// sigmoid'(r) = gy (1 - sigmoid(r)) (0 without the gate).
template <int RP, typename E>
__device__ __forceinline__ float gate_grad(const E* sg, int o, float& gq) {
  const float g = to_f32<E>(sg[o]);
  if constexpr (RP == 0) {
    gq = 0.f;
    return g;
  } else {
    const float s = sigmoid(to_f32<E>(sg[o + RP]));
    const float gy = g * s;
    gq = fmaf(-gy, s, gy);
    return gy;
  }
}

// The zero-carry adjoint at the chunk start, scaled by e^{pp there}.
template <int S, typename E = float, int RP = 0>
__device__ __forceinline__ void exact_zero_adjoint(const E* sk, const E* sv, const E* sg, int len, float w, float u,
                                                   const float* xa, const float* xb, const float* xp, float& la,
                                                   float& lb) {
  la = 0.f;
  lb = 0.f;
#pragma unroll 1
  for (int i = len - 1; i >= 0; --i) {
    float gq;
    const Local o = local_terms(State{xa[i], xb[i], xp[i]}, to_f32<E>(sk[i * S]), to_f32<E>(sv[i * S]),
                                gate_grad<RP>(sg, i * S, gq), w, u);
    la = carry(o.t, la, o.gb);
    lb = carry(o.t, lb, -o.gb * o.y);
  }
}

// gk, gv with the carry (la, lb, scaled by e^{pp after the chunk});
// out[0..1] receive the gw, gu partial sums, out[2..3] the adjoint at the
// chunk start.  With the gate (RP != 0, see gate_grad) gr goes to grp.
template <int S, typename E = float, int RP = 0>
__device__ __forceinline__ void exact_final(const E* sk, const E* sv, const E* sg, int len, float w, float u,
                                            const float* xa, const float* xb, const float* xp, float la, float lb,
                                            float* gkp, float* gvp, int64_t C, bool valid, float* out,
                                            float* grp = nullptr) {
  float gw_acc = 0.f, gu_acc = 0.f;
#pragma unroll 1
  for (int i = len - 1; i >= 0; --i) {
    const State si{xa[i], xb[i], xp[i]};
    const float k = to_f32<E>(sk[i * S]), v = to_f32<E>(sv[i * S]);
    float gq;
    const Local o = local_terms(si, k, v, gate_grad<RP>(sg, i * S, gq), w, u);
    const float cur = o.gc * o.vmy;
    const float gk = fmaf(o.t.kap, fmaf(la, v, lb), cur);
    const float gv = fmaf(o.t.kap, la, o.gc);
    gu_acc += cur;
    gw_acc = fmaf(-(o.t.dec + o.t.cor), fmaf(la, si.num, lb * si.den), gw_acc);
    // the adjoint is carried back by the transpose of the forward step
    la = carry(o.t, la, o.gb);
    lb = carry(o.t, lb, -o.gb * o.y);
    if (valid) {
      __stcs(gkp + (int64_t)i * C, gk);
      __stcs(gvp + (int64_t)i * C, gv);
      if constexpr (RP != 0) __stcs(grp + (int64_t)i * C, gq * o.y);
    }
  }
  out[0] = gw_acc;
  out[1] = gu_acc;
  out[2] = la;  // adjoint at the chunk start, scaled by e^{pp there}
  out[3] = lb;
}

}  // namespace wkv
