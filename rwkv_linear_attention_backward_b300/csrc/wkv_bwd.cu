// wkv_bwd.cu -- WKV backward pass: reverse-time chunked scan.
//
// Gradients of every parameter are needed for training (qiita "RWKV について
// の調査記録", section "Trainingについて"); the pages give no formulas, so
// they are derived by reverse-mode differentiation of the recurrence.  With
// a_t, b_t the sums before token t, D_t = b_t + e^{u+k_t}, wkv_t the output,
// gN_t = gy_t / D_t, gD_t = -gy_t wkv_t / D_t, and the adjoints
// la_t = dL/da_t, lb_t = dL/db_t (zero after the last token):
//
//   la_t = gN_t + e^{-w} la_{t+1},         lb_t = gD_t + e^{-w} lb_{t+1}
//   gk_t = (gN_t v_t + gD_t) e^{u+k_t} + (la_{t+1} v_t + lb_{t+1}) e^{k_t}
//   gv_t = gN_t e^{u+k_t} + la_{t+1} e^{k_t}
//   gu  += (gN_t v_t + gD_t) e^{u+k_t}
//   gw  += -e^{-w} (la_{t+1} a_t + lb_{t+1} b_t)
//
// The adjoint recurrence is linear with a data-independent decay, so it is
// scanned in chunks like the forward pass, from the last chunk backwards.  A
// tile is (chunk j, batch row b, 128 channels) with k, v, gy staged in
// shared memory by the producer warp (wkv_pipe.cuh).  Per tile and lane:
//
//   1. the forward state before every token of the chunk, recomputed from
//      the forward pass's checkpoint at the fixed scale e^{F}, F = max k of
//      the chunk (a kept in shared memory in place of k, b in registers);
//   2. reverse pass with a zero carry: gN per token (kept in shared memory
//      in place of gy) and the chunk's own adjoint summary, published for
//      the look-back (wkv_common.cuh);
//   3. look-back over the later chunks: the adjoint carried into the chunk's
//      end, and the inclusive record of this chunk;
//   4. reverse pass with the carry: gk, gv, and this tile's partial sums of
//      gw, gu; a second kernel adds the partials in a fixed order, so the
//      result is deterministic.
//
// At the fixed scale e^{F} (la carried as la e^{F}), every factor is a plain
// product: e^{u+k} = ek e^{u}, la e^{k} = (la e^{F}) ek, la a = (la e^{F})
// (a e^{-F}).  The bounds that keep it exact in fp32 are those of the forward
// pass (wkv_fwd.cu); lanes outside them take the per-token running-maximum
// form, with the adjoints scaled by e^{pp_t} per token.
#include "wkv_common.cuh"
#include "wkv_internal.h"
#include "wkv_pipe.cuh"

namespace wkv {

namespace {

constexpr int kBwdStages = 2;
constexpr float kFastRange = 69.f;
constexpr float kFastCeil = 60.f;

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
  const float e = exp_nat((A.f - Lw) - X.f);
  return Adj{fmaf(e, X.la, A.la), fmaf(e, X.lb, A.lb), A.f};
}

__device__ __forceinline__ Adj load_adj(const float* rec, size_t plane, size_t o) {
  return Adj{__ldcg(rec + o), __ldcg(rec + o + plane), __ldcg(rec + o + 2 * plane)};
}

__device__ __forceinline__ void store_adj(float* rec, size_t plane, size_t o, const Adj& x) {
  rec[o] = x.la;
  rec[o + plane] = x.lb;
  rec[o + 2 * plane] = x.f;
}

// The per-token (running-maximum) form for lanes outside the fixed scale's
// bounds.  Rare, so its loops stay rolled with the per-token states (num,
// den, pp before each token) in local memory, leaving the fast form's
// registers alone.  Pass 1: the states and the zero-carry adjoint at the chunk start,
// scaled by e^{P.pp}.
__device__ __forceinline__ void exact_prepass(const float* sk, const float* sv, const float* sg, int len, State s,
                                           float w, float u, float* xa, float* xb, float* xp, float* out) {
  constexpr int S = kCtaChannels;
#pragma unroll 1
  for (int i = 0; i < len; ++i) {
    xa[i] = s.num;
    xb[i] = s.den;
    xp[i] = s.pp;
    step(s, sk[i * S], sv[i * S], w);
  }
  float la = 0.f, lb = 0.f;
#pragma unroll 1
  for (int i = len - 1; i >= 0; --i) {
    const Local o = local_terms(State{xa[i], xb[i], xp[i]}, sk[i * S], sv[i * S], sg[i * S], w, u);
    la = carry(o.t, la, o.gb);
    lb = carry(o.t, lb, -o.gb * o.y);
  }
  out[0] = la;
  out[1] = lb;
  out[2] = s.pp;  // pp after the chunk
}

// Pass 2: gk, gv with the carry (la, lb, scaled by e^{pp after the chunk});
// out[0..1] receive the gw, gu partial sums.
__device__ __forceinline__ void exact_final(const float* sk, const float* sv, const float* sg, int len, float w, float u,
                                         const float* xa, const float* xb, const float* xp, float la, float lb,
                                         float* gkp, float* gvp, int64_t C, bool valid, float* out) {
  constexpr int S = kCtaChannels;
  float gw_acc = 0.f, gu_acc = 0.f;
#pragma unroll 1
  for (int i = len - 1; i >= 0; --i) {
    const State si{xa[i], xb[i], xp[i]};
    const float k = sk[i * S], v = sv[i * S];
    const Local o = local_terms(si, k, v, sg[i * S], w, u);
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
    }
  }
  out[0] = gw_acc;
  out[1] = gu_acc;
}

// One consumer warp's share (32 channels) of one tile.  The fast form also
// writes into the stage: the forward sum a in place of k, gN in place of gy.
template <bool FULL>
__device__ __forceinline__ void bwd_tile(const BwdArgs& a, float* sk, const float* sv, float* sg, int j, int b, int wg,
                                         int c, int len) {
  constexpr int L = kChunk;
  constexpr int S = kCtaChannels;
  const ScanGeometry& g = a.g;
  const int lane = threadIdx.x & 31;
  const bool valid = c < g.C;
  const int cc = valid ? c : g.C - 1;
  const float w = __ldg(a.w + cc);
  const float u = __ldg(a.u + cc);
  sk += lane;
  sv += lane;
  sg += lane;
  const size_t P3 = g.plane;
  const size_t jstride = (size_t)g.B * g.C;
  const size_t row = (size_t)b * g.C + cc;
  const size_t slot = (size_t)j * jstride + row;

  State P = empty_state();
  if (j > 0) {
    const size_t o = (size_t)(j - 1) * jstride + row;
    P = State{__ldg(a.ckpt + o), __ldg(a.ckpt + o + P3), __ldg(a.ckpt + o + 2 * P3)};
  }

  float kr[L];
  float F = -3.0e38f, kmin = 3.0e38f;
#pragma unroll
  for (int i = 0; i < L; ++i) {
    if (FULL || i < len) {
      kr[i] = sk[i * S];
      F = fmaxf(F, kr[i]);
      kmin = fminf(kmin, kr[i]);
    }
  }
  const float ew = expf(-w);
  const float eu = expf(u);
  const bool fast = (kmin + fminf(u, 0.f) >= F - kFastRange) && (u <= kFastCeil) && (P.pp - F <= kFastCeil);

  float Bd[L];                // fast form: forward sum b before each token at scale e^{F}
  float xa[L], xb[L], xp[L];  // per-token form: (num, den, pp) before each token (local memory)
  float la = 0.f, lb = 0.f;
  float pp_end = 0.f;
  float s0 = 0.f;
  if (fast) {
    // 1. forward states at scale e^{F}: b in registers, a in place of k
    const float F2 = F * kLog2e;
    s0 = exp_nat(P.pp - F);
    float na = P.num * s0, nb = P.den * s0;
#pragma unroll
    for (int i = 0; i < L; ++i) {
      if (FULL || i < len) {
        const float ek = ex2(fmaf(kr[i], kLog2e, -F2));
        kr[i] = ek;
        const float vv = sv[i * S];
        sk[i * S] = na;
        Bd[i] = nb;
        na = fmaf(na, ew, ek * vv);
        nb = fmaf(nb, ew, ek);
      }
    }
    // 2. reverse pass with a zero carry; gN kept in place of gy
#pragma unroll
    for (int i = L - 1; i >= 0; --i) {
      if (FULL || i < len) {
        const float ek = kr[i];
        const float vv = sv[i * S];
        const float ai = sk[i * S];
        const float rr = rcp(fmaf(ek, eu, Bd[i]));
        const float gi = sg[i * S] * rr;             // gN at scale e^{F}
        const float vmy = fmaf(vv, Bd[i], -ai) * rr;  // v - wkv
        sg[i * S] = gi;
        la = fmaf(la, ew, gi);
        lb = fmaf(lb, ew, -gi * (vv - vmy));
      }
    }
    // from scale e^{F} to the record's scale e^{P.pp}
    la *= s0;
    lb *= s0;
  } else {
    float res[3];
    exact_prepass(sk, sv, sg, len, P, w, u, xa, xb, xp, res);
    la = res[0];
    lb = res[1];
    pp_end = res[2];
  }

  const float Lw = (float)L * w;
  const Adj own{la, lb, P.pp};
  uint64_t* flag = a.flags + ((size_t)j * g.B + b) * g.nwg + wg;
  const bool has_pred = j > 0;
  const bool has_succ = j < g.nchunks - 1;
  const bool skip = j == a.debug_skip_chunk;  // fault injection: this tile never publishes

  // 3. look-back over the later chunks
  Adj X{0.f, 0.f, 0.f};
  if (has_succ) {
    if (has_pred && !skip) {
      if (valid) store_adj(a.ragg, P3, slot, own);
      publish(flag, a.epoch, kAgg);
    }
    const int nwin = min(g.nchunks - 1 - j, 32);
    int base = 0;
    const int rc = lookback_wait(
        [&](int i) { return a.flags + ((size_t)(j + 1 + i) * g.B + b) * g.nwg + wg; }, nwin, a.epoch, a.budget_ns,
        a.eh, base);
    if (rc != kWaitOk) {
      if (rc == kWaitTimeout && lane == 0) record_error(a.eh, kDevErrTimeout, a.epoch);
      if (has_pred && !skip) publish(flag, a.epoch, kErr);
      return;
    }
    X = load_adj(a.rinc, P3, (size_t)(j + 1 + base) * jstride + row);
    // fold the records of chunks j + base .. j + 1, the furthest first
    for (int i = base - 1; i >= 0; i -= 4) {
      Adj q[4];
#pragma unroll
      for (int m = 0; m < 4; ++m)
        if (i - m >= 0) q[m] = load_adj(a.ragg, P3, (size_t)(j + 1 + (i - m)) * jstride + row);
#pragma unroll
      for (int m = 0; m < 4; ++m)
        if (i - m >= 0) X = fold_adj(q[m], Lw, X);
    }
  }
  if (has_pred && !skip) {
    const Adj incl = has_succ ? fold_adj(own, Lw, X) : own;
    if (valid) store_adj(a.rinc, P3, slot, incl);
    publish(flag, a.epoch, kIncl);
  }

  // 4. reverse pass with the carry
  float gw_acc = 0.f, gu_acc = 0.f;
  float* gkp = a.gk + ((int64_t)b * g.T + (int64_t)j * L) * g.C + cc;
  float* gvp = a.gv + ((int64_t)b * g.T + (int64_t)j * L) * g.C + cc;
  if (fast) {
    const float f = has_succ ? exp_nat(F - X.f) : 0.f;
    la = X.la * f;
    lb = X.lb * f;
#pragma unroll
    for (int i = L - 1; i >= 0; --i) {
      if (FULL || i < len) {
        const float ek = kr[i];
        const float vv = sv[i * S];
        const float gi = sg[i * S];
        const float ai = sk[i * S];
        const float ec = ek * eu;
        const float vmy = fmaf(vv, Bd[i], -ai) * rcp(Bd[i] + ec);  // v - wkv
        const float cur = gi * vmy * ec;  // (gN v + gD) e^{u+k}
        const float gk = fmaf(fmaf(la, vv, lb), ek, cur);
        const float gv = fmaf(gi, ec, la * ek);
        gu_acc += cur;
        gw_acc = fmaf(la, ai, fmaf(lb, Bd[i], gw_acc));
        la = fmaf(la, ew, gi);
        lb = fmaf(lb, ew, -gi * (vv - vmy));
        if (valid) {
          __stcs(gkp + (int64_t)i * g.C, gk);
          __stcs(gvp + (int64_t)i * g.C, gv);
        }
      }
    }
    gw_acc *= -ew;
  } else {
    const float f = has_succ ? exp_nat(pp_end - X.f) : 0.f;
    float res[2];
    exact_final(sk, sv, sg, len, w, u, xa, xb, xp, X.la * f, X.lb * f, gkp, gvp, g.C, valid, res);
    gw_acc = res[0];
    gu_acc = res[1];
  }
  if (valid) {
    a.part[slot] = gw_acc;
    a.part[slot + P3] = gu_acc;
  }
}

__global__ void __launch_bounds__(kPipeThreads, 2) bwd_scan_kernel(const __grid_constant__ BwdArgs a) {
  constexpr int NS = kBwdStages;
  constexpr int TILE = kChunk * kCtaChannels;
  extern __shared__ __align__(1024) unsigned char smem[];
  float* stages = reinterpret_cast<float*>(smem);  // stage s: k, v, gy at (3s + 0..2) * TILE
  auto* ctl = reinterpret_cast<PipeCtl<NS>*>(smem + (size_t)NS * 3 * TILE * sizeof(float));
  pipe_init(ctl);
  const ScanGeometry& g = a.g;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int per_j = g.B * g.ncb;

  if (warp == kProducerWarp) {
    if (a.use_tma && lane == 0) {
      tma_prefetch_desc(&a.tk);
      tma_prefetch_desc(&a.tv);
      tma_prefetch_desc(&a.tg);
    }
    producer_loop<NS>(ctl, a.ticket, g.ntiles, a.use_tma != 0, (uint32_t)(3 * TILE * sizeof(float)), a.budget_ns,
                      a.eh, a.epoch, [&](unsigned int t, int s, uint64_t* bar) {
                        const int jr = t / per_j;
                        const int j = g.nchunks - 1 - jr;  // last chunk first
                        const int rem = t - jr * per_j;
                        const int b = rem / g.ncb;
                        const int cb = rem - b * g.ncb;
                        float* dk = stages + (size_t)(3 * s) * TILE;
                        if (a.use_tma) {
                          if (lane == 0) {
                            tma_load_3d(dk, &a.tk, bar, cb * kCtaChannels, j * kChunk, b);
                            tma_load_3d(dk + TILE, &a.tv, bar, cb * kCtaChannels, j * kChunk, b);
                            tma_load_3d(dk + 2 * TILE, &a.tg, bar, cb * kCtaChannels, j * kChunk, b);
                          }
                        } else {
                          copy_tile_plain(dk, a.k, g.B, g.T, g.C, b, j * kChunk, cb * kCtaChannels, kChunk);
                          copy_tile_plain(dk + TILE, a.v, g.B, g.T, g.C, b, j * kChunk, cb * kCtaChannels, kChunk);
                          copy_tile_plain(dk + 2 * TILE, a.gy, g.B, g.T, g.C, b, j * kChunk, cb * kCtaChannels,
                                          kChunk);
                        }
                      });
  } else {
    int s = 0;
    uint32_t phase = 0;
    while (true) {
      const bool ok = __all_sync(0xffffffffu, mbar_wait(&ctl->full[s], phase, a.budget_ns));
      if (!ok) {
        if (lane == 0) pipe_fail(ctl, a.eh, kDevErrTimeout, a.epoch);
        break;
      }
      const int t = *(volatile int*)&ctl->tile[s];
      if (t < 0) break;
      const int jr = t / per_j;
      const int j = g.nchunks - 1 - jr;
      const int rem = t - jr * per_j;
      const int b = rem / g.ncb;
      const int cb = rem - b * g.ncb;
      const int c0 = cb * kCtaChannels + warp * 32;
      if (c0 < g.C) {
        float* sk = stages + (size_t)(3 * s) * TILE + warp * 32;
        const int len = min(kChunk, g.T - j * kChunk);
        const int wg = cb * kConsumerWarps + warp;
        // one predicated body for full and partial chunks: the full-chunk
        // specialisation schedules more loads ahead than the register file
        // of two resident CTAs holds (it spills)
        bwd_tile<false>(a, sk, sk + TILE, sk + 2 * TILE, j, b, wg, c0 + lane, len);
        // this warp wrote into the stage; the next TMA fill must come after
        fence_proxy_async_smem();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->empty[s]);
      if (++s == NS) {
        s = 0;
        phase ^= 1u;
      }
    }
  }
  pipe_exit(a.ticket, a.exited);
}

// gw[c] = sum over the partial rows of part[0][.][c], gu likewise from
// part[1].  Block (g, sl) of 8 warps sums the rows of slice sl for the 32
// channels of group g: warp q takes rows q, q+8, ... with compensated
// (Kahan) summation, then the 8 warp sums are added in order.  The last
// block of a group to finish (counted on a launch-tagged counter) adds the
// slice sums in slice order.  Every
// order is fixed by the shape, so the result is deterministic.
__global__ void __launch_bounds__(256) reduce_kernel(const ReduceArgs a) {
  __shared__ float sw[8][32], su[8][32];
  __shared__ bool last;
  const int lane = threadIdx.x & 31, q = threadIdx.x >> 5;
  const int grp = blockIdx.x, sl = blockIdx.y;
  const int c = grp * 32 + lane;
  const int per = (a.rows + a.nslice - 1) / a.nslice;
  const int r0 = sl * per, r1 = min(a.rows, r0 + per);
  float s1 = 0.f, k1 = 0.f, s2 = 0.f, k2 = 0.f;
  if (c < a.C) {
    const size_t P = (size_t)a.rows * a.C;
    for (int r = r0 + q; r < r1; r += 8) {
      const size_t o = (size_t)r * a.C + c;
      const float y1 = a.part[o] - k1;
      const float t1 = s1 + y1;
      k1 = (t1 - s1) - y1;
      s1 = t1;
      const float y2 = a.part[o + P] - k2;
      const float t2 = s2 + y2;
      k2 = (t2 - s2) - y2;
      s2 = t2;
    }
  }
  sw[q][lane] = s1;
  su[q][lane] = s2;
  __syncthreads();
  if (q == 0) {
    float t1 = 0.f, t2 = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      t1 += sw[i][lane];
      t2 += su[i][lane];
    }
    if (c < a.C) {
      a.slices[((size_t)sl * 2) * a.C + c] = t1;
      a.slices[((size_t)sl * 2 + 1) * a.C + c] = t2;
    }
    __threadfence();
    __syncwarp();
    if (lane == 0) {
      // arrivals of this launch; a word left by another launch (another tag)
      // counts as zero, so the counters need no reset between launches
      unsigned long long old = *(volatile unsigned long long*)(a.count + grp), seen;
      do {
        seen = old;
        const unsigned long long mine = (seen >> 32) == a.tag ? seen + 1ull : ((unsigned long long)a.tag << 32) | 1ull;
        old = atomicCAS(a.count + grp, seen, mine);
      } while (old != seen);
      const unsigned int n = (seen >> 32) == a.tag ? (unsigned int)(seen & 0xffffffffu) + 1u : 1u;
      last = n == (unsigned int)a.nslice;
    }
    __syncwarp();
    if (last) {
      __threadfence();
      if (c < a.C) {
        float g1 = 0.f, g2 = 0.f;
        for (int i = 0; i < a.nslice; ++i) {
          g1 += __ldcg(a.slices + ((size_t)i * 2) * a.C + c);
          g2 += __ldcg(a.slices + ((size_t)i * 2 + 1) * a.C + c);
        }
        a.gw[c] = g1;
        a.gu[c] = g2;
      }
    }
  }
}

}  // namespace

int reduce_slices(int rows, int C) {
  const int groups = (C + 31) / 32;
  int ns = (rows + 31) / 32;
  int cap = 2 * 148 / groups;
  if (cap < 1) cap = 1;
  if (ns > cap) ns = cap;
  if (ns < 1) ns = 1;
  return ns;
}

cudaError_t launch_backward(BwdArgs& a, cudaStream_t s) {
  constexpr int NS = kBwdStages;
  const size_t smem = (size_t)NS * 3 * kChunk * kCtaChannels * sizeof(float) + sizeof(PipeCtl<NS>);
  static int grid_per_dev[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int grid = (dev >= 0 && dev < 64) ? grid_per_dev[dev] : 0;
  if (grid == 0) {
    e = cudaFuncSetAttribute(bwd_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0, sms = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, bwd_scan_kernel, kPipeThreads, smem);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    grid = (per_sm > 0 ? per_sm : 1) * sms;
    if (dev >= 0 && dev < 64) grid_per_dev[dev] = grid;
  }
  const unsigned int nblk = a.g.ntiles < (unsigned)grid ? a.g.ntiles : (unsigned)grid;
  bwd_scan_kernel<<<dim3(nblk), dim3(kPipeThreads), smem, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_reduce(const ReduceArgs& a, cudaStream_t s) {
  reduce_kernel<<<dim3((a.C + 31) / 32, a.nslice), dim3(256), 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace wkv
