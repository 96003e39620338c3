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
//   summary  the forward state from the forward pass's checkpoint at the
//            fixed scale e^{F}, F = max k of the chunk; in the same forward
//            sweep the chunk's zero-carry adjoint at its first token,
//            la = sum_t e^{-(t-t0) w} gN_t (lb likewise with gD), published
//            as a tagged record (ek = e^{k - F} is kept in place of k);
//   finish   the adjoint carried into the chunk's end, from the walker; the
//            forward states again (b in registers, a in registers), then the
//            reverse pass with the carry: gk, gv, and this tile's partial
//            sums of gw, gu (a second kernel adds the partials in a fixed
//            order, so the result is deterministic).
// Walker warps carry the adjoint along each chain from the last chunk:
// X_j = zero-carry_j + e^{-Lw} X_{j+1}, a fold in a fixed order, written as
// tagged records for the previous chunk's tiles.
//
// At the fixed scale e^{F} (la carried as la e^{F}), every factor is a plain
// product: e^{u+k} = ek e^{u}, la e^{k} = (la e^{F}) ek, la a = (la e^{F})
// (a e^{-F}).  The bounds that keep it exact in fp32 are those of the forward
// pass (wkv_fwd.cu); lanes outside them take the per-token running-maximum
// form, with the adjoints scaled by e^{pp_t} per token.
#include "wkv_adjoint.cuh"
#include "wkv_common.cuh"
#include "wkv_internal.h"
#include "wkv_pipe.cuh"

namespace wkv {

namespace {

constexpr int kBwdStages = 2;
constexpr float kFastRange = 69.f;
constexpr float kFastCeil = 60.f;
constexpr int kWalkCap = 16;   // chains per walker whose state stays in shared memory
constexpr int kWalkRing = 8;   // records requested together by a walker
// walker shared memory (see bwd_walker)
constexpr size_t kWalkSmem = (size_t)kWalkCap * (96 + 32 + 32) * sizeof(float) + (size_t)kWalkRing * 32 * 16;
static_assert((kWalkCap * (96 + 32 + 32) * sizeof(float)) % 16 == 0, "the record ring must be 16-byte aligned");
static_assert(2 * 3 * kChunk * kCtaChannels * 4 + kWalkSmem + 1024 <= 114 * 1024, "two backward CTAs per SM");

// What a consumer lane keeps of a tile between its summary and its finish.
struct BwdPend {
  int j, b, c, len;
  bool live;  // the warp has channels in this tile
  bool fast;
  float w, u, ew, eu, F, s0;
  State P;
};

__device__ __forceinline__ void bwd_summary(const BwdArgs& a, const Launch& L, float* __restrict__ sk,
                                            const float* __restrict__ sv,
                                            const float* __restrict__ sg, BwdPend& p, float* xa, float* xb,
                                            float* xp) {
  constexpr int S = kCtaChannels;
  const ScanGeometry& g = a.g;
  const int cc = p.c < g.C ? p.c : g.C - 1;
  p.P = empty_state();
  if (p.j > 0) {
    const size_t o = ((size_t)(p.j - 1) * g.B + p.b) * g.C + cc;
    p.P = State{__ldg(a.ckpt + o), __ldg(a.ckpt + o + g.plane), __ldg(a.ckpt + o + 2 * g.plane)};
  }
  float F = -3.0e38f, kmin = 3.0e38f;
#pragma unroll 8
  for (int i = 0; i < p.len; ++i) {
    const float k = sk[i * S];
    F = fmaxf(F, k);
    kmin = fminf(kmin, k);
  }
  p.F = F;
  p.fast = (kmin + fminf(p.u, 0.f) >= F - kFastRange) && (p.u <= kFastCeil) && (p.P.pp - F <= kFastCeil);
  float la, lb;
  if (p.fast) {
    // forward states at scale e^{F}; the zero-carry adjoint at the chunk
    // start accumulates in the same sweep, each token's gN, gD weighted by
    // e^{-(t - t0) w}
    const float F2 = F * kLog2e;
    p.s0 = exp_nat(p.P.pp - F);
    float na = p.P.num * p.s0, nb = p.P.den * p.s0, pw = 1.f;
    la = 0.f;
    lb = 0.f;
#pragma unroll 8
    for (int i = 0; i < p.len; ++i) {
      const float ek = ex2(fmaf(sk[i * S], kLog2e, -F2));
      sk[i * S] = ek;
      const float vv = sv[i * S];
      const float ec = ek * p.eu;
      const float rr = rcp(nb + ec);
      const float gi = sg[i * S] * rr;         // gN at scale e^{F}
      const float y = fmaf(ec, vv, na) * rr;   // wkv_t
      la = fmaf(pw, gi, la);
      lb = fmaf(-pw, gi * y, lb);
      pw *= p.ew;
      na = fmaf(na, p.ew, ek * vv);
      nb = fmaf(nb, p.ew, ek);
    }
    // from scale e^{F} to the record's scale e^{P.pp}
    la *= p.s0;
    lb *= p.s0;
  } else {
    exact_states<kCtaChannels>(sk, sv, p.len, p.P, p.w, xa, xb, xp);
    exact_zero_adjoint<kCtaChannels>(sk, sv, sg, p.len, p.w, p.u, xa, xb, xp, la, lb);
  }
  if (p.j > 0 && p.j != a.debug_skip_chunk && p.c < g.C)  // chunk 0's adjoint is never needed
    rec_store(a.ragg + ((size_t)p.j * g.B + p.b) * g.C + p.c, L.tag, la, lb, p.P.pp);
}

// gk, gv and the gw, gu partials of a tile, given the adjoint X carried
// into its chunk's end (ignored for the last chunk).
template <bool FULL>
__device__ __forceinline__ void bwd_finish(const BwdArgs& a, const float* __restrict__ sk,
                                           const float* __restrict__ sv, const float* __restrict__ sg,
                                           const BwdPend& p, const Adj& X, float* xa, float* xb, float* xp) {
  constexpr int L = kChunk;
  constexpr int S = kCtaChannels;
  const ScanGeometry& g = a.g;
  const bool valid = p.c < g.C;
  const size_t slot = ((size_t)p.j * g.B + p.b) * g.C + (valid ? p.c : g.C - 1);
  const bool has_succ = p.j < g.nchunks - 1;
  float gw_acc = 0.f, gu_acc = 0.f;
  float* __restrict__ gkp = a.gk + ((int64_t)p.b * g.T + (int64_t)p.j * L) * g.C + p.c;
  float* __restrict__ gvp = a.gv + ((int64_t)p.b * g.T + (int64_t)p.j * L) * g.C + p.c;
  if (p.fast) {
    // forward sums before each token at scale e^{F}, from the stored ek
    float A[L], Bd[L];
    float na = p.P.num * p.s0, nb = p.P.den * p.s0;
#pragma unroll
    for (int i = 0; i < L; ++i) {
      if (FULL || i < p.len) {
        const float ek = sk[i * S];
        const float vv = sv[i * S];
        A[i] = na;
        Bd[i] = nb;
        na = fmaf(na, p.ew, ek * vv);
        nb = fmaf(nb, p.ew, ek);
      }
    }
    // reverse pass with the carry (at scale e^{F})
    const float f = has_succ ? exp_nat(p.F - X.f) : 0.f;
    float la = X.la * f, lb = X.lb * f;
#pragma unroll
    for (int i = L - 1; i >= 0; --i) {
      if (FULL || i < p.len) {
        const float ek = sk[i * S];
        const float vv = sv[i * S];
        const float ec = ek * p.eu;
        const float rr = rcp(Bd[i] + ec);
        const float gi = sg[i * S] * rr;
        const float vmy = fmaf(vv, Bd[i], -A[i]) * rr;  // v - wkv
        const float cur = gi * vmy * ec;                // (gN v + gD) e^{u+k}
        const float gk = fmaf(fmaf(la, vv, lb), ek, cur);
        const float gv = fmaf(gi, ec, la * ek);
        gu_acc += cur;
        gw_acc += fmaf(la, A[i], lb * Bd[i]);  // the two nearly cancelling terms first
        la = fmaf(la, p.ew, gi);
        lb = fmaf(lb, p.ew, -gi * (vv - vmy));
        if (valid) {
          __stcs(gkp + (int64_t)i * g.C, gk);
          __stcs(gvp + (int64_t)i * g.C, gv);
        }
      }
    }
    gw_acc *= -p.ew;
  } else {
    const float pp_end = exact_states<kCtaChannels>(sk, sv, p.len, p.P, p.w, xa, xb, xp);
    const float f = has_succ ? exp_nat(pp_end - X.f) : 0.f;
    float res[4];
    exact_final<kCtaChannels>(sk, sv, sg, p.len, p.w, p.u, xa, xb, xp, X.la * f, X.lb * f, gkp, gvp, g.C, valid, res);
    gw_acc = res[0];
    gu_acc = res[1];
  }
  if (valid) {
    a.part[slot] = gw_acc;
    a.part[slot + g.plane] = gu_acc;
  }
}

// The walkers (see the forward pass): walker x owns the chains q = x + m *
// gridDim.x and takes them chunk by chunk from the last chunk (for each
// chunk, each of its chains).  Chunk 0's adjoint is never needed, so chunks
// nchunks-1 .. 1.  Walker shared memory, per chain qi < kWalkCap: adjoint
// [3][32] f32 (la, lb, f), chunk decay L*w [32] f32, this lane's element
// offset [32] i32 (bit 31 set when the lane's channel is past C); then the
// record ring [kWalkRing][32].
__device__ __forceinline__ float* walk_state(float* pst, int qi) { return pst + qi * 96; }
__device__ __forceinline__ float* walk_w(float* pst) { return pst + kWalkCap * 96; }
__device__ __forceinline__ int* walk_off(float* pst) { return reinterpret_cast<int*>(pst + kWalkCap * 128); }

__device__ __noinline__ int walk_off_slow(const ScanGeometry& g, int qi) {
  const int q = (int)blockIdx.x + qi * (int)gridDim.x;
  const int b = q / g.nwg;
  const int c = (q - b * g.nwg) * 32 + (int)(threadIdx.x & 31);
  return c < g.C ? b * g.C + c : (b * g.C + g.C - 1) | (int)0x80000000;
}

__device__ __forceinline__ int walk_offset(const ScanGeometry& g, float* pst, int mq, int qi) {
  return mq <= kWalkCap ? walk_off(pst)[qi * 32 + (threadIdx.x & 31)] : walk_off_slow(g, qi);
}

// One item: the adjoint at the start of chunk j of chain qi from the chunk's
// zero-carry record s and the adjoint at the start of chunk j + 1.
// Inlined once into the walker's rolled loop (see the forward walker).
// A walker with a single chain keeps its adjoint, chunk decay and offset
// here, in registers (the common case: fewer chains than CTAs).
struct WalkOne {
  Adj X;
  float Lw;
  int eo;
};

__device__ __forceinline__ void bwd_walk_item(const BwdArgs& a, const Launch& L, float* pst, int mq, int j, int qi,
                                              Rec s, WalkOne& one) {
  const ScanGeometry& g = a.g;
  const int lane = threadIdx.x & 31;
  const int eo = mq == 1 ? one.eo : walk_offset(g, pst, mq, qi);
  const bool valid = eo >= 0;
  const size_t o = (size_t)j * g.B * g.C + (eo & 0x7fffffff);
  const bool in_smem = mq <= kWalkCap;
  float* ps = walk_state(pst, qi) + lane;
  Adj X{rec_x(s), rec_y(s), rec_z(s)};
  if (j < g.nchunks - 1) {
    Adj nx;
    if (mq == 1) {
      nx = one.X;
    } else if (in_smem) {
      nx = Adj{ps[0], ps[32], ps[64]};
    } else {
      const Rec r = rec_load(a.rinc + o + (size_t)g.B * g.C);  // written by this lane mq items ago
      nx = Adj{rec_x(r), rec_y(r), rec_z(r)};
    }
    const float Lw = mq == 1 ? one.Lw
                             : (in_smem ? walk_w(pst)[qi * 32 + lane] : (float)kChunk * __ldg(a.w + (eo & 0x7fffffff) % g.C));
    X = fold_adj(X, Lw, nx);
  }
  if (valid) rec_store(a.rinc + o, L.tag, X.la, X.lb, X.f);
  if (mq == 1) {
    one.X = X;
  } else if (in_smem) {
    ps[0] = X.la;
    ps[32] = X.lb;
    ps[64] = X.f;
  }
}

__device__ __forceinline__ void bwd_walker(const BwdArgs& a, const Launch& L, float* pst) {
  const ScanGeometry& g = a.g;
  const int lane = threadIdx.x & 31;
  const int nchain = g.B * g.nwg;
  const int x = blockIdx.x, G = gridDim.x;
  if (x >= nchain || g.nchunks < 2) return;
  const int mq = (nchain - 1 - x) / G + 1;
  const bool in_smem = mq <= kWalkCap;
  const long nitems = (long)(g.nchunks - 1) * mq;
  const size_t jstride = (size_t)g.B * g.C;
  if (in_smem) {
    for (int qi = 0; qi < mq; ++qi) {
      const int eo = walk_off_slow(g, qi);
      walk_off(pst)[qi * 32 + lane] = eo;
      walk_w(pst)[qi * 32 + lane] = (float)kChunk * __ldg(a.w + (eo & 0x7fffffff) % g.C);
    }
  }
  Rec* ring = reinterpret_cast<Rec*>(walk_off(pst) + kWalkCap * 32);  // [kWalkRing][32]
  __syncwarp();
  WalkOne one;
  one.eo = walk_off_slow(g, 0);
  one.Lw = (float)kChunk * __ldg(a.w + (one.eo & 0x7fffffff) % g.C);
  one.X = Adj{0.f, 0.f, 0.f};
  auto offset_of = [&](int qi) { return mq == 1 ? one.eo : walk_offset(g, pst, mq, qi); };
  const uint32_t tag = L.tag;
  // Blocks of kWalkRing items, as in the forward walker.
  int bj = g.nchunks - 1, bq = 0;  // first item of the block
  for (long base = 0; base < nitems; base += kWalkRing) {
    const int nb = (int)min((long)kWalkRing, nitems - base);
    int done = 0, cj = bj, cq = bq;
    bool first = true;
    uint64_t t0 = globaltimer();
    while (done < nb) {
      int j = cj, qi = cq;
      for (int r = done; r < nb; ++r) {
        Rec* slot = ring + r * 32 + lane;
        if (first || !rec_ok(*slot, tag))
          cp_async16(slot, a.ragg + (size_t)j * jstride + (offset_of(qi) & 0x7fffffff));
        if (++qi == mq) {
          qi = 0;
          --j;
        }
      }
      cp_async_wait_all();
      __syncwarp();
      first = false;
      const int before = done;
      for (; done < nb; ++done) {
        const Rec rr = ring[done * 32 + lane];
        if (!__all_sync(0xffffffffu, offset_of(cq) < 0 || rec_ok(rr, tag))) break;
        bwd_walk_item(a, L, pst, mq, cj, cq, rr, one);
        if (++cq == mq) {
          cq = 0;
          --cj;
        }
      }
      if (done > before) {
        t0 = globaltimer();
        continue;
      }
      if (__shfl_sync(0xffffffffu, *(volatile const unsigned long long*)&a.eh->abort, 0) == L.epoch) return;
      if (__shfl_sync(0xffffffffu, globaltimer(), 0) - t0 > a.budget_ns) {
        if (lane == 0) record_error(a.eh, kDevErrTimeout, L.epoch);
        return;
      }
    }
    bj = cj;
    bq = cq;
  }
}

__global__ void __launch_bounds__(kPipeThreads, 2) bwd_scan_kernel(const __grid_constant__ BwdArgs a) {
  constexpr int NS = kBwdStages;
  constexpr int TILE = kChunk * kCtaChannels;
  extern __shared__ __align__(1024) unsigned char smem[];
  float* stages = reinterpret_cast<float*>(smem);  // stage s: k, v, gy at (3s + 0..2) * TILE
  auto* ctl = reinterpret_cast<PipeCtl<NS>*>(smem + (size_t)NS * 3 * TILE * sizeof(float));
  // walker shared memory (kWalkSmem bytes), 128-byte aligned
  float* pst = reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(ctl) + pipe_ctl_bytes<NS>());
  const Launch L = pipe_init(ctl, a.eh);
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
                      a.eh, L.epoch, [&](unsigned int t, int s, uint64_t* bar) {
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
  } else if (warp == kWalkerWarp) {
    bwd_walker(a, L, pst);
  } else {
    // Consumer: a tile is summarised as soon as its stage lands, and the
    // oldest summarised tile is finished once its carried adjoint is
    // published; neither step blocks the other (see the forward kernel).
    float xa[kChunk], xb[kChunk], xp[kChunk];  // per-token form's states (local memory)
    // Per-lane results of a tile's summary wait for its finish in registers,
    // one set per stage, selected with constant indices (a stage-indexed
    // array would live in local memory); the tile's coordinates come back
    // from its ticket, still in the control block until the stage is
    // released.
    float sF[NS], sS0[NS], sEw[NS], sEu[NS], sPn[NS], sPd[NS], sPp[NS];
    bool sFast[NS];
    auto decode = [&](int t, BwdPend& p) {
      const int jr = t / per_j;
      const int rem = t - jr * per_j;
      p.j = g.nchunks - 1 - jr;
      p.b = rem / g.ncb;
      const int c0 = (rem - p.b * g.ncb) * kCtaChannels + warp * 32;
      p.live = c0 < g.C;
      p.c = c0 + lane;
      p.len = min(kChunk, g.T - p.j * kChunk);
      const int cc = p.c < g.C ? p.c : g.C - 1;
      p.w = __ldg(a.w + cc);
      p.u = __ldg(a.u + cc);
    };
    int ns = 0, nf = 0, count = 0;
    uint32_t ps = 0;
    bool end = false, failed = false, idle = false;
    uint64_t idle_since = 0;
    while (true) {
      bool progress = false;
      while (!end && count < NS && __all_sync(0xffffffffu, mbar_test(&ctl->full[ns], ps))) {
        const int t = *(volatile int*)&ctl->tile[ns];
        if (t < 0) {
          end = true;
          break;
        }
        BwdPend p;
        decode(t, p);
        if (p.live && !failed) {
          p.ew = expf(-p.w);
          p.eu = expf(p.u);
          float* sk = stages + (size_t)(3 * ns) * TILE + warp * 32 + lane;
          bwd_summary(a, L, sk, sk + TILE, sk + 2 * TILE, p, xa, xb, xp);
#pragma unroll
          for (int q = 0; q < NS; ++q) {
            if (q == ns) {
              sF[q] = p.F;
              sS0[q] = p.s0;
              sEw[q] = p.ew;
              sEu[q] = p.eu;
              sPn[q] = p.P.num;
              sPd[q] = p.P.den;
              sPp[q] = p.P.pp;
              sFast[q] = p.fast;
            }
          }
        }
        ++count;
        if (++ns == NS) {
          ns = 0;
          ps ^= 1u;
        }
        progress = true;
      }
      if (count > 0) {
        BwdPend p;
        decode(*(volatile int*)&ctl->tile[nf], p);
        bool ready = true;
        Adj X{0.f, 0.f, 0.f};
        if (p.live && !failed && p.j < g.nchunks - 1) {
          const bool valid = p.c < g.C;
          const Rec r = rec_load(a.rinc + ((size_t)(p.j + 1) * g.B + p.b) * g.C + (valid ? p.c : 0));
          ready = __all_sync(0xffffffffu, !valid || rec_ok(r, L.tag));
          X = Adj{rec_x(r), rec_y(r), rec_z(r)};
        }
        if (ready) {
          if (p.live && !failed) {
#pragma unroll
            for (int q = 0; q < NS; ++q) {
              if (q == nf) {
                p.F = sF[q];
                p.s0 = sS0[q];
                p.ew = sEw[q];
                p.eu = sEu[q];
                p.P = State{sPn[q], sPd[q], sPp[q]};
                p.fast = sFast[q];
              }
            }
            float* sk = stages + (size_t)(3 * nf) * TILE + warp * 32 + lane;
            // one predicated body for full and partial chunks: a full-chunk
            // specialisation would not fit two CTAs' registers (it spills)
            bwd_finish<false>(a, sk, sk + TILE, sk + 2 * TILE, p, X, xa, xb, xp);
            // this warp wrote into the stage; the next TMA fill must come after
            fence_proxy_async_smem();
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&ctl->empty[nf]);
          --count;
          if (++nf == NS) nf = 0;
          progress = true;
        }
      }
      if (end && count == 0) break;
      if (progress) {
        idle = false;
        continue;
      }
      // nothing to do: bounded wait for a stage or a carried adjoint
      const uint64_t now = __shfl_sync(0xffffffffu, globaltimer(), 0);
      if (!idle) {
        idle = true;
        idle_since = now;
      } else if (now - idle_since > a.budget_ns) {
        if (failed) break;  // nothing more will arrive
        if (lane == 0) {
          record_error(a.eh, kDevErrTimeout, L.epoch);
          *(volatile int*)&ctl->abort = 1;
        }
        failed = true;  // later tiles are only drained
        idle_since = now;
      }
      if (!failed && __shfl_sync(0xffffffffu, *(volatile const unsigned long long*)&a.eh->abort, 0) == L.epoch) {
        failed = true;
        if (lane == 0) *(volatile int*)&ctl->abort = 1;
      }
    }
  }
  pipe_exit(a.ticket, a.exited, a.eh, L.epoch);
}

// gw[c] = sum over the partial rows of part[0][.][c], gu likewise from
// part[1].  Block (g, sl) of 8 warps sums the rows of slice sl for the 32
// channels of group g: warp q takes rows q, q+8, ... with compensated
// (Kahan) summation, then the 8 warp sums are added in order.  With one
// slice those sums are gw, gu; with several, the last block of a group to
// finish (counted on a launch-tagged counter) adds the slice sums in slice
// order.  Every order is fixed by the shape, so the result is
// deterministic.
__global__ void __launch_bounds__(256) reduce_kernel(const ReduceArgs a) {
  __shared__ float sw[8][32], su[8][32];
  __shared__ bool last;
  // launched as a dependent of the backward scan: wait until the scan has
  // completed and its writes (the partial rows, the sequence number) are
  // visible; a no-op when launched without that dependency
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31, q = threadIdx.x >> 5;
  const int grp = blockIdx.x, sl = blockIdx.y;
  const int c = grp * 32 + lane;
  const int per = (a.rows + a.nslice - 1) / a.nslice;
  const int r0 = sl * per, r1 = min(a.rows, r0 + per);
  float s1 = 0.f, k1 = 0.f, s2 = 0.f, k2 = 0.f;
  if (c < a.C) {
    const size_t P = (size_t)a.rows * a.C;
#pragma unroll 4
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
    if (a.nslice == 1) {  // the whole sum: no slices to combine
      if (c < a.C) {
        a.gw[c] = t1;
        a.gu[c] = t2;
      }
      return;
    }
    if (c < a.C) {
      a.slices[((size_t)sl * 2) * a.C + c] = t1;
      a.slices[((size_t)sl * 2 + 1) * a.C + c] = t2;
    }
    __threadfence();
    __syncwarp();
    if (lane == 0) {
      // arrivals of this launch, tagged with the workspace's sequence number
      // (advanced by the backward scan before this kernel runs); a word left
      // by another launch (another tag) counts as zero, so the counters need
      // no reset between launches
      const uint32_t tag = tag_of(*(volatile const unsigned long long*)&a.eh->seq);
      unsigned long long old = *(volatile unsigned long long*)(a.count + grp), seen;
      do {
        seen = old;
        const unsigned long long mine = (seen >> 32) == tag ? seen + 1ull : ((unsigned long long)tag << 32) | 1ull;
        old = atomicCAS(a.count + grp, seen, mine);
      } while (old != seen);
      const unsigned int n = (seen >> 32) == tag ? (unsigned int)(seen & 0xffffffffu) + 1u : 1u;
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
  // up to 64 rows one block per channel group sums them all (8 rows a warp
  // at most): a second pass over slices would cost more than it spreads
  if (rows <= 64) return 1;
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
  const size_t smem = (size_t)NS * 3 * kChunk * kCtaChannels * sizeof(float) + pipe_ctl_bytes<NS>() + kWalkSmem;
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
  return launch_cooperative(bwd_scan_kernel, nblk, smem, s, a);
}

// The reduction is a programmatic dependent of the backward scan launched
// just before it on the stream: it may be scheduled while the scan's last
// CTAs finish (the scan signals griddepcontrol.launch_dependents at its
// start), and its griddepcontrol.wait holds it until the scan is complete.
cudaError_t launch_reduce(const ReduceArgs& a, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((a.C + 31) / 32, a.nslice);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, reduce_kernel, a);
}

// The device-wide error record of this file's kernels (wkv_sync_status).
cudaError_t take_error_bwd(unsigned int* code) { return take_module_error(code); }

}  // namespace wkv
