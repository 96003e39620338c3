// wkv_fwd.cu -- WKV forward pass: single-pass chunked scan over time.
//
// The recurrent form of the operator ("RWKV解读：在Transformer的时代的新RNN",
// section "3、RWKV的网络架构": eq. (8) can be written recursively) is a
// linear recurrence whose decay is data independent, which is what makes the
// training form time-parallel (qiita "RWKV についての調査記録", section
// "Trainingについて").  Time is cut into chunks of kChunk tokens; a tile is
// (chunk j, batch row b, 128 channels), one channel per consumer lane, its k
// and v staged in shared memory by the producer warp (wkv_pipe.cuh).
//
// Consumer warps, per tile and lane:
//   summary  chunk statistics F = max k, the smallest k and the running
//            maximum at the chunk end r = max_i (k_i - (n-1-i) w); the
//            chunk's own summary (its tokens from the empty state) at the
//            fixed scale e^{F}: ek_i = e^{k_i - F} <= 1, num = num e^{-w} +
//            ek v, den = den e^{-w} + ek, rescaled to the canonical scale
//            e^{r}; published as a tagged record;
//   re-run   (after the summary of the next tile, so that waiting overlaps
//            work) the state P carried into the chunk, from the walker; the
//            outputs y = (a + e^{u} ek v) / (b + e^{u} ek) from P at scale
//            e^{F}.
// Walker warps carry the state along each chain (batch row, 32 channels)
// of chunks: P_{j+1} = P_j (+) summary_j, a left fold in chunk order (so the
// result is bitwise reproducible), written as the checkpoints and as tagged
// records for the next chunk's tiles.  A walker reads its summaries through
// a ring of prefetched records, so a long chain advances at several chunks
// per memory round trip.
//
// The fixed scale makes each element cost a few FMAs and exponentials.  It
// is exact in fp32 as long as every value the chunk handles stays within the
// fp32 range: here when every token's bonus weight ek e^{min(u,0)} is at
// least e^{-69} (then the current token's own term bounds the denominator
// from below, and any term that underflows is below 2^-24 of it), u <= 60
// and P's scale exceeds F by at most 60 (no overflow).  Lanes outside these
// bounds take the per-token running-maximum recurrence of wkv_common.cuh
// (step/output), which is exact for any finite input.
#include <cuda_bf16.h>

#include "wkv_common.cuh"
#include "wkv_internal.h"
#include "wkv_pipe.cuh"

namespace wkv {

namespace {


template <typename KV>
struct FwdStages {
  static constexpr int value = sizeof(KV) == 4 ? 3 : 4;
};

constexpr float kFastRange = 69.f;  // smallest bonus weight of the fixed scale: e^{-69}
constexpr float kFastCeil = 60.f;   // largest scale-up of the fixed scale: e^{60}
constexpr int kWalkCap = 16;        // chains per walker whose state stays in shared memory
constexpr int kWalkRing = 8;        // summaries requested together by a walker
// walker shared memory: chain states [kWalkCap][3][32] f32, decays [kWalkCap][32] f32, offsets [kWalkCap][32] i32,
// record ring [kWalkRing][32] of 16-byte records
constexpr size_t kWalkSmem = (size_t)kWalkCap * (96 + 32 + 32) * sizeof(float) + (size_t)kWalkRing * 32 * 16;
static_assert((kWalkCap * (96 + 32 + 32) * sizeof(float)) % 16 == 0, "the record ring must be 16-byte aligned");
static_assert(3 * 2 * kChunk * kCtaChannels * 4 + kWalkSmem + 1024 <= 114 * 1024, "two fp32 forward CTAs per SM");

// What a consumer lane keeps of a tile between its summary and its re-run.
struct FwdPend {
  int j, b, c, len, stage;
  bool live;   // the warp has channels in this tile
  bool fast;   // the summary used the fixed scale
  float w, u, ew, F, kmin;
};

template <typename KV>
__device__ __forceinline__ void fwd_summary(const FwdArgs& a, const Launch& L, const KV* __restrict__ sk,
                                            const KV* __restrict__ sv, FwdPend& p) {
  constexpr int S = kCtaChannels;
  const ScanGeometry& g = a.g;
  const int n = p.len;
  float F = -3.0e38f, kmin = 3.0e38f, r = -3.0e38f;
#pragma unroll 8
  for (int i = 0; i < n; ++i) {
    const float k = to_f32<KV>(sk[i * S]);
    F = fmaxf(F, k);
    kmin = fminf(kmin, k);
    r = fmaxf(r, fmaf(-(float)(n - 1 - i), p.w, k));
  }
  p.F = F;
  p.kmin = kmin;
  p.fast = kmin >= F - kFastRange;
  State s;
  if (p.fast) {
    const float F2 = F * kLog2e;
    float num = 0.f, den = 0.f;
#pragma unroll 8
    for (int i = 0; i < n; ++i) {
      const float ek = ex2(fmaf(to_f32<KV>(sk[i * S]), kLog2e, -F2));
      const float vv = to_f32<KV>(sv[i * S]);
      num = fmaf(num, p.ew, ek * vv);
      den = fmaf(den, p.ew, ek);
    }
    const float sc = exp_nat(F - r);  // >= 1: from scale e^{F} to e^{r}
    s = State{num * sc, den * sc, r};
  } else {
    s = empty_state();
#pragma unroll 1
    for (int i = 0; i < p.len; ++i) step(s, to_f32<KV>(sk[i * S]), to_f32<KV>(sv[i * S]), p.w);
  }
  if (p.j == a.debug_skip_chunk) return;  // fault injection: this chunk's summaries are never published
  if (p.c < g.C) rec_store(a.agg + ((size_t)p.j * g.B + p.b) * g.C + p.c, L.tag, s.num, s.den, s.pp);
}

// The outputs of a tile from the state P carried into its chunk.
template <typename KV, bool WRITE_Y>
__device__ __forceinline__ void fwd_rerun(const FwdArgs& a, const KV* __restrict__ sk, const KV* __restrict__ sv,
                                          const FwdPend& p, const State& P) {
  constexpr int L = kChunk;
  constexpr int S = kCtaChannels;
  const ScanGeometry& g = a.g;
  const bool valid = p.c < g.C;
  if constexpr (WRITE_Y) {
    float* __restrict__ yp = a.y + ((int64_t)p.b * g.T + (int64_t)p.j * L) * g.C + p.c;
    const float u = p.u;
    const bool fast = p.fast && (p.kmin + fminf(u, 0.f) >= p.F - kFastRange) && (u <= kFastCeil) &&
                      (P.pp - p.F <= kFastCeil);
    if (fast) {
      const float eu = expf(u);
      const float F2 = p.F * kLog2e;
      const float s0 = exp_nat(P.pp - p.F);  // P at scale e^{F}; 0 for the empty state
      float na = P.num * s0, nb = P.den * s0;
#pragma unroll 8
      for (int i = 0; i < p.len; ++i) {
        const float ek = ex2(fmaf(to_f32<KV>(sk[i * S]), kLog2e, -F2));
        const float ekv = ek * to_f32<KV>(sv[i * S]);
        // numerator e^{k-F} v e^u + a, denominator e^{k-F} e^u + b: the
        // sequential kernels' arithmetic, so both give the same outputs
        const float yv = fmaf(ekv, eu, na) * rcp(fmaf(ek, eu, nb));
        if (valid) __stcs(yp + (int64_t)i * g.C, yv);
        na = fmaf(na, p.ew, ekv);
        nb = fmaf(nb, p.ew, ek);
      }
    } else {
      State s = P;
#pragma unroll 1
      for (int i = 0; i < p.len; ++i) {
        const float kk = to_f32<KV>(sk[i * S]);
        const float vv = to_f32<KV>(sv[i * S]);
        const float yv = output(s, kk, vv, u);
        if (valid) __stcs(yp + (int64_t)i * g.C, yv);
        step(s, kk, vv, p.w);
      }
    }
  }
}

// The walkers.  Walker x (one warp per CTA) owns the chains q = x + m * G
// (G = gridDim.x, q = b * nwg + group of 32 channels) and takes their chunks
// chunk by chunk (for each chunk, each of its chains), so it never waits on
// a chunk before the chunks it still has to deliver.  With at most kWalkCap
// chains, a chain's state, decay and row offset stay in shared memory (each
// lane reads back only what it wrote); beyond that the state is read back
// from the checkpoints it wrote, kWalkRing items ahead.

// Walker shared memory, per chain qi < kWalkCap: state [3][32] f32 (num,
// den, pp), decay w [32] f32, and this lane's element offset within a chunk
// [32] i32 (b * C + channel; bit 31 set when the lane's channel is past C).
__device__ __forceinline__ float* walk_state(float* pst, int qi) { return pst + qi * 96; }
__device__ __forceinline__ float* walk_w(float* pst) { return pst + kWalkCap * 96; }
__device__ __forceinline__ int* walk_off(float* pst) { return reinterpret_cast<int*>(pst + kWalkCap * 128); }

// Element offset (bit 31: lane past C) of chain qi for this lane, computed.
__device__ __noinline__ int walk_off_slow(const ScanGeometry& g, int qi) {
  const int q = (int)blockIdx.x + qi * (int)gridDim.x;
  const int b = q / g.nwg;
  const int c = (q - b * g.nwg) * 32 + (int)(threadIdx.x & 31);
  return c < g.C ? b * g.C + c : (b * g.C + g.C - 1) | (int)0x80000000;
}

__device__ __forceinline__ int walk_offset(const ScanGeometry& g, float* pst, int mq, int qi) {
  return mq <= kWalkCap ? walk_off(pst)[qi * 32 + (threadIdx.x & 31)] : walk_off_slow(g, qi);
}

// A walker with a single chain keeps its state, decay and offset here, in
// registers (the common case: fewer chains than CTAs).
struct WalkOne {
  State P;
  float w;
  int eo;
};

// One item: the state after chunk j of chain qi from the one before it and
// the chunk's summary s.  Inlined once into the walker's rolled loop (a call
// would save registers to local memory, which misses the small L1 left
// beside the shared memory).
__device__ __forceinline__ void fwd_walk_item(const FwdArgs& a, const Launch& L, float* pst, int mq, int j, int qi,
                                              Rec s, WalkOne& one) {
  const ScanGeometry& g = a.g;
  const int lane = threadIdx.x & 31;
  const int eo = mq == 1 ? one.eo : walk_offset(g, pst, mq, qi);
  const bool valid = eo >= 0;
  const size_t o = (size_t)j * g.B * g.C + (eo & 0x7fffffff);
  const bool in_smem = mq <= kWalkCap;
  float* ps = walk_state(pst, qi) + lane;
  State P;
  if (j == 0) {
    P = load_state_planes(a.state_in, (size_t)g.B * g.C, eo & 0x7fffffff);
  } else if (mq == 1) {
    P = one.P;
  } else if (in_smem) {
    P = State{ps[0], ps[32], ps[64]};
  } else {
    const size_t op = o - (size_t)g.B * g.C;  // written by this lane mq items ago
    P = State{__ldcg(a.ckpt + op), __ldcg(a.ckpt + op + g.plane), __ldcg(a.ckpt + op + 2 * g.plane)};
  }
  const float w = mq == 1 ? one.w : (in_smem ? walk_w(pst)[qi * 32 + lane] : __ldg(a.w + (eo & 0x7fffffff) % g.C));
  const int n = j == g.nchunks - 1 ? g.T - j * kChunk : kChunk;
  P = combine(P, (float)n * w, State{rec_x(s), rec_y(s), rec_z(s)});
  if (valid) {
    const size_t P3 = g.plane;
    a.ckpt[o] = P.num;
    a.ckpt[o + P3] = P.den;
    a.ckpt[o + 2 * P3] = P.pp;
    if (j < g.nchunks - 1) rec_store(a.inc + o, L.tag, P.num, P.den, P.pp);
    if (j == g.nchunks - 1 && a.state_out) store_state_planes(a.state_out, (size_t)g.B * g.C, eo & 0x7fffffff, P);
  }
  if (mq == 1) {
    one.P = P;
  } else if (in_smem) {
    ps[0] = P.num;
    ps[32] = P.den;
    ps[64] = P.pp;
  }
}

__device__ __forceinline__ void fwd_walker(const FwdArgs& a, const Launch& L, float* pst) {
  const ScanGeometry& g = a.g;
  const int lane = threadIdx.x & 31;
  const int nchain = g.B * g.nwg;
  const int x = blockIdx.x, G = gridDim.x;
  if (x >= nchain) return;
  const int mq = (nchain - 1 - x) / G + 1;
  const bool in_smem = mq <= kWalkCap;
  const long nitems = (long)g.nchunks * mq;
  const size_t jstride = (size_t)g.B * g.C;
  if (in_smem) {
    for (int qi = 0; qi < mq; ++qi) {
      const int eo = walk_off_slow(g, qi);
      walk_off(pst)[qi * 32 + lane] = eo;
      walk_w(pst)[qi * 32 + lane] = __ldg(a.w + (eo & 0x7fffffff) % g.C);
    }
  }
  Rec* ring = reinterpret_cast<Rec*>(walk_off(pst) + kWalkCap * 32);  // [kWalkRing][32]
  __syncwarp();
  WalkOne one;
  one.eo = walk_off_slow(g, 0);
  one.w = __ldg(a.w + (one.eo & 0x7fffffff) % g.C);
  one.P = empty_state();
  auto offset_of = [&](int qi) { return mq == 1 ? one.eo : walk_offset(g, pst, mq, qi); };
  const uint32_t tag = L.tag;
  // Items are taken in blocks of kWalkRing: every record of the block not yet
  // current is copied into the ring together (one memory round trip), then
  // the current prefix is folded in order; the rest is copied again.
  int bj = 0, bq = 0;  // first item of the block
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
          cp_async16(slot, a.agg + (size_t)j * jstride + (offset_of(qi) & 0x7fffffff));
        if (++qi == mq) {
          qi = 0;
          ++j;
        }
      }
      cp_async_wait_all();
      __syncwarp();
      first = false;
      const int before = done;
      for (; done < nb; ++done) {
        const Rec rr = ring[done * 32 + lane];
        if (!__all_sync(0xffffffffu, offset_of(cq) < 0 || rec_ok(rr, tag))) break;
        fwd_walk_item(a, L, pst, mq, cj, cq, rr, one);
        if (++cq == mq) {
          cq = 0;
          ++cj;
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

template <typename KV, bool WRITE_Y>
__global__ void __launch_bounds__(kPipeThreads, 2) fwd_scan_kernel(const __grid_constant__ FwdArgs a) {
  constexpr int NS = FwdStages<KV>::value;
  constexpr int TILE = kChunk * kCtaChannels;
  extern __shared__ __align__(1024) unsigned char smem[];
  KV* stages = reinterpret_cast<KV*>(smem);  // stage s: k at 2s*TILE, v at (2s+1)*TILE
  auto* ctl = reinterpret_cast<PipeCtl<NS>*>(smem + (size_t)NS * 2 * TILE * sizeof(KV));
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
    }
    producer_loop<NS>(ctl, a.ticket, g.ntiles, a.use_tma != 0, (uint32_t)(2 * TILE * sizeof(KV)), a.budget_ns, a.eh,
                      L.epoch, [&](unsigned int t, int s, uint64_t* bar) {
                        const int j = t / per_j;
                        const int rem = t - j * per_j;
                        const int b = rem / g.ncb;
                        const int cb = rem - b * g.ncb;
                        KV* dk = stages + (size_t)(2 * s) * TILE;
                        KV* dv = dk + TILE;
                        if (a.use_tma) {
                          if (lane == 0) {
                            tma_load_3d(dk, &a.tk, bar, cb * kCtaChannels, j * kChunk, b);
                            tma_load_3d(dv, &a.tv, bar, cb * kCtaChannels, j * kChunk, b);
                          }
                        } else {
                          copy_tile_plain(dk, static_cast<const KV*>(a.k), g.B, g.T, g.C, b, j * kChunk,
                                          cb * kCtaChannels, kChunk);
                          copy_tile_plain(dv, static_cast<const KV*>(a.v), g.B, g.T, g.C, b, j * kChunk,
                                          cb * kCtaChannels, kChunk);
                        }
                      });
  } else if (warp == kWalkerWarp) {
    fwd_walker(a, L, pst);
  } else {
    // Consumer: a tile is summarised as soon as its stage lands (every
    // ticketed tile's summary reaches the walkers without waiting on other
    // tiles), and the oldest summarised tile is re-run once its carried state
    // is published; neither step blocks the other.
    // Per-lane results of a tile's summary wait for its re-run in registers,
    // one set per stage, selected with constant indices (a stage-indexed
    // array would live in local memory).  The tile's coordinates come back
    // from its ticket, still in the control block until the stage is
    // released.
    float sF[NS], sK[NS], sE[NS];
    bool sFast[NS];
    auto decode = [&](int t, FwdPend& p) {
      const int j = t / per_j;
      const int rem = t - j * per_j;
      p.j = j;
      p.b = rem / g.ncb;
      const int c0 = (rem - p.b * g.ncb) * kCtaChannels + warp * 32;
      p.live = c0 < g.C;
      p.c = c0 + lane;
      p.len = min(kChunk, g.T - j * kChunk);
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
        FwdPend p;
        decode(t, p);
        if (p.live && !failed) {
          p.ew = expf(-p.w);
          const KV* sk = stages + (size_t)(2 * ns) * TILE + warp * 32 + lane;
          fwd_summary<KV>(a, L, sk, sk + TILE, p);
#pragma unroll
          for (int q = 0; q < NS; ++q) {
            if (q == ns) {
              sF[q] = p.F;
              sK[q] = p.kmin;
              sE[q] = p.ew;
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
        FwdPend p;
        decode(*(volatile int*)&ctl->tile[nf], p);
        bool ready = true;
        State P = empty_state();
        if (p.live && !failed && p.j > 0) {
          const bool valid = p.c < g.C;
          const Rec r = rec_load(a.inc + ((size_t)(p.j - 1) * g.B + p.b) * g.C + (valid ? p.c : 0));
          ready = __all_sync(0xffffffffu, !valid || rec_ok(r, L.tag));
          P = State{rec_x(r), rec_y(r), rec_z(r)};
        } else if (p.live && p.j == 0) {
          P = load_state_planes(a.state_in, (size_t)g.B * g.C, (size_t)p.b * g.C + (p.c < g.C ? p.c : g.C - 1));
        }
        if (ready) {
          if (p.live && !failed) {
#pragma unroll
            for (int q = 0; q < NS; ++q) {
              if (q == nf) {
                p.F = sF[q];
                p.kmin = sK[q];
                p.ew = sE[q];
                p.fast = sFast[q];
              }
            }
            const KV* sk = stages + (size_t)(2 * nf) * TILE + warp * 32 + lane;
            fwd_rerun<KV, WRITE_Y>(a, sk, sk + TILE, p, P);
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
      // nothing to do: bounded wait for a stage or a carried state
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

template <typename KV, bool WRITE_Y>
cudaError_t launch_fwd_t(const FwdArgs& a, cudaStream_t s) {
  constexpr int NS = FwdStages<KV>::value;
  const size_t smem = (size_t)NS * 2 * kChunk * kCtaChannels * sizeof(KV) + pipe_ctl_bytes<NS>() + kWalkSmem;
  auto kern = fwd_scan_kernel<KV, WRITE_Y>;
  // per device: the opt-in to large dynamic shared memory and the resident CTAs per SM
  static int grid_per_dev[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int grid = (dev >= 0 && dev < 64) ? grid_per_dev[dev] : 0;
  if (grid == 0) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0, sms = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kPipeThreads, smem);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    grid = (per_sm > 0 ? per_sm : 1) * sms;
    if (dev >= 0 && dev < 64) grid_per_dev[dev] = grid;
  }
  const unsigned int nblk = a.g.ntiles < (unsigned)grid ? a.g.ntiles : (unsigned)grid;
  return launch_cooperative(kern, nblk, smem, s, a);
}

}  // namespace

cudaError_t launch_forward(FwdArgs& a, int kv_dtype, bool write_y, cudaStream_t s) {
  if (kv_dtype == 0)
    return write_y ? launch_fwd_t<float, true>(a, s) : launch_fwd_t<float, false>(a, s);
  return write_y ? launch_fwd_t<__nv_bfloat16, true>(a, s) : launch_fwd_t<__nv_bfloat16, false>(a, s);
}

// The device-wide error record of this file's kernels (wkv_sync_status).
cudaError_t take_error_fwd(unsigned int* code) { return take_module_error(code); }

}  // namespace wkv
