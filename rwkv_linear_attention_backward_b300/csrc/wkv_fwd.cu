// wkv_fwd.cu -- WKV forward pass: single-pass chunked scan over time.
//
// The recurrent form of the operator ("RWKV解读：在Transformer的时代的新RNN",
// section "3、RWKV的网络架构": eq. (8) can be written recursively) is a
// linear recurrence whose decay is data independent, which is what makes the
// training form time-parallel (qiita "RWKV についての調査記録", section
// "Trainingについて").  Time is cut into chunks of kChunk tokens; a tile is
// (chunk j, batch row b, 128 channels), one channel per consumer lane, its k
// and v staged in shared memory by the producer warp (wkv_pipe.cuh).  Per
// tile and lane:
//
//   1. chunk statistics: F = max k, the smallest k, and the state's running
//      maximum at the chunk end r = max_i (k_i - (n-1-i) w);
//   2. the chunk's own summary (its tokens from the empty state), computed at
//      the fixed scale e^{F}: ek_i = e^{k_i - F} <= 1, num = num e^{-w} +
//      ek v, den = den e^{-w} + ek, then rescaled to the canonical scale
//      e^{r}; published for the look-back (wkv_common.cuh);
//   3. look-back: the state carried into the chunk, P;
//   4. the state after the chunk, P (+) summary, written as the checkpoint
//      and published as the inclusive record;
//   5. the outputs: the chunk re-run from P at scale e^{F}:
//      y = (a + e^{u} ek v) / (b + e^{u} ek).
//
// The fixed scale makes each element cost one exponential and a few FMAs.  It
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
__device__ __forceinline__ float to_f32(KV x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) {
  return x;
}
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}

template <typename KV>
struct FwdStages {
  static constexpr int value = sizeof(KV) == 4 ? 3 : 4;
};

constexpr float kFastRange = 69.f;   // smallest bonus weight of the fixed scale: e^{-69}
constexpr float kFastCeil = 60.f;    // largest scale-up of the fixed scale: e^{60}

__device__ __forceinline__ State load_state(const float* rec, size_t plane, size_t o) {
  return State{__ldcg(rec + o), __ldcg(rec + o + plane), __ldcg(rec + o + 2 * plane)};
}

__device__ __forceinline__ void store_state(float* rec, size_t plane, size_t o, const State& s) {
  rec[o] = s.num;
  rec[o + plane] = s.den;
  rec[o + 2 * plane] = s.pp;
}

// One consumer warp's share (32 channels) of one tile.
template <typename KV, bool WRITE_Y, bool FULL>
__device__ __forceinline__ void fwd_tile(const FwdArgs& a, const KV* sk, const KV* sv, int j, int b, int wg, int c,
                                         int len) {
  constexpr int L = kChunk;
  const ScanGeometry& g = a.g;
  const int lane = threadIdx.x & 31;
  const bool valid = c < g.C;
  const int cc = valid ? c : g.C - 1;  // out-of-range lanes shadow the last channel, never store
  const int n = FULL ? L : len;
  const float w = __ldg(a.w + cc);
  const float u = __ldg(a.u + cc);
  sk += lane;
  sv += lane;

  // 1. chunk statistics
  float kr[L];
  float F = -3.0e38f, kmin = 3.0e38f, r = -3.0e38f;
#pragma unroll
  for (int i = 0; i < L; ++i) {
    if (FULL || i < len) {
      kr[i] = to_f32<KV>(sk[i * kCtaChannels]);
      F = fmaxf(F, kr[i]);
      kmin = fminf(kmin, kr[i]);
      r = fmaxf(r, fmaf(-(float)(n - 1 - i), w, kr[i]));
    }
  }

  // 2. the chunk's own summary
  const bool fast_sum = kmin >= F - kFastRange;
  const float ew = expf(-w);
  State S;
  if (fast_sum) {
    const float F2 = F * kLog2e;
    float num = 0.f, den = 0.f;
#pragma unroll
    for (int i = 0; i < L; ++i) {
      if (FULL || i < len) {
        const float ek = ex2(fmaf(kr[i], kLog2e, -F2));
        kr[i] = ek;
        const float vv = to_f32<KV>(sv[i * kCtaChannels]);
        num = fmaf(num, ew, ek * vv);
        den = fmaf(den, ew, ek);
      }
    }
    const float sc = exp_nat(F - r);  // >= 1: from scale e^{F} to e^{r}
    S = State{num * sc, den * sc, r};
  } else {
    State s = empty_state();
#pragma unroll
    for (int i = 0; i < L; ++i)
      if (FULL || i < len) step(s, kr[i], to_f32<KV>(sv[i * kCtaChannels]), w);
    S = s;
  }

  const size_t P3 = g.plane;
  const size_t slot = ((size_t)j * g.B + b) * g.C + cc;
  uint64_t* flag = a.flags + ((size_t)j * g.B + b) * g.nwg + wg;
  const bool has_succ = j < g.nchunks - 1;
  const bool skip = j == a.debug_skip_chunk;  // fault injection: this tile never publishes
  const float Lw = (float)L * w;              // decay over a whole chunk

  // 3. look-back for the state carried into the chunk
  State P = empty_state();
  if (j > 0) {
    if (has_succ && !skip) {
      if (valid) store_state(a.agg, P3, slot, S);
      publish(flag, a.epoch, kAgg);
    }
    const int nwin = min(j, 32);
    int base = 0;
    const int rc = lookback_wait(
        [&](int i) { return a.flags + ((size_t)(j - 1 - i) * g.B + b) * g.nwg + wg; }, nwin, a.epoch, a.budget_ns,
        a.eh, base);
    if (rc != kWaitOk) {
      if (rc == kWaitTimeout && lane == 0) record_error(a.eh, kDevErrTimeout, a.epoch);
      if (has_succ && !skip) publish(flag, a.epoch, kErr);
      return;
    }
    const size_t row = (size_t)b * g.C + cc;
    const size_t jstride = (size_t)g.B * g.C;
    P = load_state(a.inc, P3, (size_t)(j - 1 - base) * jstride + row);
    // fold the summaries of chunks j - base .. j - 1, oldest first, four loads in flight
    for (int i = base - 1; i >= 0; i -= 4) {
      State q[4];
#pragma unroll
      for (int m = 0; m < 4; ++m)
        if (i - m >= 0) q[m] = load_state(a.agg, P3, (size_t)(j - 1 - (i - m)) * jstride + row);
#pragma unroll
      for (int m = 0; m < 4; ++m)
        if (i - m >= 0) P = combine(P, Lw, q[m]);
    }
  }

  // 4. the state after the chunk: checkpoint and inclusive record
  const State incl = combine(P, (float)n * w, S);
  if (valid) store_state(a.inc, P3, slot, incl);
  if (has_succ && !skip) publish(flag, a.epoch, kIncl);

  if constexpr (WRITE_Y) {
    // 5. outputs
    float* yp = a.y + ((int64_t)b * g.T + (int64_t)j * L) * g.C + cc;
    const bool fast_run = fast_sum && (kmin + fminf(u, 0.f) >= F - kFastRange) && (u <= kFastCeil) &&
                          (P.pp - F <= kFastCeil);
    if (fast_run) {
      const float eu = expf(u);
      const float s0 = exp_nat(P.pp - F);  // P at scale e^{F}; 0 for the empty state
      float na = P.num * s0, nb = P.den * s0;
#pragma unroll
      for (int i = 0; i < L; ++i) {
        if (FULL || i < len) {
          const float ek = kr[i];
          const float vv = to_f32<KV>(sv[i * kCtaChannels]);
          const float ec = ek * eu;
          const float yv = fmaf(ec, vv, na) * rcp(nb + ec);
          if (valid) __stcs(yp + (int64_t)i * g.C, yv);
          na = fmaf(na, ew, ek * vv);
          nb = fmaf(nb, ew, ek);
        }
      }
    } else {
      State s = P;
#pragma unroll
      for (int i = 0; i < L; ++i) {
        if (FULL || i < len) {
          const float kk = to_f32<KV>(sk[i * kCtaChannels]);
          const float vv = to_f32<KV>(sv[i * kCtaChannels]);
          const float yv = output(s, kk, vv, u);
          if (valid) __stcs(yp + (int64_t)i * g.C, yv);
          step(s, kk, vv, w);
        }
      }
    }
  }
}

template <typename KV, bool WRITE_Y>
__global__ void __launch_bounds__(kPipeThreads, 1) fwd_scan_kernel(const __grid_constant__ FwdArgs a) {
  constexpr int NS = FwdStages<KV>::value;
  constexpr int TILE = kChunk * kCtaChannels;
  extern __shared__ __align__(1024) unsigned char smem[];
  KV* stages = reinterpret_cast<KV*>(smem);  // stage s: k at 2s*TILE, v at (2s+1)*TILE
  auto* ctl = reinterpret_cast<PipeCtl<NS>*>(smem + (size_t)NS * 2 * TILE * sizeof(KV));
  pipe_init(ctl);
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
                      a.epoch, [&](unsigned int t, int s, uint64_t* bar) {
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
      const int j = t / per_j;
      const int rem = t - j * per_j;
      const int b = rem / g.ncb;
      const int cb = rem - b * g.ncb;
      const int c0 = cb * kCtaChannels + warp * 32;
      if (c0 < g.C) {
        const KV* sk = stages + (size_t)(2 * s) * TILE + warp * 32;
        const KV* sv = sk + TILE;
        const int len = min(kChunk, g.T - j * kChunk);
        const int wg = cb * kConsumerWarps + warp;
        if (len == kChunk)
          fwd_tile<KV, WRITE_Y, true>(a, sk, sv, j, b, wg, c0 + lane, len);
        else
          fwd_tile<KV, WRITE_Y, false>(a, sk, sv, j, b, wg, c0 + lane, len);
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

template <typename KV, bool WRITE_Y>
cudaError_t launch_fwd_t(const FwdArgs& a, cudaStream_t s) {
  constexpr int NS = FwdStages<KV>::value;
  const size_t smem = (size_t)NS * 2 * kChunk * kCtaChannels * sizeof(KV) + sizeof(PipeCtl<NS>);
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
  kern<<<dim3(nblk), dim3(kPipeThreads), smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_forward(FwdArgs& a, int kv_dtype, bool write_y, cudaStream_t s) {
  if (kv_dtype == 0)
    return write_y ? launch_fwd_t<float, true>(a, s) : launch_fwd_t<float, false>(a, s);
  return write_y ? launch_fwd_t<__nv_bfloat16, true>(a, s) : launch_fwd_t<__nv_bfloat16, false>(a, s);
}

}  // namespace wkv
