// wkv_seq.cu -- WKV forward and backward as one sequential walk over time
// per column, for shapes with enough independent columns to fill the GPU.
//
// Channels and batch rows are independent (the recurrence of
// "RWKV解读：在Transformer的时代的新RNN", section "3、RWKV的网络架构",
// eq. (8), runs per channel), so a column -- one batch row and 32
// consecutive channels, one channel per lane -- needs nothing from any other
// column.  One warp (one CTA) walks a column's time chunks in order (the
// forward pass) or in reverse order (the backward pass) and carries the
// state, or the adjoint, from chunk to chunk in registers: there is no chunk
// summary to publish and no wait on another CTA.  The warp stages its own
// chunks, k and v (and gy) as [kChunk tokens x 32 channels] boxes, into a
// ring of shared-memory stages by TMA, several chunks ahead, so each column
// keeps its next loads in flight while it computes.
//
// The per-chunk arithmetic is that of the chunked scans (wkv_fwd.cu,
// wkv_bwd.cu): the fixed scale e^{F}, F = the chunk's largest k, under the
// same bounds, and the per-token running-maximum form for lanes outside
// them.  The carried state crosses a chunk boundary the way the chunked
// scan's walkers carry it -- the chunk's own summary combined with the
// state before it decayed by e^{-n w} in one exponential -- not through n
// products of the rounded e^{-w}, whose rounding error would otherwise grow
// with T.  The adjoint crosses chunk boundaries the same way.  Outputs and
// checkpoints of fixed-scale lanes therefore match the chunked forward
// pass's bit for bit.
#include <cuda_bf16.h>

#include <type_traits>

#include "wkv_adjoint.cuh"
#include "wkv_common.cuh"
#include "wkv_internal.h"
#include "wkv_pipe.cuh"

namespace wkv {

namespace {

constexpr int kSeqTile = kChunk * kSeqChannels;  // elements of one array in one stage
constexpr float kFastRange = 69.f;  // smallest bonus weight of the fixed scale: e^{-69}
constexpr float kFastCeil = 60.f;   // largest scale-up of the fixed scale: e^{60}


// Column q (batch row q / nwg, channels from 32 (q % nwg)): batch row,
// first channel, this lane's channel.
struct Column {
  int b, c0, c;
  bool valid;  // c < C
  int cc;      // c clamped into [0, C)
};

__device__ __forceinline__ Column column_of(const ScanGeometry& g, int q) {
  Column o;
  o.b = q / g.nwg;
  o.c0 = (q - o.b * g.nwg) * kSeqChannels;
  o.c = o.c0 + (int)(threadIdx.x & 31);
  o.valid = o.c < g.C;
  o.cc = o.valid ? o.c : g.C - 1;
  return o;
}

// Plain-load copy of one [kChunk x 32] box of a [B, T, C] tensor, zero
// outside the tensor (TMA's fill value); the whole warp takes part, lane l
// writing column l of the box.
template <typename E>
__device__ __forceinline__ void copy_box_plain(E* dst, const E* src, const ScanGeometry& g, const Column& col,
                                               int t0) {
#pragma unroll 4
  for (int i = 0; i < kChunk; ++i) {
    const int t = t0 + i;
    E val = E(0.f);
    if (t < g.T && col.valid) val = src[((int64_t)col.b * g.T + t) * g.C + col.c];
    dst[i * kSeqChannels + (threadIdx.x & 31)] = val;
  }
}

// Waits (bounded) for stage s's TMA bytes of phase `parity`; every lane
// waits, so every lane's later reads see the copied bytes.
__device__ __forceinline__ bool stage_wait(uint64_t* bar, uint32_t parity, uint64_t budget_ns) {
  const bool ok = mbar_wait(bar, parity, budget_ns);
  return __all_sync(0xffffffffu, ok);
}

// After an expired wait: give the copies still in flight into this CTA's
// shared memory (stages of chunks issued after the one that expired) one
// more shared, bounded chance to land before the CTA exits.  The limit is
// fixed (not the adjustable wait budget), long against any copy.
constexpr uint64_t kDrainNs = 200ull * 1000 * 1000;

template <int NS>
__device__ __forceinline__ void drain_stages(uint64_t* full, int first, int issued) {
  const uint64_t t0 = globaltimer();
  for (int it = first + 1; it < issued; ++it) {
    const int s = it % NS;
    const uint32_t parity = (uint32_t)((it / NS) & 1);
    while (!mbar_try_wait(&full[s], parity)) {
      if (globaltimer() - t0 > kDrainNs) return;
    }
  }
}

// Three-input max / min (single PTX instructions on sm_100 and later).
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

__device__ __forceinline__ float min3f(float a, float b, float c) {
  float r;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Largest / smallest of x[0..N): a balanced ternary tree (max and min are
// exact, so the result is that of any order), with many independent
// operations per level instead of a chain of N.
template <int N>
__device__ __forceinline__ float tree_max(const float* x) {
  if constexpr (N == 1) {
    return x[0];
  } else if constexpr (N == 2) {
    return fmaxf(x[0], x[1]);
  } else {
    constexpr int a = N / 3, b = N / 3;
    return max3f(tree_max<a>(x), tree_max<b>(x + a), tree_max<N - a - b>(x + a + b));
  }
}

template <int N>
__device__ __forceinline__ float tree_min(const float* x) {
  if constexpr (N == 1) {
    return x[0];
  } else if constexpr (N == 2) {
    return fminf(x[0], x[1]);
  } else {
    constexpr int a = N / 3, b = N / 3;
    return min3f(tree_min<a>(x), tree_min<b>(x + a), tree_min<N - a - b>(x + a + b));
  }
}

// ------------------------------------------------------------------ forward
// What a forward walk writes per token: nothing (a state-only pass), wkv_t,
// or the gated output sigmoid(r_t) wkv_t.
constexpr int kYNone = 0, kYWkv = 1, kYGated = 2;

// The gate's input for output i of a chunk (rp: r at the chunk's first
// token of this lane's channel, token stride `stride`); 0 unless gated.
template <typename KV, int YM>
__device__ __forceinline__ float load_r(const KV* __restrict__ rp, int i, int64_t stride, bool valid) {
  if constexpr (YM == kYGated) return valid ? to_f32<KV>(__ldg(rp + (int64_t)i * stride)) : 0.f;
  return 0.f;
}

// Stores output i of a chunk (yp: y at the chunk's first token): wkv_t, or
// sigmoid(r) wkv_t when gated.
template <int YM>
__device__ __forceinline__ void put_y(float* __restrict__ yp, int i, int64_t stride, float yv, float r, bool valid) {
  if (!valid) return;
  if constexpr (YM == kYGated) yv *= sigmoid(r);
  __stcs(yp + (int64_t)i * stride, yv);
}

// A whole chunk of the forward pass for this lane, with every loop fully
// unrolled and no per-token branch: the one warp of a column has no other
// warp to hide latencies behind, so each phase is written as independent
// work per token (the k values and then ek in registers; the statistics by
// trees) and only the carried sums form chains.  Same arithmetic, in the
// same order per value, as the generic form below.
template <typename KV, int YM>
__device__ __forceinline__ void seq_fwd_full(const KV* __restrict__ sk, const KV* __restrict__ sv, float w, float u,
                                             float ew, float eu, State& P, float* __restrict__ yp,
                                             const KV* __restrict__ rp, int64_t ystride, bool valid) {
  constexpr int L = kChunk;
  constexpr int S = kSeqChannels;
  // the gate's r for the whole chunk first: independent global loads, in
  // flight while the chunk is computed (loaded one by one next to the y
  // stores, each would wait for the last)
  float rg[L];
  if constexpr (YM == kYGated) {
#pragma unroll
    for (int i = 0; i < L; ++i) rg[i] = load_r<KV, YM>(rp, i, ystride, valid);
  }
  float kr[L], rr[L];
#pragma unroll
  for (int i = 0; i < L; ++i) {
    kr[i] = to_f32<KV>(sk[i * S]);
    rr[i] = fmaf(-(float)(L - 1 - i), w, kr[i]);
  }
  const float F = tree_max<L>(kr);
  const float kmin = tree_min<L>(kr);
  const float r = tree_max<L>(rr);
  const bool fast = (kmin + fminf(u, 0.f) >= F - kFastRange) && (u <= kFastCeil) && (P.pp - F <= kFastCeil);
  if (fast) {
    // Phase by phase over the whole chunk (independent work per token in
    // each, so one warp keeps several in flight): ek; the carried sums
    // before each token (four chains); the outputs.
    const float F2 = F * kLog2e;
    const float s0 = exp_nat(P.pp - F);
    // per token the pair {e^{k-F} v, e^{k-F}}: the addends of both pairs of
    // chains (the sums with P, for the outputs; the chunk's own, for the
    // carried state) and, times e^u, of the output's numerator and
    // denominator
    Pk2 kv[L];
#pragma unroll
    for (int i = 0; i < L; ++i) {
      const float ek = ex2(fmaf(kr[i], kLog2e, -F2));
      kv[i] = f2(ek * to_f32<KV>(sv[i * S]), ek);
    }
    const Pk2 ew2 = f2(ew, ew);
    Pk2 nab = f2(P.num * s0, P.den * s0);  // sums with P before each token
    Pk2 own = f2(0.f, 0.f);                // the chunk's own sums
    Pk2 AB[L];
#pragma unroll
    for (int i = 0; i < L; ++i) {
      if constexpr (YM != kYNone) {
        AB[i] = nab;
        nab = fma2(nab, ew2, kv[i]);
      }
      own = fma2(own, ew2, kv[i]);
    }
    if constexpr (YM != kYNone) {
      const Pk2 eu2 = f2(eu, eu);
#pragma unroll
      for (int i = 0; i < L; ++i) {
        const Pk2 nd = fma2(kv[i], eu2, AB[i]);  // {numerator, denominator}
        const float yv = f2_lo(nd) * rcp(f2_hi(nd));
        put_y<YM>(yp, i, ystride, yv, YM == kYGated ? rg[i] : 0.f, valid);
      }
    }
    const float sc = exp_nat(F - r);
    P = combine(P, (float)L * w, State{f2_lo(own) * sc, f2_hi(own) * sc, r});
  } else {
#pragma unroll 1
    for (int i = 0; i < L; ++i) {
      const float kk = to_f32<KV>(sk[i * S]);
      const float vv = to_f32<KV>(sv[i * S]);
      if constexpr (YM != kYNone) {
        const float yv = output(P, kk, vv, u);
        put_y<YM>(yp, i, ystride, yv, load_r<KV, YM>(rp, i, ystride, valid), valid);
      }
      step(P, kk, vv, w);
    }
  }
}

// One chunk of n <= kChunk tokens (the generic form, for the partial last
// chunk): outputs from the carried state P (unless YM is kYNone), then P advanced
// past the chunk.
template <typename KV, int YM>
__device__ __forceinline__ void seq_fwd_chunk(const KV* __restrict__ sk, const KV* __restrict__ sv, int n, float w,
                                              float u, float ew, float eu, State& P, float* __restrict__ yp,
                                              const KV* __restrict__ rp, int64_t ystride, bool valid) {
  constexpr int S = kSeqChannels;
  float F = -3.0e38f, kmin = 3.0e38f, r = -3.0e38f;
#pragma unroll 8
  for (int i = 0; i < n; ++i) {
    const float k = to_f32<KV>(sk[i * S]);
    F = fmaxf(F, k);
    kmin = fminf(kmin, k);
    r = fmaxf(r, fmaf(-(float)(n - 1 - i), w, k));
  }
  const bool fast = (kmin + fminf(u, 0.f) >= F - kFastRange) && (u <= kFastCeil) && (P.pp - F <= kFastCeil);
  if (fast) {
    const float F2 = F * kLog2e;
    const float s0 = exp_nat(P.pp - F);  // P at scale e^{F}; 0 for the empty state
    float na = P.num * s0, nb = P.den * s0;  // sums before each token, with P (for the outputs)
    float on = 0.f, od = 0.f;                // the chunk's own sums (for the carried state)
#pragma unroll 8
    for (int i = 0; i < n; ++i) {
      const float ek = ex2(fmaf(to_f32<KV>(sk[i * S]), kLog2e, -F2));
      const float vv = to_f32<KV>(sv[i * S]);
      const float ekv = ek * vv;
      if constexpr (YM != kYNone) {
        // the full-chunk body's arithmetic (numerator e^{k-F} v e^u + a,
        // denominator e^{k-F} e^u + b)
        const float yv = fmaf(ekv, eu, na) * rcp(fmaf(ek, eu, nb));
        put_y<YM>(yp, i, ystride, yv, load_r<KV, YM>(rp, i, ystride, valid), valid);
        na = fmaf(na, ew, ekv);
        nb = fmaf(nb, ew, ek);
      }
      on = fmaf(on, ew, ekv);
      od = fmaf(od, ew, ek);
    }
    // the chunk's own summary at its running-maximum scale e^{r}, then
    // P decayed by the chunk's length combined with it
    const float sc = exp_nat(F - r);
    P = combine(P, (float)n * w, State{on * sc, od * sc, r});
  } else {
#pragma unroll 1
    for (int i = 0; i < n; ++i) {
      const float kk = to_f32<KV>(sk[i * S]);
      const float vv = to_f32<KV>(sv[i * S]);
      if constexpr (YM != kYNone) {
        const float yv = output(P, kk, vv, u);
        put_y<YM>(yp, i, ystride, yv, load_r<KV, YM>(rp, i, ystride, valid), valid);
      }
      step(P, kk, vv, w);
    }
  }
}

// Phase 1 of the forward walk for one chunk of n tokens: S, the state a run
// carries from the empty one, advanced past the chunk.  The chunk's own sums
// are formed directly: token i enters the sums after the chunk with exponent
// rr_i = k_i - (n-1-i) w; with r = max_i rr_i every weight e^{rr_i - r} is at
// most 1 and their sum at least 1, so this form is exact in fp32 for any
// finite input (no fixed scale to leave, no per-token fallback) and needs no
// chain through the tokens.  S is then decayed over the chunk and combined
// with the chunk's sums at scale e^{r}.  Phase 2 keeps the chained form,
// which also yields the outputs, so the checkpoints of every kernel that
// walks a chunk in phase 2 are the same bit for bit.
template <bool FULL, typename KV>
__device__ __forceinline__ void seq_fwd_summary(const KV* __restrict__ sk, const KV* __restrict__ sv, int n, float w,
                                                State& S) {
  constexpr int L = kChunk;
  constexpr int Sd = kSeqChannels;
  float r, on = 0.f, od = 0.f;
  if constexpr (FULL) {
    float rr[L];
#pragma unroll
    for (int i = 0; i < L; ++i) rr[i] = fmaf(-(float)(L - 1 - i), w, to_f32<KV>(sk[i * Sd]));
    r = tree_max<L>(rr);
    const float r2 = r * kLog2e;
    float on1 = 0.f, od1 = 0.f;  // odd tokens: two chains per sum
#pragma unroll
    for (int i = 0; i < L; i += 2) {
      const float e0 = ex2(fmaf(rr[i], kLog2e, -r2)), e1 = ex2(fmaf(rr[i + 1], kLog2e, -r2));
      on = fmaf(e0, to_f32<KV>(sv[i * Sd]), on);
      on1 = fmaf(e1, to_f32<KV>(sv[(i + 1) * Sd]), on1);
      od += e0;
      od1 += e1;
    }
    on += on1;
    od += od1;
  } else {
    r = -3.0e38f;
#pragma unroll 8
    for (int i = 0; i < n; ++i) r = fmaxf(r, fmaf(-(float)(n - 1 - i), w, to_f32<KV>(sk[i * Sd])));
    const float r2 = r * kLog2e;
#pragma unroll 8
    for (int i = 0; i < n; ++i) {
      const float e = ex2(fmaf(fmaf(-(float)(n - 1 - i), w, to_f32<KV>(sk[i * Sd])), kLog2e, -r2));
      on = fmaf(e, to_f32<KV>(sv[i * Sd]), on);
      od += e;
    }
  }
  S = combine(S, (float)n * w, State{on, od, r});
}

// Runs of a column's walk: the chunks in walk order (time order for the
// forward pass, reverse time order for the backward pass) cut into nseg
// equal contiguous runs (the first nchunks % nseg one chunk longer); run s
// of column q is CTA q * nseg + s, one warp.  Every run but the last first
// summarises its chunks (phase 1: the state, or the adjoint, it carries from
// the empty one) and publishes the summary as tagged records; then each run
// folds the summaries of the runs before it into its carry and walks its
// chunks again with it (phase 2, reading them a second time, from L2 while
// they fit there).  The runs of a column wait only on phase-1 results, which
// every run produces before it waits, and the launch is cooperative (all
// runs resident), so the waits always end.  With nseg == 1 this is the
// plain sequential walk and nothing is exchanged.
__device__ __forceinline__ void segment_of(int nchunks, int nseg, int s, int& first, int& count) {
  const int base = nchunks / nseg, rem = nchunks - base * nseg;
  first = s * base + min(s, rem);
  count = base + (s < rem ? 1 : 0);
}

// Shared memory of a run's CTA: its ring of NS stages of `arrays`
// [kChunk x 32] boxes of E, then the stages' mbarriers.
template <typename E, int NS>
__host__ __device__ constexpr size_t seq_ring_elems(int arrays) {
  return (size_t)NS * arrays * kSeqTile;
}

template <typename E, int NS>
__host__ __device__ constexpr size_t seq_smem_bytes(int arrays) {
  return seq_ring_elems<E, NS>(arrays) * sizeof(E) + 128;
}

// The launch's identity: 1 + the workspace's sequence number, read by every
// CTA at its start, before the last CTA to finish can advance it (seq_exit).
__device__ __forceinline__ Launch seq_launch(const WsHeader* h) {
  unsigned long long e = 0;
  if ((threadIdx.x & 31) == 0) e = *(volatile const unsigned long long*)&h->seq + 1ull;
  e = __shfl_sync(0xffffffffu, e, 0);
  return Launch{e, tag_of(e)};
}

// The last CTA out resets the exit counter and advances the sequence number.
// Both matter only to later launches, which the end of this one orders
// after every write of it, so no fence is needed (a fence here would wait
// for the CTA's streaming stores to drain).
__device__ __forceinline__ void seq_exit(unsigned int* exited, WsHeader* h, unsigned long long epoch) {
  __syncwarp();
  if (threadIdx.x == 0) {
    if (atomicAdd(exited, 1u) == gridDim.x - 1) {
      atomicExch(exited, 0u);
      atomicExch(&h->seq, epoch);
    }
  }
}

// Waits (bounded) until the record at p carries this launch's tag on every
// valid lane.  False when the wait expired (recorded) or the launch gave up
// elsewhere.  The poll reloads the record back to back (one L2 round trip
// per try, no sleep: the wait sits on the critical path of the runs that
// follow) and looks at the abort flag and the clock every 16th try only.
__device__ __forceinline__ bool wait_rec(const Rec* p, bool valid, const Launch& L, WsHeader* h, uint64_t budget_ns,
                                         Rec& r) {
  r = rec_load(p);
  if (__all_sync(0xffffffffu, !valid || rec_ok(r, L.tag))) return true;
  const uint64_t t0 = globaltimer();
  for (unsigned int n = 1;; ++n) {
    r = rec_load(p);
    if (__all_sync(0xffffffffu, !valid || rec_ok(r, L.tag))) return true;
    if ((n & 15u) != 0) continue;
    if (__shfl_sync(0xffffffffu, *(volatile const unsigned long long*)&h->abort, 0) == L.epoch) return false;
    if (__shfl_sync(0xffffffffu, globaltimer(), 0) - t0 > budget_ns) {
      if ((threadIdx.x & 31) == 0) record_error(h, kDevErrTimeout, L.epoch);
      return false;
    }
  }
}

template <typename KV, int NS, int YM>
__device__ __forceinline__ void seq_fwd_run(const SeqFwdArgs& a, const Launch& L, unsigned char* smem) {
  KV* ring = reinterpret_cast<KV*>(smem);  // stage s: k at 2s*kSeqTile, v at (2s+1)*kSeqTile
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + seq_ring_elems<KV, NS>(2) * sizeof(KV));
  const int lane = threadIdx.x;
  const ScanGeometry& g = a.g;
  const int nseg = a.nseg;
  const int q = blockIdx.x / nseg, run = blockIdx.x - q * nseg;
  const Column col = column_of(g, q);
  const float w = __ldg(a.w + col.cc), u = __ldg(a.u + col.cc);
  const float ew = expf(-w), eu = expf(u);
  const bool tma = a.use_tma != 0;
  constexpr uint32_t kStageBytes = 2 * kSeqTile * sizeof(KV);

  int first, count;
  segment_of(g.nchunks, nseg, run, first, count);
  const int n1 = run < nseg - 1 ? count : 0;  // phase-1 items, then the same chunks again
  const int nitems = n1 + count;
  auto chunk_of = [&](int it) { return first + (it < n1 ? it : it - n1); };
  auto issue = [&](int it) {  // lane 0: item it into its stage
    const int s = it % NS;
    const int j = chunk_of(it);
    KV* dk = ring + (size_t)(2 * s) * kSeqTile;
    mbar_arrive_expect_tx(&full[s], kStageBytes);
    tma_load_3d(dk, &a.tk, &full[s], col.c0, j * kChunk, col.b);
    tma_load_3d(dk + kSeqTile, &a.tv, &full[s], col.c0, j * kChunk, col.b);
  };
  int issued = 0;
  if (tma) {
    if (lane == 0) {
      for (int s = 0; s < NS; ++s) mbar_init(&full[s], 1);
      mbar_init_fence();
      tma_prefetch_desc(&a.tk);
      tma_prefetch_desc(&a.tv);
      for (int it = 0; it < NS && it < nitems; ++it) issue(it);
    }
    issued = min(NS, nitems);
    __syncwarp();
  }
  // Takes item it's stage (false: the wait expired); `release` after use.
  auto acquire = [&](int it, KV*& dk) {
    const int s = it % NS;
    dk = ring + (size_t)(2 * s) * kSeqTile;
    if (tma) return stage_wait(&full[s], (uint32_t)((it / NS) & 1), a.budget_ns);
    const int j = chunk_of(it);
    copy_box_plain(dk, static_cast<const KV*>(a.k), g, col, j * kChunk);
    copy_box_plain(dk + kSeqTile, static_cast<const KV*>(a.v), g, col, j * kChunk);
    __syncwarp();
    return true;
  };
  auto release = [&](int it) {
    // Every lane's reads of the stage come before the copy that refills it:
    // their values have been used before this point, so the reads are
    // complete; the stage is only read, so no proxy fence is needed.
    __syncwarp();
    if (tma && it + NS < nitems) {
      if (lane == 0) issue(it + NS);
      ++issued;
    }
  };
  auto fail = [&](int it) {
    if (lane == 0) record_error(a.eh, kDevErrTimeout, L.epoch);
    drain_stages<NS>(full, it, issued);
  };
  const size_t rec0 = (size_t)col.b * g.C + col.cc;  // + run * B * C
  const size_t jstride = (size_t)g.B * g.C;

  // phase 1: this run's own summary (the state it carries from the empty one)
  State P = empty_state();
  int it = 0;
  for (; it < n1; ++it) {
    KV* dk;
    if (!acquire(it, dk)) return fail(it);
    const int j = chunk_of(it);
    const int n = min(kChunk, g.T - j * kChunk);
    if (n == kChunk)
      seq_fwd_summary<true, KV>(dk + lane, dk + kSeqTile + lane, n, w, P);
    else
      seq_fwd_summary<false, KV>(dk + lane, dk + kSeqTile + lane, n, w, P);
    release(it);
  }
  const bool skip = a.debug_skip_chunk >= first && a.debug_skip_chunk < first + count;  // fault injection
  if (n1 > 0 && col.valid && !skip) rec_store(a.recs + (size_t)run * jstride + rec0, L.tag, P.num, P.den, P.pp);

  // the carry into this run: the state given before the first token, then
  // the runs before this one, in order
  P = load_state_planes(a.state_in, jstride, rec0);
  for (int r = 0; r < run; ++r) {
    int fr, cr;
    segment_of(g.nchunks, nseg, r, fr, cr);
    Rec rec;
    if (!wait_rec(a.recs + (size_t)r * jstride + rec0, col.valid, L, a.eh, a.budget_ns, rec)) return fail(it - 1);
    P = combine(P, (float)(cr * kChunk) * w, State{rec_x(rec), rec_y(rec), rec_z(rec)});
  }

  // phase 2: outputs and checkpoints
  for (; it < nitems; ++it) {
    KV* dk;
    if (!acquire(it, dk)) return fail(it);
    const int j = chunk_of(it);
    const int n = min(kChunk, g.T - j * kChunk);
    const int64_t row = ((int64_t)col.b * g.T + (int64_t)j * kChunk) * g.C + col.c;
    float* yp = YM != kYNone ? a.y + row : nullptr;
    const KV* rp = YM == kYGated ? static_cast<const KV*>(a.r) + row : nullptr;
    if (n == kChunk)
      seq_fwd_full<KV, YM>(dk + lane, dk + kSeqTile + lane, w, u, ew, eu, P, yp, rp, g.C, col.valid);
    else
      seq_fwd_chunk<KV, YM>(dk + lane, dk + kSeqTile + lane, n, w, u, ew, eu, P, yp, rp, g.C, col.valid);
    if (col.valid) {
      const size_t o = (size_t)j * jstride + rec0;
      a.ckpt[o] = P.num;
      a.ckpt[o + g.plane] = P.den;
      a.ckpt[o + 2 * g.plane] = P.pp;
      if (j == g.nchunks - 1 && a.state_out) store_state_planes(a.state_out, jstride, rec0, P);
    }
    release(it);
  }
}

// Chained runs, for columns whose inputs do not fit in L2 while the columns
// alone leave SMs idle (a long sequence): a column's chunks are cut into R
// short runs of `chain` chunks, and warp wi of the column's nseg warps walks
// runs wi, wi + nseg, ... in order.  For each run the warp summarises it
// (phase 1), waits for the state after the previous run (a tagged record
// written by the warp that walked it), publishes the state after its own run
// (that state combined with its summary: a fixed order of folds, so the
// results are reproducible), and walks the run again from the carried state
// (phase 2), a few microseconds after phase 1 read it, so from L2.  Only the
// runs in flight sit in L2, whatever T is.  Run r waits only on run r - 1,
// which its warp reaches before any later run of its own, and every warp is
// resident (cooperative launch), so the waits always end.  The last run
// publishes nothing and needs no phase 1.
//
// The walk moves in items of chain_chunks(sizeof(KV)) chunks: one stage, one
// TMA box per array and one wait per item.  With bf16 inputs an item is two
// chunks, so a box row is 128 bytes (64 tokens x 32 channels) and the
// per-item work of the pipeline (waits, copies issued, bookkeeping) is paid
// once per 64 tokens.  The last item of a run's phase holds the run's last
// chunk alone when the run has an odd length (its box then also carries the
// next chunk, unused).  Each chunk is computed exactly as with one-chunk
// items, so the results do not depend on the item size.
template <typename KV, int NS, int YM>
__device__ __forceinline__ void seq_fwd_chain(const SeqFwdArgs& a, const Launch& L, unsigned char* smem) {
  constexpr int CP = chain_chunks(sizeof(KV));  // chunks per item
  constexpr int kBox = CP * kSeqTile;           // elements of one array's box
  KV* ring = reinterpret_cast<KV*>(smem);       // stage s: k at 2s*kBox, v at (2s+1)*kBox
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)NS * 2 * kBox * sizeof(KV));
  const int lane = threadIdx.x;
  const ScanGeometry& g = a.g;
  const int W = a.nseg, len = a.chain;
  const int q = blockIdx.x / W, wi = blockIdx.x - q * W;
  const int R = (g.nchunks + len - 1) / len;
  const Column col = column_of(g, q);
  const float w = __ldg(a.w + col.cc), u = __ldg(a.u + col.cc);
  const float ew = expf(-w), eu = expf(u);
  const bool tma = a.use_tma != 0;
  constexpr uint32_t kStageBytes = 2 * kBox * sizeof(KV);
  const size_t rec0 = (size_t)col.b * g.C + col.cc;  // + run * B * C
  const size_t jstride = (size_t)g.B * g.C;

  // The warp's item stream: per run, its items (phase 1) then the same items
  // again (phase 2); the last run of the column has phase 2 only.  Items
  // per phase: ip for a full run, il for the last one.
  const int last_len = g.nchunks - (R - 1) * len;
  const int ip = (len + CP - 1) / CP, il = (last_len + CP - 1) / CP;
  int nitems = 0;
  for (int r = wi; r < R; r += W) nitems += r == R - 1 ? il : 2 * ip;
  // A position in the warp's item stream: m-th run of the warp, item off of
  // that run; advanced one item at a time (no division per item).
  struct Cur {
    int m, off;
  };
  auto advance = [&](Cur& c) {
    const int n = wi + c.m * W == R - 1 ? il : 2 * ip;
    if (++c.off == n) {
      c.off = 0;
      ++c.m;
    }
  };
  struct Item {
    int r, j, nc;           // run; first chunk; chunks of the run in the item
    bool p1, first, last;  // phase 1 item; first / last item of its phase
  };
  auto item = [&](const Cur& c) {
    Item o;
    o.r = wi + c.m * W;
    int k, rl, np;  // item of the phase; chunks in the run; items in the phase
    if (o.r == R - 1) {
      o.p1 = false;
      k = c.off;
      rl = last_len;
      np = il;
    } else {
      o.p1 = c.off < ip;
      k = o.p1 ? c.off : c.off - ip;
      rl = len;
      np = ip;
    }
    o.j = o.r * len + k * CP;
    o.nc = min(CP, rl - k * CP);
    o.first = k == 0;
    o.last = k == np - 1;
    return o;
  };
  auto issue = [&](int it, const Cur& c) {  // lane 0: item it (at c) into its stage
    const int s = it % NS;
    const int j = item(c).j;
    KV* dk = ring + (size_t)(2 * s) * kBox;
    mbar_arrive_expect_tx(&full[s], kStageBytes);
    tma_load_3d(dk, &a.tk2, &full[s], col.c0, j * kChunk, col.b);
    tma_load_3d(dk + kBox, &a.tv2, &full[s], col.c0, j * kChunk, col.b);
  };
  int issued = 0;
  Cur ahead{0, 0};  // the next item to stage
  if (tma) {
    if (lane == 0) {
      for (int s = 0; s < NS; ++s) mbar_init(&full[s], 1);
      mbar_init_fence();
      tma_prefetch_desc(&a.tk2);
      tma_prefetch_desc(&a.tv2);
    }
    for (int it = 0; it < NS && it < nitems; ++it) {
      if (lane == 0) issue(it, ahead);
      advance(ahead);
    }
    issued = min(NS, nitems);
    __syncwarp();
  }
  auto fail = [&](int it) {
    if (lane == 0) record_error(a.eh, kDevErrTimeout, L.epoch);
    drain_stages<NS>(full, it, issued);
  };
  // the state after run r - 1 (empty before run 0)
  auto carry_in = [&](int r, State& P) {
    if (r == 0) {
      P = load_state_planes(a.state_in, jstride, rec0);  // the state given before the first token
      return true;
    }
    Rec rec;
    if (!wait_rec(a.recs + (size_t)(r - 1) * jstride + rec0, col.valid, L, a.eh, a.budget_ns, rec)) return false;
    P = State{rec_x(rec), rec_y(rec), rec_z(rec)};
    return true;
  };

  State S = empty_state(), P = empty_state();
  Cur cur{0, 0};
  for (int it = 0; it < nitems; ++it, advance(cur)) {
    const Item m = item(cur);
    const int s = it % NS;
    KV* dk = ring + (size_t)(2 * s) * kBox;
    if (tma) {
      if (!stage_wait(&full[s], (uint32_t)((it / NS) & 1), a.budget_ns)) return fail(it);
    } else {
      for (int h = 0; h < m.nc; ++h) {
        copy_box_plain(dk + h * kSeqTile, static_cast<const KV*>(a.k), g, col, (m.j + h) * kChunk);
        copy_box_plain(dk + kBox + h * kSeqTile, static_cast<const KV*>(a.v), g, col, (m.j + h) * kChunk);
      }
      __syncwarp();
    }
    if (m.p1 && m.first) S = empty_state();
    if (!m.p1 && m.first && m.r == R - 1 && !carry_in(m.r, P)) return fail(it);
#pragma unroll 1
    for (int h = 0; h < m.nc; ++h) {
      const int j = m.j + h;
      const KV* sk = dk + h * kSeqTile + lane;
      const KV* sv = dk + kBox + h * kSeqTile + lane;
      const int n = min(kChunk, g.T - j * kChunk);
      if (m.p1) {
        if (n == kChunk)
          seq_fwd_summary<true, KV>(sk, sv, n, w, S);
        else
          seq_fwd_summary<false, KV>(sk, sv, n, w, S);
      } else {
        const int64_t row = ((int64_t)col.b * g.T + (int64_t)j * kChunk) * g.C + col.c;
        float* yp = YM != kYNone ? a.y + row : nullptr;
        const KV* rp = YM == kYGated ? static_cast<const KV*>(a.r) + row : nullptr;
        if (n == kChunk)
          seq_fwd_full<KV, YM>(sk, sv, w, u, ew, eu, P, yp, rp, g.C, col.valid);
        else
          seq_fwd_chunk<KV, YM>(sk, sv, n, w, u, ew, eu, P, yp, rp, g.C, col.valid);
        if (col.valid) {
          const size_t o = (size_t)j * jstride + rec0;
          a.ckpt[o] = P.num;
          a.ckpt[o + g.plane] = P.den;
          a.ckpt[o + 2 * g.plane] = P.pp;
          if (j == g.nchunks - 1 && a.state_out) store_state_planes(a.state_out, jstride, rec0, P);
        }
      }
    }
    // release the stage (only read: see seq_fwd_run)
    __syncwarp();
    if (tma && it + NS < nitems) {
      if (lane == 0) issue(it + NS, ahead);
      advance(ahead);
      ++issued;
    }
    if (m.p1 && m.last) {
      // the state after the previous run, then the state after this one
      if (!carry_in(m.r, P)) return fail(it);
      const State I = combine(P, (float)(len * kChunk) * w, S);
      const bool skip = a.debug_skip_chunk >= m.r * len && a.debug_skip_chunk < (m.r + 1) * len;
      if (col.valid && !skip) rec_store(a.recs + (size_t)m.r * jstride + rec0, L.tag, I.num, I.den, I.pp);
    }
  }
}

// CHAIN: chained runs (seq_fwd_chain), else runs exchanging summaries
// (seq_fwd_run); separate kernels, so that each holds only its own code
// (both in one kernel overflowed the instruction cache).
template <typename KV, int NS, int YM, bool CHAIN>
__global__ void __launch_bounds__(kSeqChannels) seq_fwd_kernel(const __grid_constant__ SeqFwdArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  const Launch L = seq_launch(a.eh);
  if constexpr (CHAIN)
    seq_fwd_chain<KV, NS, YM>(a, L, smem);
  else
    seq_fwd_run<KV, NS, YM>(a, L, smem);
  seq_exit(a.exited, a.eh, L.epoch);
}

// ----------------------------------------------------------------- backward
// The adjoint recurrence and the gradients are those of the chunked
// backward pass (wkv_bwd.cu).  Per chunk, last chunk first: the forward
// sums before each token from the checkpoint before the chunk (the sums in
// registers, ek written over k in the stage), then the reverse sweep with
// the adjoint X carried in from the next chunk.  The sweep keeps the
// chunk's zero-carry adjoint (la0, lb0) apart from X's decayed share, so X
// crosses the chunk in one exponential (fold_adj) rather than n products of
// the rounded e^{-w}.
struct BwdColumn {
  float w, u, ew, eu;
  float gw_s, gw_k, gu_s, gu_k;  // compensated sums over the chunks
};

__device__ __forceinline__ void kahan_add(float& s, float& k, float x) {
  const float y = x - k;
  const float t = s + y;
  k = (t - s) - y;
  s = t;
}

// FULL: a whole chunk (n == kChunk), every loop fully unrolled with no
// per-token branch and ek kept in registers (see seq_fwd_full); otherwise
// the first n tokens, each token under its own predicate, ek computed again
// where the reverse sweep needs it.  KV: the staged element type (float or
// bf16; the arithmetic is fp32).  RP: 0, or for the gated output the offset
// of the staged r plane from the output-gradient plane sg (gate_grad); then
// gr_t = gout_t sigmoid'(r_t) wkv_t goes to grp.
template <bool FULL, typename KV, int RP>
__device__ __forceinline__ void seq_bwd_chunk(const KV* __restrict__ sk, const KV* __restrict__ sv,
                                              const KV* __restrict__ sg, int n, const BwdColumn& cw,
                                              const State& P, bool has_succ, Adj& X, float* __restrict__ gkp,
                                              float* __restrict__ gvp, float* __restrict__ grp, int64_t stride,
                                              bool valid, float& gw_acc, float& gu_acc, float* xa, float* xb,
                                              float* xp) {
  constexpr int L = kChunk;
  constexpr int S = kSeqChannels;
  if constexpr (FULL) n = L;
  float kr[L];
  float F, kmin;
  if constexpr (FULL) {
#pragma unroll
    for (int i = 0; i < L; ++i) kr[i] = to_f32<KV>(sk[i * S]);
    F = tree_max<L>(kr);
    kmin = tree_min<L>(kr);
  } else {
    F = -3.0e38f;
    kmin = 3.0e38f;
#pragma unroll 8
    for (int i = 0; i < n; ++i) {
      const float k = to_f32<KV>(sk[i * S]);
      F = fmaxf(F, k);
      kmin = fminf(kmin, k);
    }
  }
  const bool fast =
      (kmin + fminf(cw.u, 0.f) >= F - kFastRange) && (cw.u <= kFastCeil) && (P.pp - F <= kFastCeil);
  gw_acc = 0.f;
  gu_acc = 0.f;
  if (fast) {
    const float F2 = F * kLog2e;
    const float s0 = exp_nat(P.pp - F);
    float A[L], Bd[L];
    float na = P.num * s0, nb = P.den * s0;
    if constexpr (FULL) {
#pragma unroll
      for (int i = 0; i < L; ++i) kr[i] = ex2(fmaf(kr[i], kLog2e, -F2));  // ek
    }
#pragma unroll
    for (int i = 0; i < L; ++i) {
      if (FULL || i < n) {
        float ek;
        if constexpr (FULL) {
          ek = kr[i];
        } else {
          ek = ex2(fmaf(to_f32<KV>(sk[i * S]), kLog2e, -F2));
        }
        const float vv = to_f32<KV>(sv[i * S]);
        A[i] = na;
        Bd[i] = nb;
        na = fmaf(na, cw.ew, ek * vv);
        nb = fmaf(nb, cw.ew, ek);
      }
    }
    // X at scale e^{F}; its share of the adjoint after token i is
    // X e^{-(n-1-i) w} (pw)
    const float f = has_succ ? exp_nat(F - X.f) : 0.f;
    const float xla = X.la * f, xlb = X.lb * f;
    float la0 = 0.f, lb0 = 0.f, pw = 1.f;
    if constexpr (FULL) {
      // the per-token terms that need no adjoint, for the whole chunk first
      // (independent work), then the reverse sweep's chains
      float GI[L], VM[L];
#pragma unroll
      for (int i = 0; i < L; ++i) {
        const float ec = kr[i] * cw.eu;
        const float rr = rcp(Bd[i] + ec);
        const float vv = to_f32<KV>(sv[i * S]);
        float gq;
        GI[i] = gate_grad<RP>(sg, i * S, gq) * rr;  // gN at scale e^{F}
        VM[i] = fmaf(vv, Bd[i], -A[i]) * rr;        // v - wkv
        if constexpr (RP != 0) {
          if (valid) __stcs(grp + (int64_t)i * stride, gq * (fmaf(ec, vv, A[i]) * rr));
        }
      }
#pragma unroll
      for (int i = L - 1; i >= 0; --i) {
        const float la = fmaf(xla, pw, la0);  // adjoints after token i, at scale e^{F}
        const float lb = fmaf(xlb, pw, lb0);
        const float ek = kr[i];
        const float vv = to_f32<KV>(sv[i * S]);
        const float ec = ek * cw.eu;
        const float gi = GI[i];
        const float cur = gi * VM[i] * ec;  // (gN v + gD) e^{u+k}
        const float gk = fmaf(fmaf(la, vv, lb), ek, cur);
        const float gv = fmaf(gi, ec, la * ek);
        gu_acc += cur;
        // the token's two terms first: they nearly cancel (lb ~ -la wkv), so
        // summing each over the chunk apart would round at ~32 times the size
        // of what is left after the cancellation
        gw_acc += fmaf(la, A[i], lb * Bd[i]);
        la0 = fmaf(la0, cw.ew, gi);
        lb0 = fmaf(lb0, cw.ew, -gi * (vv - VM[i]));
        pw *= cw.ew;
        if (valid) {
          __stcs(gkp + (int64_t)i * stride, gk);
          __stcs(gvp + (int64_t)i * stride, gv);
        }
      }
    }
#pragma unroll
    for (int i = L - 1; i >= 0; --i) {
      if (!FULL && i < n) {
        const float la = fmaf(xla, pw, la0);
        const float lb = fmaf(xlb, pw, lb0);
        const float ek = ex2(fmaf(to_f32<KV>(sk[i * S]), kLog2e, -F2));
        const float vv = to_f32<KV>(sv[i * S]);
        const float ec = ek * cw.eu;
        const float rr = rcp(Bd[i] + ec);
        float gq;
        const float gi = gate_grad<RP>(sg, i * S, gq) * rr;
        const float vmy = fmaf(vv, Bd[i], -A[i]) * rr;  // v - wkv
        const float cur = gi * vmy * ec;                // (gN v + gD) e^{u+k}
        const float gk = fmaf(fmaf(la, vv, lb), ek, cur);
        const float gv = fmaf(gi, ec, la * ek);
        gu_acc += cur;
        // the token's two terms first: they nearly cancel (lb ~ -la wkv), so
        // summing each over the chunk apart would round at ~32 times the size
        // of what is left after the cancellation
        gw_acc += fmaf(la, A[i], lb * Bd[i]);
        la0 = fmaf(la0, cw.ew, gi);
        lb0 = fmaf(lb0, cw.ew, -gi * (vv - vmy));
        pw *= cw.ew;
        if (valid) {
          __stcs(gkp + (int64_t)i * stride, gk);
          __stcs(gvp + (int64_t)i * stride, gv);
          if constexpr (RP != 0) __stcs(grp + (int64_t)i * stride, gq * (fmaf(ec, vv, A[i]) * rr));
        }
      }
    }
    gw_acc = -cw.ew * gw_acc;
    // the adjoint at the chunk start, at the scale of P (the record form)
    const Adj A0{la0 * s0, lb0 * s0, P.pp};
    X = has_succ ? fold_adj(A0, (float)n * cw.w, X) : A0;
  } else {
    const float pp_end = exact_states<kSeqChannels, KV>(sk, sv, n, P, cw.w, xa, xb, xp);
    const float f = has_succ ? exp_nat(pp_end - X.f) : 0.f;
    float res[4];
    exact_final<kSeqChannels, KV, RP>(sk, sv, sg, n, cw.w, cw.u, xa, xb, xp, X.la * f, X.lb * f, gkp, gvp, stride,
                                      valid, res, grp);
    gw_acc = res[0];
    gu_acc = res[1];
    X = Adj{res[2], res[3], P.pp};
  }
}

// Phase 1 of the backward walk for one chunk: the chunk's zero-carry
// adjoint at its first token (its own gy only), in the record form: scaled
// by e^{P.pp}, P the state before the chunk.  The forward sums and the
// adjoint accumulate in one forward sweep, each token's gN, gD weighted by
// e^{-(t - t0) w} (pw), as in the chunked backward pass's summary.
template <bool FULL, typename KV, int RP>
__device__ __forceinline__ Adj seq_bwd_summary(const KV* __restrict__ sk, const KV* __restrict__ sv,
                                               const KV* __restrict__ sg, int n, const BwdColumn& cw,
                                               const State& P, float* xa, float* xb, float* xp) {
  constexpr int L = kChunk;
  constexpr int S = kSeqChannels;
  if constexpr (FULL) n = L;
  float kr[L];
  float F, kmin;
  if constexpr (FULL) {
#pragma unroll
    for (int i = 0; i < L; ++i) kr[i] = to_f32<KV>(sk[i * S]);
    F = tree_max<L>(kr);
    kmin = tree_min<L>(kr);
  } else {
    F = -3.0e38f;
    kmin = 3.0e38f;
#pragma unroll 8
    for (int i = 0; i < n; ++i) {
      const float k = to_f32<KV>(sk[i * S]);
      F = fmaxf(F, k);
      kmin = fminf(kmin, k);
    }
  }
  const bool fast =
      (kmin + fminf(cw.u, 0.f) >= F - kFastRange) && (cw.u <= kFastCeil) && (P.pp - F <= kFastCeil);
  float la = 0.f, lb = 0.f;
  if (fast) {
    const float F2 = F * kLog2e;
    const float s0 = exp_nat(P.pp - F);
    float na = P.num * s0, nb = P.den * s0, pw = 1.f;
    if constexpr (FULL) {
#pragma unroll
      for (int i = 0; i < L; ++i) kr[i] = ex2(fmaf(kr[i], kLog2e, -F2));  // ek
#pragma unroll
      for (int i = 0; i < L; ++i) {
        const float ek = kr[i];
        const float vv = to_f32<KV>(sv[i * S]);
        const float ec = ek * cw.eu;
        const float rr = rcp(nb + ec);
        float gq;
        const float gi = gate_grad<RP>(sg, i * S, gq) * rr;  // gN at scale e^{F}
        const float y = fmaf(ec, vv, na) * rr;  // wkv_t
        la = fmaf(pw, gi, la);
        lb = fmaf(-pw, gi * y, lb);
        pw *= cw.ew;
        na = fmaf(na, cw.ew, ek * vv);
        nb = fmaf(nb, cw.ew, ek);
      }
    } else {
#pragma unroll 8
      for (int i = 0; i < n; ++i) {
        const float ek = ex2(fmaf(to_f32<KV>(sk[i * S]), kLog2e, -F2));
        const float vv = to_f32<KV>(sv[i * S]);
        const float ec = ek * cw.eu;
        const float rr = rcp(nb + ec);
        float gq;
        const float gi = gate_grad<RP>(sg, i * S, gq) * rr;
        const float y = fmaf(ec, vv, na) * rr;
        la = fmaf(pw, gi, la);
        lb = fmaf(-pw, gi * y, lb);
        pw *= cw.ew;
        na = fmaf(na, cw.ew, ek * vv);
        nb = fmaf(nb, cw.ew, ek);
      }
    }
    la *= s0;  // from scale e^{F} to the record's e^{P.pp}
    lb *= s0;
  } else {
    exact_states<kSeqChannels, KV>(sk, sv, n, P, cw.w, xa, xb, xp);
    exact_zero_adjoint<kSeqChannels, KV, RP>(sk, sv, sg, n, cw.w, cw.u, xa, xb, xp, la, lb);
  }
  return Adj{la, lb, P.pp};
}

// GATE: the gated output (SeqBwdArgs::r): the staged planes are k, v, the
// output's gradient and r.
template <typename KV, int NS, bool GATE>
__device__ __forceinline__ void seq_bwd_run(const SeqBwdArgs& a, const Launch& L, unsigned char* smem) {
  constexpr int NP = GATE ? 4 : 3;              // planes per stage
  constexpr int RP = GATE ? kSeqTile : 0;       // r's plane after the gradient's
  KV* ring = reinterpret_cast<KV*>(smem);  // stage s: k, v, gy (, r) at (NP s + 0..NP-1) * kSeqTile
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + seq_ring_elems<KV, NS>(NP) * sizeof(KV));
  const int lane = threadIdx.x;
  const ScanGeometry& g = a.g;
  const int nseg = a.nseg;
  const int q = blockIdx.x / nseg, run = blockIdx.x - q * nseg;
  const Column col = column_of(g, q);
  BwdColumn cw;
  cw.w = __ldg(a.w + col.cc);
  cw.u = __ldg(a.u + col.cc);
  cw.ew = expf(-cw.w);
  cw.eu = expf(cw.u);
  cw.gw_s = cw.gw_k = cw.gu_s = cw.gu_k = 0.f;
  const bool tma = a.use_tma != 0;
  constexpr uint32_t kStageBytes = NP * kSeqTile * sizeof(KV);
  const int last = g.nchunks - 1;

  int first, count;  // in walk order: position p is chunk last - p
  segment_of(g.nchunks, nseg, run, first, count);
  // A summary pass (no gk, gv): every run summarises its chunks, and the run
  // holding chunk 0 folds the summaries and writes the start state's
  // gradient; nothing else is computed.
  const bool summary = a.gk == nullptr;
  const int n1 = summary || run < nseg - 1 ? count : 0;
  const int nitems = summary ? n1 : n1 + count;
  auto chunk_of = [&](int it) { return last - (first + (it < n1 ? it : it - n1)); };
  auto issue = [&](int it) {  // lane 0: item it into its stage
    const int s = it % NS;
    const int j = chunk_of(it);
    KV* dk = ring + (size_t)(NP * s) * kSeqTile;
    mbar_arrive_expect_tx(&full[s], kStageBytes);
    tma_load_3d(dk, &a.tk, &full[s], col.c0, j * kChunk, col.b);
    tma_load_3d(dk + kSeqTile, &a.tv, &full[s], col.c0, j * kChunk, col.b);
    tma_load_3d(dk + 2 * kSeqTile, &a.tg, &full[s], col.c0, j * kChunk, col.b);
    if constexpr (GATE) tma_load_3d(dk + 3 * kSeqTile, &a.tr, &full[s], col.c0, j * kChunk, col.b);
  };
  int issued = 0;
  if (tma) {
    if (lane == 0) {
      for (int s = 0; s < NS; ++s) mbar_init(&full[s], 1);
      mbar_init_fence();
      tma_prefetch_desc(&a.tk);
      tma_prefetch_desc(&a.tv);
      tma_prefetch_desc(&a.tg);
      if constexpr (GATE) tma_prefetch_desc(&a.tr);
      for (int it = 0; it < NS && it < nitems; ++it) issue(it);
    }
    issued = min(NS, nitems);
    __syncwarp();
  }
  auto acquire = [&](int it, KV*& dk) {
    const int s = it % NS;
    dk = ring + (size_t)(NP * s) * kSeqTile;
    if (tma) return stage_wait(&full[s], (uint32_t)((it / NS) & 1), a.budget_ns);
    const int j = chunk_of(it);
    copy_box_plain(dk, static_cast<const KV*>(a.k), g, col, j * kChunk);
    copy_box_plain(dk + kSeqTile, static_cast<const KV*>(a.v), g, col, j * kChunk);
    copy_box_plain(dk + 2 * kSeqTile, static_cast<const KV*>(a.gy), g, col, j * kChunk);
    if constexpr (GATE) copy_box_plain(dk + 3 * kSeqTile, static_cast<const KV*>(a.r), g, col, j * kChunk);
    __syncwarp();
    return true;
  };
  auto release = [&](int it) {
    // the stage is only read (see seq_fwd_run): no proxy fence
    __syncwarp();
    if (tma && it + NS < nitems) {
      if (lane == 0) issue(it + NS);
      ++issued;
    }
  };
  auto fail = [&](int it) {
    if (lane == 0) record_error(a.eh, kDevErrTimeout, L.epoch);
    drain_stages<NS>(full, it, issued);
  };

  float xa[kChunk], xb[kChunk], xp[kChunk];  // per-token form's states (local memory)
  const size_t o0 = (size_t)col.b * g.C + col.cc;
  const size_t jstride = (size_t)g.B * g.C;
  auto load_state = [&](int j) {  // the checkpoint before chunk j (the given start state before chunk 0)
    if (j <= 0) return load_state_planes(a.state_in, jstride, o0);
    const size_t o = (size_t)(j - 1) * jstride + o0;
    return State{__ldg(a.ckpt + o), __ldg(a.ckpt + o + g.plane), __ldg(a.ckpt + o + 2 * g.plane)};
  };

  // phase 1: this run's zero-carry adjoint at its first token (in time)
  State Pn = nitems > 0 ? load_state(chunk_of(0)) : empty_state();
  Adj X{0.f, 0.f, 0.f};
  int it = 0;
  for (; it < n1; ++it) {
    const State P = Pn;
    if (it + 1 < nitems) Pn = load_state(chunk_of(it + 1));  // one chunk ahead
    KV* dk;
    if (!acquire(it, dk)) return fail(it);
    const int j = chunk_of(it);
    const int n = min(kChunk, g.T - j * kChunk);
    const Adj A = n == kChunk ? seq_bwd_summary<true, KV, RP>(dk + lane, dk + kSeqTile + lane,
                                                                dk + 2 * kSeqTile + lane, n, cw, P, xa, xb, xp)
                              : seq_bwd_summary<false, KV, RP>(dk + lane, dk + kSeqTile + lane,
                                                                 dk + 2 * kSeqTile + lane, n, cw, P, xa, xb, xp);
    X = it == 0 ? A : fold_adj(A, (float)n * cw.w, X);
    release(it);
  }
  // fault injection: the run holding this chunk never publishes
  const bool skip = a.debug_skip_chunk >= 0 && last - a.debug_skip_chunk >= first &&
                    last - a.debug_skip_chunk < first + count;
  if (n1 > 0 && run < nseg - 1 && col.valid && !skip)
    rec_store(a.recs + (size_t)run * jstride + o0, L.tag, X.la, X.lb, X.f);
  if (summary && run < nseg - 1) return;
  const Adj own = X;  // this run's summary (the summary pass's last run)

  // the carry into this run's end (in time): the gradient given on the
  // state after the last token, if any (the num, den gradients of a state
  // at the given pp: exactly the record form), then the runs after this
  // one, nearest last.  Run 0 holds the last chunks, the only partial one
  // among them, so its span is counted in tokens.
  const bool has_end = a.gstate_end != nullptr;
  X = Adj{0.f, 0.f, 0.f};
  if (has_end)
    X = Adj{__ldg(a.gstate_end + o0), __ldg(a.gstate_end + jstride + o0), __ldg(a.gstate_end + 2 * jstride + o0)};
  for (int r = 0; r < run; ++r) {
    int fr, cr;
    segment_of(g.nchunks, nseg, r, fr, cr);
    Rec rec;
    if (!wait_rec(a.recs + (size_t)r * jstride + o0, col.valid, L, a.eh, a.budget_ns, rec)) return fail(it - 1);
    const Adj Ar{rec_x(rec), rec_y(rec), rec_z(rec)};
    const int span = r == 0 ? g.T - (g.nchunks - cr) * kChunk : cr * kChunk;
    X = (r == 0 && !has_end) ? Ar : fold_adj(Ar, (float)span * cw.w, X);
  }

  // phase 2: gk, gv, and this run's gw, gu
  for (; it < nitems; ++it) {
    const State P = Pn;
    if (it + 1 < nitems) Pn = load_state(chunk_of(it + 1));
    KV* dk;
    if (!acquire(it, dk)) return fail(it);
    const int j = chunk_of(it);
    const int n = min(kChunk, g.T - j * kChunk);
    const int64_t row = ((int64_t)col.b * g.T + (int64_t)j * kChunk) * g.C + col.c;
    float gw_acc, gu_acc;
    float* grp = GATE ? a.gr + row : nullptr;
    const bool has_succ = j < last || has_end;
    if (n == kChunk)
      seq_bwd_chunk<true, KV, RP>(dk + lane, dk + kSeqTile + lane, dk + 2 * kSeqTile + lane, n, cw, P, has_succ, X,
                                  a.gk + row, a.gv + row, grp, g.C, col.valid, gw_acc, gu_acc, xa, xb, xp);
    else
      seq_bwd_chunk<false, KV, RP>(dk + lane, dk + kSeqTile + lane, dk + 2 * kSeqTile + lane, n, cw, P, has_succ,
                                   X, a.gk + row, a.gv + row, grp, g.C, col.valid, gw_acc, gu_acc, xa, xb, xp);
    kahan_add(cw.gw_s, cw.gw_k, gw_acc);
    kahan_add(cw.gu_s, cw.gu_k, gu_acc);
    release(it);
  }
  if (summary) {  // the run holding chunk 0: its own summary after the carry
    const int span = run == 0 ? g.T : count * kChunk;
    X = (run == 0 && !has_end) ? own : fold_adj(own, (float)span * cw.w, X);
    if (a.gstate_in && col.valid) {
      a.gstate_in[o0] = X.la;
      a.gstate_in[jstride + o0] = X.lb;
      a.gstate_in[2 * jstride + o0] = X.f;
    }
    return;
  }
  // the run holding chunk 0 ends at the sequence's start: X is then the
  // gradient of the start state's num, den, in record form at its pp
  if (run == nseg - 1 && a.gstate_in && col.valid) {
    a.gstate_in[o0] = X.la;
    a.gstate_in[jstride + o0] = X.lb;
    a.gstate_in[2 * jstride + o0] = X.f;
  }
  // one gw, gu row per (run, batch row): row run * B + b of [2][nseg * B][C]
  // (added up in row order by the reduction kernel that follows)
  if (col.valid) {
    const size_t o = (size_t)run * jstride + o0;
    a.part[o] = cw.gw_s;
    a.part[(size_t)nseg * jstride + o] = cw.gu_s;
  }
}

template <typename KV, int NS, bool GATE>
__global__ void __launch_bounds__(kSeqChannels) seq_bwd_kernel(const __grid_constant__ SeqBwdArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  // the gw, gu reduction that follows may be launched now (its CTAs start as
  // this launch's CTAs leave SMs, and wait for its completion before reading)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const Launch L = seq_launch(a.eh);
  seq_bwd_run<KV, NS, GATE>(a, L, smem);
  seq_exit(a.exited, a.eh, L.epoch);
}

// ------------------------------------------------------------------ launch
struct DevInfo {
  int sms = 0;
  size_t smem_per_sm = 0;
  size_t l2 = 0;
};

cudaError_t dev_info(DevInfo& d) {
  static DevInfo cache[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && cache[dev].sms > 0) {
    d = cache[dev];
    return cudaSuccess;
  }
  int sms = 0, smem = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
  if (e != cudaSuccess) return e;
  int l2 = 0;
  e = cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev);
  if (e != cudaSuccess) return e;
  d.sms = sms;
  d.smem_per_sm = (size_t)smem;
  d.l2 = (size_t)l2;
  if (dev >= 0 && dev < 64) cache[dev] = d;
  return cudaSuccess;
}

// Per device and kernel: the opt-in to the kernel's shared memory and its
// resident CTAs per SM at that size (one warp each), queried once (the first
// call on a device, before any stream capture, as for the other kernels).
template <class Args, void (*K)(Args)>
cudaError_t resident_per_sm(size_t smem, int& per_sm) {
  static int cache[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && cache[dev] > 0) {
    per_sm = cache[dev];
    return cudaSuccess;
  }
  e = cudaFuncSetAttribute(K, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, K, kSeqChannels, smem);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64) cache[dev] = per_sm;
  return cudaSuccess;
}

template <class Args>
cudaError_t launch_runs(void (*kern)(Args), unsigned int nblk, size_t smem, bool cooperative, cudaStream_t s,
                        const Args& a) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(nblk);
  cfg.blockDim = dim3(kSeqChannels);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = cooperative ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

// Runs per column: about `warps` warps per SM in all (every run is
// resident, so no more than the SMs hold at two stages per run), at most
// kSeqMaxRuns and one per chunk; and 1 when the inputs that phase 2
// re-reads would not fit in L2 (60% of it) while the columns alone fill
// every SM.
int choose_runs(const DevInfo& d, const ScanGeometry& g, int per_sm2, size_t input_bytes, int warps, bool chained) {
  const long long cols = (long long)g.B * g.nwg;
  const long long cap = (long long)per_sm2 * d.sms;
  // when phase 2 re-reads from DRAM anyway, more runs only add phase-1 work
  if (!chained && (double)input_bytes > 0.6 * (double)d.l2 && warps > 8) warps = 8;
  const long long target = cap < (long long)warps * d.sms ? cap : (long long)warps * d.sms;
  long long nseg = target / cols;
  if (nseg > kSeqMaxRuns) nseg = kSeqMaxRuns;
  if (nseg > g.nchunks) nseg = g.nchunks;
  if (nseg < 1) nseg = 1;
  const double reread = (double)input_bytes * (double)(nseg - 1) / (double)nseg;
  if (cols >= d.sms && reread > 0.6 * (double)d.l2) nseg = 1;
  return (int)nseg;
}

// Launches `K<NS>::fn` for the largest NS of 8, 4, 3, 2 at which all `nblk`
// CTAs are resident at once (needed when runs wait on each other, and it
// spares a second wave otherwise).
template <class Args, template <int> class K>
cudaError_t launch_staged(const DevInfo& d, const Args& a, unsigned int nblk, size_t stage, bool coop,
                          cudaStream_t s) {
  const unsigned int need = (nblk + d.sms - 1) / d.sms;
  if (a.use_tma) {
    int per_sm = 0;
    cudaError_t e = resident_per_sm<Args, K<8>::fn>(8 * stage + 128, per_sm);
    if (e != cudaSuccess) return e;
    if ((unsigned)per_sm >= need) return launch_runs(K<8>::fn, nblk, 8 * stage + 128, coop, s, a);
    e = resident_per_sm<Args, K<4>::fn>(4 * stage + 128, per_sm);
    if (e != cudaSuccess) return e;
    if ((unsigned)per_sm >= need) return launch_runs(K<4>::fn, nblk, 4 * stage + 128, coop, s, a);
    e = resident_per_sm<Args, K<3>::fn>(3 * stage + 128, per_sm);
    if (e != cudaSuccess) return e;
    if ((unsigned)per_sm >= need) return launch_runs(K<3>::fn, nblk, 3 * stage + 128, coop, s, a);
  }
  int per_sm2 = 0;
  cudaError_t e = resident_per_sm<Args, K<2>::fn>(2 * stage + 128, per_sm2);
  if (e != cudaSuccess) return e;
  return launch_runs(K<2>::fn, nblk, 2 * stage + 128, coop, s, a);
}

// Plans the runs (a.nseg, and a.chain for the forward pass) and launches
// Kern, or KernChain for chained runs.
template <class Args, template <int> class Kern, template <int> class KernChain>
cudaError_t launch_planned(const DevInfo& d, Args& a, int arrays, size_t elem, size_t input_bytes, int warps,
                           cudaStream_t s) {
  const unsigned int cols = (unsigned int)a.g.B * a.g.nwg;
  const size_t stage = (size_t)arrays * kSeqTile * elem;
  const int cap_runs = a.nseg;
  bool chained = false;
  int forced = 0;
  if constexpr (std::is_same<Args, SeqFwdArgs>::value) {
    // Chained runs when phase 2 would re-read from DRAM (inputs beyond L2)
    // while the columns alone leave SMs idle; a positive a.chain on entry
    // forces chained runs of that length.
    forced = a.chain;
    chained = forced > 0 || ((long long)cols < d.sms && (double)input_bytes > 0.6 * (double)d.l2);
    // Chained runs take the caller's warps per SM too: on the long-context
    // forward (B=1 T=131072 C=2560 bf16) 12 per SM give 22 runs per column;
    // 29 runs (16 per SM) were 8% slower, 23 or 24 runs 30-40%, 20 runs 10%
    // (one GPU call, one-chunk items).
  }
  // a stage of the chained walk holds chain_chunks(elem) chunks
  const size_t cstage = chained ? stage * chain_chunks(elem) : stage;
  // resident CTAs per SM of the kernel that will run, at two stages
  int per_sm2 = 0;
  cudaError_t e = chained ? resident_per_sm<Args, KernChain<2>::fn>(2 * cstage + 128, per_sm2)
                          : resident_per_sm<Args, Kern<2>::fn>(2 * stage + 128, per_sm2);
  if (e != cudaSuccess) return e;
  a.nseg = choose_runs(d, a.g, per_sm2, input_bytes, warps, chained);
  if (cap_runs > 0 && a.nseg > cap_runs) a.nseg = cap_runs;
  if constexpr (std::is_same<Args, SeqFwdArgs>::value) {
    a.chain = 0;
    if (chained) {
      // runs of `len` chunks, the runs in flight (nseg per column) within 35%
      // of L2 (longer runs fall out of L2 before phase 2; shorter ones make
      // the chain of carried states the bound).  Long-context forward, 22
      // runs per column: 0.57 ms at 6 chunks (42 MB in flight), 0.60 at 5,
      // 0.65 at 4, 0.68 at 8.
      long long len = forced;
      if (len <= 0) {
        const double per_run_chunk = (double)cols * a.nseg * stage;  // one chunk of every run in flight
        len = (long long)(0.35 * (double)d.l2 / per_run_chunk);
        if (len < 4) len = 4;
        if (len > 64) len = 64;
      }
      a.chain = (int)len;
      const int R = (a.g.nchunks + a.chain - 1) / a.chain;
      if (a.nseg > R) a.nseg = R;  // a warp per run at most
    }
  }
  const unsigned int nblk = cols * (unsigned int)a.nseg;
  const bool coop = a.nseg > 1;  // runs wait on each other
  if (chained) return launch_staged<Args, KernChain>(d, a, nblk, cstage, coop, s);
  return launch_staged<Args, Kern>(d, a, nblk, stage, coop, s);
}

template <typename KV, int YM, bool CHAIN>
struct FwdKern {
  template <int NS>
  struct At {
    static constexpr void (*fn)(SeqFwdArgs) = seq_fwd_kernel<KV, NS, YM, CHAIN>;
  };
};

template <typename KV, bool GATE>
struct BwdKern {
  template <int NS>
  struct At {
    static constexpr void (*fn)(SeqBwdArgs) = seq_bwd_kernel<KV, NS, GATE>;
  };
};

template <typename KV, int YM>
cudaError_t launch_seq_fwd_t(SeqFwdArgs& a, cudaStream_t s) {
  DevInfo d;
  cudaError_t e = dev_info(d);
  if (e != cudaSuccess) return e;
  const size_t input_bytes = (size_t)a.g.B * a.g.T * a.g.C * 2 * sizeof(KV);
  // the forward kernel's registers allow more warps than its two stages of
  // shared memory: aim at 12 per SM
  return launch_planned<SeqFwdArgs, FwdKern<KV, YM, false>::template At, FwdKern<KV, YM, true>::template At>(
      d, a, 2, sizeof(KV), input_bytes, 12, s);
}

}  // namespace

cudaError_t launch_seq_forward(SeqFwdArgs& a, int kv_dtype, bool write_y, cudaStream_t s) {
  const int ym = !write_y ? kYNone : (a.r ? kYGated : kYWkv);
  if (kv_dtype == 0) {
    if (ym == kYGated) return launch_seq_fwd_t<float, kYGated>(a, s);
    return ym == kYWkv ? launch_seq_fwd_t<float, kYWkv>(a, s) : launch_seq_fwd_t<float, kYNone>(a, s);
  }
  if (ym == kYGated) return launch_seq_fwd_t<__nv_bfloat16, kYGated>(a, s);
  return ym == kYWkv ? launch_seq_fwd_t<__nv_bfloat16, kYWkv>(a, s) : launch_seq_fwd_t<__nv_bfloat16, kYNone>(a, s);
}

template <typename KV, bool GATE>
cudaError_t launch_seq_bwd_t(SeqBwdArgs& a, cudaStream_t s) {
  DevInfo d;
  cudaError_t e = dev_info(d);
  if (e != cudaSuccess) return e;
  constexpr int NP = GATE ? 4 : 3;
  const size_t input_bytes = (size_t)a.g.B * a.g.T * a.g.C * NP * sizeof(KV);
  // the backward kernel's registers (up to 255 per thread) allow 8 warps per SM
  return launch_planned<SeqBwdArgs, BwdKern<KV, GATE>::template At, BwdKern<KV, GATE>::template At>(
      d, a, NP, sizeof(KV), input_bytes, 8, s);
}

cudaError_t launch_seq_backward(SeqBwdArgs& a, int kv_dtype, cudaStream_t s) {
  if (a.r) return kv_dtype == 0 ? launch_seq_bwd_t<float, true>(a, s) : launch_seq_bwd_t<__nv_bfloat16, true>(a, s);
  return kv_dtype == 0 ? launch_seq_bwd_t<float, false>(a, s) : launch_seq_bwd_t<__nv_bfloat16, false>(a, s);
}

// The device-wide error record of this file's kernels (wkv_sync_status).
cudaError_t take_error_seq(unsigned int* code) { return take_module_error(code); }

}  // namespace wkv
