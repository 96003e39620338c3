// wkv_pipe.cuh -- the tile pipeline of the persistent scan kernels (sm_103a).
//
// A scan kernel runs a fixed number of CTAs (a multiple of the SM count's
// resident capacity), each with one producer warp, kConsumerWarps consumer
// warps and one walker warp (the walkers carry chunk results from chunk to
// chunk; see the scan kernels).  The producer takes tile tickets from a counter in the
// workspace header, in increasing order, and stages every tile's input
// arrays ([chunk of tokens] x [128 channels] each) into a ring of shared
// memory stages: by TMA (cp.async.bulk.tensor, completion counted on the
// stage's `full` mbarrier) when the tensors meet TMA's alignment rules, else
// by plain loads.  Consumer warps take the stages in the same order, and
// release each one on its `empty` mbarrier.  Tickets are handed out in scan
// order and each CTA handles its tickets in increasing order; a tile only
// waits on results of earlier chunks, which the walkers (one warp per CTA,
// each with a fixed set of chains, all resident: the kernels are launched
// cooperatively) derive from tiles with smaller tickets.  The oldest
// unfinished tile can therefore always progress: the kernels cannot
// deadlock.
//
// Every wait is bounded (%globaltimer budget); an expired wait records
// WKV_ERR_TIMEOUT in the workspace header and the kernel winds down.
#pragma once

#include <cuda.h>
#include <cstdint>

#include "wkv_common.cuh"

namespace wkv {

constexpr int kConsumerWarps = 4;                       // one channel per lane: 128 channels per tile
constexpr int kProducerWarp = kConsumerWarps;            // stages the tiles
constexpr int kWalkerWarp = kConsumerWarps + 1;          // carries chunk results along the chains
constexpr int kPipeThreads = (kConsumerWarps + 2) * 32;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking: whether the phase of `bar` with the given parity completed.
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase of `bar` with the given parity to complete, for at
// most budget_ns.  Returns false on expiry.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t budget_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer() - t0 > budget_ns) return false;
  }
}

// 16-byte asynchronous copy global -> shared that bypasses L1 (so a copy
// issued again reads the current value in L2), and the wait for all of this
// thread's copies.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// Orders this thread's generic-proxy accesses to shared memory before later
// async-proxy (TMA) writes to the same place.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// One TMA tile load of a rank-3 tensor map: box at coordinates (x, y, z),
// innermost first; completion is counted on `bar`.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Pipeline control block in shared memory.
template <int NSTAGE>
struct PipeCtl {
  uint64_t full[NSTAGE];   // one arrival (producer) + the stage's TMA bytes
  uint64_t empty[NSTAGE];  // one arrival per consumer warp
  int tile[NSTAGE];        // ticket staged in the stage, -1 = no more tiles
  int abort;               // set when this CTA gave up a wait
  unsigned long long epoch;  // this launch's epoch (see Launch)
};

// Bytes reserved for the control block: a multiple of 128, so that what
// follows it in shared memory (16-byte records) stays aligned.
template <int NSTAGE>
__host__ __device__ constexpr size_t pipe_ctl_bytes() {
  return (sizeof(PipeCtl<NSTAGE>) + 127) / 128 * 128;
}

// Initialises the control block and returns this launch's identity: every
// CTA reads the workspace's sequence number before any CTA of the launch can
// advance it (that happens in pipe_exit, after every CTA has finished).
template <int NSTAGE>
__device__ __forceinline__ Launch pipe_init(PipeCtl<NSTAGE>* ctl, const WsHeader* h) {
  if (threadIdx.x == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], kConsumerWarps);
    }
    ctl->abort = 0;
    ctl->epoch = *(volatile const unsigned long long*)&h->seq + 1ull;
    mbar_init_fence();
  }
  __syncthreads();
  const unsigned long long e = ctl->epoch;
  return Launch{e, tag_of(e)};
}

// Records that this launch (epoch) gave up a wait, CTA-wide and device-wide.
template <int NSTAGE>
__device__ __forceinline__ void pipe_fail(PipeCtl<NSTAGE>* ctl, WsHeader* h, unsigned int code, uint64_t epoch) {
  *(volatile int*)&ctl->abort = 1;
  record_error(h, code, epoch);
}

// The producer warp's loop.  `stage_fill(tile, stage, bar)` is called by the
// whole warp for each ticket below ntiles; with TMA it must have lane 0 issue
// the copies after lane 0 armed `bar` for `tx_bytes`, else it copies with all
// lanes and the helper arrives for it.
template <int NSTAGE, class Fill>
__device__ __forceinline__ void producer_loop(PipeCtl<NSTAGE>* ctl, unsigned int* ticket, unsigned int ntiles,
                                              bool use_tma, uint32_t tx_bytes, uint64_t budget_ns, WsHeader* h,
                                              uint64_t epoch, Fill stage_fill) {
  const int lane = threadIdx.x & 31;
  int s = 0;
  uint32_t phase = 0;
  for (int it = 0;; ++it) {
    if (it >= NSTAGE) {
      // wait until every consumer warp released the stage's previous tile
      bool ok = true;
      if (lane == 0) ok = mbar_wait(&ctl->empty[s], phase ^ 1u, budget_ns);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        pipe_fail(ctl, h, kDevErrTimeout, epoch);
        // the stage may still be read: nothing more is issued; consumers stop at their own bounded waits
        return;
      }
    }
    unsigned int t = 0;
    if (lane == 0) t = *(volatile int*)&ctl->abort ? ntiles : atomicAdd(ticket, 1u);
    t = __shfl_sync(0xffffffffu, t, 0);
    if (t >= ntiles) {
      if (lane == 0) {
        ctl->tile[s] = -1;
        mbar_arrive(&ctl->full[s]);
      }
      return;
    }
    if (lane == 0) ctl->tile[s] = static_cast<int>(t);
    if (use_tma) {
      if (lane == 0) mbar_arrive_expect_tx(&ctl->full[s], tx_bytes);
      stage_fill(t, s, &ctl->full[s]);
    } else {
      stage_fill(t, s, &ctl->full[s]);
      __threadfence_block();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->full[s]);
    }
    if (++s == NSTAGE) {
      s = 0;
      phase ^= 1u;
    }
  }
}

// Last CTA out resets the launch's ticket counter for the next launch that
// uses the same workspace (every CTA has stopped taking tickets by then) and
// advances the workspace's sequence number to this launch's epoch.
__device__ __forceinline__ void pipe_exit(unsigned int* ticket, unsigned int* exited, WsHeader* h,
                                          unsigned long long epoch) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(exited, 1u) == gridDim.x - 1) {
      atomicExch(ticket, 0u);
      atomicExch(exited, 0u);
      atomicExch(&h->seq, epoch);
    }
  }
}

// Plain-load copy of one [rows x 128] tile of a [B, T, C] tensor into shared
// memory, zero outside the tensor (the TMA path's fill value): the whole
// producer warp takes part.
template <typename E>
__device__ __forceinline__ void copy_tile_plain(E* dst, const E* src, int B, int T, int C, int b, int t0, int c0,
                                                int rows) {
  const int lane = threadIdx.x & 31;
  for (int i = 0; i < rows; ++i) {
    const int t = t0 + i;
    for (int q = lane; q < 128; q += 32) {
      const int c = c0 + q;
      E val = E(0.f);
      if (t < T && c < C) val = src[((int64_t)b * T + t) * C + c];
      dst[i * 128 + q] = val;
    }
  }
}

// Launches a scan kernel cooperatively: all its CTAs are resident at once
// (or the launch fails), which the walkers' fixed chain assignment needs.
template <class Args>
inline cudaError_t launch_cooperative(void (*kern)(Args), unsigned int nblk, size_t smem, cudaStream_t s,
                                      const Args& args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(nblk);
  cfg.blockDim = dim3(kPipeThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args);
}

}  // namespace wkv
