// wkv_fwd.cu -- WKV forward pass: single-pass chunked scan over time.
//
// The recurrent form of the operator ("RWKV解读：在Transformer的时代的新RNN",
// section "3、RWKV的网络架构": eq. (8) can be written recursively) is a
// linear recurrence whose decay is data independent, which is what makes the
// training form time-parallel (qiita "RWKV についての調査記録", section
// "Trainingについて").  Time is cut into chunks of kChunk tokens.  One tile
// is (chunk, batch row, 128 channels); one lane owns one channel.
//
//   1. load the tile's k, v into registers (coalesced along C);
//   2. summarise the chunk from the empty state -> (num, den, pp);
//   3. publish the summary as a leaf of the binary-indexed tree over chunks
//      (wkv_common.cuh), wait for the popcount(j) tree nodes that make up
//      the prefix before chunk j, combine them in a fixed order into the
//      state at the chunk start, and publish the tree nodes this chunk
//      completes;
//   4. write the state after the chunk (the checkpoint the backward pass
//      restarts from), then re-run the chunk from the start state writing
//      wkv_t.
//
// k and v cross HBM once.  Results are bitwise reproducible: no step
// depends on which tile finished first.
#include <cuda_bf16.h>

#include "wkv_common.cuh"
#include "wkv_internal.h"

namespace wkv {

template <typename KV>
__device__ __forceinline__ float load_kv(const KV* p);
template <>
__device__ __forceinline__ float load_kv<float>(const float* p) {
  return __ldg(p);
}
template <>
__device__ __forceinline__ float load_kv<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}

template <typename KV, int L, bool WRITE_Y>
__global__ void __launch_bounds__(kCtaChannels, 4) fwd_scan_kernel(const FwdArgs a) {
  const ScanGeometry& g = a.g;
  const unsigned int ticket = take_ticket(a.ticket, g.ntiles);
  if (ticket >= g.ntiles) return;  // only if the counter was not zeroed: never touch memory then
  const int per_j = g.B * g.ncb;
  const int j = ticket / per_j;
  const int rem = ticket - j * per_j;
  const int b = rem / g.ncb;
  const int cb = rem - b * g.ncb;
  const int c = cb * kCtaChannels + threadIdx.x;
  const bool valid = c < g.C;
  const int cc = valid ? c : g.C - 1;  // out-of-range lanes shadow the last channel, never store
  const int t0 = j * L;
  const int len = min(L, g.T - t0);

  const KV* kp = static_cast<const KV*>(a.k);
  const KV* vp = static_cast<const KV*>(a.v);
  const int64_t base = ((int64_t)b * g.T + t0) * g.C + cc;

  float kr[L], vr[L];
#pragma unroll
  for (int i = 0; i < L; ++i) {
    if (i < len) {
      kr[i] = load_kv<KV>(kp + base + (int64_t)i * g.C);
      vr[i] = load_kv<KV>(vp + base + (int64_t)i * g.C);
    } else {
      kr[i] = 0.f;
      vr[i] = 0.f;
    }
  }
  const float w = __ldg(a.w + cc);
  const float u = __ldg(a.u + cc);

  // 2. summary of this chunk alone
  State agg = empty_state();
#pragma unroll
  for (int i = 0; i < L; ++i)
    if (i < len) step(agg, kr[i], vr[i], w);

  if (j == a.debug_skip_chunk) return;  // fault injection: this tile never publishes

  const int wg = cb * 4 + (threadIdx.x >> 5);
  uint64_t* flags = a.flags + ((int64_t)b * g.nwg + wg) * g.nnodes;
  const size_t NP = g.nplane;
  const float* nodes = a.nodes;
  auto nslot = [&](int nd) -> size_t { return ((size_t)nd * g.B + b) * g.C + cc; };
  const bool has_succ = j < g.nchunks - 1;  // nodes of the last chunk are never read
  auto put_node = [&](int level, const State& st, uint64_t status) {
    const int nd = node_index(g.level_off, j, level);
    if (valid && status == kNodeReady) {
      const size_t o = nslot(nd);
      a.nodes[o] = st.num;
      a.nodes[o + NP] = st.den;
      a.nodes[o + 2 * NP] = st.pp;
    }
    publish(flags + nd, a.epoch, status);
  };

  if (has_succ) put_node(0, agg, kNodeReady);
  const int nf = __popc(j);      // nodes in the prefix list of chunk j
  const int nup = __ffs(~j) - 1; // trailing ones of j: tree nodes completed here
  const int rc = wait_flags(
      [&](int i) {
        int e, l;
        fenwick_node(j, i, e, l);
        return flags + node_index(g.level_off, e, l);
      },
      nf, a.epoch, a.budget_ns, a.eh);
  if (rc != kWaitOk) {
    if (rc == kWaitTimeout && (threadIdx.x & 31) == 0) record_error(a.eh, kDevErrTimeout, a.epoch);
    if (has_succ)
      for (int s = 1; s <= nup; ++s) put_node(s, agg, kNodeErr);
    return;
  }

  // prefix before chunk j, nearest node first; nodes are read four at a time
  State prefix = empty_state();
  State node = agg;
  int x = j, i = 0;
  while (x) {
    State nv[4];
    int ne[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      ne[q] = -1;
      if (x) {
        const int lvl = __ffs(x) - 1;
        ne[q] = x - 1;
        const size_t o = nslot(node_index(g.level_off, x - 1, lvl));
        nv[q] = State{ld_cg(nodes + o), ld_cg(nodes + o + NP), ld_cg(nodes + o + 2 * NP)};
        x &= x - 1;
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (ne[q] >= 0) {
        // the node ends (j - 1 - end) whole chunks before chunk j starts
        prefix = combine(nv[q], (float)((j - 1 - ne[q]) * L) * w, prefix);
        if (i < nup && has_succ) {
          // node (j, i+1) = node (j - 2^i, i) followed by node (j, i)
          node = combine(nv[q], (float)((1 << i) * L) * w, node);
          put_node(i + 1, node, kNodeReady);
        }
        ++i;
      }
    }
  }

  if (valid) {
    const State incl = combine(prefix, (float)len * w, agg);
    const size_t P = g.plane;
    const size_t o = ((size_t)j * g.B + b) * g.C + cc;
    a.incl[o] = incl.num;
    a.incl[o + P] = incl.den;
    a.incl[o + 2 * P] = incl.pp;
  }

  if constexpr (WRITE_Y) {
    // 4. re-run from the state at the chunk start
    State s = prefix;
    float* yp = a.y + base;
#pragma unroll
    for (int i = 0; i < L; ++i) {
      if (i < len) {
        const float yv = output(s, kr[i], vr[i], u);
        if (valid) __stcs(yp + (int64_t)i * g.C, yv);
        step(s, kr[i], vr[i], w);
      }
    }
  }
}

cudaError_t launch_forward(const FwdArgs& a, int kv_dtype, bool write_y, cudaStream_t s) {
  const dim3 grid(a.g.ntiles), block(kCtaChannels);
  if (kv_dtype == 0) {
    if (write_y)
      fwd_scan_kernel<float, kChunk, true><<<grid, block, 0, s>>>(a);
    else
      fwd_scan_kernel<float, kChunk, false><<<grid, block, 0, s>>>(a);
  } else {
    if (write_y)
      fwd_scan_kernel<__nv_bfloat16, kChunk, true><<<grid, block, 0, s>>>(a);
    else
      fwd_scan_kernel<__nv_bfloat16, kChunk, false><<<grid, block, 0, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace wkv
