// wkv_state.cu -- the state after consecutive segments of one sequence, from
// each segment's own state (after its tokens, from the empty state) and its
// length.  The decay does not depend on the data ("RWKV についての調査記録",
// section "Trainingについて"), so a segment acts on the carried state as
// "decay by its length, then add its own sums": the associative combine of
// the scan kernels (wkv_common.cuh), folded over the segments in order.
// This is what lets the segments of one long sequence run on different
// devices: each summarises its own, the summaries are exchanged, and each
// folds those before it into the state it starts from.
//
// One thread per (batch row, channel), segments in order: a few bytes per
// segment and element, far from any bound.
#include <cstdint>
#include <cuda_runtime.h>

#include "wkv_common.cuh"
#include "wkv_internal.h"

namespace wkv {

namespace {

__global__ void __launch_bounds__(256) state_fold_kernel(const FoldArgs a) {
  const size_t bc = (size_t)a.B * a.C;
  for (size_t o = (size_t)blockIdx.x * blockDim.x + threadIdx.x; o < bc; o += (size_t)gridDim.x * blockDim.x) {
    const float w = __ldg(a.w + o % a.C);
    State P = empty_state();
    for (int i = 0; i < a.n; ++i)
      P = combine(P, (float)a.len[i] * w, load_state_planes(a.states + (size_t)i * 3 * bc, bc, o));
    store_state_planes(a.out, bc, o, P);
  }
}

}  // namespace

cudaError_t launch_state_fold(const FoldArgs& a, cudaStream_t s) {
  state_fold_kernel<<<elementwise_grid((int64_t)a.B * a.C, 256), 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace wkv
