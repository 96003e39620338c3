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

#include "wkv_adjoint.cuh"
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

// The backward counterpart: the gradient of a segment's start state is its
// own (from its outputs' gradients, with nothing after it) plus the next
// segment's start-state gradient decayed over the segment's length (the
// adjoint recurrence run backwards over tokens with no output gradient:
// la <- e^{-w} la, lb alike), folded from the last segment to the first.
// Planes (g_num, g_den, pp): the gradients of a state's num, den at its pp.
__global__ void __launch_bounds__(256) adjoint_fold_kernel(const AdjFoldArgs a) {
  const size_t bc = (size_t)a.B * a.C;
  for (size_t o = (size_t)blockIdx.x * blockDim.x + threadIdx.x; o < bc; o += (size_t)gridDim.x * blockDim.x) {
    const float w = __ldg(a.w + o % a.C);
    bool have = a.gend != nullptr;
    Adj X{0.f, 0.f, 0.f};
    if (have) X = Adj{__ldg(a.gend + o), __ldg(a.gend + bc + o), __ldg(a.gend + 2 * bc + o)};
    for (int i = a.n - 1; i >= 0; --i) {
      const float* p = a.adj + (size_t)i * 3 * bc;
      const Adj A{__ldg(p + o), __ldg(p + bc + o), __ldg(p + 2 * bc + o)};
      X = have ? fold_adj(A, (float)a.len[i] * w, X) : A;
      have = true;
    }
    a.out[o] = X.la;
    a.out[bc + o] = X.lb;
    a.out[2 * bc + o] = X.f;
  }
}

}  // namespace

cudaError_t launch_adjoint_fold(const AdjFoldArgs& a, cudaStream_t s) {
  adjoint_fold_kernel<<<elementwise_grid((int64_t)a.B * a.C, 256), 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_state_fold(const FoldArgs& a, cudaStream_t s) {
  state_fold_kernel<<<elementwise_grid((int64_t)a.B * a.C, 256), 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace wkv
