// wkv_cmix.cu -- the pointwise parts of channel mixing, forward and backward.
//
// Channel mixing computes K from the token-shifted input, V from K, and
// gates the result with a sigmoid of the receptance ("RWKV についての調査記録",
// the Time Mixing / Channel Mixing walk-through); the non-linearity between
// the key and value projections is a squared ReLU ("Инновационная
// архитектура RWKV", section "Механизмы взаимодействия"; "RWKV解读" section
// "3、RWKV的网络架构", eq. (10)).  Around the three projections, elementwise:
//
//   a   = max(k, 0)^2             gk  = 2 max(k, 0) ga
//   out = sigmoid(r) vk           gvk = gout sigmoid(r)
//                                 gr  = gvk (1 - sigmoid(r)) vk
//
// Bound by HBM bandwidth: 8, 12, 12 and 20 bytes per element.  Four elements
// per thread with 16-byte accesses when every pointer is 16-byte aligned (the
// last n % 4 elements one per thread), one per thread otherwise.  Each
// element is read before it is written, by the same thread, so an output may
// be the very buffer of an input (in place).
#include <cstdint>
#include <cuda_runtime.h>

#include "wkv_common.cuh"
#include "wkv_internal.h"

namespace wkv {

namespace {

enum { kSqrelu = 0, kSqreluBwd = 1, kGate = 2, kGateBwd = 3 };

template <int OP>
__device__ __forceinline__ void cmix_op(float x, float y, float z, float& p, float& q) {
  if constexpr (OP == kSqrelu) {
    const float m = fmaxf(x, 0.f);
    p = m * m;
  } else if constexpr (OP == kSqreluBwd) {
    p = 2.f * fmaxf(x, 0.f) * y;
  } else if constexpr (OP == kGate) {
    p = sigmoid(x) * y;
  } else {
    const float s = sigmoid(x);
    const float gv = z * s;
    q = gv;
    p = fmaf(-gv, s, gv) * y;
  }
}

template <int OP>
__device__ __forceinline__ void cmix_one(const CmixArgs& a, int64_t i) {
  const float x = a.x[i];
  const float y = OP != kSqrelu ? a.y[i] : 0.f;
  const float z = OP == kGateBwd ? a.z[i] : 0.f;
  float p, q = 0.f;
  cmix_op<OP>(x, y, z, p, q);
  a.o1[i] = p;
  if constexpr (OP == kGateBwd) a.o2[i] = q;
}

// V = 4: float4 items (the caller checked the alignment), then the tail of
// n % 4 elements by the first threads of CTA 0.  V = 1: one element each.
template <int OP, int V>
__global__ void __launch_bounds__(256) cmix_kernel(const CmixArgs a) {
  const int64_t items = a.n / V;
  for (int64_t it = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; it < items; it += (int64_t)gridDim.x * blockDim.x) {
    if constexpr (V == 1) {
      cmix_one<OP>(a, it);
    } else {
      const float4 x = reinterpret_cast<const float4*>(a.x)[it];
      float4 y = make_float4(0.f, 0.f, 0.f, 0.f), z = y, p, q = y;
      if constexpr (OP != kSqrelu) y = reinterpret_cast<const float4*>(a.y)[it];
      if constexpr (OP == kGateBwd) z = reinterpret_cast<const float4*>(a.z)[it];
      cmix_op<OP>(x.x, y.x, z.x, p.x, q.x);
      cmix_op<OP>(x.y, y.y, z.y, p.y, q.y);
      cmix_op<OP>(x.z, y.z, z.z, p.z, q.z);
      cmix_op<OP>(x.w, y.w, z.w, p.w, q.w);
      reinterpret_cast<float4*>(a.o1)[it] = p;
      if constexpr (OP == kGateBwd) reinterpret_cast<float4*>(a.o2)[it] = q;
    }
  }
  if constexpr (V > 1) {
    const int64_t tail = a.n - items * V;
    if (blockIdx.x == 0 && threadIdx.x < tail) cmix_one<OP>(a, items * V + threadIdx.x);
  }
}

bool aligned16(const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

template <int OP>
cudaError_t launch_op(const CmixArgs& a, cudaStream_t s) {
  const bool vec4 = aligned16(a.x) && aligned16(a.y) && aligned16(a.z) && aligned16(a.o1) && aligned16(a.o2);
  if (vec4)
    cmix_kernel<OP, 4><<<elementwise_grid(a.n / 4, 256), 256, 0, s>>>(a);
  else
    cmix_kernel<OP, 1><<<elementwise_grid(a.n, 256), 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_cmix(int op, const CmixArgs& a, cudaStream_t s) {
  switch (op) {
    case kSqrelu:
      return launch_op<kSqrelu>(a, s);
    case kSqreluBwd:
      return launch_op<kSqreluBwd>(a, s);
    case kGate:
      return launch_op<kGate>(a, s);
    default:
      return launch_op<kGateBwd>(a, s);
  }
}

}  // namespace wkv
