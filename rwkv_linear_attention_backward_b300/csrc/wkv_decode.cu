// wkv_decode.cu -- one RNN-mode step of the WKV time mixing (decode).
//
// In inference the layer takes the current token and a state and returns an
// output and the new state ("RWKV についての調査記録", section "RWKVとは？";
// "介绍RWKV – 具有Transformer优势的RNN", section
// "RWKV作为RNN和transformer的结合体").  Fused per element (l, b, c):
//
//   token shift, eq. (7) of "RWKV解读：在Transformer的时代的新RNN":
//       xk = mu_k x + (1 - mu_k) x_prev   (xv, xr alike; optional outputs)
//   wkv of this token from the carried state (num, den, pp) and (k, v, u);
//   gate, eq. (9): y = sigmoid(r) * wkv;
//   state update: consume (k, v) with decay w (same step as the scans).
//
// Pure streaming: every element is independent, 60 bytes move per element
// with the mix outputs, 48 without (fp32 token inputs).  With bf16 token
// inputs (x, x_prev, r, k, v; state, parameters and outputs stay fp32) it is
// 50 and 38.  Four consecutive channels per thread: 16-byte accesses of the
// fp32 arrays and 8-byte accesses of the bf16 ones, when C % 4 == 0 and
// every pointer is aligned to that access.
#include <cuda_bf16.h>

#include "wkv_common.cuh"
#include "wkv_internal.h"

namespace wkv {

namespace {

struct Elem {
  float y, xk, xv, xr;
};

__device__ __forceinline__ Elem decode_one(float x, float xp, float mk, float mv, float mr, float r, float k, float v,
                                           float w, float u, float& num, float& den, float& pp) {
  Elem o;
  // mu x + (1 - mu) x_prev as written: one rounding per product (forming
  // x - x_prev first would add its rounding, large where the terms cancel)
  o.xk = fmaf(mk, x, (1.f - mk) * xp);
  o.xv = fmaf(mv, x, (1.f - mv) * xp);
  o.xr = fmaf(mr, x, (1.f - mr) * xp);
  State s{num, den, pp};
  const float wkv_t = output(s, k, v, u);
  const float gate = rcp(1.f + exp_nat(-r));  // sigmoid(r)
  o.y = wkv_t * gate;
  step(s, k, v, w);
  num = s.num;
  den = s.den;
  pp = s.pp;
  return o;
}

// Four consecutive token inputs as fp32: one 16-byte load of fp32, or one
// 8-byte load of bf16 widened exactly (a bf16 is the top half of an fp32).
__device__ __forceinline__ float4 load4(const float* p, int64_t i) {
  return __ldcs(reinterpret_cast<const float4*>(p) + i);
}
__device__ __forceinline__ float4 load4(const __nv_bfloat16* p, int64_t i) {
  const uint2 raw = __ldcs(reinterpret_cast<const uint2*>(p) + i);
  return make_float4(__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xffff0000u),
                     __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xffff0000u));
}

// E: the type of the token inputs x, x_prev, r, k, v (float or bf16).
template <typename E>
__global__ void __launch_bounds__(256) decode_kernel_vec4(const DecodeArgs a) {
  const int64_t n4 = (int64_t)a.L * a.B * a.C / 4;
  const int C4 = a.C / 4;
  const int64_t BC4 = (int64_t)a.B * C4;
  const E* ax = static_cast<const E*>(a.x);
  const E* axp = static_cast<const E*>(a.x_prev);
  const E* ar = static_cast<const E*>(a.r);
  const E* ak = static_cast<const E*>(a.k);
  const E* av = static_cast<const E*>(a.v);
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n4; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t l = i / BC4;
    const int64_t pc = l * C4 + (i % C4);  // index of the (l, c) parameters
    const float4 x = load4(ax, i);
    const float4 xp = load4(axp, i);
    const float4 r = load4(ar, i);
    const float4 k = load4(ak, i);
    const float4 v = load4(av, i);
    float4 num = __ldcs(reinterpret_cast<const float4*>(a.num) + i);
    float4 den = __ldcs(reinterpret_cast<const float4*>(a.den) + i);
    float4 pp = __ldcs(reinterpret_cast<const float4*>(a.pp) + i);
    const float4 mk = __ldg(reinterpret_cast<const float4*>(a.mu_k) + pc);
    const float4 mv = __ldg(reinterpret_cast<const float4*>(a.mu_v) + pc);
    const float4 mr = __ldg(reinterpret_cast<const float4*>(a.mu_r) + pc);
    const float4 w = __ldg(reinterpret_cast<const float4*>(a.w) + pc);
    const float4 u = __ldg(reinterpret_cast<const float4*>(a.u) + pc);
    const Elem e0 = decode_one(x.x, xp.x, mk.x, mv.x, mr.x, r.x, k.x, v.x, w.x, u.x, num.x, den.x, pp.x);
    const Elem e1 = decode_one(x.y, xp.y, mk.y, mv.y, mr.y, r.y, k.y, v.y, w.y, u.y, num.y, den.y, pp.y);
    const Elem e2 = decode_one(x.z, xp.z, mk.z, mv.z, mr.z, r.z, k.z, v.z, w.z, u.z, num.z, den.z, pp.z);
    const Elem e3 = decode_one(x.w, xp.w, mk.w, mv.w, mr.w, r.w, k.w, v.w, w.w, u.w, num.w, den.w, pp.w);
    __stcs(reinterpret_cast<float4*>(a.y) + i, make_float4(e0.y, e1.y, e2.y, e3.y));
    __stcs(reinterpret_cast<float4*>(a.num) + i, num);
    __stcs(reinterpret_cast<float4*>(a.den) + i, den);
    __stcs(reinterpret_cast<float4*>(a.pp) + i, pp);
    if (a.xk) __stcs(reinterpret_cast<float4*>(a.xk) + i, make_float4(e0.xk, e1.xk, e2.xk, e3.xk));
    if (a.xv) __stcs(reinterpret_cast<float4*>(a.xv) + i, make_float4(e0.xv, e1.xv, e2.xv, e3.xv));
    if (a.xr) __stcs(reinterpret_cast<float4*>(a.xr) + i, make_float4(e0.xr, e1.xr, e2.xr, e3.xr));
  }
}

template <typename E>
__global__ void __launch_bounds__(256) decode_kernel_scalar(const DecodeArgs a) {
  const int64_t n = (int64_t)a.L * a.B * a.C;
  const int64_t BC = (int64_t)a.B * a.C;
  const E* ax = static_cast<const E*>(a.x);
  const E* axp = static_cast<const E*>(a.x_prev);
  const E* ar = static_cast<const E*>(a.r);
  const E* ak = static_cast<const E*>(a.k);
  const E* av = static_cast<const E*>(a.v);
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t l = i / BC;
    const int64_t pc = l * a.C + (i % a.C);
    float num = a.num[i], den = a.den[i], pp = a.pp[i];
    const Elem e = decode_one(to_f32<E>(ax[i]), to_f32<E>(axp[i]), a.mu_k[pc], a.mu_v[pc], a.mu_r[pc],
                              to_f32<E>(ar[i]), to_f32<E>(ak[i]), to_f32<E>(av[i]), a.w[pc], a.u[pc], num, den, pp);
    a.y[i] = e.y;
    a.num[i] = num;
    a.den[i] = den;
    a.pp[i] = pp;
    if (a.xk) a.xk[i] = e.xk;
    if (a.xv) a.xv[i] = e.xv;
    if (a.xr) a.xr[i] = e.xr;
  }
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, bool vec4, int token_dtype, cudaStream_t s) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t n = (int64_t)a.L * a.B * a.C;
  const int64_t work = vec4 ? n / 4 : n;
  const int threads = 256;
  int64_t blocks = (work + threads - 1) / threads;
  const int64_t cap = (int64_t)sms * 8;  // 8 resident CTAs of 256 threads per SM, grid-stride beyond
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  const dim3 grid((unsigned)blocks), block(threads);
  if (token_dtype == 0) {
    if (vec4)
      decode_kernel_vec4<float><<<grid, block, 0, s>>>(a);
    else
      decode_kernel_scalar<float><<<grid, block, 0, s>>>(a);
  } else {
    if (vec4)
      decode_kernel_vec4<__nv_bfloat16><<<grid, block, 0, s>>>(a);
    else
      decode_kernel_scalar<__nv_bfloat16><<<grid, block, 0, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace wkv
