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
// with the mix outputs, 48 without.  Four consecutive channels per thread
// with 16-byte accesses when C % 4 == 0 and every pointer is 16-byte aligned.
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
  const float dx = x - xp;
  o.xk = fmaf(mk, dx, xp);
  o.xv = fmaf(mv, dx, xp);
  o.xr = fmaf(mr, dx, xp);
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

__global__ void __launch_bounds__(256) decode_kernel_vec4(const DecodeArgs a) {
  const int64_t n4 = (int64_t)a.L * a.B * a.C / 4;
  const int C4 = a.C / 4;
  const int64_t BC4 = (int64_t)a.B * C4;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n4; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t l = i / BC4;
    const int64_t pc = l * C4 + (i % C4);  // index of the (l, c) parameters
    const float4 x = __ldcs(reinterpret_cast<const float4*>(a.x) + i);
    const float4 xp = __ldcs(reinterpret_cast<const float4*>(a.x_prev) + i);
    const float4 r = __ldcs(reinterpret_cast<const float4*>(a.r) + i);
    const float4 k = __ldcs(reinterpret_cast<const float4*>(a.k) + i);
    const float4 v = __ldcs(reinterpret_cast<const float4*>(a.v) + i);
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

__global__ void __launch_bounds__(256) decode_kernel_scalar(const DecodeArgs a) {
  const int64_t n = (int64_t)a.L * a.B * a.C;
  const int64_t BC = (int64_t)a.B * a.C;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t l = i / BC;
    const int64_t pc = l * a.C + (i % a.C);
    float num = a.num[i], den = a.den[i], pp = a.pp[i];
    const Elem e = decode_one(a.x[i], a.x_prev[i], a.mu_k[pc], a.mu_v[pc], a.mu_r[pc], a.r[i], a.k[i], a.v[i],
                              a.w[pc], a.u[pc], num, den, pp);
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

cudaError_t launch_decode(const DecodeArgs& a, bool vec4, cudaStream_t s) {
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
  if (vec4)
    decode_kernel_vec4<<<dim3((unsigned)blocks), dim3(threads), 0, s>>>(a);
  else
    decode_kernel_scalar<<<dim3((unsigned)blocks), dim3(threads), 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace wkv
