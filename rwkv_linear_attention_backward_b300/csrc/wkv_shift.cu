// wkv_shift.cu -- the token shift of the training path, forward and backward.
//
// Each projection of a time-mixing block takes a weighted sum of the current
// and the previous token ("RWKV解读：在Transformer的时代的新RNN", section
// "3、RWKV的网络架构", eq. (7); "Инновационная архитектура RWKV", section
// "Механизмы взаимодействия"): per (b, t, c), with x_{-1} = x0 (the token
// before the sequence; zeros when none is given),
//
//   xk_t = mu_k x_t + (1 - mu_k) x_{t-1},   xv_t, xr_t alike with mu_v, mu_r.
//
// The three mixes are written in one pass over x (one read of x and of the
// previous row, which the neighbouring CTAs have just brought into L2).  The
// backward pass gives
//
//   gx_t  = sum_m mu_m gxm_t + (1 - mu_m) gxm_{t+1}   (no t+1 term at T-1)
//   gx0   = sum_m (1 - mu_m) gxm_0
//   gmu_m = sum_{b,t} gxm_t (x_t - x_{t-1}),
//
// gmu summed per CTA slice of rows (compensated, in row order) and then over
// the slices in slice order by a second kernel: deterministic.  Both passes
// are bound by HBM bandwidth (16 and 20 bytes per element); channels go
// four to a thread with 16-byte accesses when C % 4 == 0 and every pointer is
// 16-byte aligned, one to a thread otherwise.
#include <cstdint>
#include <cuda_runtime.h>

#include "wkv_common.cuh"
#include "wkv_internal.h"

namespace wkv {

namespace {

template <int V>
struct Vec;
template <>
struct Vec<4> {
  using T = float4;
  __device__ static float4 load(const float* p) { return __ldg(reinterpret_cast<const float4*>(p)); }
  __device__ static void store(float* p, const float4& v) { __stcs(reinterpret_cast<float4*>(p), v); }
  __device__ static float get(const float4& v, int i) { return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w; }
  __device__ static void set(float4& v, int i, float x) {
    if (i == 0) v.x = x;
    else if (i == 1) v.y = x;
    else if (i == 2) v.z = x;
    else v.w = x;
  }
  __device__ static float4 zero() { return make_float4(0.f, 0.f, 0.f, 0.f); }
};
template <>
struct Vec<1> {
  using T = float;
  __device__ static float load(const float* p) { return __ldg(p); }
  __device__ static void store(float* p, const float& v) { __stcs(p, v); }
  __device__ static float get(const float& v, int) { return v; }
  __device__ static void set(float& v, int, float x) { v = x; }
  __device__ static float zero() { return 0.f; }
};

// Forward: item = (row b*T + t, V consecutive channels); grid-stride.
template <int V>
__global__ void __launch_bounds__(256) shift_fwd_kernel(const ShiftArgs a) {
  using W = Vec<V>;
  using VT = typename W::T;
  const int64_t per_row = a.C / V;
  const int64_t n = (int64_t)a.B * a.T * per_row;
  for (int64_t it = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; it < n; it += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = it / per_row;
    const int c = (int)(it - row * per_row) * V;
    const int b = (int)(row / a.T);
    const int t = (int)(row - (int64_t)b * a.T);
    const int64_t o = row * a.C + c;
    const VT cur = W::load(a.x + o);  // kept in L2: the next row reads it as its previous token
    VT prev;
    if (t > 0) prev = W::load(a.x + o - a.C);
    else prev = a.x0 ? W::load(a.x0 + (int64_t)b * a.C + c) : W::zero();
    const VT mk = W::load(a.mu_k + c), mv = W::load(a.mu_v + c), mr = W::load(a.mu_r + c);
    VT ok, ov, orr;
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const float x = W::get(cur, i), p = W::get(prev, i);
      // mu x + (1 - mu) x_prev as written in eq. (7): one rounding per
      // product, where mu (x - x_prev) + x_prev would first round
      // x - x_prev, a larger error wherever the two terms nearly cancel
      W::set(ok, i, fmaf(W::get(mk, i), x, (1.f - W::get(mk, i)) * p));
      W::set(ov, i, fmaf(W::get(mv, i), x, (1.f - W::get(mv, i)) * p));
      W::set(orr, i, fmaf(W::get(mr, i), x, (1.f - W::get(mr, i)) * p));
    }
    W::store(a.xk + o, ok);
    W::store(a.xv + o, ov);
    W::store(a.xr + o, orr);
  }
}

__device__ __forceinline__ void kahan(float& s, float& k, float x) {
  const float y = x - k;
  const float t = s + y;
  k = (t - s) - y;
  s = t;
}

// Backward: block (channel group of 32 V channels, row slice); the slice's
// rows are cut into 8 contiguous ranges, one per warp, and a warp walks its
// range from the last row to the first.  Walking down, the mix gradients of
// row t+1 (the "next" terms of row t) are the ones loaded one step before,
// and the x_{t-1} loaded for row t is the x_t of the next step, so a row
// costs four loads (gxk, gxv, gxr and x_{t-1}) instead of eight.  gmu
// partials of the slice go to part[slice][3][C], the 8 warps' sums added in
// warp order.
template <int V>
__global__ void __launch_bounds__(256, 2) shift_bwd_kernel(const ShiftArgs a) {
  using W = Vec<V>;
  using VT = typename W::T;
  __shared__ float red[8][3][32 * V];
  const int lane = threadIdx.x & 31, wy = threadIdx.x >> 5;
  const int c = (blockIdx.x * 32 + lane) * V;
  const bool valid = c < a.C;
  const int64_t rows = (int64_t)a.B * a.T;
  const int64_t per = (rows + a.nslice - 1) / a.nslice;
  const int64_t r0 = (int64_t)blockIdx.y * per, r1 = r0 + per < rows ? r0 + per : rows;
  const int64_t pw = r1 > r0 ? (r1 - r0 + 7) / 8 : 0;  // rows per warp
  const int64_t w0 = r0 + wy * pw, w1 = w0 + pw < r1 ? w0 + pw : r1;
  float sk[V], kk[V], sv[V], kv[V], sr[V], kr[V];
#pragma unroll
  for (int i = 0; i < V; ++i) sk[i] = kk[i] = sv[i] = kv[i] = sr[i] = kr[i] = 0.f;
  if (valid && w0 < w1) {
    const VT mk = W::load(a.mu_k + c), mv = W::load(a.mu_v + c), mr = W::load(a.mu_r + c);
    int64_t row = w1 - 1;
    int b = (int)(row / a.T);
    int t = (int)(row - (int64_t)b * a.T);
    // the row after the range (none past the end of a sequence)
    VT nk = W::zero(), nv = W::zero(), nr = W::zero();
    if (t + 1 < a.T) {
      const int64_t o = (row + 1) * a.C + c;
      nk = W::load(a.gxk + o);
      nv = W::load(a.gxv + o);
      nr = W::load(a.gxr + o);
    }
    VT cur = W::load(a.x + row * a.C + c);
    for (; row >= w0; --row) {
      const int64_t o = row * a.C + c;
      const VT gk = W::load(a.gxk + o), gv = W::load(a.gxv + o), gr = W::load(a.gxr + o);
      VT prev;
      if (t > 0) prev = W::load(a.x + o - a.C);
      else prev = a.x0 ? W::load(a.x0 + (int64_t)b * a.C + c) : W::zero();
      VT g;
      VT g0 = W::zero();
#pragma unroll
      for (int i = 0; i < V; ++i) {
        const float mki = W::get(mk, i), mvi = W::get(mv, i), mri = W::get(mr, i);
        const float gki = W::get(gk, i), gvi = W::get(gv, i), gri = W::get(gr, i);
        // explicit fused multiply-adds: every instantiation rounds alike
        const float own = fmaf(mki, gki, fmaf(mvi, gvi, mri * gri));
        const float nxt = fmaf(1.f - mki, W::get(nk, i), fmaf(1.f - mvi, W::get(nv, i), (1.f - mri) * W::get(nr, i)));
        W::set(g, i, own + nxt);
        if (t == 0) W::set(g0, i, fmaf(1.f - mki, gki, fmaf(1.f - mvi, gvi, (1.f - mri) * gri)));
        const float d = W::get(cur, i) - W::get(prev, i);
        kahan(sk[i], kk[i], gki * d);
        kahan(sv[i], kv[i], gvi * d);
        kahan(sr[i], kr[i], gri * d);
      }
      W::store(a.gx + o, g);
      if (t == 0 && a.gx0) W::store(a.gx0 + (int64_t)b * a.C + c, g0);
      // one row down: this row's mix gradients are the next terms of the
      // row below, and its x_{t-1} is that row's x_t; below a sequence's
      // first row lies the previous sequence's last row (no next terms)
      if (t > 0) {
        nk = gk;
        nv = gv;
        nr = gr;
        cur = prev;
        --t;
      } else {
        nk = nv = nr = W::zero();
        t = a.T - 1;
        --b;
        if (row > w0) cur = W::load(a.x + (row - 1) * a.C + c);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < V; ++i) {
    red[wy][0][lane * V + i] = sk[i];
    red[wy][1][lane * V + i] = sv[i];
    red[wy][2][lane * V + i] = sr[i];
  }
  __syncthreads();
  // warp m (< 3) adds the 8 warps' sums of mix m in warp order
  if (wy < 3) {
#pragma unroll
    for (int i = 0; i < V; ++i) {
      float s = 0.f;
#pragma unroll
      for (int q = 0; q < 8; ++q) s += red[q][wy][lane * V + i];
      const int ci = c + i;
      if (ci < a.C) a.part[((int64_t)blockIdx.y * 3 + wy) * a.C + ci] = s;
    }
  }
}

// gmu_m[c] = the slice sums part[s][m][c], added in slice order.
__global__ void __launch_bounds__(256) shift_reduce_kernel(const ShiftArgs a) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= 3 * (int64_t)a.C) return;
  const int m = (int)(i / a.C);
  const int c = (int)(i - (int64_t)m * a.C);
  float s = 0.f, k = 0.f;
  for (int sl = 0; sl < a.nslice; ++sl) kahan(s, k, a.part[((int64_t)sl * 3 + m) * a.C + c]);
  float* out = m == 0 ? a.gmu_k : (m == 1 ? a.gmu_v : a.gmu_r);
  out[c] = s;
}

}  // namespace

// CTAs for `items` work items of a grid-stride kernel: enough for the items,
// at most 8 CTAs of `threads` threads per SM of the current device.
int elementwise_grid(int64_t items, int threads) {
  static int sms_per_dev[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  int sms = (dev >= 0 && dev < 64) ? sms_per_dev[dev] : 0;
  if (sms == 0) {
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 148;
    if (dev >= 0 && dev < 64) sms_per_dev[dev] = sms;
  }
  const int64_t want = (items + threads - 1) / threads;
  const int64_t cap = (int64_t)sms * 8;
  return (int)(want < cap ? (want > 0 ? want : 1) : cap);
}

int shift_slices(int B, int T, int C, bool vec4) {
  const int per_group = vec4 ? 128 : 32;
  const int groups = (C + per_group - 1) / per_group;
  const int64_t rows = (int64_t)B * T;
  int64_t ns = (2 * 148) / groups;  // two CTAs per SM at most: one wave
  if (ns > (rows + 7) / 8) ns = (rows + 7) / 8;
  if (ns < 1) ns = 1;
  return (int)ns;
}

cudaError_t launch_shift_forward(const ShiftArgs& a, bool vec4, cudaStream_t s) {
  if (vec4) {
    shift_fwd_kernel<4><<<elementwise_grid((int64_t)a.B * a.T * (a.C / 4), 256), 256, 0, s>>>(a);
  } else {
    shift_fwd_kernel<1><<<elementwise_grid((int64_t)a.B * a.T * a.C, 256), 256, 0, s>>>(a);
  }
  return cudaGetLastError();
}

cudaError_t launch_shift_backward(const ShiftArgs& a, bool vec4, cudaStream_t s) {
  const int per_group = vec4 ? 128 : 32;
  const dim3 grid((a.C + per_group - 1) / per_group, a.nslice);
  if (vec4) {
    shift_bwd_kernel<4><<<grid, 256, 0, s>>>(a);
  } else {
    shift_bwd_kernel<1><<<grid, 256, 0, s>>>(a);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  shift_reduce_kernel<<<(unsigned)((3 * (int64_t)a.C + 255) / 256), 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace wkv
