// wkv_bwd.cu -- WKV backward pass: reverse-time chunked scan.
//
// Gradients of every parameter are needed for training (qiita "RWKV について
// の調査記録", section "Trainingについて"); the pages give no formulas, so
// they are derived by reverse-mode differentiation of the recurrence.  With
// the state before token t written a_t = num e^{pp}, b_t = den e^{pp}, the
// denominator D_t = b_t + e^{u+k_t}, gN_t = gy_t / D_t, gD_t = -gy_t wkv_t /
// D_t, and the adjoints la_t = dL/da_t, lb_t = dL/db_t (zero after the last
// token):
//
//   la_t = gN_t + e^{-w} la_{t+1},         lb_t = gD_t + e^{-w} lb_{t+1}
//   gk_t = (gN_t v_t + gD_t) e^{u+k_t} + (la_{t+1} v_t + lb_{t+1}) e^{k_t}
//   gv_t = gN_t e^{u+k_t} + la_{t+1} e^{k_t}
//   gu  += (gN_t v_t + gD_t) e^{u+k_t}
//   gw  += -e^{-w} (la_{t+1} a_t + lb_{t+1} b_t)
//
// The adjoints are carried scaled by the forward maximum, La_t = la_t e^{pp_t},
// so every factor below is an exponential of a non-positive number.
//
// The adjoint recurrence is linear with a data-independent decay, so it is
// scanned in chunks like the forward pass, but from the last chunk backwards.
// One tile is (chunk, batch row, 128 channels), one lane one channel:
//
//   1. load k, v, gy of the tile and the forward state at the chunk start
//      (the forward pass's checkpoint);
//   2. re-run the forward recurrence over the chunk, keeping each step's
//      state in shared memory;
//   3. reverse pass with a zero carry -> the chunk's adjoint summary; publish
//      it as a leaf of the binary-indexed tree over chunks counted from the
//      end (wkv_common.cuh), wait for the tree nodes that make up the
//      following chunks, combine them in a fixed order into the carry at the
//      chunk end, and publish the tree nodes this chunk completes (tiles are
//      handed out last chunk first);
//   4. reverse pass with the carry, writing gk, gv and this tile's partial
//      sums of gw, gu; a separate kernel adds the partials in a fixed order,
//      so the result is deterministic.
#include "wkv_common.cuh"
#include "wkv_internal.h"

namespace wkv {

namespace {

// Everything the reverse pass needs at one token, from the state before it.
struct Local {
  float gb;  // gy e^{pp-q} / Dhat : scaled gN
  float gc;  // gy e^{u+k-q} / Dhat : gN e^{u+k}
  float y;   // wkv_t
  float vmy; // v_t - wkv_t, formed without subtracting the two
  Decay t;   // carry factors of the forward step (same as the forward pass)
};

__device__ __forceinline__ Local local_terms(const State& s, float k, float v, float g, float w, float u) {
  Local o;
  const float d1 = s.pp - (u + k);
  const float e1 = exp_neg_abs(d1);
  const bool past = d1 >= 0.f;
  const float cp = past ? 1.f : e1;
  const float cc = past ? e1 : 1.f;
  const float inv = rcp(fmaf(cp, s.den, cc));
  o.y = fmaf(cp, s.num, cc * v) * inv;
  // v - wkv = cp (den v - num) / Dhat: exact cancellation of the current
  // token's own share, so no rounding noise when the bonus dominates
  o.vmy = cp * fmaf(s.den, v, -s.num) * inv;
  const float gi = g * inv;
  o.gb = gi * cp;
  o.gc = gi * cc;
  o.t = decay_terms(s.pp, k, w);
  return o;
}

}  // namespace

template <int L>
__global__ void __launch_bounds__(kCtaChannels, 3) bwd_scan_kernel(const BwdArgs a) {
  extern __shared__ float sm[];  // [3][L][kCtaChannels]: num, den, pp before each token
  const ScanGeometry& g = a.g;
  const unsigned int ticket = take_ticket(a.ticket, g.ntiles);
  if (ticket >= g.ntiles) return;  // only if the counter was not zeroed: never touch memory then
  const int per_j = g.B * g.ncb;
  const int jr = ticket / per_j;
  const int j = g.nchunks - 1 - jr;  // last chunk first
  const int rem = ticket - jr * per_j;
  const int b = rem / g.ncb;
  const int cb = rem - b * g.ncb;
  const int tid = threadIdx.x;
  const int c = cb * kCtaChannels + tid;
  const bool valid = c < g.C;
  const int cc = valid ? c : g.C - 1;
  const int t0 = j * L;
  const int len = min(L, g.T - t0);
  const int64_t base = ((int64_t)b * g.T + t0) * g.C + cc;
  const size_t P = g.plane;
  auto slot = [&](int jj) -> size_t { return ((size_t)jj * g.B + b) * g.C + cc; };

  float kr[L], vr[L], gr[L];
#pragma unroll
  for (int i = 0; i < L; ++i) {
    if (i < len) {
      const int64_t o = base + (int64_t)i * g.C;
      kr[i] = __ldg(a.k + o);
      vr[i] = __ldg(a.v + o);
      gr[i] = __ldg(a.gy + o);
    } else {
      kr[i] = vr[i] = gr[i] = 0.f;
    }
  }
  const float w = __ldg(a.w + cc);
  const float u = __ldg(a.u + cc);

  State s0 = empty_state();
  if (j > 0) {
    const size_t o = slot(j - 1);
    s0 = State{a.ckpt[o], a.ckpt[o + P], a.ckpt[o + 2 * P]};
  }

  // 2. forward re-run, states kept per token
  float* sm_num = sm;
  float* sm_den = sm + L * kCtaChannels;
  float* sm_pp = sm + 2 * L * kCtaChannels;
  State s = s0;
#pragma unroll
  for (int i = 0; i < L; ++i) {
    if (i < len) {
      sm_num[i * kCtaChannels + tid] = s.num;
      sm_den[i * kCtaChannels + tid] = s.den;
      sm_pp[i * kCtaChannels + tid] = s.pp;
      step(s, kr[i], vr[i], w);
    }
  }
  const float pp_end = s.pp;

  // 3. adjoint summary of the chunk with nothing after it, scaled by
  // e^{pp at the chunk start}
  float la = 0.f, lb = 0.f;
#pragma unroll
  for (int i = L - 1; i >= 0; --i) {
    if (i < len) {
      const State si{sm_num[i * kCtaChannels + tid], sm_den[i * kCtaChannels + tid], sm_pp[i * kCtaChannels + tid]};
      const Local o = local_terms(si, kr[i], vr[i], gr[i], w, u);
      // the adjoint is carried back by the transpose of the forward step
      la = carry(o.t, la, o.gb);
      lb = carry(o.t, lb, -o.gb * o.y);
    }
  }

  if (j == a.debug_skip_chunk) return;  // fault injection: this tile never publishes

  // Tree over the reverse chunk index rj: a node value (la, lb, ex) is the
  // adjoint at the start of its span, from the span alone, scaled by e^{ex}
  // with ex the forward pp there.
  const int wg = cb * 4 + (tid >> 5);
  uint64_t* flags = a.flags + ((int64_t)b * g.nwg + wg) * g.nnodes;
  const size_t NP = g.nplane;
  const float* rn = a.rnodes;
  auto nslot = [&](int nd) -> size_t { return ((size_t)nd * g.B + b) * g.C + cc; };
  const bool has_pred = j > 0;  // earlier chunks will read this chunk's nodes
  auto put_node = [&](int level, float na, float nb, float ne, uint64_t status) {
    const int nd = node_index(g.level_off, jr, level);
    if (valid && status == kNodeReady) {
      const size_t o = nslot(nd);
      a.rnodes[o] = na;
      a.rnodes[o + NP] = nb;
      a.rnodes[o + 2 * NP] = ne;
    }
    publish(flags + nd, a.epoch, status);
  };

  if (has_pred) put_node(0, la, lb, s0.pp, kNodeReady);
  const int nf = __popc(jr);
  const int nup = __ffs(~jr) - 1;
  const int rc = wait_flags(
      [&](int i) {
        int e, l;
        fenwick_node(jr, i, e, l);
        return flags + node_index(g.level_off, e, l);
      },
      nf, a.epoch, a.budget_ns, a.eh);
  if (rc != kWaitOk) {
    if (rc == kWaitTimeout && (tid & 31) == 0) record_error(a.eh, kDevErrTimeout, a.epoch);
    if (has_pred)
      for (int s = 1; s <= nup; ++s) put_node(s, 0.f, 0.f, 0.f, kNodeErr);
    return;
  }

  // carry at the start of chunk j+1: (xa, xb) e^{-ex}; nodes nearest first
  float xa = 0.f, xb = 0.f, ex = 0.f;
  float na = la, nb = lb;  // node (jr, i) of this chunk, exponent s0.pp
  int x = jr, i = 0;
  while (x) {
    float va[4], vb[4], ve[4];
    int ne[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      ne[q] = -1;
      if (x) {
        const int lvl = __ffs(x) - 1;
        ne[q] = x - 1;
        const size_t o = nslot(node_index(g.level_off, x - 1, lvl));
        va[q] = ld_cg(rn + o);
        vb[q] = ld_cg(rn + o + NP);
        ve[q] = ld_cg(rn + o + 2 * NP);
        x &= x - 1;
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (ne[q] >= 0) {
        if (i == 0) {
          xa = va[q];
          xb = vb[q];
          ex = ve[q];
        } else {
          // the node starts (jr - 1 - end) whole chunks after chunk j+1 starts
          const float f = exp_nat(ex - ve[q] - (float)((jr - 1 - ne[q]) * L) * w);
          xa = fmaf(va[q], f, xa);
          xb = fmaf(vb[q], f, xb);
        }
        if (i < nup && has_pred) {
          // node (jr, i+1) = node (jr, i) then, later in time, node (jr - 2^i, i)
          const float f = exp_nat(s0.pp - ve[q] - (float)((1 << i) * L) * w);
          na = fmaf(va[q], f, na);
          nb = fmaf(vb[q], f, nb);
          put_node(i + 1, na, nb, s0.pp, kNodeReady);
        }
        ++i;
      }
    }
  }
  float ca = 0.f, cbv = 0.f;  // carry at this chunk's end, scaled by e^{pp_end}
  if (nf > 0) {
    const float f = exp_nat(pp_end - ex);
    ca = xa * f;
    cbv = xb * f;
  }

  // 4. reverse pass with the carry
  la = ca;
  lb = cbv;
  float gw_acc = 0.f, gu_acc = 0.f;
#pragma unroll
  for (int i = L - 1; i >= 0; --i) {
    if (i < len) {
      const State si{sm_num[i * kCtaChannels + tid], sm_den[i * kCtaChannels + tid], sm_pp[i * kCtaChannels + tid]};
      const float k = kr[i], v = vr[i];
      const Local o = local_terms(si, k, v, gr[i], w, u);
      const float cur = o.gc * o.vmy;
      const float gk = fmaf(o.t.kap, fmaf(la, v, lb), cur);
      const float gv = fmaf(o.t.kap, la, o.gc);
      gu_acc += cur;
      gw_acc = fmaf(-(o.t.dec + o.t.cor), fmaf(la, si.num, lb * si.den), gw_acc);
      // the adjoint is carried back by the transpose of the forward step
      la = carry(o.t, la, o.gb);
      lb = carry(o.t, lb, -o.gb * o.y);
      if (valid) {
        const int64_t off = base + (int64_t)i * g.C;
        __stcs(a.gk + off, gk);
        __stcs(a.gv + off, gv);
      }
    }
  }
  if (valid) {
    const size_t o = slot(j);
    a.part[o] = gw_acc;
    a.part[o + P] = gu_acc;
  }
}

// gw[c] = sum over (chunk, row) of the partials, gu likewise.  Block of 256
// threads = 8 warps for 32 channels; warp q sums rows q, q+8, ... with
// compensated (Kahan) summation, then the 8 results are added in order.
__global__ void __launch_bounds__(256) reduce_kernel(const ReduceArgs a) {
  __shared__ float sw[8][32], su[8][32];
  const int lane = threadIdx.x & 31, q = threadIdx.x >> 5;
  const int c = blockIdx.x * 32 + lane;
  float s1 = 0.f, k1 = 0.f, s2 = 0.f, k2 = 0.f;
  if (c < a.C) {
    const size_t P = (size_t)a.rows * a.C;
    for (int r = q; r < a.rows; r += 8) {
      const size_t o = (size_t)r * a.C + c;
      float y1 = a.part[o] - k1;
      float t1 = s1 + y1;
      k1 = (t1 - s1) - y1;
      s1 = t1;
      float y2 = a.part[o + P] - k2;
      float t2 = s2 + y2;
      k2 = (t2 - s2) - y2;
      s2 = t2;
    }
  }
  sw[q][lane] = s1;
  su[q][lane] = s2;
  __syncthreads();
  if (q == 0 && c < a.C) {
    float t1 = 0.f, t2 = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      t1 += sw[i][lane];
      t2 += su[i][lane];
    }
    a.gw[c] = t1;
    a.gu[c] = t2;
  }
}

cudaError_t launch_backward(const BwdArgs& a, cudaStream_t s) {
  const size_t smem = 3 * kChunk * kCtaChannels * sizeof(float);
  // The opt-in for more than 48 KB of dynamic shared memory is per device.
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(bwd_scan_kernel<kChunk>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  bwd_scan_kernel<kChunk><<<dim3(a.g.ntiles), dim3(kCtaChannels), smem, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_reduce(const ReduceArgs& a, cudaStream_t s) {
  reduce_kernel<<<dim3((a.C + 31) / 32), dim3(256), 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace wkv
