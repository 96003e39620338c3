// wkv_common.cuh -- device helpers shared by the WKV kernels (sm_103a).
//
// The operator (RWKV time mixing, "RWKV解读：在Transformer的时代的新RNN",
// section "3、RWKV的网络架构", eq. (8); qiita "RWKV についての調査記録",
// section "wkvとは"): per batch row and channel, with decay w > 0 and bonus u,
//
//   wkv_t = (sum_{i<t} e^{-(t-1-i)w + k_i} v_i + e^{u+k_t} v_t)
//         / (sum_{i<t} e^{-(t-1-i)w + k_i}     + e^{u+k_t}),
//
// computed through a carried state.  The state after t tokens is the triple
// (num, den, pp) with a_t = num e^{pp}, b_t = den e^{pp}, where
// a_t = sum_{i<t} e^{-(t-1-i)w+k_i} v_i, b_t likewise without v, and pp is
// the running maximum of the exponents, so den >= 1 once a token is seen and
// no exponential overflows.  The empty state is (0, 0, -1e38).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace wkv {

// Element of an input array (k, v, gy) as fp32: inputs may be fp32 or bf16,
// the arithmetic is fp32.
template <typename E>
__device__ __forceinline__ float to_f32(E x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) {
  return x;
}
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}

constexpr float kLog2e = 1.4426950408889634f;  // log2(e)
constexpr float kEmptyPP = -1e38f;             // pp of the empty state

// Error codes written to the workspace header by a kernel.
constexpr unsigned int kDevErrTimeout = 6;

// ---------------------------------------------------------------- math
// 2^x with the MUFU unit.  Flushes subnormal results to zero, which only
// ever drops weights below 2^-126 relative to the running maximum.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float rcp(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// e^{-|d|}: the one exponential needed for a pair e^{x-q}, e^{y-q} with
// q = max(x, y) and d = x - y (the larger one gets exactly 1).
__device__ __forceinline__ float exp_neg_abs(float d) { return ex2(-fabsf(d) * kLog2e); }

__device__ __forceinline__ float exp_nat(float x) { return ex2(x * kLog2e); }

// Two fp32 values in one 64-bit register pair, for the packed fp32
// instructions of sm_100 and later: one fma.rn.f32x2 is two IEEE fmas, lane
// by lane, so a packed chain gives the scalar chain's values bit for bit.
struct Pk2 {
  unsigned long long v;
};
__device__ __forceinline__ Pk2 f2(float lo, float hi) {
  Pk2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r.v) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float f2_lo(Pk2 a) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(a.v));
  return lo;
}
__device__ __forceinline__ float f2_hi(Pk2 a) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(a.v));
  return hi;
}
__device__ __forceinline__ Pk2 fma2(Pk2 a, Pk2 b, Pk2 c) {  // a * b + c, per lane
  Pk2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d.v) : "l"(a.v), "l"(b.v), "l"(c.v));
  return d;
}

// sigmoid(r) = 1 / (1 + e^{-r}), the receptance gate on the time-mixing
// output: 0 once e^{-r} overflows (r below about -88), 1 once e^{-r} is
// below half an ulp of 1.
__device__ __forceinline__ float sigmoid(float r) { return rcp(1.f + exp_nat(-r)); }

struct State {
  float num, den, pp;
};

__device__ __forceinline__ State empty_state() { return State{0.f, 0.f, kEmptyPP}; }

// A state given per (batch row, channel) as planes [3][B][C] (num, den, pp;
// bc = B * C, o = b * C + c); NULL is the empty state.
__device__ __forceinline__ State load_state_planes(const float* s, size_t bc, size_t o) {
  if (s == nullptr) return empty_state();
  return State{__ldg(s + o), __ldg(s + o + bc), __ldg(s + o + 2 * bc)};
}

__device__ __forceinline__ void store_state_planes(float* s, size_t bc, size_t o, const State& P) {
  s[o] = P.num;
  s[o + bc] = P.den;
  s[o + 2 * bc] = P.pp;
}

// Consume one token (k, v): a' = e^{-w} a + e^{k} v, b' = e^{-w} b + e^{k},
// pp' = max(pp - w, k).  The old state is carried over by the factor
// e^{(pp - w) - pp'} = dec * (1 + res), where res = (pp - w) - fl(pp - w) is
// the rounding residual of the new exponent (Fast2Sum).  Adding the term
// dec * res * num separately keeps that correction at full precision (1 + res
// itself would round to 1), so a long run of steps where the decayed past
// stays the maximum does not drift the carried sums.
struct Decay {
  float dec;  // e^{fl(pp - w) - pp'}
  float cor;  // dec * res
  float kap;  // e^{k - pp'}
  float pp;   // pp'
};

__device__ __forceinline__ Decay decay_terms(float pp, float k, float w) {
  Decay o;
  const float sw = pp - w;
  const float res = (pp - sw) - w;
  const float d = sw - k;
  const float e = exp_neg_abs(d);
  const bool keep = d >= 0.f;  // decayed past is still the maximum
  o.dec = keep ? 1.f : e;
  o.kap = keep ? e : 1.f;
  o.cor = o.dec * res;
  o.pp = keep ? sw : k;
  return o;
}

// x' = e^{(pp - w) - pp'} x + add, with the correction term kept separate.
__device__ __forceinline__ float carry(const Decay& t, float x, float add) {
  return fmaf(t.dec, x, fmaf(t.cor, x, add));
}

__device__ __forceinline__ void step(State& s, float k, float v, float w) {
  const Decay t = decay_terms(s.pp, k, w);
  s.num = carry(t, s.num, t.kap * v);
  s.den = carry(t, s.den, t.kap);
  s.pp = t.pp;
}

// wkv for the current token (k, v) given the state before it.
__device__ __forceinline__ float output(const State& s, float k, float v, float u) {
  const float d = s.pp - (u + k);
  const float e = exp_neg_abs(d);
  const bool past = d >= 0.f;
  const float cp = past ? 1.f : e;  // weight of the carried past
  const float cc = past ? e : 1.f;  // weight of the current token (bonus u)
  const float n = fmaf(cp, s.num, cc * v);
  const float dd = fmaf(cp, s.den, cc);
  return n * rcp(dd);
}

// x decayed over `decay` (= steps * w) followed by y: the associative combine
// of chunk results (the decay is data independent, so a chunk's effect on
// the carried state is "decay by its length, then add its own summary").
// One exponential: the larger of the two scales gets exactly 1.  Written with
// explicit roundings (fmaf, and __fsub_rn, which the compiler never fuses
// with the multiply that formed `decay` at the call site) so that every
// kernel performs the same roundings: the forward pass and the state-only
// pass must give bitwise equal states, and the look-back relies on bitwise
// equal folds.
__device__ __forceinline__ State combine(const State& x, float decay, const State& y) {
  const float px = __fsub_rn(x.pp, decay);
  const float d = px - y.pp;
  const float e = exp_neg_abs(d);
  const bool keep = d >= 0.f;
  const float ex = keep ? 1.f : e;
  const float ey = keep ? e : 1.f;
  return State{fmaf(ex, x.num, ey * y.num), fmaf(ex, x.den, ey * y.den), keep ? px : y.pp};
}

// ------------------------------------------------------------- timing
__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Workspace header: the first 256 bytes of a workspace, at the same place for
// every shape, so a workspace zero-filled once stays valid when it is reused
// for other shapes (everything after the header is either epoch-tagged or
// written before it is read within a call).
struct WsHeader {
  unsigned int ticket[4];    // dynamic tile counters, one per kind of launch
  unsigned int exited[4];    // CTAs of that launch that have finished (the last one resets both)
  unsigned int error;        // first device error code since the last check, 0 if none
  unsigned int pad0;
  unsigned long long abort;  // epoch of the last launch that gave up a wait
  unsigned long long seq;    // epoch of the last launch that used this workspace
  unsigned int pad[50];
};
static_assert(sizeof(WsHeader) == 256, "header size");

// A launch's identity: its epoch (1 + the workspace's sequence number when
// the launch starts, read on the device, so that a launch replayed from a
// CUDA graph still gets a new one) and the record tag derived from it.
struct Launch {
  unsigned long long epoch;
  uint32_t tag;
};

__host__ __device__ __forceinline__ uint32_t tag_of(unsigned long long epoch) {
  return (uint32_t)((epoch - 1) % 0xFFFFFFFFull) + 1u;  // never 0: the tag of a zero-filled workspace
}

// The first device error code of any launch of this compilation unit's
// kernels on a device since the host last took it (take_module_error):
// what wkv_sync_status reports, whatever workspace the launch used.  One
// copy per compilation unit (each .cu file is its own device module), zero
// when the library loads.
static __device__ unsigned int g_module_error;

// Records that this launch (epoch) gave up: the code for the host (in the
// workspace, and device-wide for wkv_sync_status), the epoch so the
// launch's other waits stop at once.
__device__ __forceinline__ void record_error(WsHeader* h, unsigned int code, uint64_t epoch) {
  atomicCAS(&h->error, 0u, code);
  atomicCAS(&g_module_error, 0u, code);
  atomicExch(&h->abort, (unsigned long long)epoch);
}

// Host side: reads this compilation unit's g_module_error on the current
// device into *code and clears it when set.  Synchronous.
static inline cudaError_t take_module_error(unsigned int* code) {
  unsigned int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_module_error, sizeof(v));
  if (e == cudaSuccess && v != 0) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_module_error, &zero, sizeof(zero));
  }
  *code = v;
  return e;
}

}  // namespace wkv

namespace wkv {

// ------------------------------------------------------ tagged records
// Chunk results pass between warps of different CTAs as 16-byte records, one
// per channel: three values and a check word, written and read as 128-bit
// accesses with no fence and no separate flag.  The check word is the
// launch tag mixed with the bits of the three values (rec_check), so a
// reader accepts a record only when the values it holds are the ones the
// current launch wrote with that word.  A read that saw part of a record
// from one write and part from another (an older launch's record, the
// zero-filled workspace, or a write not yet complete) fails the check and is
// read again, so correctness does not rest on 128-bit accesses being
// indivisible: should one be split, the pieces would not match (a random
// match has probability 2^-31).  Tags come from the launch epoch and are
// never 0; epochs increase from launch to launch on a workspace, so records
// left by earlier launches never pass as current.
struct Rec {
  unsigned long long lo;  // value 0 | value 1 << 32
  unsigned long long hi;  // value 2 | check << 32
};

// The check word of a record: tag and value bits through a multiplicative
// mix; odd, so never the 0 of a zero-filled workspace.
__device__ __forceinline__ uint32_t rec_check(uint32_t tag, uint32_t x, uint32_t y, uint32_t z) {
  uint32_t h = tag * 0x9E3779B1u;
  h = (h ^ x) * 0x85EBCA77u;
  h = (h ^ (h >> 15) ^ y) * 0xC2B2AE3Du;
  h = (h ^ (h >> 13) ^ z) * 0x27D4EB2Fu;
  return (h ^ (h >> 16)) | 1u;
}

__device__ __forceinline__ Rec rec_load(const Rec* p) {
  Rec r;
  asm volatile(
      "{\n\t.reg .b128 t;\n\t"
      "ld.relaxed.gpu.global.b128 t, [%2];\n\t"
      "mov.b128 {%0, %1}, t;\n\t}"
      : "=l"(r.lo), "=l"(r.hi)
      : "l"(p)
      : "memory");
  return r;
}

__device__ __forceinline__ void rec_store(Rec* p, uint32_t tag, float x, float y, float z) {
  const uint32_t bx = __float_as_uint(x), by = __float_as_uint(y), bz = __float_as_uint(z);
  const unsigned long long lo = ((unsigned long long)by << 32) | bx;
  const unsigned long long hi = ((unsigned long long)rec_check(tag, bx, by, bz) << 32) | bz;
  asm volatile(
      "{\n\t.reg .b128 t;\n\t"
      "mov.b128 t, {%0, %1};\n\t"
      "st.relaxed.gpu.global.b128 [%2], t;\n\t}" ::"l"(lo),
      "l"(hi), "l"(p)
      : "memory");
}

__device__ __forceinline__ bool rec_ok(const Rec& r, uint32_t tag) {
  return (uint32_t)(r.hi >> 32) == rec_check(tag, (uint32_t)r.lo, (uint32_t)(r.lo >> 32), (uint32_t)r.hi);
}
__device__ __forceinline__ float rec_x(const Rec& r) { return __uint_as_float((uint32_t)r.lo); }
__device__ __forceinline__ float rec_y(const Rec& r) { return __uint_as_float((uint32_t)(r.lo >> 32)); }
__device__ __forceinline__ float rec_z(const Rec& r) { return __uint_as_float((uint32_t)r.hi); }

constexpr int kWaitOk = 0;
constexpr int kWaitTimeout = 1;
constexpr int kWaitError = 2;

}  // namespace wkv
