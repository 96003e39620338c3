// wkv_abi.cu -- the extern "C" boundary of libwkv.so (declared in
// include/wkv.h): argument checks, workspace layout, launch plans.
#include <atomic>
#include <climits>
#include <cstdio>
#include <cstring>

#include "wkv.h"
#include "wkv_common.cuh"
#include "wkv_internal.h"

namespace wkv {

namespace {

constexpr long long kDefaultBudgetNs = 500LL * 1000 * 1000;

std::atomic<uint64_t> g_epoch{0};
std::atomic<long long> g_budget_ns{kDefaultBudgetNs};
std::atomic<int> g_skip_chunk{-1};
thread_local char g_last_error[256] = "";

void clear_error() { g_last_error[0] = '\0'; }

wkv_status cuda_fail(cudaError_t e, const char* where) {
  std::snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
  return WKV_ERR_CUDA;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

bool sizes_ok(int B, int T, int C) {
  if (B <= 0 || T <= 0 || C <= 0) return false;
  const double n = (double)B * (double)T * (double)C;
  if (n >= 1099511627776.0) return false;  // 2^40 elements
  const ScanGeometry g = make_geometry(B, T, C);
  return (double)g.nchunks * g.B * g.ncb <= (double)INT_MAX;
}

// Forward workspace: header (tile counters, error record) | flags
// [B][nwg][nnodes] u64 | tree nodes
// [3][nnodes][B][C] f32 | checkpoints [3][nchunks][B][C] f32 (used when the
// caller passes none).
struct FwdLayout {
  size_t flags, nodes, incl, total;
};

FwdLayout fwd_layout(const ScanGeometry& g) {
  FwdLayout l;
  size_t off = sizeof(WsHeader);
  l.flags = off;
  off += align256((size_t)g.B * g.nwg * g.nnodes * sizeof(uint64_t));
  l.nodes = off;
  off += align256(3 * g.nplane * sizeof(float));
  l.incl = off;
  off += align256(3 * g.plane * sizeof(float));
  l.total = off;
  return l;
}

// Backward workspace: header | flags [B][nwg][nnodes] u64 | adjoint tree
// nodes [3][nnodes][B][C] f32 | gw, gu partials [2][nchunks][B][C] f32 |
// a forward workspace for recomputing the checkpoints when none are given.
struct BwdLayout {
  size_t flags, rnodes, part, fwd, total;
};

BwdLayout bwd_layout(const ScanGeometry& g) {
  BwdLayout l;
  size_t off = sizeof(WsHeader);
  l.flags = off;
  off += align256((size_t)g.B * g.nwg * g.nnodes * sizeof(uint64_t));
  l.rnodes = off;
  off += align256(3 * g.nplane * sizeof(float));
  l.part = off;
  off += align256(2 * g.plane * sizeof(float));
  l.fwd = off;  // nested forward workspace, used when no checkpoint is given
  off += fwd_layout(g).total;
  l.total = off;
  return l;
}

uint64_t next_epoch() { return g_epoch.fetch_add(1) + 1; }

char* bytes(void* p) { return static_cast<char*>(p); }

}  // namespace

void set_last_error(const char* msg) {
  std::snprintf(g_last_error, sizeof(g_last_error), "%s", msg);
}

ScanGeometry make_geometry(int B, int T, int C) {
  ScanGeometry g;
  g.B = B;
  g.T = T;
  g.C = C;
  g.nchunks = (T + kChunk - 1) / kChunk;
  g.ncb = (C + kCtaChannels - 1) / kCtaChannels;
  g.nwg = g.ncb * (kCtaChannels / 32);
  g.ntiles = (unsigned int)((size_t)g.nchunks * B * g.ncb);
  g.plane = (size_t)g.nchunks * B * C;
  g.nnodes = 0;
  g.nlevels = 0;
  for (int s = 0; s < 32; ++s) {
    g.level_off[s] = g.nnodes;
    const int cnt = g.nchunks >> s;
    if (cnt > 0) {
      g.nnodes += cnt;
      g.nlevels = s + 1;
    }
  }
  g.nplane = (size_t)g.nnodes * B * C;
  return g;
}

}  // namespace wkv

using namespace wkv;

extern "C" {

const char* wkv_status_string(int status) {
  switch (status) {
    case WKV_OK: return "WKV_OK";
    case WKV_ERR_INVALID_ARG: return "WKV_ERR_INVALID_ARG";
    case WKV_ERR_UNSUPPORTED: return "WKV_ERR_UNSUPPORTED";
    case WKV_ERR_MISALIGNED: return "WKV_ERR_MISALIGNED";
    case WKV_ERR_WORKSPACE: return "WKV_ERR_WORKSPACE";
    case WKV_ERR_CUDA: return "WKV_ERR_CUDA";
    case WKV_ERR_TIMEOUT: return "WKV_ERR_TIMEOUT";
    default: return "WKV_ERR_UNKNOWN";
  }
}

const char* wkv_last_error_string(void) { return g_last_error; }

int wkv_version(void) { return 1; }

int wkv_chunk_len(void) { return kChunk; }

size_t wkv_checkpoint_floats(int B, int T, int C) {
  if (!sizes_ok(B, T, C)) return 0;
  return 3 * make_geometry(B, T, C).plane;
}

size_t wkv_forward_workspace_bytes(int B, int T, int C) {
  if (!sizes_ok(B, T, C)) return 0;
  return fwd_layout(make_geometry(B, T, C)).total;
}

size_t wkv_backward_workspace_bytes(int B, int T, int C) {
  if (!sizes_ok(B, T, C)) return 0;
  return bwd_layout(make_geometry(B, T, C)).total;
}

wkv_status wkv_workspace_init(void* workspace, size_t nbytes, void* stream) {
  clear_error();
  if (!workspace || nbytes < sizeof(WsHeader)) return WKV_ERR_INVALID_ARG;
  cudaError_t e = cudaMemsetAsync(workspace, 0, nbytes, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? WKV_OK : cuda_fail(e, "wkv_workspace_init");
}

wkv_status wkv_workspace_check(void* workspace, void* stream) {
  clear_error();
  if (!workspace) return WKV_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "wkv_workspace_check: synchronize");
  unsigned int code = 0;
  WsHeader* h = static_cast<WsHeader*>(workspace);
  e = cudaMemcpy(&code, &h->error, sizeof(code), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "wkv_workspace_check: read");
  if (code == 0) return WKV_OK;
  const unsigned int zero = 0;
  e = cudaMemcpy(&h->error, &zero, sizeof(zero), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(e, "wkv_workspace_check: clear");
  return code == kDevErrTimeout ? WKV_ERR_TIMEOUT : WKV_ERR_CUDA;
}

wkv_status wkv_forward(int B, int T, int C, int kv_dtype, const float* w, const float* u, const void* k,
                       const void* v, float* y, float* ckpt, void* workspace, size_t workspace_bytes,
                       void* stream) {
  clear_error();
  if (!sizes_ok(B, T, C) || !w || !u || !k || !v || !y) return WKV_ERR_INVALID_ARG;
  if (kv_dtype != WKV_F32 && kv_dtype != WKV_BF16) return WKV_ERR_INVALID_ARG;
  const ScanGeometry g = make_geometry(B, T, C);
  const FwdLayout l = fwd_layout(g);
  if (!workspace || workspace_bytes < l.total) return WKV_ERR_WORKSPACE;
  FwdArgs a;
  a.w = w;
  a.u = u;
  a.k = k;
  a.v = v;
  a.y = y;
  a.nodes = reinterpret_cast<float*>(bytes(workspace) + l.nodes);
  a.incl = ckpt ? ckpt : reinterpret_cast<float*>(bytes(workspace) + l.incl);
  a.flags = reinterpret_cast<uint64_t*>(bytes(workspace) + l.flags);
  a.eh = static_cast<WsHeader*>(workspace);
  a.ticket = &a.eh->ticket[0];
  a.g = g;
  a.epoch = next_epoch();
  a.budget_ns = (uint64_t)g_budget_ns.load();
  a.debug_skip_chunk = g_skip_chunk.load();
  cudaError_t e = launch_forward(a, kv_dtype, true, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? WKV_OK : cuda_fail(e, "wkv_forward");
}

wkv_status wkv_backward(int B, int T, int C, int kv_dtype, const float* w, const float* u, const void* k,
                        const void* v, const float* gy, const float* ckpt, float* gw, float* gu, float* gk,
                        float* gv, void* workspace, size_t workspace_bytes, void* stream) {
  clear_error();
  if (!sizes_ok(B, T, C) || !w || !u || !k || !v || !gy || !gw || !gu || !gk || !gv) return WKV_ERR_INVALID_ARG;
  if (kv_dtype != WKV_F32 && kv_dtype != WKV_BF16) return WKV_ERR_INVALID_ARG;
  if (kv_dtype != WKV_F32) return WKV_ERR_UNSUPPORTED;
  const ScanGeometry g = make_geometry(B, T, C);
  const BwdLayout l = bwd_layout(g);
  if (!workspace || workspace_bytes < l.total) return WKV_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  WsHeader* hdr = static_cast<WsHeader*>(workspace);
  const int skip = g_skip_chunk.load();
  const uint64_t budget = (uint64_t)g_budget_ns.load();

  const float* states = ckpt;
  if (!states) {
    // recompute the chunk-boundary states: forward scan without outputs
    char* fws = bytes(workspace) + l.fwd;
    const FwdLayout fl = fwd_layout(g);
    FwdArgs f;
    f.w = w;
    f.u = u;
    f.k = k;
    f.v = v;
    f.y = nullptr;
    f.nodes = reinterpret_cast<float*>(fws + fl.nodes);
    f.incl = reinterpret_cast<float*>(fws + fl.incl);
    f.flags = reinterpret_cast<uint64_t*>(fws + fl.flags);
    f.ticket = &hdr->ticket[1];  // counters stay in the outer header: its place never moves
    f.eh = hdr;
    f.g = g;
    f.epoch = next_epoch();
    f.budget_ns = budget;
    f.debug_skip_chunk = -1;
    cudaError_t e = launch_forward(f, WKV_F32, false, s);
    if (e != cudaSuccess) return cuda_fail(e, "wkv_backward: state pass");
    states = f.incl;
  }

  BwdArgs a;
  a.w = w;
  a.u = u;
  a.k = static_cast<const float*>(k);
  a.v = static_cast<const float*>(v);
  a.gy = gy;
  a.ckpt = states;
  a.gk = gk;
  a.gv = gv;
  a.rnodes = reinterpret_cast<float*>(bytes(workspace) + l.rnodes);
  a.part = reinterpret_cast<float*>(bytes(workspace) + l.part);
  a.flags = reinterpret_cast<uint64_t*>(bytes(workspace) + l.flags);
  a.ticket = &hdr->ticket[2];
  a.eh = hdr;
  a.g = g;
  a.epoch = next_epoch();
  a.budget_ns = budget;
  a.debug_skip_chunk = skip;
  cudaError_t e = launch_backward(a, s);
  if (e != cudaSuccess) return cuda_fail(e, "wkv_backward");

  ReduceArgs r;
  r.part = a.part;
  r.gw = gw;
  r.gu = gu;
  r.rows = g.nchunks * g.B;
  r.C = C;
  e = launch_reduce(r, s);
  return e == cudaSuccess ? WKV_OK : cuda_fail(e, "wkv_backward: reduce");
}

wkv_status wkv_decode_step(int L, int B, int C, const float* x, const float* x_prev, const float* mu_k,
                           const float* mu_v, const float* mu_r, const float* r, const float* k, const float* v,
                           const float* w, const float* u, float* num, float* den, float* pp, float* y, float* xk,
                           float* xv, float* xr, void* stream) {
  clear_error();
  if (L <= 0 || B <= 0 || C <= 0) return WKV_ERR_INVALID_ARG;
  if ((double)L * B * C >= 1099511627776.0) return WKV_ERR_INVALID_ARG;
  if (!x || !x_prev || !mu_k || !mu_v || !mu_r || !r || !k || !v || !w || !u || !num || !den || !pp || !y)
    return WKV_ERR_INVALID_ARG;
  DecodeArgs a{x, x_prev, mu_k, mu_v, mu_r, r, k, v, w, u, num, den, pp, y, xk, xv, xr, L, B, C};
  auto al16 = [](const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  const bool vec4 = (C % 4 == 0) && al16(x) && al16(x_prev) && al16(mu_k) && al16(mu_v) && al16(mu_r) && al16(r) &&
                    al16(k) && al16(v) && al16(w) && al16(u) && al16(num) && al16(den) && al16(pp) && al16(y) &&
                    al16(xk) && al16(xv) && al16(xr);
  cudaError_t e = launch_decode(a, vec4, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? WKV_OK : cuda_fail(e, "wkv_decode_step");
}

wkv_status wkv_debug_set_wait_budget_ns(long long ns) {
  g_budget_ns.store(ns > 0 ? ns : kDefaultBudgetNs);
  return WKV_OK;
}

wkv_status wkv_debug_set_skip_chunk(int chunk) {
  g_skip_chunk.store(chunk < 0 ? -1 : chunk);
  return WKV_OK;
}

}  // extern "C"
