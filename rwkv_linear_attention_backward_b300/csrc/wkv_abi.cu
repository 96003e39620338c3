// wkv_abi.cu -- the extern "C" boundary of libwkv.so (declared in
// include/wkv.h): argument checks, workspace layout, launch plans.
#include <algorithm>
#include <atomic>
#include <mutex>
#include <cudaTypedefs.h>
#include <climits>
#include <cstdio>
#include <cstring>

#include "wkv.h"
#include "wkv_common.cuh"
#include "wkv_internal.h"

namespace wkv {

namespace {

constexpr long long kDefaultBudgetNs = 500LL * 1000 * 1000;

std::atomic<long long> g_budget_ns{kDefaultBudgetNs};
std::atomic<int> g_skip_chunk{-1};
std::atomic<int> g_scan_mode{WKV_SCAN_AUTO};
std::atomic<int> g_max_runs{0};
std::atomic<int> g_chain_len{0};
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

// Forward workspace: header (tile counters, error record) | chunk summaries
// [nchunks][B][C] tagged 16-byte records | carried states [nchunks][B][C]
// records | checkpoints [3][nchunks][B][C] f32 (used when the caller passes
// none).
struct FwdLayout {
  size_t agg, inc, ckpt, total;
};

FwdLayout fwd_layout(const ScanGeometry& g) {
  FwdLayout l;
  size_t off = sizeof(WsHeader);
  l.agg = off;
  off += align256(g.plane * sizeof(Rec));
  l.inc = off;
  off += align256(g.plane * sizeof(Rec));
  l.ckpt = off;
  off += align256(3 * g.plane * sizeof(float));
  l.total = off;
  return l;
}

// Backward workspace: header | adjoint records, zero-carry and carried,
// [nchunks][B][C] tagged 16-byte records each | gw, gu partials [2][nchunks][B][C]
// f32 | reduction slices [nslice][2][C] f32 | launch-tagged reduction
// counters [ceil(C/32)] u64 | a forward workspace for recomputing the
// checkpoints when none are given.
struct BwdLayout {
  size_t ragg, rinc, part, slices, count, fwd, total;
  int nslice;
};

BwdLayout bwd_layout(const ScanGeometry& g) {
  BwdLayout l;
  size_t off = sizeof(WsHeader);
  l.ragg = off;
  off += align256(g.plane * sizeof(Rec));
  l.rinc = off;
  off += align256(g.plane * sizeof(Rec));
  l.part = off;
  off += align256(2 * g.plane * sizeof(float));
  l.nslice = reduce_slices(g.nchunks * g.B, g.C);
  l.slices = off;
  off += align256((size_t)l.nslice * 2 * g.C * sizeof(float));
  l.count = off;
  off += align256((size_t)((g.C + 31) / 32) * sizeof(unsigned long long));
  l.fwd = off;  // nested forward workspace, used when no checkpoint is given
  off += fwd_layout(g).total;
  l.total = off;
  return l;
}



char* bytes(void* p) { return static_cast<char*>(p); }

// Whether a call takes the sequential column kernels (wkv_seq.cu) or the
// chunked scan (wkv_fwd.cu, wkv_bwd.cu).  Automatic: sequential for every
// shape.  Measured on B300 (forward + backward per call, fp32; forward only,
// bf16, for the last two): B=1 T=64 C=64 0.060 vs 0.061 ms; 1x1024x768 0.068
// vs 0.074; 2x4096x512 0.080 vs 0.137; 1x65536x32 0.317 vs 1.288;
// 4x2048x1024 0.099 vs 0.125; 8x1024x768 0.088 vs 0.102; 1x16384x2048 0.339
// vs 0.451; 1x131072x2560 0.970 vs 1.623; 1x32768x4096 0.345 vs 0.456.  The
// chunked scan stays selectable (wkv_debug_set_scan_mode) and tested.
cudaError_t sequential_mode(const ScanGeometry& g, bool& seq) {
  (void)g;
  seq = g_scan_mode.load() != WKV_SCAN_CHUNKED;
  return cudaSuccess;
}

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
  g.nwg = (C + 31) / 32;
  g.ntiles = (unsigned int)((size_t)g.nchunks * B * g.ncb);
  g.plane = (size_t)g.nchunks * B * C;
  return g;
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

}  // namespace

bool make_tile_map(CUtensorMap* map, const void* base, int B, int T, int C, int elem_bytes, int box_c, int box_t) {
  if ((reinterpret_cast<uintptr_t>(base) & 15u) != 0) return false;
  if (((size_t)C * elem_bytes) % 16 != 0) return false;
  PFN_cuTensorMapEncodeTiled_v12000 fn = tensor_map_encoder();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)C, (cuuint64_t)T, (cuuint64_t)B};
  const cuuint64_t strides[2] = {(cuuint64_t)C * elem_bytes, (cuuint64_t)T * C * elem_bytes};
  const cuuint32_t box[3] = {(cuuint32_t)box_c, (cuuint32_t)box_t, 1u};
  const cuuint32_t estride[3] = {1u, 1u, 1u};
  const CUresult r = fn(map, elem_bytes == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                        const_cast<void*>(base), dims, strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace wkv

namespace wkv {
namespace {

// The tensor maps of the sequential forward walk: k and v in boxes of one
// chunk, and in boxes of one chained item (chain_chunks chunks).  False when
// the inputs do not allow TMA (the kernels then copy with plain loads).
bool seq_forward_maps(SeqFwdArgs& a, const void* k, const void* v, int B, int T, int C, int eb) {
  const int box_t = chain_chunks((size_t)eb) * kChunk;
  return make_tile_map(&a.tk, k, B, T, C, eb, kSeqChannels) && make_tile_map(&a.tv, v, B, T, C, eb, kSeqChannels) &&
         make_tile_map(&a.tk2, k, B, T, C, eb, kSeqChannels, box_t) &&
         make_tile_map(&a.tv2, v, B, T, C, eb, kSeqChannels, box_t);
}

// The backward pass with the sequential column kernels: the checkpoints
// (recomputed by a state-only forward walk when the caller has none), the
// reverse walk writing gk, gv (and gr for the gated output, r non-null) and
// one gw, gu row per (run, batch row), then the reduction of those rows.
wkv_status backward_sequential(const ScanGeometry& g, const BwdLayout& l, int kv_dtype, const float* w,
                               const float* u, const void* k, const void* v, const void* gy, const void* r,
                               const float* state_in, const float* gstate_end, const float* ckpt, float* gw,
                               float* gu, float* gk, float* gv, float* gr, float* gstate_in, WsHeader* hdr,
                               void* workspace, uint64_t budget, cudaStream_t s) {
  const int B = g.B, T = g.T, C = g.C;
  const int eb = kv_dtype == WKV_F32 ? 4 : 2;
  const float* states = ckpt;
  if (!states) {
    SeqFwdArgs f;
    std::memset(&f, 0, sizeof(f));
    f.w = w;
    f.u = u;
    f.k = k;
    f.v = v;
    f.y = nullptr;
    f.state_in = state_in;
    f.ckpt = reinterpret_cast<float*>(bytes(workspace) + l.fwd + fwd_layout(g).ckpt);
    f.recs = reinterpret_cast<Rec*>(bytes(workspace) + l.fwd + fwd_layout(g).agg);
    f.exited = &hdr->exited[1];
    f.nseg = g_max_runs.load();
    f.chain = g_chain_len.load();
    f.debug_skip_chunk = -1;
    f.eh = hdr;
    f.g = g;
    f.budget_ns = budget;
    f.use_tma = seq_forward_maps(f, k, v, B, T, C, eb);
    cudaError_t e = launch_seq_forward(f, kv_dtype, false, s);
    if (e != cudaSuccess) return cuda_fail(e, "wkv_backward: state pass");
    states = f.ckpt;
  }
  SeqBwdArgs a;
  std::memset(&a, 0, sizeof(a));
  a.w = w;
  a.u = u;
  a.k = k;
  a.v = v;
  a.gy = gy;
  a.r = r;
  a.ckpt = states;
  a.state_in = state_in;
  a.gstate_end = gstate_end;
  a.gstate_in = gstate_in;
  a.gk = gk;
  a.gv = gv;
  a.gr = gr;
  a.part = reinterpret_cast<float*>(bytes(workspace) + l.part);  // [2][nseg * B][C]
  a.recs = reinterpret_cast<Rec*>(bytes(workspace) + l.ragg);
  a.exited = &hdr->exited[2];
  a.nseg = g_max_runs.load();
  a.debug_skip_chunk = g_skip_chunk.load();
  a.eh = hdr;
  a.g = g;
  a.budget_ns = budget;
  a.use_tma = make_tile_map(&a.tk, k, B, T, C, eb, kSeqChannels) &&
              make_tile_map(&a.tv, v, B, T, C, eb, kSeqChannels) && make_tile_map(&a.tg, gy, B, T, C, eb, kSeqChannels) &&
              (!r || make_tile_map(&a.tr, r, B, T, C, eb, kSeqChannels));
  cudaError_t e = launch_seq_backward(a, kv_dtype, s);
  if (e != cudaSuccess) return cuda_fail(e, "wkv_backward");
  if (!gk) return WKV_OK;  // a summary pass: no gw, gu to reduce
  const int rows = a.nseg * B;
  ReduceArgs red;
  red.part = a.part;
  red.slices = reinterpret_cast<float*>(bytes(workspace) + l.slices);
  red.count = reinterpret_cast<unsigned long long*>(bytes(workspace) + l.count);
  red.eh = hdr;
  red.gw = gw;
  red.gu = gu;
  red.rows = rows;
  red.C = C;
  red.nslice = reduce_slices(rows, C);
  e = launch_reduce(red, s);
  return e == cudaSuccess ? WKV_OK : cuda_fail(e, "wkv_backward: reduce");
}

}  // namespace
}  // namespace wkv

using namespace wkv;

namespace wkv {
namespace {

// wkv_forward_with_state, and wkv_forward_gated when r is non-null.
wkv_status forward_impl(int B, int T, int C, int kv_dtype, const float* w, const float* u, const void* k,
                        const void* v, const void* r, const float* state_in, float* y, float* state_out, float* ckpt,
                        void* workspace, size_t workspace_bytes, void* stream) {
  clear_error();
  // no y: a state-only pass, which must return the state (or checkpoints)
  if (!sizes_ok(B, T, C) || !w || !u || !k || !v || (!y && !state_out && !ckpt) || (r && !y))
    return WKV_ERR_INVALID_ARG;
  if (kv_dtype != WKV_F32 && kv_dtype != WKV_BF16) return WKV_ERR_INVALID_ARG;
  const ScanGeometry g = make_geometry(B, T, C);
  const FwdLayout l = fwd_layout(g);
  if (!workspace || workspace_bytes < l.total) return WKV_ERR_WORKSPACE;
  const int eb = kv_dtype == WKV_F32 ? 4 : 2;
  bool seq = false;
  cudaError_t e = sequential_mode(g, seq);
  if (e != cudaSuccess) return cuda_fail(e, "wkv_forward");
  if (r && !seq) {
    set_last_error("wkv_forward_gated: the gated output is written by the sequential kernels only (the chunked scan "
                   "is forced)");
    return WKV_ERR_UNSUPPORTED;
  }
  if (seq) {
    SeqFwdArgs q;
    std::memset(&q, 0, sizeof(q));
    q.w = w;
    q.u = u;
    q.k = k;
    q.v = v;
    q.y = y;
    q.r = r;
    q.state_in = state_in;
    q.state_out = state_out;
    q.ckpt = ckpt ? ckpt : reinterpret_cast<float*>(bytes(workspace) + l.ckpt);
    q.recs = reinterpret_cast<Rec*>(bytes(workspace) + l.agg);
    q.eh = static_cast<WsHeader*>(workspace);
    q.exited = &q.eh->exited[0];
    q.nseg = g_max_runs.load();  // 0: the launcher's choice
    q.chain = g_chain_len.load();
    q.debug_skip_chunk = g_skip_chunk.load();
    q.g = g;
    q.budget_ns = (uint64_t)g_budget_ns.load();
    q.use_tma = seq_forward_maps(q, k, v, B, T, C, eb);
    e = launch_seq_forward(q, kv_dtype, y != nullptr, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? WKV_OK : cuda_fail(e, "wkv_forward");
  }
  FwdArgs a;
  std::memset(&a, 0, sizeof(a));
  a.w = w;
  a.u = u;
  a.k = k;
  a.v = v;
  a.y = y;
  a.state_in = state_in;
  a.state_out = state_out;
  a.agg = reinterpret_cast<Rec*>(bytes(workspace) + l.agg);
  a.inc = reinterpret_cast<Rec*>(bytes(workspace) + l.inc);
  a.ckpt = ckpt ? ckpt : reinterpret_cast<float*>(bytes(workspace) + l.ckpt);
  a.eh = static_cast<WsHeader*>(workspace);
  a.ticket = &a.eh->ticket[0];
  a.exited = &a.eh->exited[0];
  a.g = g;
  a.budget_ns = (uint64_t)g_budget_ns.load();
  a.debug_skip_chunk = g_skip_chunk.load();
  a.use_tma = make_tile_map(&a.tk, k, B, T, C, eb, kCtaChannels) && make_tile_map(&a.tv, v, B, T, C, eb, kCtaChannels);
  e = launch_forward(a, kv_dtype, y != nullptr, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? WKV_OK : cuda_fail(e, "wkv_forward");
}

// wkv_backward, wkv_backward_gated when r is non-null (then gy is the
// gated output's gradient and gr receives r's), and wkv_backward_with_state
// (state_in, gstate_end, gstate_in).
wkv_status backward_impl(int B, int T, int C, int kv_dtype, const float* w, const float* u, const void* k,
                         const void* v, const void* gy, const void* r, const float* state_in,
                         const float* gstate_end, const float* ckpt, float* gw, float* gu, float* gk, float* gv,
                         float* gr, float* gstate_in, void* workspace, size_t workspace_bytes, void* stream) {
  clear_error();
  // gk, gv both NULL: the summary pass (the start state's gradient only)
  const bool summary = !gk && !gv && gstate_in && !r;
  if (!sizes_ok(B, T, C) || !w || !u || !k || !v || !gy) return WKV_ERR_INVALID_ARG;
  if (!summary && (!gw || !gu || !gk || !gv)) return WKV_ERR_INVALID_ARG;
  if (r && !gr) return WKV_ERR_INVALID_ARG;
  if (kv_dtype != WKV_F32 && kv_dtype != WKV_BF16) return WKV_ERR_INVALID_ARG;
  const ScanGeometry g = make_geometry(B, T, C);
  const BwdLayout l = bwd_layout(g);
  if (!workspace || workspace_bytes < l.total) return WKV_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  WsHeader* hdr = static_cast<WsHeader*>(workspace);
  const int skip = g_skip_chunk.load();
  const uint64_t budget = (uint64_t)g_budget_ns.load();
  bool seq = false;
  cudaError_t e = sequential_mode(g, seq);
  if (e != cudaSuccess) return cuda_fail(e, "wkv_backward");
  if (seq)
    return backward_sequential(g, l, kv_dtype, w, u, k, v, gy, r, state_in, gstate_end, ckpt, gw, gu, gk, gv, gr,
                               gstate_in, hdr, workspace, budget, s);
  if (state_in || gstate_end || gstate_in) {
    set_last_error("wkv_backward_with_state: carried states are taken by the sequential kernels only (the chunked "
                   "scan is forced)");
    return WKV_ERR_UNSUPPORTED;
  }
  if (r) {
    set_last_error("wkv_backward_gated: the gated output's backward pass runs on the sequential kernels only (the "
                   "chunked scan is forced)");
    return WKV_ERR_UNSUPPORTED;
  }
  if (kv_dtype != WKV_F32) {
    set_last_error("wkv_backward: bf16 inputs are taken by the sequential kernels only (the chunked scan is forced)");
    return WKV_ERR_UNSUPPORTED;
  }

  const float* states = ckpt;
  if (!states) {
    // recompute the chunk-boundary states: forward scan without outputs
    char* fws = bytes(workspace) + l.fwd;
    const FwdLayout fl = fwd_layout(g);
    FwdArgs f;
    std::memset(&f, 0, sizeof(f));
    f.w = w;
    f.u = u;
    f.k = k;
    f.v = v;
    f.y = nullptr;
    f.agg = reinterpret_cast<Rec*>(fws + fl.agg);
    f.inc = reinterpret_cast<Rec*>(fws + fl.inc);
    f.ckpt = reinterpret_cast<float*>(fws + fl.ckpt);
    f.ticket = &hdr->ticket[1];  // counters stay in the outer header: its place never moves
    f.exited = &hdr->exited[1];
    f.eh = hdr;
    f.g = g;
    f.budget_ns = budget;
    f.debug_skip_chunk = -1;
    f.use_tma = make_tile_map(&f.tk, k, B, T, C, 4, kCtaChannels) && make_tile_map(&f.tv, v, B, T, C, 4, kCtaChannels);
    e = launch_forward(f, WKV_F32, false, s);
    if (e != cudaSuccess) return cuda_fail(e, "wkv_backward: state pass");
    states = f.ckpt;
  }

  BwdArgs a;
  std::memset(&a, 0, sizeof(a));
  a.w = w;
  a.u = u;
  a.k = static_cast<const float*>(k);
  a.v = static_cast<const float*>(v);
  a.gy = static_cast<const float*>(gy);
  a.ckpt = states;
  a.gk = gk;
  a.gv = gv;
  a.ragg = reinterpret_cast<Rec*>(bytes(workspace) + l.ragg);
  a.rinc = reinterpret_cast<Rec*>(bytes(workspace) + l.rinc);
  a.part = reinterpret_cast<float*>(bytes(workspace) + l.part);
  a.ticket = &hdr->ticket[2];
  a.exited = &hdr->exited[2];
  a.eh = hdr;
  a.g = g;
  a.budget_ns = budget;
  a.debug_skip_chunk = skip;
  a.use_tma = make_tile_map(&a.tk, k, B, T, C, 4, kCtaChannels) && make_tile_map(&a.tv, v, B, T, C, 4, kCtaChannels) &&
              make_tile_map(&a.tg, gy, B, T, C, 4, kCtaChannels);
  e = launch_backward(a, s);
  if (e != cudaSuccess) return cuda_fail(e, "wkv_backward");

  ReduceArgs red;
  red.part = a.part;
  red.slices = reinterpret_cast<float*>(bytes(workspace) + l.slices);
  red.count = reinterpret_cast<unsigned long long*>(bytes(workspace) + l.count);
  red.eh = hdr;
  red.gw = gw;
  red.gu = gu;
  red.rows = g.nchunks * g.B;
  red.C = C;
  red.nslice = l.nslice;
  e = launch_reduce(red, s);
  return e == cudaSuccess ? WKV_OK : cuda_fail(e, "wkv_backward: reduce");
}

}  // namespace
}  // namespace wkv


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

wkv_status wkv_sync_status(void* stream) {
  clear_error();
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "wkv_sync_status: synchronize");
  unsigned int first = 0;
  cudaError_t (*const takers[])(unsigned int*) = {take_error_seq, take_error_fwd, take_error_bwd};
  for (auto take : takers) {  // every record is taken (and cleared), the first one reported
    unsigned int code = 0;
    e = take(&code);
    if (e != cudaSuccess) return cuda_fail(e, "wkv_sync_status: read");
    if (first == 0) first = code;
  }
  if (first == 0) return WKV_OK;
  set_last_error("wkv_sync_status: a bounded device-side wait expired; the outputs of that call are invalid");
  return first == kDevErrTimeout ? WKV_ERR_TIMEOUT : WKV_ERR_CUDA;
}

wkv_status wkv_forward(int B, int T, int C, int kv_dtype, const float* w, const float* u, const void* k,
                       const void* v, float* y, float* ckpt, void* workspace, size_t workspace_bytes,
                       void* stream) {
  if (!y) {
    clear_error();
    return WKV_ERR_INVALID_ARG;
  }
  return wkv_forward_with_state(B, T, C, kv_dtype, w, u, k, v, nullptr, y, nullptr, ckpt, workspace,
                                workspace_bytes, stream);
}

wkv_status wkv_forward_with_state(int B, int T, int C, int kv_dtype, const float* w, const float* u, const void* k,
                                  const void* v, const float* state_in, float* y, float* state_out, float* ckpt,
                                  void* workspace, size_t workspace_bytes, void* stream) {
  return forward_impl(B, T, C, kv_dtype, w, u, k, v, nullptr, state_in, y, state_out, ckpt, workspace,
                      workspace_bytes, stream);
}

wkv_status wkv_forward_gated(int B, int T, int C, int kv_dtype, const float* w, const float* u, const void* k,
                             const void* v, const void* r, const float* state_in, float* out, float* state_out,
                             float* ckpt, void* workspace, size_t workspace_bytes, void* stream) {
  clear_error();
  if (!r) return WKV_ERR_INVALID_ARG;
  return forward_impl(B, T, C, kv_dtype, w, u, k, v, r, state_in, out, state_out, ckpt, workspace, workspace_bytes,
                      stream);
}

wkv_status wkv_backward(int B, int T, int C, int kv_dtype, const float* w, const float* u, const void* k,
                        const void* v, const void* gy, const float* ckpt, float* gw, float* gu, float* gk,
                        float* gv, void* workspace, size_t workspace_bytes, void* stream) {
  return backward_impl(B, T, C, kv_dtype, w, u, k, v, gy, nullptr, nullptr, nullptr, ckpt, gw, gu, gk, gv, nullptr,
                       nullptr, workspace, workspace_bytes, stream);
}

wkv_status wkv_backward_with_state(int B, int T, int C, int kv_dtype, const float* w, const float* u, const void* k,
                                   const void* v, const void* gy, const float* state_in, const float* gstate_end,
                                   const float* ckpt, float* gw, float* gu, float* gk, float* gv, float* gstate_in,
                                   void* workspace, size_t workspace_bytes, void* stream) {
  return backward_impl(B, T, C, kv_dtype, w, u, k, v, gy, nullptr, state_in, gstate_end, ckpt, gw, gu, gk, gv,
                       nullptr, gstate_in, workspace, workspace_bytes, stream);
}

wkv_status wkv_backward_gated(int B, int T, int C, int kv_dtype, const float* w, const float* u, const void* k,
                              const void* v, const void* r, const void* gout, const float* ckpt, float* gw, float* gu,
                              float* gk, float* gv, float* gr, void* workspace, size_t workspace_bytes, void* stream) {
  clear_error();
  if (!r || !gr) return WKV_ERR_INVALID_ARG;
  return backward_impl(B, T, C, kv_dtype, w, u, k, v, gout, r, nullptr, nullptr, ckpt, gw, gu, gk, gv, gr, nullptr,
                       workspace, workspace_bytes, stream);
}

namespace {

// The decode step with fp32 (token_dtype 0) or bf16 (1) token inputs.
wkv_status decode_impl(int L, int B, int C, int token_dtype, const void* x, const void* x_prev, const float* mu_k,
                       const float* mu_v, const float* mu_r, const void* r, const void* k, const void* v,
                       const float* w, const float* u, float* num, float* den, float* pp, float* y, float* xk,
                       float* xv, float* xr, void* stream, const char* where) {
  clear_error();
  if (L <= 0 || B <= 0 || C <= 0) return WKV_ERR_INVALID_ARG;
  if ((double)L * B * C >= 1099511627776.0) return WKV_ERR_INVALID_ARG;
  if (!x || !x_prev || !mu_k || !mu_v || !mu_r || !r || !k || !v || !w || !u || !num || !den || !pp || !y)
    return WKV_ERR_INVALID_ARG;
  DecodeArgs a{x, x_prev, mu_k, mu_v, mu_r, r, k, v, w, u, num, den, pp, y, xk, xv, xr, L, B, C};
  auto al = [](const void* p, unsigned m) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & m) == 0; };
  // four channels per thread: 16-byte accesses of fp32 arrays, 8-byte of bf16 ones
  const unsigned tm = token_dtype == 0 ? 15u : 7u;
  const bool vec4 = (C % 4 == 0) && al(x, tm) && al(x_prev, tm) && al(r, tm) && al(k, tm) && al(v, tm) &&
                    al(mu_k, 15u) && al(mu_v, 15u) && al(mu_r, 15u) && al(w, 15u) && al(u, 15u) && al(num, 15u) &&
                    al(den, 15u) && al(pp, 15u) && al(y, 15u) && al(xk, 15u) && al(xv, 15u) && al(xr, 15u);
  cudaError_t e = launch_decode(a, vec4, token_dtype, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? WKV_OK : cuda_fail(e, where);
}

}  // namespace

wkv_status wkv_decode_step(int L, int B, int C, const float* x, const float* x_prev, const float* mu_k,
                           const float* mu_v, const float* mu_r, const float* r, const float* k, const float* v,
                           const float* w, const float* u, float* num, float* den, float* pp, float* y, float* xk,
                           float* xv, float* xr, void* stream) {
  return decode_impl(L, B, C, 0, x, x_prev, mu_k, mu_v, mu_r, r, k, v, w, u, num, den, pp, y, xk, xv, xr, stream,
                     "wkv_decode_step");
}

wkv_status wkv_decode_step_bf16(int L, int B, int C, const void* x, const void* x_prev, const float* mu_k,
                                const float* mu_v, const float* mu_r, const void* r, const void* k, const void* v,
                                const float* w, const float* u, float* num, float* den, float* pp, float* y,
                                float* xk, float* xv, float* xr, void* stream) {
  return decode_impl(L, B, C, 1, x, x_prev, mu_k, mu_v, mu_r, r, k, v, w, u, num, den, pp, y, xk, xv, xr, stream,
                     "wkv_decode_step_bf16");
}

size_t wkv_token_shift_backward_workspace_bytes(int B, int T, int C) {
  if (B <= 0 || T <= 0 || C <= 0 || (double)B * T * C >= 1099511627776.0) return 0;
  const bool vec4 = C % 4 == 0;  // the larger of the two slice counts
  const int ns = std::max(shift_slices(B, T, C, vec4), shift_slices(B, T, C, false));
  return std::max<size_t>(align256((size_t)ns * 3 * C * sizeof(float)), 256);
}

wkv_status wkv_token_shift(int B, int T, int C, const float* x, const float* x0, const float* mu_k,
                           const float* mu_v, const float* mu_r, float* xk, float* xv, float* xr, void* stream) {
  clear_error();
  if (B <= 0 || T <= 0 || C <= 0 || (double)B * T * C >= 1099511627776.0) return WKV_ERR_INVALID_ARG;
  if (!x || !mu_k || !mu_v || !mu_r || !xk || !xv || !xr) return WKV_ERR_INVALID_ARG;
  ShiftArgs a;
  std::memset(&a, 0, sizeof(a));
  a.x = x;
  a.x0 = x0;
  a.mu_k = mu_k;
  a.mu_v = mu_v;
  a.mu_r = mu_r;
  a.xk = xk;
  a.xv = xv;
  a.xr = xr;
  a.B = B;
  a.T = T;
  a.C = C;
  auto al16 = [](const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  const bool vec4 = C % 4 == 0 && al16(x) && al16(x0) && al16(mu_k) && al16(mu_v) && al16(mu_r) && al16(xk) &&
                    al16(xv) && al16(xr);
  cudaError_t e = launch_shift_forward(a, vec4, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? WKV_OK : cuda_fail(e, "wkv_token_shift");
}

wkv_status wkv_token_shift_backward(int B, int T, int C, const float* x, const float* x0, const float* mu_k,
                                    const float* mu_v, const float* mu_r, const float* gxk, const float* gxv,
                                    const float* gxr, float* gx, float* gx0, float* gmu_k, float* gmu_v,
                                    float* gmu_r, void* workspace, size_t workspace_bytes, void* stream) {
  clear_error();
  if (B <= 0 || T <= 0 || C <= 0 || (double)B * T * C >= 1099511627776.0) return WKV_ERR_INVALID_ARG;
  if (!x || !mu_k || !mu_v || !mu_r || !gxk || !gxv || !gxr || !gx || !gmu_k || !gmu_v || !gmu_r)
    return WKV_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < wkv_token_shift_backward_workspace_bytes(B, T, C)) return WKV_ERR_WORKSPACE;
  ShiftArgs a;
  std::memset(&a, 0, sizeof(a));
  a.x = x;
  a.x0 = x0;
  a.mu_k = mu_k;
  a.mu_v = mu_v;
  a.mu_r = mu_r;
  a.gxk = gxk;
  a.gxv = gxv;
  a.gxr = gxr;
  a.gx = gx;
  a.gx0 = gx0;
  a.gmu_k = gmu_k;
  a.gmu_v = gmu_v;
  a.gmu_r = gmu_r;
  a.part = static_cast<float*>(workspace);
  a.B = B;
  a.T = T;
  a.C = C;
  auto al16 = [](const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  const bool vec4 = C % 4 == 0 && al16(x) && al16(x0) && al16(mu_k) && al16(mu_v) && al16(mu_r) && al16(gxk) &&
                    al16(gxv) && al16(gxr) && al16(gx) && al16(gx0);
  a.nslice = shift_slices(B, T, C, vec4);
  cudaError_t e = launch_shift_backward(a, vec4, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? WKV_OK : cuda_fail(e, "wkv_token_shift_backward");
}

namespace {
// The channel-mix calls: nothing to do for n == 0; every pointer required
// for n > 0.
wkv_status cmix_call(int op, long long n, const float* x, const float* y, const float* z, float* o1, float* o2,
                     void* stream, const char* who) {
  clear_error();
  if (n < 0) return WKV_ERR_INVALID_ARG;
  if (n == 0) return WKV_OK;
  if (!x || !o1 || (op != 0 && !y) || (op == 3 && (!z || !o2))) return WKV_ERR_INVALID_ARG;
  CmixArgs a;
  a.x = x;
  a.y = op != 0 ? y : nullptr;
  a.z = op == 3 ? z : nullptr;
  a.o1 = o1;
  a.o2 = op == 3 ? o2 : nullptr;
  a.n = n;
  cudaError_t e = launch_cmix(op, a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? WKV_OK : cuda_fail(e, who);
}
}  // namespace

wkv_status wkv_channel_mix_sqrelu(long long n, const float* k, float* a, void* stream) {
  return cmix_call(0, n, k, nullptr, nullptr, a, nullptr, stream, "wkv_channel_mix_sqrelu");
}

wkv_status wkv_channel_mix_sqrelu_backward(long long n, const float* k, const float* ga, float* gk, void* stream) {
  return cmix_call(1, n, k, ga, nullptr, gk, nullptr, stream, "wkv_channel_mix_sqrelu_backward");
}

wkv_status wkv_channel_mix_gate(long long n, const float* r, const float* vk, float* out, void* stream) {
  return cmix_call(2, n, r, vk, nullptr, out, nullptr, stream, "wkv_channel_mix_gate");
}

wkv_status wkv_channel_mix_gate_backward(long long n, const float* r, const float* vk, const float* gout, float* gr,
                                         float* gvk, void* stream) {
  return cmix_call(3, n, r, vk, gout, gr, gvk, stream, "wkv_channel_mix_gate_backward");
}

wkv_status wkv_state_fold(int B, int C, const float* w, int n, const float* states, const long long* lengths,
                          float* out, void* stream) {
  clear_error();
  if (B <= 0 || C <= 0 || (double)B * C >= 1099511627776.0 || !w || !out || n < 0 || n > kMaxFoldSegments)
    return WKV_ERR_INVALID_ARG;
  if (n > 0 && (!states || !lengths)) return WKV_ERR_INVALID_ARG;
  FoldArgs a;
  std::memset(&a, 0, sizeof(a));
  for (int i = 0; i < n; ++i) {
    if (lengths[i] < 0) return WKV_ERR_INVALID_ARG;
    a.len[i] = lengths[i];
  }
  a.w = w;
  a.states = states;
  a.out = out;
  a.B = B;
  a.C = C;
  a.n = n;
  cudaError_t e = launch_state_fold(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? WKV_OK : cuda_fail(e, "wkv_state_fold");
}

wkv_status wkv_adjoint_fold(int B, int C, const float* w, int n, const float* adj, const long long* lengths,
                            const float* gstate_end, float* out, void* stream) {
  clear_error();
  if (B <= 0 || C <= 0 || (double)B * C >= 1099511627776.0 || !w || !out || n < 0 || n > kMaxFoldSegments)
    return WKV_ERR_INVALID_ARG;
  if (n > 0 && (!adj || !lengths)) return WKV_ERR_INVALID_ARG;
  if (n == 0 && !gstate_end) return WKV_ERR_INVALID_ARG;
  AdjFoldArgs a;
  std::memset(&a, 0, sizeof(a));
  for (int i = 0; i < n; ++i) {
    if (lengths[i] < 0) return WKV_ERR_INVALID_ARG;
    a.len[i] = lengths[i];
  }
  a.w = w;
  a.adj = adj;
  a.gend = gstate_end;
  a.out = out;
  a.B = B;
  a.C = C;
  a.n = n;
  cudaError_t e = launch_adjoint_fold(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? WKV_OK : cuda_fail(e, "wkv_adjoint_fold");
}

wkv_status wkv_debug_set_wait_budget_ns(long long ns) {
  g_budget_ns.store(ns > 0 ? ns : kDefaultBudgetNs);
  return WKV_OK;
}

wkv_status wkv_debug_set_skip_chunk(int chunk) {
  g_skip_chunk.store(chunk < 0 ? -1 : chunk);
  return WKV_OK;
}

int wkv_scan_strategy(int B, int T, int C) {
  if (!sizes_ok(B, T, C)) return -1;
  bool seq = false;
  if (sequential_mode(make_geometry(B, T, C), seq) != cudaSuccess) return -1;
  return seq ? WKV_SCAN_SEQUENTIAL : WKV_SCAN_CHUNKED;
}

wkv_status wkv_debug_set_chain_len(int chunks) {
  g_chain_len.store(chunks > 0 ? chunks : 0);
  return WKV_OK;
}

wkv_status wkv_debug_set_max_runs(int runs) {
  g_max_runs.store(runs > 0 ? runs : 0);
  return WKV_OK;
}

wkv_status wkv_debug_set_scan_mode(int mode) {
  if (mode != WKV_SCAN_AUTO && mode != WKV_SCAN_CHUNKED && mode != WKV_SCAN_SEQUENTIAL) return WKV_ERR_INVALID_ARG;
  g_scan_mode.store(mode);
  return WKV_OK;
}

}  // extern "C"
