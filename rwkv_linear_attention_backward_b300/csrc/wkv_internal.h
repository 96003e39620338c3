// wkv_internal.h -- host-side declarations shared by the library's .cu files.
// Not part of the public ABI (that is include/wkv.h).
#pragma once

#include <cuda.h>
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace wkv {

struct WsHeader;

// Time-chunk length of the chunked scans.  One value for every shape, so the
// chunk-boundary states written by the forward pass line up with the chunks
// of the backward pass.
constexpr int kChunk = 32;
// Channels per tile of the scan kernels (4 consumer warps x 32 lanes, one
// channel per lane).
constexpr int kCtaChannels = 128;

struct ScanGeometry {
  int B, T, C;
  int nchunks;          // ceil(T / kChunk)
  int ncb;              // ceil(C / kCtaChannels): channel blocks per (chunk, row)
  int nwg;              // ceil(C / 32): 32-channel groups per row (one chain of chunks each)
  unsigned int ntiles;  // nchunks * B * ncb
  size_t plane;         // nchunks * B * C: floats per record plane
};

ScanGeometry make_geometry(int B, int T, int C);

struct Rec;  // a 16-byte tagged record (wkv_common.cuh)

// Forward scan.  Records are [nchunks][B][C] arrays of tagged 16-byte
// records (wkv_common.cuh) holding states (num, den, pp).
struct FwdArgs {
  CUtensorMap tk, tv;  // rank-3 maps {C, T, B} of k and v, box {128, kChunk, 1} (when use_tma)
  const float* w;
  const float* u;
  const void* k;
  const void* v;
  float* y;            // may be null (state-only pass)
  const float* state_in;  // [3][B][C] state before the first token (num, den, pp planes); null: empty
  float* state_out;       // [3][B][C] state after the last token; may be null
  Rec* agg;            // each chunk's own summary (from the empty state), written by the tiles
  Rec* inc;            // the state after each chunk, written by the walkers for the next chunk's tiles
  float* ckpt;         // [3][nchunks][B][C] f32: the state after each chunk (the checkpoints)
  unsigned int* ticket;  // tile counter of this launch (in a workspace header)
  unsigned int* exited;  // CTAs of this launch that have finished
  WsHeader* eh;          // where an expired wait is recorded (checked by the host)
  ScanGeometry g;
  uint64_t budget_ns;
  int debug_skip_chunk;  // -1: off
  int use_tma;
};

// Backward scan.  Adjoint records (tagged, [nchunks][B][C]) hold (la, lb,
// f): the adjoints of the sums a, b at a chunk's first token, scaled by
// e^{f}, with f the forward state's pp there.
struct BwdArgs {
  CUtensorMap tk, tv, tg;  // rank-3 maps of k, v, gy (when use_tma)
  const float* w;
  const float* u;
  const float* k;
  const float* v;
  const float* gy;
  const float* ckpt;   // [3][nchunks][B][C] state after each chunk (forward)
  float* gk;
  float* gv;
  Rec* ragg;           // zero-carry adjoint of each chunk, written by the tiles
  Rec* rinc;           // adjoint at each chunk's start with everything after it, written by the walkers
  float* part;         // [2][nchunks][B][C] per-tile gw, gu partial sums
  unsigned int* ticket;
  unsigned int* exited;
  WsHeader* eh;
  ScanGeometry g;
  uint64_t budget_ns;
  int debug_skip_chunk;
  int use_tma;
};

struct ReduceArgs {
  const float* part;    // [2][rows][C]
  float* slices;        // [nslice][2][C] per-slice sums
  unsigned long long* count;  // [ceil(C / 32)] arrival counters, (tag << 32) | arrivals
  const WsHeader* eh;         // its sequence number tags the counters: another tag reads as zero
  float* gw;
  float* gu;
  int rows;             // nchunks * B
  int C;
  int nslice;           // row slices (blockIdx.y)
};

struct DecodeArgs {
  const void *x, *x_prev;           // token inputs [L, B, C]: float or bf16 (the launch's token dtype)
  const float *mu_k, *mu_v, *mu_r;  // [L, C]
  const void *r, *k, *v;            // token inputs, as x
  const float *w, *u;               // [L, C]
  float *num, *den, *pp, *y, *xk, *xv, *xr;
  int L, B, C;
};

// Sets the text returned by wkv_last_error_string() on this thread.
void set_last_error(const char* msg);

// Each file's device-wide record of an expired wait on the current device:
// read and cleared (wkv_sync_status).
cudaError_t take_error_seq(unsigned int* code);
cudaError_t take_error_fwd(unsigned int* code);
cudaError_t take_error_bwd(unsigned int* code);

// Rank-3 TMA descriptor of a [B, T, C] tensor with a {box_c, kChunk, 1} box
// (elem_bytes 4 = fp32, 2 = bf16).  False when TMA cannot address it (the
// base not 16-byte aligned or C * elem_bytes not a multiple of 16) or the
// driver has no encoder; the kernels then stage tiles with plain loads.
bool make_tile_map(CUtensorMap* map, const void* base, int B, int T, int C, int elem_bytes, int box_c,
                   int box_t = kChunk);

// Sequential column kernels (wkv_seq.cu): a column is one batch row and 32
// channels; its chunks are walked in order (forward) or in reverse order
// (backward) by nseg runs, one warp (CTA) each, which exchange one summary
// each through tagged records.  Used when there are at least as many
// columns as SMs (wkv_abi.cu).
constexpr int kSeqChannels = 32;
constexpr int kSeqMaxRuns = 32;  // runs per column

// Chunks per item of the chained forward walk (one stage and one TMA box
// per array): two for 2-byte elements (a box row of 32 channels is then 128
// bytes), one for 4-byte ones.
__host__ __device__ constexpr int chain_chunks(size_t elem_bytes) { return elem_bytes == 2 ? 2 : 1; }

struct SeqFwdArgs {
  CUtensorMap tk, tv;    // box {32, kChunk, 1} (when use_tma)
  CUtensorMap tk2, tv2;  // box {32, chain_chunks(element size) * kChunk, 1}: the chained walk's items
  const float* w;
  const float* u;
  const void* k;
  const void* v;
  float* y;               // may be null (state-only pass)
  const void* r;          // [B, T, C] of the k, v type, or null: y = sigmoid(r) wkv (the gated output)
  float* ckpt;            // [3][nchunks][B][C] state after each chunk
  const float* state_in;  // [3][B][C] state before the first token (num, den, pp planes); null: empty
  float* state_out;       // [3][B][C] state after the last token; may be null
  Rec* recs;              // [nseg][B][C] run summaries (tagged records)
  unsigned int* exited;   // CTAs of this launch that have finished (in a workspace header)
  WsHeader* eh;
  ScanGeometry g;
  uint64_t budget_ns;
  int nseg;               // runs per column: in, an upper bound (0: none); out, the runs launched
  int debug_skip_chunk;   // -1: off; else the run holding this chunk never publishes its summary
  int chain;              // 0: runs exchange summaries; > 0: chained runs of this many chunks (set by the launcher)
  int use_tma;
};

struct SeqBwdArgs {
  CUtensorMap tk, tv, tg, tr;  // tr: of r (gated launches)
  const float* w;
  const float* u;
  const void* k;   // k, v, gy, r: float or bf16 (kv_dtype of the launch)
  const void* v;
  const void* gy;  // with r: the gradient of the gated output sigmoid(r) wkv
  const void* r;   // null: ungated
  const float* ckpt;
  const float* state_in;    // [3][B][C] state before the first token, or null (empty)
  const float* gstate_end;  // [3][B][C] gradient of the last state's num, den at the given pp, or null
  float* gstate_in;         // [3][B][C] out: gradient of state_in's num, den, and state_in's pp; or null
  float* gk;
  float* gv;
  float* gr;       // [B, T, C] (gated launches)
  float* part;            // [2][nseg * B][C] gw, gu sums per (run, batch row)
  Rec* recs;              // [nseg][B][C] run summaries (tagged records)
  unsigned int* exited;
  WsHeader* eh;
  ScanGeometry g;
  uint64_t budget_ns;
  int nseg;               // as for the forward pass
  int debug_skip_chunk;
  int use_tma;
};

// Choose the runs per column (written to a.nseg) and launch; a.r non-null
// selects the gated kernels.
cudaError_t launch_seq_forward(SeqFwdArgs& a, int kv_dtype, bool write_y, cudaStream_t s);
cudaError_t launch_seq_backward(SeqBwdArgs& a, int kv_dtype, cudaStream_t s);

// Token shift of the training path (wkv_shift.cu).
struct ShiftArgs {
  const float *x, *x0, *mu_k, *mu_v, *mu_r;  // x [B, T, C]; x0 [B, C] or null (zeros); mu [C]
  float *xk, *xv, *xr;                        // forward outputs [B, T, C]
  const float *gxk, *gxv, *gxr;               // backward inputs [B, T, C]
  float *gx, *gx0, *gmu_k, *gmu_v, *gmu_r;    // backward outputs; gx0 may be null
  float* part;                                // [nslice][3][C] per-slice gmu sums
  int B, T, C, nslice;
};

// CTAs of `threads` threads for a grid-stride kernel over `items` items: at
// most 8 per SM of the current device (wkv_shift.cu).
int elementwise_grid(int64_t items, int threads);

// Row slices of the backward pass (a function of the shape only).
int shift_slices(int B, int T, int C, bool vec4);
cudaError_t launch_shift_forward(const ShiftArgs& a, bool vec4, cudaStream_t s);
cudaError_t launch_shift_backward(const ShiftArgs& a, bool vec4, cudaStream_t s);

// Pointwise parts of channel mixing (wkv_cmix.cu), elementwise over n:
// op 0 a = max(k, 0)^2 (x = k; o1 = a); op 1 gk = 2 max(k, 0) ga (x = k,
// y = ga; o1 = gk); op 2 out = sigmoid(r) vk (x = r, y = vk; o1 = out);
// op 3 gvk = gout sigmoid(r), gr = gvk (1 - sigmoid(r)) vk (x = r, y = vk,
// z = gout; o1 = gr, o2 = gvk).
struct CmixArgs {
  const float *x, *y, *z;
  float *o1, *o2;
  int64_t n;
};
cudaError_t launch_cmix(int op, const CmixArgs& a, cudaStream_t s);

// The state after n consecutive segments (wkv_state.cu): states [n][3][B][C]
// (each segment's own state), len[i] segment i's tokens, out [3][B][C].
constexpr int kMaxFoldSegments = 256;
struct FoldArgs {
  const float* w;
  const float* states;
  float* out;
  int B, C, n;
  long long len[kMaxFoldSegments];
};
cudaError_t launch_state_fold(const FoldArgs& a, cudaStream_t s);

// Start-state gradients of consecutive segments (each with a zero gradient
// on its end state), folded last to first after the gradient on the last
// segment's end state (gend, or null): the start-state gradient of the first.
struct AdjFoldArgs {
  const float* w;
  const float* adj;   // [n][3][B][C] planes (g_num, g_den, pp)
  const float* gend;  // [3][B][C] or null
  float* out;         // [3][B][C]
  int B, C, n;
  long long len[kMaxFoldSegments];
};
cudaError_t launch_adjoint_fold(const AdjFoldArgs& a, cudaStream_t s);

// Grid of a persistent scan kernel: resident CTAs per SM x SMs, at most ntiles.
cudaError_t launch_forward(FwdArgs& a, int kv_dtype, bool write_y, cudaStream_t s);
cudaError_t launch_backward(BwdArgs& a, cudaStream_t s);
cudaError_t launch_reduce(const ReduceArgs& a, cudaStream_t s);
// token_dtype: 0 fp32 token inputs, 1 bf16.
cudaError_t launch_decode(const DecodeArgs& a, bool vec4, int token_dtype, cudaStream_t s);

// Row slices of the gw/gu reduction for `rows` partial rows over C channels
// (a function of the shape only, so the summation order is fixed).
int reduce_slices(int rows, int C);

}  // namespace wkv
