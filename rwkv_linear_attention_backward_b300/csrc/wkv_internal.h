// wkv_internal.h -- host-side declarations shared by the library's .cu files.
// Not part of the public ABI (that is include/wkv.h).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace wkv {

struct WsHeader;

// Time-chunk length of the chunked scans.  One value for every shape, so the
// chunk-boundary states written by the forward pass line up with the chunks
// of the backward pass.
constexpr int kChunk = 32;
// Channels per CTA of the scan kernels (4 warps x 32 lanes, one channel per
// lane).
constexpr int kCtaChannels = 128;

struct ScanGeometry {
  int B, T, C;
  int nchunks;   // ceil(T / kChunk)
  int ncb;       // ceil(C / kCtaChannels): channel blocks (CTAs) per (chunk, row)
  int nwg;       // ncb * 4: 32-channel groups per row (one flag each per node)
  unsigned int ntiles;  // nchunks * B * ncb
  size_t plane;  // nchunks * B * C: floats per checkpoint plane
  int nnodes;    // nodes of the binary-indexed tree over chunks
  int nlevels;   // levels of that tree (level s holds nchunks >> s nodes)
  int level_off[32];
  size_t nplane; // nnodes * B * C: floats per node plane
};

ScanGeometry make_geometry(int B, int T, int C);

struct FwdArgs {
  const float* w;
  const float* u;
  const void* k;
  const void* v;
  float* y;          // may be null (state-only pass)
  float* nodes;      // [3][nnodes][B][C] tree nodes: (num, den, pp)
  float* incl;       // [3][nchunks][B][C] state after each chunk (checkpoints)
  uint64_t* flags;   // [B][nwg][nnodes]
  unsigned int* ticket;   // tile counter of this launch (in a workspace header)
  WsHeader* eh;           // where an expired wait is recorded (checked by the host)
  ScanGeometry g;
  uint64_t epoch;
  uint64_t budget_ns;
  int debug_skip_chunk;  // -1: off
};

struct BwdArgs {
  const float* w;
  const float* u;
  const float* k;
  const float* v;
  const float* gy;
  const float* ckpt;   // [3][nchunks][B][C] state after each chunk (forward)
  float* gk;
  float* gv;
  float* rnodes;       // [3][nnodes][B][C] tree nodes of the adjoint: (la, lb, exponent)
  float* part;         // [2][nchunks][B][C] per-tile gw, gu partial sums
  uint64_t* flags;     // [B][nwg][nnodes]
  unsigned int* ticket;
  WsHeader* eh;
  ScanGeometry g;
  uint64_t epoch;
  uint64_t budget_ns;
  int debug_skip_chunk;
};

struct ReduceArgs {
  const float* part;  // [2][rows][C]
  float* gw;
  float* gu;
  int rows;           // nchunks * B
  int C;
};

struct DecodeArgs {
  const float *x, *x_prev, *mu_k, *mu_v, *mu_r, *r, *k, *v, *w, *u;
  float *num, *den, *pp, *y, *xk, *xv, *xr;
  int L, B, C;
};

// Sets the text returned by wkv_last_error_string() on this thread.
void set_last_error(const char* msg);

cudaError_t launch_forward(const FwdArgs& a, int kv_dtype, bool write_y, cudaStream_t s);
cudaError_t launch_backward(const BwdArgs& a, cudaStream_t s);
cudaError_t launch_reduce(const ReduceArgs& a, cudaStream_t s);
cudaError_t launch_decode(const DecodeArgs& a, bool vec4, cudaStream_t s);

}  // namespace wkv
