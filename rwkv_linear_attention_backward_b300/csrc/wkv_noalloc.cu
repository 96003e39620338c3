// wkv_noalloc.cu -- a forward pass for callers that cannot allocate device
// memory.
//
// wkv_forward needs a scratch workspace of wkv_forward_workspace_bytes bytes
// from its caller.  Some callers cannot provide one: a plugin or embedded
// host whose device memory belongs to another allocator, or a latency-bound
// loop that must never call cudaMalloc (which can synchronise the device and
// stall every stream).  wkv_forward_noalloc runs the same forward pass with
// its scratch in a fixed array compiled into this library instead.
#include <cstdio>
#include <mutex>

#include "wkv.h"
#include "wkv_common.cuh"
#include "wkv_internal.h"

namespace wkv {

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB

// Scratch of every wkv_forward_noalloc call on a device.  Every GPU that
// loads this library holds it until the process exits.  Zero at load.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};  // device address of the array, per device

// The array's name is only a host-side stand-in in host code; the device
// address comes from the runtime, once per device, with that device current.
wkv_status scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    set_last_error("wkv_forward_noalloc: cudaGetDevice failed");
    return WKV_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    set_last_error("wkv_forward_noalloc: device index out of range");
    return WKV_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      char msg[200];
      std::snprintf(msg, sizeof(msg), "wkv_forward_noalloc: cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
      set_last_error(msg);
      return WKV_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return WKV_OK;
}

}  // namespace

}  // namespace wkv

extern "C" wkv_status wkv_forward_noalloc(int B, int T, int C, int kv_dtype, const float* w, const float* u,
                                          const void* k, const void* v, float* y, float* ckpt, void* stream) {
  using namespace wkv;
  set_last_error("");  // a rejection below must not leave an earlier call's message in place
  if (!w || !u || !k || !v || !y || B <= 0 || T <= 0 || C <= 0) {
    set_last_error("wkv_forward_noalloc: a required pointer is null or a size is not positive");
    return WKV_ERR_INVALID_ARG;
  }
  const size_t need = wkv_forward_workspace_bytes(B, T, C);
  if (need == 0) {
    set_last_error("wkv_forward_noalloc: B * T * C is beyond the sizes the library takes");
    return WKV_ERR_INVALID_ARG;
  }
  if (need > kNoAllocScratchBytes) {
    char msg[200];
    std::snprintf(msg, sizeof(msg),
                  "wkv_forward_noalloc: shape (B=%d, T=%d, C=%d) needs %zu bytes of scratch, the built-in array "
                  "holds %zu; use wkv_forward with a workspace",
                  B, T, C, need, kNoAllocScratchBytes);
    set_last_error(msg);
    return WKV_ERR_WORKSPACE;
  }
  void* scratch = nullptr;
  const wkv_status st = scratch_address(&scratch);
  if (st != WKV_OK) return st;
  // The array keeps the previous call's contents, and nothing in it needs
  // clearing: it is zero when the library loads, every launch leaves its
  // tile counters at zero, and the sequence number in its header must carry
  // on from call to call (the tag of each call's records comes from it, so
  // records of an earlier call never read as current).
  return wkv_forward(B, T, C, kv_dtype, w, u, k, v, y, ckpt, scratch, kNoAllocScratchBytes, stream);
}
