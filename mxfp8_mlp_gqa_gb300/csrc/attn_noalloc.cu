// gqa_decode_attn_noalloc: the split-KV decode attention of gqa_decode_attn, with its scratch
// (the per-split partial outputs and log-sum-exp values) held in a fixed device array that the
// library owns, so the caller passes no workspace and nothing is ever allocated.
//
// Why it exists: some callers cannot allocate device memory at the point where they run
// attention -- code that runs while a CUDA graph is being captured (cudaMalloc is not allowed
// there), real-time decode threads that must never block in an allocator, and host
// applications that own the whole device-memory budget and forbid plugins from allocating.
// They cannot size and hand over a workspace for every batch shape, so this entry point uses
// a static array instead.
//
// Scratch: kNoAllocScratchBytes (8 MiB) in a file-scope __device__ array. Every GPU that loads
// the library keeps it until the process exits. All calls share it and it keeps the last
// call's contents (no kernel here needs it zeroed: every partial is written before it is
// read). Calls whose kernels overlap on the GPU -- e.g. on two streams without ordering --
// race on the array; order them on one stream.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace mxg {

namespace {

constexpr size_t kNoAllocScratchBytes = 8u << 20;
constexpr int kMaxDevices = 64;

__device__ __align__(256) uint8_t g_attn_scratch[kNoAllocScratchBytes];

// Device address of g_attn_scratch for each device, looked up once per device with that
// device current (the host-side symbol is only a stand-in, never a device address).
void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

cudaError_t scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_attn_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

}  // namespace mxg

using namespace mxg;

extern "C" {

size_t gqa_decode_attn_noalloc_capacity(void) { return kNoAllocScratchBytes; }

mxg_status gqa_decode_attn_noalloc(const void* q, int64_t ld_q, const void* k_cache, const void* v_cache,
                                   const int32_t* kv_len, int64_t bs, int64_t Hq, int64_t Hkv, int64_t D, int64_t cap,
                                   int64_t max_kv_len, float scale, void* out, int32_t* err_flag, void* stream) {
  void* scratch = nullptr;
  if (scratch_for_current_device(&scratch) != cudaSuccess) return MXG_ELAUNCH;
  // the same checks and launch as gqa_decode_attn, with the fixed array as the workspace; a
  // problem whose partials do not fit in it is refused before anything is enqueued
  const mxg_status st = decode_attn_call(q, ld_q, k_cache, v_cache, kv_len, bs, Hq, Hkv, D, cap, max_kv_len, scale,
                                         out, err_flag, scratch, kNoAllocScratchBytes, stream);
  return st == MXG_EWORKSPACE ? MXG_ESCRATCH : st;
}

}  // extern "C"
