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

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

}  // namespace mxg

using namespace mxg;

extern "C" {

size_t gqa_decode_attn_noalloc_capacity(void) { return kNoAllocScratchBytes; }

mxg_status gqa_decode_attn_noalloc(const void* q, int64_t ld_q, const void* k_cache, const void* v_cache,
                                   const int32_t* kv_len, int64_t bs, int64_t Hq, int64_t Hkv, int64_t D, int64_t cap,
                                   int64_t max_kv_len, float scale, void* out, int32_t* err_flag, void* stream) {
  if (!q || !k_cache || !v_cache || !kv_len || !out) return MXG_EINVAL;
  if (!(scale > 0.f) || !(scale < 1e30f)) return MXG_EINVAL;
  if (bs < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || Hq / Hkv > 8 || (D != 64 && D != 128) || cap <= 0 ||
      max_kv_len <= 0 || ld_q < Hq * D)
    return MXG_ESHAPE;
  if (bs * Hkv * cap >= ((int64_t)1 << 31) || bs * Hkv > 65535 || max_kv_len > ((int64_t)1 << 30)) return MXG_ESHAPE;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) || ld_q % 8) return MXG_EALIGN;
  if (bs == 0) return MXG_OK;
  if (attn_workspace_bytes(bs, Hq, Hkv, D, max_kv_len) > kNoAllocScratchBytes) return MXG_ESCRATCH;
  void* scratch = nullptr;
  if (scratch_for_current_device(&scratch) != cudaSuccess) return MXG_ELAUNCH;
  CUtensorMap tk, tv;
  const uint64_t rows = (uint64_t)(bs * Hkv * cap);
  if (!make_tensor_map_2d(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, k_cache, (uint64_t)D, rows, (uint64_t)D * 2, 64, 64,
                          CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tensor_map_2d(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, v_cache, (uint64_t)D, rows, (uint64_t)D * 2, 64, 64,
                          CU_TENSOR_MAP_SWIZZLE_128B))
    return MXG_ENOTSUP;
  const cudaError_t e = launch_gqa_decode_attn(tk, tv, static_cast<const uint16_t*>(q), ld_q, kv_len, bs, Hq, Hkv, D,
                                               cap, max_kv_len, scale, static_cast<uint16_t*>(out), err_flag, scratch,
                                               (cudaStream_t)stream);
  return e == cudaSuccess ? MXG_OK : MXG_ELAUNCH;
}

}  // extern "C"
