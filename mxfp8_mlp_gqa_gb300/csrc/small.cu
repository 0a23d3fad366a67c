// Small per-step data-movement kernels: the Dual-AR prev-tokens window shift and the KV
// cache append.
#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"

namespace mxg {

// [S2.1] "DualAR: S2-Specific Batching Constraints": prev int32 [bs, W, cw] slides by one
// frame and next_tokens int32 [bs, cw] becomes the newest frame. One CTA per sequence: the
// whole window is read into shared memory before any element is written, so the in-place
// update never reads a value it has already overwritten.
__global__ void __launch_bounds__(256) prev_tokens_shift_kernel(int32_t* __restrict__ prev,
                                                                const int32_t* __restrict__ next, int W, int cw) {
  MXG_TL_SCOPE(kTlShift);
  extern __shared__ int32_t win[];
  pdl_wait();
  MXG_TL_WAITED();
  pdl_trigger();
  const int n = W * cw;
  int32_t* p = prev + (int64_t)blockIdx.x * n;
  const int32_t* nx = next + (int64_t)blockIdx.x * cw;
  for (int i = threadIdx.x; i < n; i += blockDim.x) win[i] = p[i];
  __syncthreads();
  const int keep = n - cw;
  for (int i = threadIdx.x; i < n; i += blockDim.x) p[i] = i < keep ? win[i + cw] : nx[i - keep];
}

// Byte copy by a kernel in 16-byte moves. Either side may be page-locked host memory mapped
// into the device address space (the host entry point resolves the mapping), so a step's small
// host <-> device transfers cost a kernel that PDL chains to its neighbours instead of a
// copy-engine operation with its own start-up latency.
__global__ void __launch_bounds__(256) copy16_kernel(uint4* __restrict__ dst, const uint4* __restrict__ src,
                                                     int64_t n16) {
  MXG_TL_SCOPE(kTlCopy16);
  pdl_wait();
  MXG_TL_WAITED();
  // no early trigger: the bytes may be kv_len or K/V cache rows that the next kernel (decode
  // attention) reads before its own wait, so the successor starts only once this one completes
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n16; i += (int64_t)gridDim.x * blockDim.x)
    dst[i] = src[i];
}

cudaError_t launch_copy16(void* dst, const void* src, int64_t n16, cudaStream_t st) {
  int64_t blocks = (n16 + 255) / 256;
  if (blocks > 4 * 152) blocks = 4 * 152;
  return launch_k(copy16_kernel, dim3((unsigned)blocks), dim3(256), 0, st, 1, static_cast<uint4*>(dst),
                  static_cast<const uint4*>(src), n16);
}

// [FSKV] §5 (kv_cache.update, in place): K/V rows of this step land at position kv_len-1.
// One warp per (sequence, kv head); each lane moves 16 bytes of K and of V. With a page table
// the row is looked up as in the paged attention (a bad page id sets the error flag, no write).
__global__ void __launch_bounds__(256) kv_append_kernel(uint16_t* __restrict__ kc, uint16_t* __restrict__ vc,
                                                        const uint16_t* __restrict__ kn,
                                                        const uint16_t* __restrict__ vn, int64_t ld_new,
                                                        const int32_t* __restrict__ kv_len, int bs, int Hkv, int D,
                                                        int64_t cap, int32_t* err, KvPages pg) {
  MXG_TL_SCOPE(kTlKvAppend);
  pdl_wait();
  MXG_TL_WAITED();
  pdl_trigger();
  const int gw = (int)((blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (gw >= bs * Hkv) return;
  const int b = gw / Hkv, g = gw - b * Hkv;
  const int n = kv_len[b];
  if (n < 1 || (int64_t)n > cap) {
    if (lane == 0 && g == 0) set_error(err, MXG_EDEVICE);
    return;
  }
  int64_t dst = (((int64_t)b * Hkv + g) * cap + (n - 1)) * D;
  if (pg.table) {
    const int page = pg.table[(int64_t)b * pg.max_pages + (n - 1) / pg.page_size];
    if (page < 0 || page >= pg.num_pages) {
      if (lane == 0 && g == 0) set_error(err, MXG_EDEVICE);
      return;
    }
    dst = (((int64_t)page * Hkv + g) * pg.page_size + (n - 1) % pg.page_size) * D;
  }
  const int64_t src = (int64_t)b * ld_new + (int64_t)g * D;
  for (int i = lane * 8; i < D; i += 256) {
    *reinterpret_cast<uint4*>(kc + dst + i) = *reinterpret_cast<const uint4*>(kn + src + i);
    *reinterpret_cast<uint4*>(vc + dst + i) = *reinterpret_cast<const uint4*>(vn + src + i);
  }
}

cudaError_t launch_prev_tokens_shift(int32_t* prev, const int32_t* next, int64_t bs, int64_t W, int64_t cw,
                                     cudaStream_t st) {
  const size_t smem = (size_t)W * cw * sizeof(int32_t);
  return launch_k(prev_tokens_shift_kernel, dim3((unsigned)bs), dim3(256), smem, st, 1, prev, next, (int)W, (int)cw);
}

// kv_append into an MXFP8 cache: the K and V rows of this step are MX-quantised along D ([S2.1]
// "FP8 Quantization Strategy": 1x32 blocks, E4M3 + UE8M0) and land at position kv_len-1.
// One warp per (sequence, kv head); lane i holds element i of each 32-wide block.
__global__ void __launch_bounds__(256) kv_append_mx_kernel(uint8_t* __restrict__ kc, uint8_t* __restrict__ ks,
                                                           uint8_t* __restrict__ vc, uint8_t* __restrict__ vs,
                                                           const uint16_t* __restrict__ kn,
                                                           const uint16_t* __restrict__ vn, int64_t ld_new,
                                                           const int32_t* __restrict__ kv_len, int bs, int Hkv, int D,
                                                           int64_t cap, int32_t* err, KvPages pg) {
  pdl_wait();
  pdl_trigger();
  const int gw = (int)((blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (gw >= bs * Hkv) return;
  const int b = gw / Hkv, g = gw - b * Hkv;
  const int n = kv_len[b];
  if (n < 1 || (int64_t)n > cap) {
    if (lane == 0 && g == 0) set_error(err, MXG_EDEVICE);
    return;
  }
  int64_t row = ((int64_t)b * Hkv + g) * cap + (n - 1);
  if (pg.table) {
    const int page = pg.table[(int64_t)b * pg.max_pages + (n - 1) / pg.page_size];
    if (page < 0 || page >= pg.num_pages) {
      if (lane == 0 && g == 0) set_error(err, MXG_EDEVICE);
      return;
    }
    row = ((int64_t)page * Hkv + g) * pg.page_size + (n - 1) % pg.page_size;
  }
  const int64_t src = (int64_t)b * ld_new + (int64_t)g * D;
  const int nb = D >> 5;
  for (int j = 0; j < nb; ++j) {
    const float kv = __uint_as_float((uint32_t)kn[src + 32 * j + lane] << 16);
    const float vv = __uint_as_float((uint32_t)vn[src + 32 * j + lane] << 16);
    mx_quant_warp_store(kv, kc + row * D + 32 * j + lane, ks + row * nb + j);
    mx_quant_warp_store(vv, vc + row * D + 32 * j + lane, vs + row * nb + j);
  }
}

cudaError_t launch_kv_append(uint16_t* kc, uint16_t* vc, const uint16_t* kn, const uint16_t* vn, int64_t ld_new,
                             const int32_t* kv_len, int64_t bs, int64_t Hkv, int64_t D, int64_t cap, int32_t* err,
                             cudaStream_t st, const KvPages* pages) {
  const int64_t warps = bs * Hkv;
  const int64_t blocks = (warps * 32 + 255) / 256;
  const KvPages pg = pages ? *pages : KvPages{};
  return launch_k(kv_append_kernel, dim3((unsigned)blocks), dim3(256), 0, st, 1, kc, vc, kn, vn, ld_new, kv_len,
                  (int)bs, (int)Hkv, (int)D, cap, err, pg);
}

cudaError_t launch_kv_append_mx(uint8_t* kc, uint8_t* ks, uint8_t* vc, uint8_t* vs, const uint16_t* kn,
                                const uint16_t* vn, int64_t ld_new, const int32_t* kv_len, int64_t bs, int64_t Hkv,
                                int64_t D, int64_t cap, int32_t* err, cudaStream_t st, const KvPages* pages) {
  const int64_t warps = bs * Hkv;
  const int64_t blocks = (warps * 32 + 255) / 256;
  const KvPages pg = pages ? *pages : KvPages{};
  return launch_k(kv_append_mx_kernel, dim3((unsigned)blocks), dim3(256), 0, st, 1, kc, ks, vc, vs, kn, vn, ld_new,
                  kv_len, (int)bs, (int)Hkv, (int)D, cap, err, pg);
}

}  // namespace mxg

MXG_TL_UNIT(small)
