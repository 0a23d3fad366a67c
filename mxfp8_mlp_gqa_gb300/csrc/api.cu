// C ABI of libmxg: argument checks, workspace sizing and kernel dispatch. Nothing here
// allocates, frees or synchronises; each entry point only enqueues work on `stream`.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace mxg {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_tiled_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline mxg_status launched(cudaError_t e) { return e == cudaSuccess ? MXG_OK : MXG_ELAUNCH; }

int g_tc_path = 1;  // 1: tcgen05 kernels where the shape allows, 0: CUDA-core kernels only

}  // namespace

bool tensor_core_path_enabled() { return g_tc_path != 0; }

bool make_tensor_map_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                        uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz) {
  auto fn = encode_tiled_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D tensor map (innermost dimension first; strides of dimensions 1 and 2 in bytes).
bool make_tensor_map_3d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, const uint64_t (&dims)[3],
                        const uint64_t (&stride_bytes)[2], const uint32_t (&box)[3], CUtensorMapSwizzle swz) {
  auto fn = encode_tiled_fn();
  if (!fn) return false;
  cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
  cuuint64_t st[2] = {stride_bytes[0], stride_bytes[1]};
  cuuint32_t bx[3] = {box[0], box[1], box[2]};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, dt, 3, const_cast<void*>(base), d, st, bx, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace mxg

using namespace mxg;

extern "C" {

const char* mxg_status_str(int s) {
  switch (s) {
    case MXG_OK: return "ok";
    case MXG_EINVAL: return "invalid argument";
    case MXG_ESHAPE: return "unsupported shape";
    case MXG_EALIGN: return "misaligned pointer or stride";
    case MXG_EWORKSPACE: return "workspace too small";
    case MXG_ELAUNCH: return "kernel launch failed";
    case MXG_ETIMEOUT: return "device wait timed out";
    case MXG_EDEVICE: return "device-side input out of range";
    case MXG_ENOTSUP: return "not supported on this device/configuration";
    case MXG_ESCRATCH: return "problem exceeds the fixed scratch of the allocation-free entry point";
    default: return "unknown status";
  }
}

int mxg_version(void) { return 100; }

int mxg_set_tensor_core_path(int enable) {
  const int prev = g_tc_path;
  g_tc_path = enable ? 1 : 0;
  return prev;
}

mxg_status mxg_debug_stall_attn_loads(int on) { return launched(set_attn_load_stall(on)); }

mxg_status mxfp8_quantize(const void* x, int64_t M, int64_t K, int64_t ld_x, uint8_t* q, uint8_t* s, void* stream) {
  if (M < 0 || K <= 0 || K % 32 || ld_x < K) return MXG_ESHAPE;
  if (M == 0) return MXG_OK;  // nothing to read or write (empty tensors may carry null pointers)
  if (!x || !q || !s) return MXG_EINVAL;
  if (!aligned16(x) || !aligned16(q) || ld_x % 8) return MXG_EALIGN;
  return launched(launch_mxfp8_quantize(static_cast<const uint16_t*>(x), M, K, ld_x, q, s, (cudaStream_t)stream));
}

mxg_status rmsnorm_mxfp8_quantize(const void* x, const void* gamma, float eps, int64_t M, int64_t K, int64_t ld_x,
                                  uint8_t* q, uint8_t* s, void* stream) {
  if (!(eps >= 0.f)) return MXG_EINVAL;
  if (M < 0 || K <= 0 || K % 32 || K > 17920 || ld_x < K || M > 0x7fffffff) return MXG_ESHAPE;
  if (M == 0) return MXG_OK;
  if (!x || !gamma || !q || !s) return MXG_EINVAL;
  if (!aligned16(x) || !aligned16(gamma) || !aligned16(q) || ld_x % 8) return MXG_EALIGN;
  return launched(launch_rmsnorm_mxfp8_quantize(static_cast<const uint16_t*>(x), static_cast<const uint16_t*>(gamma),
                                                eps, M, K, ld_x, q, s, (cudaStream_t)stream));
}

size_t mxfp8_gemm_workspace(int64_t M, int64_t N, int64_t K) {
  // sized for the tensor-core plan even when the CUDA-core path is forced, so that a buffer
  // sized once stays valid if the path changes
  return tc_gemm_workspace(M, N, K);
}

mxg_status mxfp8_gemm(const uint8_t* aq, const uint8_t* as, const uint8_t* bq, const uint8_t* bs, int64_t M,
                      int64_t N, int64_t K, const void* residual, void* c, void* workspace, size_t ws_bytes,
                      void* stream) {
  (void)workspace;
  if (M < 0 || N <= 0 || K <= 0 || K % 32 || N % 8 || M > 0x7fffffff || N > 0x7fffffff || K > 0x7fffffff)
    return MXG_ESHAPE;
  if (M == 0) return MXG_OK;
  if (!aq || !as || !bq || !bs || !c) return MXG_EINVAL;
  if (!aligned16(aq) || !aligned16(bq) || !aligned16(c) || (residual && !aligned16(residual))) return MXG_EALIGN;
  const size_t need = mxfp8_gemm_workspace(M, N, K);
  if (ws_bytes < need || (need && !workspace)) return MXG_EWORKSPACE;
  if (need && !aligned16(workspace)) return MXG_EALIGN;
  if (tensor_core_path_enabled() && tc_gemm_supported(M, N, K)) {
    bool unsupported = false;
    cudaError_t e = launch_mx_gemm_tc(aq, as, bq, bs, M, N, K, static_cast<const uint16_t*>(residual),
                                      static_cast<uint16_t*>(c), workspace, nullptr, (cudaStream_t)stream, &unsupported);
    if (!unsupported) return launched(e);
  }
  return launched(launch_mx_gemm_simt(aq, as, bq, bs, M, N, K, static_cast<const uint16_t*>(residual),
                                      static_cast<uint16_t*>(c), (cudaStream_t)stream));
}

mxg_status mlp_gate_up_swiglu_mxfp8(const uint8_t* xq, const uint8_t* xs, int64_t M, int64_t d_model, int64_t d_ff,
                                    const uint8_t* w13q, const uint8_t* w13s, uint8_t* hq, uint8_t* hs,
                                    void* stream) {
  if (M < 0 || d_model <= 0 || d_ff <= 0 || d_model % 32 || d_ff % 128 || M > 0x7fffffff) return MXG_ESHAPE;
  if (M == 0) return MXG_OK;
  if (!xq || !xs || !w13q || !w13s || !hq || !hs) return MXG_EINVAL;
  if (!aligned16(xq) || !aligned16(w13q) || !aligned16(hq)) return MXG_EALIGN;
  if (tensor_core_path_enabled() && d_model % 128 == 0) {
    bool unsupported = false;
    cudaError_t e = launch_gate_up_swiglu_tc(xq, xs, M, d_model, d_ff, w13q, w13s, hq, hs, nullptr,
                                             (cudaStream_t)stream, &unsupported);
    if (!unsupported) return launched(e);
  }
  return launched(launch_gate_up_swiglu_simt(xq, xs, M, d_model, d_ff, w13q, w13s, hq, hs, (cudaStream_t)stream));
}

size_t mlp_swiglu_mxfp8_workspace(int64_t M, int64_t d_model, int64_t d_ff) {
  const size_t h = (size_t)M * (size_t)d_ff;
  size_t off = (h + h / 32 + 255) / 256 * 256;
  return off + mxfp8_gemm_workspace(M, d_model, d_ff);
}

mxg_status mlp_swiglu_mxfp8(const uint8_t* xq, const uint8_t* xs, int64_t M, int64_t d_model, int64_t d_ff,
                            const uint8_t* w13q, const uint8_t* w13s, const uint8_t* w2q, const uint8_t* w2s,
                            const void* residual, void* y, void* workspace, size_t ws_bytes, void* stream) {
  if (M < 0 || d_model <= 0 || d_ff <= 0 || d_model % 32 || d_ff % 128 || M > 0x7fffffff) return MXG_ESHAPE;
  if (M == 0) return MXG_OK;
  if (!xq || !xs || !w13q || !w13s || !w2q || !w2s || !y) return MXG_EINVAL;
  if (!workspace || ws_bytes < mlp_swiglu_mxfp8_workspace(M, d_model, d_ff)) return MXG_EWORKSPACE;
  if (!aligned16(workspace)) return MXG_EALIGN;
  uint8_t* hq = static_cast<uint8_t*>(workspace);
  uint8_t* hs = hq + M * d_ff;
  const size_t off = ((size_t)M * d_ff + (size_t)M * d_ff / 32 + 255) / 256 * 256;
  mxg_status st = mlp_gate_up_swiglu_mxfp8(xq, xs, M, d_model, d_ff, w13q, w13s, hq, hs, stream);
  if (st != MXG_OK) return st;
  return mxfp8_gemm(hq, hs, w2q, w2s, M, d_model, d_ff, residual, y, static_cast<uint8_t*>(workspace) + off,
                    ws_bytes - off, stream);
}

size_t gqa_decode_attn_workspace(int64_t bs, int64_t Hq, int64_t Hkv, int64_t D, int64_t max_kv_len) {
  if (bs <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || max_kv_len <= 0) return 0;
  return attn_workspace_bytes(bs, Hq, Hkv, D, max_kv_len);
}

namespace {

mxg_status attn_call(const void* q, int64_t ld_q, const void* k_cache, const void* v_cache, const int32_t* kv_len,
                     int64_t bs, int64_t Hq, int64_t Hkv, int64_t D, int64_t cap, int64_t max_kv_len, float scale,
                     void* out, uint8_t* oq, uint8_t* os, int32_t* err_flag, void* workspace, size_t ws_bytes,
                     void* stream, const KvPages* pages = nullptr) {
  if (!q || !k_cache || !v_cache || !kv_len || !out) return MXG_EINVAL;
  if (!(scale > 0.f) || !(scale < 1e30f)) return MXG_EINVAL;
  if (bs < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || Hq / Hkv > 8 || (D != 64 && D != 128) || cap <= 0 ||
      max_kv_len <= 0 || ld_q < Hq * D)
    return MXG_ESHAPE;
  // TMA row coordinates are 32-bit: the cache (or page pool) has < 2^31 rows
  const int64_t rows_total = pages ? pages->num_pages * Hkv * pages->page_size : bs * Hkv * cap;
  if (rows_total >= ((int64_t)1 << 31) || bs * Hkv > 65535 || max_kv_len > ((int64_t)1 << 30)) return MXG_ESHAPE;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) || ld_q % 8) return MXG_EALIGN;
  if (bs == 0) return MXG_OK;
  const size_t need = attn_workspace_bytes(bs, Hq, Hkv, D, max_kv_len);
  if (need && (!workspace || ws_bytes < need)) return MXG_EWORKSPACE;
  if (need && !aligned16(workspace)) return MXG_EALIGN;
  CUtensorMap tk, tv;
  const uint64_t rows = (uint64_t)rows_total;
  if (!make_tensor_map_2d(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, k_cache, (uint64_t)D, rows, (uint64_t)D * 2, 64, 64,
                          CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tensor_map_2d(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, v_cache, (uint64_t)D, rows, (uint64_t)D * 2, 64, 64,
                          CU_TENSOR_MAP_SWIZZLE_128B))
    return MXG_ENOTSUP;
  return launched(launch_gqa_decode_attn(tk, tv, static_cast<const uint16_t*>(q), ld_q, kv_len, bs, Hq, Hkv, D, cap,
                                         max_kv_len, scale, static_cast<uint16_t*>(out), err_flag, workspace,
                                         (cudaStream_t)stream, oq, os, pages));
}

// Decode attention over an MXFP8 K/V cache (codes [rows, D] E4M3, scales [rows, D/32] UE8M0).
mxg_status attn_kv_mx_call(const void* q, int64_t ld_q, const uint8_t* kc, const uint8_t* ks, const uint8_t* vc,
                           const uint8_t* vs, const int32_t* kv_len, int64_t bs, int64_t Hq, int64_t Hkv, int64_t D,
                           int64_t cap, int64_t max_kv_len, float scale, void* out, int32_t* err_flag,
                           void* workspace, size_t ws_bytes, void* stream, const KvPages* pages = nullptr) {
  if (!q || !kc || !ks || !vc || !vs || !kv_len || !out) return MXG_EINVAL;
  if (!(scale > 0.f) || !(scale < 1e30f)) return MXG_EINVAL;
  if (bs < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || Hq / Hkv > 8 || (D != 64 && D != 128) || cap <= 0 ||
      max_kv_len <= 0 || ld_q < Hq * D)
    return MXG_ESHAPE;
  // scales are copied as 16-byte lines: a (b, g) row block must start on one (cap % 16 == 0)
  if (!pages && cap % 16) return MXG_ESHAPE;
  const int64_t rows_total = pages ? pages->num_pages * Hkv * pages->page_size : bs * Hkv * cap;
  if (rows_total >= ((int64_t)1 << 31) || bs * Hkv > 65535 || max_kv_len > ((int64_t)1 << 30)) return MXG_ESHAPE;
  if (!aligned16(q) || !aligned16(kc) || !aligned16(ks) || !aligned16(vc) || !aligned16(vs) || !aligned16(out) ||
      ld_q % 8)
    return MXG_EALIGN;
  if (bs == 0) return MXG_OK;
  const size_t need = attn_workspace_bytes(bs, Hq, Hkv, D, max_kv_len);
  if (need && (!workspace || ws_bytes < need)) return MXG_EWORKSPACE;
  if (need && !aligned16(workspace)) return MXG_EALIGN;
  const uint64_t rows = (uint64_t)rows_total;
  const uint64_t lines = rows * (uint64_t)(D / 32) / 16;
  const CUtensorMapSwizzle swz = D == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  const uint32_t sbox = (uint32_t)(64 * (D / 32) / 16);
  CUtensorMap tk, tv, tks, tvs;
  if (!make_tensor_map_2d(&tk, CU_TENSOR_MAP_DATA_TYPE_UINT8, kc, (uint64_t)D, rows, (uint64_t)D, (uint32_t)D, 64,
                          swz) ||
      !make_tensor_map_2d(&tv, CU_TENSOR_MAP_DATA_TYPE_UINT8, vc, (uint64_t)D, rows, (uint64_t)D, (uint32_t)D, 64,
                          swz) ||
      !make_tensor_map_2d(&tks, CU_TENSOR_MAP_DATA_TYPE_UINT8, ks, 16, lines, 16, 16, sbox,
                          CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !make_tensor_map_2d(&tvs, CU_TENSOR_MAP_DATA_TYPE_UINT8, vs, 16, lines, 16, 16, sbox,
                          CU_TENSOR_MAP_SWIZZLE_NONE))
    return MXG_ENOTSUP;
  return launched(launch_gqa_decode_attn_kv_mx(tk, tv, tks, tvs, static_cast<const uint16_t*>(q), ld_q, kv_len, bs,
                                               Hq, Hkv, D, cap, max_kv_len, scale, static_cast<uint16_t*>(out),
                                               err_flag, workspace, (cudaStream_t)stream, pages));
}

mxg_status kv_append_mx_call(uint8_t* kc, uint8_t* ks, uint8_t* vc, uint8_t* vs, const void* k_new,
                             const void* v_new, int64_t ld_new, const int32_t* kv_len, int64_t bs, int64_t Hkv,
                             int64_t D, int64_t cap, int32_t* err_flag, void* stream, const KvPages* pages) {
  if (!kc || !ks || !vc || !vs || !k_new || !v_new || !kv_len) return MXG_EINVAL;
  if (bs < 0 || Hkv <= 0 || D <= 0 || D % 32 || D > 1024 || cap <= 0 || ld_new < Hkv * D || bs * Hkv > (1 << 26))
    return MXG_ESHAPE;
  if (!aligned16(k_new) || !aligned16(v_new) || ld_new % 8) return MXG_EALIGN;
  if (bs == 0) return MXG_OK;
  return launched(launch_kv_append_mx(kc, ks, vc, vs, static_cast<const uint16_t*>(k_new),
                                      static_cast<const uint16_t*>(v_new), ld_new, kv_len, bs, Hkv, D, cap, err_flag,
                                      (cudaStream_t)stream, pages));
}

// Causal prefill / extend attention (D = 128) over contiguous caches or paged pools.
mxg_status prefill_call(const void* q, int64_t ld_q, const void* k_cache, const void* v_cache,
                        const int32_t* q_start, const int32_t* kv_len, int64_t bs, int64_t total_q, int64_t Hq,
                        int64_t Hkv, int64_t D, int64_t cap, int64_t max_q_len, float scale, void* out,
                        int32_t* err_flag, void* stream, const KvPages* pages = nullptr) {
  if (!q || !k_cache || !v_cache || !q_start || !kv_len || !out) return MXG_EINVAL;
  if (!(scale > 0.f) || !(scale < 1e30f)) return MXG_EINVAL;
  if (bs < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || D != 128 || cap <= 0 || total_q < 0 || max_q_len < 0 ||
      ld_q < Hq * D)
    return MXG_ESHAPE;
  const int64_t G = Hq / Hkv;
  if (128 % G || G > 16) return MXG_ESHAPE;
  const int64_t rows_total = pages ? pages->num_pages * Hkv * pages->page_size : bs * Hkv * cap;
  if (rows_total >= ((int64_t)1 << 31) || bs * Hkv > 65535 || total_q >= ((int64_t)1 << 31) ||
      max_q_len > ((int64_t)1 << 30))
    return MXG_ESHAPE;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) || ld_q % 8) return MXG_EALIGN;
  if (bs == 0 || total_q == 0 || max_q_len == 0) return MXG_OK;
  CUtensorMap tq, tk, tv;
  const uint64_t qdims[3] = {(uint64_t)D, (uint64_t)Hq, (uint64_t)total_q};
  const uint64_t qstr[2] = {(uint64_t)D * 2, (uint64_t)ld_q * 2};
  const uint32_t qbox[3] = {64, (uint32_t)G, (uint32_t)(128 / G)};
  if (!make_tensor_map_3d(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, q, qdims, qstr, qbox, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tensor_map_2d(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, k_cache, (uint64_t)D, (uint64_t)rows_total,
                          (uint64_t)D * 2, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tensor_map_2d(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, v_cache, (uint64_t)D, (uint64_t)rows_total,
                          (uint64_t)D * 2, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B))
    return MXG_ENOTSUP;
  return launched(launch_gqa_prefill_attn(tq, tk, tv, q_start, kv_len, bs, Hq, Hkv, cap, total_q, max_q_len, scale,
                                          static_cast<uint16_t*>(out), err_flag, (cudaStream_t)stream, pages));
}

mxg_status append_extend_call(void* k_cache, void* v_cache, const void* k_new, const void* v_new, int64_t ld_new,
                              const int32_t* q_start, const int32_t* kv_len, int64_t bs, int64_t total_q,
                              int64_t Hkv, int64_t D, int64_t cap, int64_t max_q_len, int32_t* err_flag,
                              void* stream, const KvPages* pages = nullptr) {
  if (!k_cache || !v_cache || !k_new || !v_new || !q_start || !kv_len) return MXG_EINVAL;
  if (bs < 0 || Hkv <= 0 || D <= 0 || D % 8 || D > 1024 || cap <= 0 || total_q < 0 || max_q_len < 0 ||
      ld_new < Hkv * D || bs > 65535)
    return MXG_ESHAPE;
  if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_new) || !aligned16(v_new) || ld_new % 8)
    return MXG_EALIGN;
  if (bs == 0 || total_q == 0 || max_q_len == 0) return MXG_OK;
  return launched(launch_kv_append_extend(static_cast<uint16_t*>(k_cache), static_cast<uint16_t*>(v_cache),
                                          static_cast<const uint16_t*>(k_new), static_cast<const uint16_t*>(v_new),
                                          ld_new, q_start, kv_len, bs, Hkv, D, cap, total_q, max_q_len, err_flag,
                                          (cudaStream_t)stream, pages));
}

// The page-table arguments shared by the paged entry points; 0 if valid.
mxg_status check_pages(const int32_t* table, int64_t max_pages, int64_t page_size, int64_t num_pages) {
  if (!table) return MXG_EINVAL;
  if (max_pages <= 0 || num_pages <= 0 || page_size <= 0 || page_size % 64 || max_pages * page_size >= ((int64_t)1 << 31))
    return MXG_ESHAPE;
  return MXG_OK;
}

}  // namespace

}  // extern "C"

namespace mxg {
// The checks, tensor maps and launch of gqa_decode_attn, for other entry points of the library
// that supply the workspace themselves.
mxg_status decode_attn_call(const void* q, int64_t ld_q, const void* k_cache, const void* v_cache,
                            const int32_t* kv_len, int64_t bs, int64_t Hq, int64_t Hkv, int64_t D, int64_t cap,
                            int64_t max_kv_len, float scale, void* out, int32_t* err_flag, void* workspace,
                            size_t ws_bytes, void* stream) {
  return attn_call(q, ld_q, k_cache, v_cache, kv_len, bs, Hq, Hkv, D, cap, max_kv_len, scale, out, nullptr, nullptr,
                   err_flag, workspace, ws_bytes, stream);
}
}  // namespace mxg

extern "C" {

mxg_status gqa_decode_attn(const void* q, int64_t ld_q, const void* k_cache, const void* v_cache,
                           const int32_t* kv_len, int64_t bs, int64_t Hq, int64_t Hkv, int64_t D, int64_t cap,
                           int64_t max_kv_len, float scale, void* out, int32_t* err_flag, void* workspace,
                           size_t ws_bytes, void* stream) {
  return attn_call(q, ld_q, k_cache, v_cache, kv_len, bs, Hq, Hkv, D, cap, max_kv_len, scale, out, nullptr, nullptr,
                   err_flag, workspace, ws_bytes, stream);
}

mxg_status gqa_decode_attn_mxfp8(const void* q, int64_t ld_q, const void* k_cache, const void* v_cache,
                                 const int32_t* kv_len, int64_t bs, int64_t Hq, int64_t Hkv, int64_t D, int64_t cap,
                                 int64_t max_kv_len, float scale, void* out, uint8_t* oq, uint8_t* os,
                                 int32_t* err_flag, void* workspace, size_t ws_bytes, void* stream) {
  if (bs > 0 && (!oq || !os)) return MXG_EINVAL;
  return attn_call(q, ld_q, k_cache, v_cache, kv_len, bs, Hq, Hkv, D, cap, max_kv_len, scale, out, oq, os, err_flag,
                   workspace, ws_bytes, stream);
}

mxg_status gqa_decode_attn_paged(const void* q, int64_t ld_q, const void* k_pool, const void* v_pool,
                                 const int32_t* block_table, int64_t max_pages, int64_t page_size, int64_t num_pages,
                                 const int32_t* kv_len, int64_t bs, int64_t Hq, int64_t Hkv, int64_t D,
                                 int64_t max_kv_len, float scale, void* out, int32_t* err_flag, void* workspace,
                                 size_t ws_bytes, void* stream) {
  const mxg_status c = check_pages(block_table, max_pages, page_size, num_pages);
  if (c != MXG_OK) return c;
  if (max_kv_len > max_pages * page_size) return MXG_ESHAPE;
  KvPages pg;
  pg.table = block_table;
  pg.max_pages = (int)max_pages;
  pg.page_size = (int)page_size;
  pg.num_pages = num_pages;
  return attn_call(q, ld_q, k_pool, v_pool, kv_len, bs, Hq, Hkv, D, max_pages * page_size, max_kv_len, scale, out,
                   nullptr, nullptr, err_flag, workspace, ws_bytes, stream, &pg);
}

mxg_status mxfp8_gemm_qkv_kv_append(const uint8_t* xq, const uint8_t* xs, const uint8_t* wq, const uint8_t* ws,
                                    int64_t M, int64_t K, int64_t Hq, int64_t Hkv, int64_t D, void* qkv,
                                    void* k_cache, void* v_cache, const int32_t* kv_len, int64_t cap,
                                    int32_t* err_flag, void* stream) {
  const int64_t N = (Hq + 2 * Hkv) * D;
  if (M < 0 || K <= 0 || K % 128 || Hq <= 0 || Hkv <= 0 || D <= 0 || D % 8 || cap <= 0 || M > 0x7fffffff ||
      N > 0x7fffffff)
    return MXG_ESHAPE;
  if (M == 0) return MXG_OK;
  if (!xq || !xs || !wq || !ws || !qkv || !k_cache || !v_cache || !kv_len) return MXG_EINVAL;
  if (!aligned16(xq) || !aligned16(wq) || !aligned16(qkv) || !aligned16(k_cache) || !aligned16(v_cache))
    return MXG_EALIGN;
  if (!tc_gemm_supported(M, N, K)) return MXG_ENOTSUP;
  KvScatter kv;
  kv.q_cols = (int)(Hq * D);
  kv.Hkv = (int)Hkv;
  kv.D = (int)D;
  kv.cap = cap;
  kv.kc = static_cast<uint16_t*>(k_cache);
  kv.vc = static_cast<uint16_t*>(v_cache);
  kv.kv_len = kv_len;
  bool unsupported = false;
  const cudaError_t e = launch_mx_gemm_tc(xq, xs, wq, ws, M, N, K, nullptr, static_cast<uint16_t*>(qkv), nullptr,
                                          err_flag, (cudaStream_t)stream, &unsupported, &kv);
  if (unsupported) return MXG_ENOTSUP;
  return launched(e);
}

mxg_status kv_append(void* k_cache, void* v_cache, const void* k_new, const void* v_new, int64_t ld_new,
                     const int32_t* kv_len, int64_t bs, int64_t Hkv, int64_t D, int64_t cap, int32_t* err_flag,
                     void* stream) {
  if (!k_cache || !v_cache || !k_new || !v_new || !kv_len) return MXG_EINVAL;
  if (bs < 0 || Hkv <= 0 || D <= 0 || D % 8 || D > 256 || cap <= 0 || ld_new < Hkv * D || bs * Hkv > (1 << 26))
    return MXG_ESHAPE;
  if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_new) || !aligned16(v_new) || ld_new % 8)
    return MXG_EALIGN;
  if (bs == 0) return MXG_OK;
  return launched(launch_kv_append(static_cast<uint16_t*>(k_cache), static_cast<uint16_t*>(v_cache),
                                   static_cast<const uint16_t*>(k_new), static_cast<const uint16_t*>(v_new), ld_new,
                                   kv_len, bs, Hkv, D, cap, err_flag, (cudaStream_t)stream));
}

mxg_status kv_append_paged(void* k_pool, void* v_pool, const int32_t* block_table, int64_t max_pages,
                           int64_t page_size, int64_t num_pages, const void* k_new, const void* v_new, int64_t ld_new,
                           const int32_t* kv_len, int64_t bs, int64_t Hkv, int64_t D, int32_t* err_flag, void* stream) {
  const mxg_status c = check_pages(block_table, max_pages, page_size, num_pages);
  if (c != MXG_OK) return c;
  if (!k_pool || !v_pool || !k_new || !v_new || !kv_len) return MXG_EINVAL;
  if (bs < 0 || Hkv <= 0 || D <= 0 || D % 8 || D > 256 || ld_new < Hkv * D || bs * Hkv > (1 << 26)) return MXG_ESHAPE;
  if (!aligned16(k_pool) || !aligned16(v_pool) || !aligned16(k_new) || !aligned16(v_new) || ld_new % 8)
    return MXG_EALIGN;
  if (bs == 0) return MXG_OK;
  KvPages pg;
  pg.table = block_table;
  pg.max_pages = (int)max_pages;
  pg.page_size = (int)page_size;
  pg.num_pages = num_pages;
  return launched(launch_kv_append(static_cast<uint16_t*>(k_pool), static_cast<uint16_t*>(v_pool),
                                   static_cast<const uint16_t*>(k_new), static_cast<const uint16_t*>(v_new), ld_new,
                                   kv_len, bs, Hkv, D, max_pages * page_size, err_flag, (cudaStream_t)stream, &pg));
}

mxg_status gqa_decode_attn_kv_mxfp8(const void* q, int64_t ld_q, const uint8_t* k_codes, const uint8_t* k_scales,
                                   const uint8_t* v_codes, const uint8_t* v_scales, const int32_t* kv_len, int64_t bs,
                                   int64_t Hq, int64_t Hkv, int64_t D, int64_t cap, int64_t max_kv_len, float scale,
                                   void* out, int32_t* err_flag, void* workspace, size_t ws_bytes, void* stream) {
  return attn_kv_mx_call(q, ld_q, k_codes, k_scales, v_codes, v_scales, kv_len, bs, Hq, Hkv, D, cap, max_kv_len,
                         scale, out, err_flag, workspace, ws_bytes, stream);
}

mxg_status gqa_decode_attn_kv_mxfp8_paged(const void* q, int64_t ld_q, const uint8_t* k_codes,
                                         const uint8_t* k_scales, const uint8_t* v_codes, const uint8_t* v_scales,
                                         const int32_t* block_table, int64_t max_pages, int64_t page_size,
                                         int64_t num_pages, const int32_t* kv_len, int64_t bs, int64_t Hq,
                                         int64_t Hkv, int64_t D, int64_t max_kv_len, float scale, void* out,
                                         int32_t* err_flag, void* workspace, size_t ws_bytes, void* stream) {
  const mxg_status c = check_pages(block_table, max_pages, page_size, num_pages);
  if (c != MXG_OK) return c;
  if (max_kv_len > max_pages * page_size) return MXG_ESHAPE;
  KvPages pg;
  pg.table = block_table;
  pg.max_pages = (int)max_pages;
  pg.page_size = (int)page_size;
  pg.num_pages = num_pages;
  return attn_kv_mx_call(q, ld_q, k_codes, k_scales, v_codes, v_scales, kv_len, bs, Hq, Hkv, D, max_pages * page_size,
                         max_kv_len, scale, out, err_flag, workspace, ws_bytes, stream, &pg);
}

mxg_status kv_append_mxfp8(uint8_t* k_codes, uint8_t* k_scales, uint8_t* v_codes, uint8_t* v_scales,
                           const void* k_new, const void* v_new, int64_t ld_new, const int32_t* kv_len, int64_t bs,
                           int64_t Hkv, int64_t D, int64_t cap, int32_t* err_flag, void* stream) {
  return kv_append_mx_call(k_codes, k_scales, v_codes, v_scales, k_new, v_new, ld_new, kv_len, bs, Hkv, D, cap,
                           err_flag, stream, nullptr);
}

mxg_status kv_append_mxfp8_paged(uint8_t* k_codes, uint8_t* k_scales, uint8_t* v_codes, uint8_t* v_scales,
                                 const int32_t* block_table, int64_t max_pages, int64_t page_size, int64_t num_pages,
                                 const void* k_new, const void* v_new, int64_t ld_new, const int32_t* kv_len,
                                 int64_t bs, int64_t Hkv, int64_t D, int32_t* err_flag, void* stream) {
  const mxg_status c = check_pages(block_table, max_pages, page_size, num_pages);
  if (c != MXG_OK) return c;
  KvPages pg;
  pg.table = block_table;
  pg.max_pages = (int)max_pages;
  pg.page_size = (int)page_size;
  pg.num_pages = num_pages;
  return kv_append_mx_call(k_codes, k_scales, v_codes, v_scales, k_new, v_new, ld_new, kv_len, bs, Hkv, D,
                           max_pages * page_size, err_flag, stream, &pg);
}

mxg_status gqa_prefill_attn(const void* q, int64_t ld_q, const void* k_cache, const void* v_cache,
                            const int32_t* q_start, const int32_t* kv_len, int64_t bs, int64_t total_q, int64_t Hq,
                            int64_t Hkv, int64_t D, int64_t cap, int64_t max_q_len, float scale, void* out,
                            int32_t* err_flag, void* stream) {
  return prefill_call(q, ld_q, k_cache, v_cache, q_start, kv_len, bs, total_q, Hq, Hkv, D, cap, max_q_len, scale, out,
                      err_flag, stream);
}

mxg_status gqa_prefill_attn_paged(const void* q, int64_t ld_q, const void* k_pool, const void* v_pool,
                                  const int32_t* block_table, int64_t max_pages, int64_t page_size, int64_t num_pages,
                                  const int32_t* q_start, const int32_t* kv_len, int64_t bs, int64_t total_q,
                                  int64_t Hq, int64_t Hkv, int64_t D, int64_t max_q_len, float scale, void* out,
                                  int32_t* err_flag, void* stream) {
  const mxg_status c = check_pages(block_table, max_pages, page_size, num_pages);
  if (c != MXG_OK) return c;
  KvPages pg;
  pg.table = block_table;
  pg.max_pages = (int)max_pages;
  pg.page_size = (int)page_size;
  pg.num_pages = num_pages;
  return prefill_call(q, ld_q, k_pool, v_pool, q_start, kv_len, bs, total_q, Hq, Hkv, D, max_pages * page_size,
                      max_q_len, scale, out, err_flag, stream, &pg);
}

mxg_status kv_append_extend(void* k_cache, void* v_cache, const void* k_new, const void* v_new, int64_t ld_new,
                            const int32_t* q_start, const int32_t* kv_len, int64_t bs, int64_t total_q, int64_t Hkv,
                            int64_t D, int64_t cap, int64_t max_q_len, int32_t* err_flag, void* stream) {
  return append_extend_call(k_cache, v_cache, k_new, v_new, ld_new, q_start, kv_len, bs, total_q, Hkv, D, cap,
                            max_q_len, err_flag, stream);
}

mxg_status kv_append_extend_paged(void* k_pool, void* v_pool, const int32_t* block_table, int64_t max_pages,
                                  int64_t page_size, int64_t num_pages, const void* k_new, const void* v_new,
                                  int64_t ld_new, const int32_t* q_start, const int32_t* kv_len, int64_t bs,
                                  int64_t total_q, int64_t Hkv, int64_t D, int64_t max_q_len, int32_t* err_flag,
                                  void* stream) {
  const mxg_status c = check_pages(block_table, max_pages, page_size, num_pages);
  if (c != MXG_OK) return c;
  KvPages pg;
  pg.table = block_table;
  pg.max_pages = (int)max_pages;
  pg.page_size = (int)page_size;
  pg.num_pages = num_pages;
  return append_extend_call(k_pool, v_pool, k_new, v_new, ld_new, q_start, kv_len, bs, total_q, Hkv, D,
                            max_pages * page_size, max_q_len, err_flag, stream, &pg);
}

mxg_status bs_quantize_act(const void* x, int64_t M, int64_t K, int64_t ld_x, uint8_t* q, float* s, void* stream) {
  if (!x || !q || !s) return MXG_EINVAL;
  if (M < 0 || K <= 0 || K % 128 || ld_x < K || M >= ((int64_t)1 << 31)) return MXG_ESHAPE;
  if (!aligned16(x) || !aligned16(q) || !aligned16(s) || ld_x % 8) return MXG_EALIGN;
  if (M == 0) return MXG_OK;
  return launched(launch_bs_quantize_act(static_cast<const uint16_t*>(x), M, K, ld_x, q, s, (cudaStream_t)stream));
}

mxg_status bs_quantize_weight(const void* w, int64_t N, int64_t K, uint8_t* q, float* s, void* stream) {
  if (!w || !q || !s) return MXG_EINVAL;
  if (N < 0 || K <= 0 || K % 128 || N >= ((int64_t)1 << 31) || (N + 127) / 128 > 65535) return MXG_ESHAPE;
  if (!aligned16(w) || !aligned16(q) || !aligned16(s)) return MXG_EALIGN;
  if (N == 0) return MXG_OK;
  return launched(launch_bs_quantize_weight(static_cast<const uint16_t*>(w), N, K, q, s, (cudaStream_t)stream));
}

size_t bs_gemm_workspace(int64_t M, int64_t N, int64_t K) { return bs_gemm_workspace_bytes(M, N, K); }

mxg_status bs_gemm(const uint8_t* xq, const float* xs, const uint8_t* wq, const float* ws, int64_t M, int64_t N,
                   int64_t K, void* out, void* workspace, size_t ws_bytes, int32_t* err_flag, void* stream) {
  if (!xq || !xs || !wq || !ws || !out) return MXG_EINVAL;
  if (M < 0 || N <= 0 || K <= 0 || K % 128 || M >= ((int64_t)1 << 31) || N >= ((int64_t)1 << 31) ||
      (N + 127) / 128 > 65535)
    return MXG_ESHAPE;
  if (!aligned16(xq) || !aligned16(xs) || !aligned16(wq) || !aligned16(ws) || !aligned16(out)) return MXG_EALIGN;
  if (M == 0) return MXG_OK;
  const size_t need = bs_gemm_workspace_bytes(M, N, K);
  if (need && (!workspace || ws_bytes < need)) return MXG_EWORKSPACE;
  if (need && !aligned16(workspace)) return MXG_EALIGN;
  return launched(launch_bs_gemm(xq, xs, wq, ws, M, N, K, static_cast<uint16_t*>(out), workspace, err_flag,
                                 (cudaStream_t)stream));
}

// The address a kernel may use for `p`: device or managed memory as it is, page-locked host
// memory through its mapping into the device address space; nullptr for anything else
// (pageable host memory is never handed to a kernel).
static const void* device_view(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) return p;
  if (a.type == cudaMemoryTypeHost) return a.devicePointer;
  return nullptr;
}

mxg_status copy_bytes(void* dst, const void* src, int64_t n, void* stream) {
  if (!dst || !src || n < 0) return MXG_EINVAL;
  if (n == 0) return MXG_OK;
  if (n % 16 || !aligned16(dst) || !aligned16(src)) return MXG_EALIGN;
  const void* s = device_view(src);
  const void* d = device_view(dst);
  if (!s || !d || !aligned16(s) || !aligned16(d)) return MXG_EINVAL;
  return launched(launch_copy16(const_cast<void*>(d), s, n / 16, (cudaStream_t)stream));
}

mxg_status prev_tokens_shift(int32_t* prev, const int32_t* next_tokens, int64_t bs, int64_t W, int64_t cw,
                             void* stream) {
  if (!prev || !next_tokens) return MXG_EINVAL;
  if (bs < 0 || W <= 0 || cw <= 0 || W * cw > 12288 || bs > 0x7fffffff) return MXG_ESHAPE;
  if (bs == 0) return MXG_OK;
  return launched(launch_prev_tokens_shift(prev, next_tokens, bs, W, cw, (cudaStream_t)stream));
}

}  // extern "C"
