// Internal launchers shared between the kernel translation units and the C ABI layer.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "mxg.h"

namespace mxg {

cudaError_t launch_mxfp8_quantize(const uint16_t* x, int64_t M, int64_t K, int64_t ld_x, uint8_t* q, uint8_t* s,
                                  cudaStream_t st);
cudaError_t launch_rmsnorm_mxfp8_quantize(const uint16_t* x, const uint16_t* gamma, float eps, int64_t M, int64_t K,
                                          int64_t ld_x, uint8_t* q, uint8_t* s, cudaStream_t st);

cudaError_t launch_prev_tokens_shift(int32_t* prev, const int32_t* next, int64_t bs, int64_t W, int64_t cw,
                                     cudaStream_t st);
cudaError_t launch_copy16(void* dst, const void* src, int64_t n16, cudaStream_t st);
struct KvPages;
cudaError_t launch_kv_append(uint16_t* kc, uint16_t* vc, const uint16_t* kn, const uint16_t* vn, int64_t ld_new,
                             const int32_t* kv_len, int64_t bs, int64_t Hkv, int64_t D, int64_t cap, int32_t* err,
                             cudaStream_t st, const KvPages* pages = nullptr);

int attn_chunk(int64_t bs, int64_t Hkv, int64_t max_kv_len);
size_t attn_workspace_bytes(int64_t bs, int64_t Hq, int64_t Hkv, int64_t D, int64_t max_kv_len);
// Paged KV caches: pools [num_pages, Hkv, page_size, D]; table [bs, max_pages] of page ids.
struct KvPages {
  const int32_t* table = nullptr;
  int max_pages = 0, page_size = 0;
  int64_t num_pages = 0;
};
cudaError_t launch_gqa_decode_attn(const CUtensorMap& tmK, const CUtensorMap& tmV, const uint16_t* q, int64_t ld_q,
                                   const int32_t* kv_len, int64_t bs, int64_t Hq, int64_t Hkv, int64_t D, int64_t cap,
                                   int64_t max_kv_len, float scale, uint16_t* out, int32_t* err, void* ws,
                                   cudaStream_t st, uint8_t* oq = nullptr, uint8_t* os = nullptr,
                                   const KvPages* pages = nullptr);
// Test hook: on != 0 makes the split-KV decode kernel's copy warp issue no loads (its waits
// then run out: MXG_ETIMEOUT). Synchronous copy to a device variable of the current device.
cudaError_t set_attn_load_stall(int on);
// gqa_decode_attn's host checks, tensor maps and launch (api.cu), for entry points that
// provide the workspace themselves (gqa_decode_attn_noalloc).
mxg_status decode_attn_call(const void* q, int64_t ld_q, const void* k_cache, const void* v_cache,
                            const int32_t* kv_len, int64_t bs, int64_t Hq, int64_t Hkv, int64_t D, int64_t cap,
                            int64_t max_kv_len, float scale, void* out, int32_t* err_flag, void* workspace,
                            size_t ws_bytes, void* stream);
// MXFP8 K/V: tmK/tmV map E4M3 codes [rows, D]; tmKS/tmVS the UE8M0 scales [rows, D/32] as
// 16-byte lines [rows * D/32 / 16, 16].
cudaError_t launch_gqa_decode_attn_kv_mx(const CUtensorMap& tmK, const CUtensorMap& tmV, const CUtensorMap& tmKS,
                                         const CUtensorMap& tmVS, const uint16_t* q, int64_t ld_q,
                                         const int32_t* kv_len, int64_t bs, int64_t Hq, int64_t Hkv, int64_t D,
                                         int64_t cap, int64_t max_kv_len, float scale, uint16_t* out, int32_t* err,
                                         void* ws, cudaStream_t st, const KvPages* pages = nullptr);
// Causal prefill / extend attention (tcgen05, D = 128): tmQ maps q as [total_q, Hq, 128] bf16
// (box {64, G, 128/G}), tmK/tmV the cache rows [rows, 128] bf16 (box {64, 64}, 128-byte swizzle).
cudaError_t launch_gqa_prefill_attn(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                                    const int32_t* q_start, const int32_t* kv_len, int64_t bs, int64_t Hq,
                                    int64_t Hkv, int64_t cap, int64_t total_q, int64_t max_q_len, float scale,
                                    uint16_t* out, int32_t* err, cudaStream_t st, const KvPages* pages = nullptr);
cudaError_t launch_kv_append_extend(uint16_t* kc, uint16_t* vc, const uint16_t* kn, const uint16_t* vn,
                                    int64_t ld_new, const int32_t* q_start, const int32_t* kv_len, int64_t bs,
                                    int64_t Hkv, int64_t D, int64_t cap, int64_t total_q, int64_t max_q_len,
                                    int32_t* err, cudaStream_t st, const KvPages* pages = nullptr);
// Block-scaled FP8 (bsgemm recipe): 1x128 activation and 128x128 weight blocks, fp32 scales.
cudaError_t launch_bs_quantize_act(const uint16_t* x, int64_t M, int64_t K, int64_t ld_x, uint8_t* q, float* s,
                                   cudaStream_t st);
cudaError_t launch_bs_quantize_weight(const uint16_t* w, int64_t N, int64_t K, uint8_t* q, float* s, cudaStream_t st);
size_t bs_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K);
cudaError_t launch_bs_gemm(const uint8_t* xq, const float* xs, const uint8_t* wq, const float* ws, int64_t M,
                           int64_t N, int64_t K, uint16_t* out, void* workspace, int32_t* err, cudaStream_t st);
// kv_append into an MXFP8 cache (codes [.., D] + scales [.., D/32]); the rows are MX-quantised.
cudaError_t launch_kv_append_mx(uint8_t* kc, uint8_t* ks, uint8_t* vc, uint8_t* vs, const uint16_t* kn,
                                const uint16_t* vn, int64_t ld_new, const int32_t* kv_len, int64_t bs, int64_t Hkv,
                                int64_t D, int64_t cap, int32_t* err, cudaStream_t st, const KvPages* pages = nullptr);

cudaError_t launch_mx_gemm_simt(const uint8_t* aq, const uint8_t* as, const uint8_t* bq, const uint8_t* bs,
                                int64_t M, int64_t N, int64_t K, const uint16_t* res, uint16_t* c, cudaStream_t st);
cudaError_t launch_gate_up_swiglu_simt(const uint8_t* xq, const uint8_t* xs, int64_t M, int64_t d_model,
                                       int64_t d_ff, const uint8_t* w13q, const uint8_t* w13s, uint8_t* hq,
                                       uint8_t* hs, cudaStream_t st);

bool tc_gemm_supported(int64_t M, int64_t N, int64_t K);
size_t tc_gemm_workspace(int64_t M, int64_t N, int64_t K);
// Optional fused KV append of a QKV projection: output columns [q_cols, q_cols + Hkv*D) are K
// and the next Hkv*D are V; they are written to the caches at row kv_len[m]-1 instead of `out`.
struct KvScatter {
  int q_cols = 0, Hkv = 0, D = 0;
  int64_t cap = 0;
  uint16_t* kc = nullptr;
  uint16_t* vc = nullptr;
  const int32_t* kv_len = nullptr;
};
cudaError_t launch_mx_gemm_tc(const uint8_t* xq, const uint8_t* xs, const uint8_t* wq, const uint8_t* ws, int64_t M,
                              int64_t N, int64_t K, const uint16_t* residual, uint16_t* out, void* workspace,
                              int32_t* err, cudaStream_t st, bool* unsupported, const KvScatter* kv = nullptr);
cudaError_t launch_gate_up_swiglu_tc(const uint8_t* xq, const uint8_t* xs, int64_t M, int64_t d_model, int64_t d_ff,
                                     const uint8_t* w13q, const uint8_t* w13s, uint8_t* hq, uint8_t* hs, int32_t* err,
                                     cudaStream_t st, bool* unsupported);

// Kernel-path selection: true unless the caller forced the CUDA-core path.
bool tensor_core_path_enabled();

// 2-D row-major tensor map (inner dimension first) for TMA; false if the driver refused it.
bool make_tensor_map_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                        uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz);

}  // namespace mxg
