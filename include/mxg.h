/*
 * libmxg -- C ABI of the GB300 (sm_103a) kernels for one slow-AR decoder-layer step of
 * Dual-AR TTS decoding: MXFP8 activation quantisation, the MXFP8 SwiGLU MLP, GQA decode
 * attention over the active prefix of a preallocated KV cache, and the prev-tokens window
 * shift.
 *
 * Pages that define the operations (cited by title and section):
 *   [S2.1] "How We Made Our Text-to-Speech API Free: The Inference Engineering Behind
 *          S2.1 Pro" -- sections "FP8 Quantization Strategy", "Kernel Benchmark Results",
 *          "DualAR: S2-Specific Batching Constraints", "What's Open Source".
 *   [FSKV] "Fish Speech KV Cache 推理优化记录" -- §4 (bottleneck: the full cache is passed
 *          although a causal mask exists), §5 (keep the capacity, read only the active
 *          prefix), §7 (review: defining correctness).
 *
 * Conventions shared by every entry point
 *   - Every pointer is a DEVICE pointer unless stated otherwise; the caller owns every
 *     buffer. The library never allocates, frees or synchronises, so each call only
 *     enqueues kernels on `stream` (a cudaStream_t; NULL = the legacy default stream).
 *   - bf16 tensors are IEEE bfloat16 bit patterns (uint16). MXFP8 tensors are two arrays:
 *     `q` = E4M3 bytes [rows, K] row-major and `s` = UE8M0 scale bytes [rows, K/32]
 *     row-major, one scale per 32 consecutive elements along K (OCP MX, 1x32 blocks).
 *     Value of element (r, k) = E4M3(q[r,k]) * 2^(s[r, k/32] - 127).
 *   - Sizes are int64 element counts; strides ("ld") are in elements.
 *   - Host-detectable errors (bad sizes, misalignment, too small a workspace) return a
 *     status and enqueue nothing. Errors only the device can see (a kv_len out of range,
 *     a bounded in-kernel wait that ran out) are written to an optional device int32
 *     `err_flag` (first error code wins; the caller zeroes it) -- no kernel ever traps.
 *   - Launch failures return MXG_ELAUNCH.
 *   - Alignment: every pointer 16-byte aligned; ld values multiples of 8 (bf16) / 16 (bytes).
 *   - Kernels are chained with programmatic dependent launch: a GEMM / MLP call starts copying
 *     its WEIGHT operand (bq/bs of mxfp8_gemm, the W13/W2/Wqkv codes and scales, the RMSNorm
 *     gain) before the previous kernel on the stream has finished, so a weight must not be
 *     written by the kernel that immediately precedes the call on that stream (prepare
 *     weights at setup). Every kernel of the library lets its successor start only after
 *     its own predecessor has completed, so at most two library kernels of a stream are in
 *     flight at once and everything before the immediately preceding kernel is complete.
 *     The decode attention calls (gqa_decode_attn*) likewise read kv_len, and over a
 *     contiguous cache the K/V rows (codes and scales) below kv_len - 1 of each sequence,
 *     before the previous kernel has finished: that kernel may write row kv_len - 1 (the
 *     step's KV append: kv_append*, mxfp8_gemm_qkv_kv_append) but no other row of the prefix
 *     and not kv_len. The library's kernels that write other cache rows or arbitrary bytes
 *     (kv_append_extend*, copy_bytes) let their successor start only after they complete.
 *     Paged cache rows and the page table are read only after the previous kernel completes,
 *     as are all other activations and outputs. Environment variable MXG_PDL=0 turns the
 *     chaining off.
 */
#ifndef MXG_H
#define MXG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MXG_OK = 0,
  MXG_EINVAL = 1,     /* null pointer or invalid scalar argument */
  MXG_ESHAPE = 2,     /* sizes outside what the kernel supports */
  MXG_EALIGN = 3,     /* pointer or stride misaligned */
  MXG_EWORKSPACE = 4, /* workspace too small */
  MXG_ELAUNCH = 5,    /* a CUDA launch failed */
  MXG_ETIMEOUT = 6,   /* device: a bounded wait ran out */
  MXG_EDEVICE = 7,    /* device: an input value out of range (e.g. kv_len) */
  MXG_ENOTSUP = 8,    /* no kernel for this device / configuration */
  MXG_ESCRATCH = 9    /* the problem needs more scratch than the library's fixed device array */
} mxg_status;

/* Static string for a status code (never NULL). */
const char* mxg_status_str(int status);
/* Library ABI version (major*10000 + minor*100 + patch). */
int mxg_version(void);
/* Kernel-path switch for diagnostics and cross-checks: enable != 0 (the default) lets the
 * GEMM / MLP entry points use the tcgen05 tensor-core kernels wherever the shape allows
 * (K % 128 == 0); enable == 0 forces the CUDA-core kernels. Process-wide, not thread-safe;
 * returns the previous setting. */
int mxg_set_tensor_core_path(int enable);
/* Failure-detection test hook. on != 0: until it is called again with 0, the split-KV decode
 * attention kernels (every gqa_decode_attn* entry point) issue no K/V loads, so their
 * consumer warps wait on pipeline stages that nothing fills; each such wait gives up after
 * its bound (2 s), the kernel records MXG_ETIMEOUT in err_flag, writes zeros for the heads it
 * owns and returns -- the device-side wind-down path, exercised without a fault and with no
 * copy in flight. The setting lives in device memory of the current device and is written
 * synchronously (all prior work on the legacy default stream completes first). Returns
 * MXG_OK or MXG_ELAUNCH. Not for production use. */
mxg_status mxg_debug_stall_attn_loads(int on);

/*
 * mxfp8_quantize -- fused activation quantisation + UE8M0 scale pack in one launch
 * ([S2.1] "Kernel Benchmark Results": the fused kernel that quantises activations and
 * packs the UE8M0 scales; "FP8 Quantization Strategy": mxfp8 = 1x32 blocks, OCP UE8M0).
 *   x      bf16 [M, K], row stride ld_x (>= K)
 *   q      E4M3 [M, K] (row-major, dense), s UE8M0 [M, K/32]
 * Per 32-block: s = clamp(floor(log2 max|x|) - 8, -127, 127), q = E4M3_rne_satfinite(x/2^s);
 * an all-zero block gets s = -127. Requires K % 32 == 0.  Bit-exact with the oracle.
 */
mxg_status mxfp8_quantize(const void* x, int64_t M, int64_t K, int64_t ld_x, uint8_t* q, uint8_t* s,
                          void* stream);

/*
 * rmsnorm_mxfp8_quantize -- RMSNorm fused into the activation quantiser (decoder-layer
 * step: RMSNorm -> attention -> RMSNorm -> MLP).
 *   y = bf16( (x * r) * gamma ), r = fp32( 1 / sqrt( mean_fp64(x^2) + eps ) ), products
 *   in fp32, then the MX rule above on y.  x bf16 [M, K] (row stride ld_x), gamma bf16 [K].
 * Requires K % 32 == 0 and K <= 17920.
 */
mxg_status rmsnorm_mxfp8_quantize(const void* x, const void* gamma, float eps, int64_t M, int64_t K, int64_t ld_x,
                                  uint8_t* q, uint8_t* s, void* stream);

/*
 * mxfp8_gemm -- C = A' B'^T (+ residual), both operands MXFP8 along K, fp32 accumulation,
 * bf16 output ([S2.1] "FP8 Quantization Strategy" / "Kernel Benchmark Results": the MXFP8
 * GEMM, square 1024^3..16384^3 and decode shapes).
 *   aq [M, K], as [M, K/32]; bq [N, K], bs [N, K/32] (weights: N = output features)
 *   residual bf16 [M, N] or NULL; c bf16 [M, N]. K % 32 == 0, N % 8 == 0.
 *   workspace: device scratch of mxfp8_gemm_workspace(M, N, K) bytes (may be NULL if 0).
 */
size_t mxfp8_gemm_workspace(int64_t M, int64_t N, int64_t K);
mxg_status mxfp8_gemm(const uint8_t* aq, const uint8_t* as, const uint8_t* bq, const uint8_t* bs, int64_t M,
                      int64_t N, int64_t K, const void* residual, void* c, void* workspace, size_t ws_bytes,
                      void* stream);

/*
 * mlp_gate_up_swiglu_mxfp8 -- the gate/up GEMM with the SwiGLU + re-quantisation epilogue
 * ([S2.1] "Kernel Benchmark Results": SwiGLU fused into the down-GEMM's activation
 * quantisation, so no bf16 intermediate is written): g = X' Wg'^T, u = X' Wu'^T (fp32),
 * h = silu(g) * u (fp32), (hq, hs) = MX(h) along d_ff.
 *   xq [M, d_model], xs [M, d_model/32]
 *   w13q [2*d_ff, d_model], w13s [2*d_ff, d_model/32]: rows 0..d_ff-1 = gate, d_ff.. = up
 *   hq [M, d_ff], hs [M, d_ff/32] (outputs).  d_model % 32 == 0, d_ff % 128 == 0.
 */
mxg_status mlp_gate_up_swiglu_mxfp8(const uint8_t* xq, const uint8_t* xs, int64_t M, int64_t d_model, int64_t d_ff,
                                    const uint8_t* w13q, const uint8_t* w13s, uint8_t* hq, uint8_t* hs,
                                    void* stream);

/*
 * mlp_swiglu_mxfp8 -- the whole Qwen3-4B-shaped SwiGLU MLP ([S2.1] "Kernel Benchmark
 * Results": quantise -> gate/up -> SwiGLU -> quantise -> down): the call above into the
 * workspace, then y = H' W2'^T (+ residual) in bf16.
 *   w2q [d_model, d_ff], w2s [d_model, d_ff/32]; residual bf16 [M, d_model] or NULL;
 *   y bf16 [M, d_model].
 *   workspace: mlp_swiglu_mxfp8_workspace(M, d_model, d_ff) bytes; it holds hq at offset 0
 *   (M*d_ff bytes) and hs right after (M*d_ff/32 bytes), then the down GEMM's scratch.
 */
size_t mlp_swiglu_mxfp8_workspace(int64_t M, int64_t d_model, int64_t d_ff);
mxg_status mlp_swiglu_mxfp8(const uint8_t* xq, const uint8_t* xs, int64_t M, int64_t d_model, int64_t d_ff,
                            const uint8_t* w13q, const uint8_t* w13s, const uint8_t* w2q, const uint8_t* w2s,
                            const void* residual, void* y, void* workspace, size_t ws_bytes, void* stream);

/*
 * gqa_decode_attn -- decode attention with grouped KV heads over the active prefix of a
 * preallocated cache ([FSKV] §5: the cache keeps its capacity; attention reads only
 * K[:, :, :kv_len] / V[:, :, :kv_len]; query head h reads KV head h / (Hq/Hkv) with no
 * head expansion -- [S2.1] "What's Open Source": native GQA by stride-0 K/V broadcast).
 *   q        bf16 [bs, Hq, D] with row stride ld_q elements between sequences (>= Hq*D)
 *   k_cache, v_cache  bf16 [bs, Hkv, cap, D] (contiguous)
 *   kv_len   int32 [bs] on the device: filled prefix length (the decode query is the last
 *            position, so nothing inside the prefix is masked). Positions >= kv_len are
 *            never used and may hold any finite values.
 *   out      bf16 [bs, Hq, D]
 *   max_kv_len  host-side bound on every kv_len (sets the grid; keeps the call capturable)
 *   scale    softmax scale (e.g. 1/sqrt(D))
 *   err_flag device int32 or NULL: MXG_EDEVICE if some kv_len is outside [1, min(cap,
 *            max_kv_len)] (that sequence's output is zeroed), MXG_ETIMEOUT on a wait limit.
 *   workspace gqa_decode_attn_workspace(bs, Hq, Hkv, D, max_kv_len) bytes (split-KV partials).
 * Supported: D in {64, 128}, Hq % Hkv == 0, Hq/Hkv <= 8, cap < 2^31.
 */
size_t gqa_decode_attn_workspace(int64_t bs, int64_t Hq, int64_t Hkv, int64_t D, int64_t max_kv_len);
mxg_status gqa_decode_attn(const void* q, int64_t ld_q, const void* k_cache, const void* v_cache,
                           const int32_t* kv_len, int64_t bs, int64_t Hq, int64_t Hkv, int64_t D, int64_t cap,
                           int64_t max_kv_len, float scale, void* out, int32_t* err_flag, void* workspace,
                           size_t ws_bytes, void* stream);

/*
 * gqa_decode_attn_mxfp8 -- gqa_decode_attn that also writes its output MX-quantised for the
 * O projection (decoder-layer step: attention -> quantise -> O projection), so that no
 * separate quantise launch is needed: oq E4M3 [bs, Hq*D], os UE8M0 [bs, Hq*D/32], the MX
 * rule of mxfp8_quantize applied to the bf16 output (bit-identical to mxfp8_quantize(out)).
 */
mxg_status gqa_decode_attn_mxfp8(const void* q, int64_t ld_q, const void* k_cache, const void* v_cache,
                                 const int32_t* kv_len, int64_t bs, int64_t Hq, int64_t Hkv, int64_t D, int64_t cap,
                                 int64_t max_kv_len, float scale, void* out, uint8_t* oq, uint8_t* os,
                                 int32_t* err_flag, void* workspace, size_t ws_bytes, void* stream);

/*
 * gqa_decode_attn_noalloc -- the same computation, kernels and arguments as gqa_decode_attn,
 * minus the workspace: the split-KV scratch lives in a fixed device array owned by the
 * library. (The pages have no counterpart of this entry point; it is an interface addition.)
 *
 * For callers that cannot allocate device memory where they run attention: code executing
 * while a CUDA graph is being captured (cudaMalloc is not permitted there), real-time decode
 * threads that must not block inside an allocator, and host applications that own the whole
 * device-memory budget and do not let plugins allocate.
 *   - Limit: gqa_decode_attn_noalloc_capacity() bytes (8 MiB) of scratch, i.e. problems with
 *     gqa_decode_attn_workspace(bs, Hq, Hkv, D, max_kv_len) <= 8 MiB (e.g. bs 64, Hq 32, D 128,
 *     max_kv_len up to ~4.2k tokens of split partials); larger problems return MXG_ESCRATCH
 *     and launch nothing. Every GPU that loads the library holds the array until exit.
 *   - Nothing is allocated or freed: no cudaMalloc/cudaFree or allocating library call.
 *   - The first call on a device looks up that device's address of the array (with the device
 *     current); make that first call before any stream capture on the device.
 *   - All calls share the array and it keeps the last call's contents; calls whose kernels
 *     overlap on the GPU (e.g. unordered streams) race on it -- order them on one stream.
 */
size_t gqa_decode_attn_noalloc_capacity(void);
mxg_status gqa_decode_attn_noalloc(const void* q, int64_t ld_q, const void* k_cache, const void* v_cache,
                                   const int32_t* kv_len, int64_t bs, int64_t Hq, int64_t Hkv, int64_t D, int64_t cap,
                                   int64_t max_kv_len, float scale, void* out, int32_t* err_flag, void* stream);

/*
 * mxfp8_gemm_qkv_kv_append -- the QKV projection of a decoder-layer step fused with the KV
 * append ([FSKV] §5, kv_cache.update): qkv = X' Wqkv'^T with X MXFP8 [M, K] and Wqkv MXFP8
 * [(Hq + 2 Hkv) D, K]; columns [0, Hq D) (q) go to qkv bf16 [M, (Hq + 2 Hkv) D], columns of K
 * and V go straight to row kv_len[m]-1 of k_cache / v_cache [M, Hkv, cap, D] (the K/V part of
 * qkv is left unwritten). err_flag: MXG_EDEVICE if some kv_len is outside [1, cap] (that
 * row is skipped). Requires K % 128 == 0, D % 8 == 0 (tensor-core path only).
 */
mxg_status mxfp8_gemm_qkv_kv_append(const uint8_t* xq, const uint8_t* xs, const uint8_t* wq, const uint8_t* ws,
                                    int64_t M, int64_t K, int64_t Hq, int64_t Hkv, int64_t D, void* qkv,
                                    void* k_cache, void* v_cache, const int32_t* kv_len, int64_t cap,
                                    int32_t* err_flag, void* stream);

/*
 * kv_append -- in-place cache update of this step's K/V rows at position kv_len[b]-1
 * ([FSKV] §5, kv_cache.update; kv_len counts the new row: prefill T, i-th decode T+i+1).
 *   k_new, v_new bf16 [bs, Hkv, D] with row stride ld_new elements between sequences.
 *   err_flag as above (MXG_EDEVICE if kv_len[b] is outside [1, cap]; that row is skipped).
 */
mxg_status kv_append(void* k_cache, void* v_cache, const void* k_new, const void* v_new, int64_t ld_new,
                     const int32_t* kv_len, int64_t bs, int64_t Hkv, int64_t D, int64_t cap, int32_t* err_flag,
                     void* stream);

/*
 * gqa_decode_attn_paged -- gqa_decode_attn over paged K/V caches ([S2.1] "What's Open
 * Source": paged decode with native GQA by stride-0 K/V broadcast; [FSKV] §5: only the active
 * prefix is read).
 *   k_pool, v_pool bf16 [num_pages, Hkv, page_size, D] (contiguous): a page holds page_size
 *            consecutive positions of one sequence for all Hkv heads.
 *   block_table int32 [bs, max_pages] on the device: positions [j*page_size, (j+1)*page_size)
 *            of sequence b live in pool page block_table[b*max_pages + j]; only the first
 *            ceil(kv_len[b] / page_size) entries of a row are read.
 *   page_size a multiple of 64; max_kv_len <= max_pages * page_size; the pools hold fewer
 *            than 2^31 rows (num_pages * Hkv * page_size).
 *   err_flag as gqa_decode_attn with capacity max_pages * page_size; also MXG_EDEVICE for a
 *            page id outside [0, num_pages) (that 64-token tile is read as zeros).
 *   q, ld_q, kv_len, out, scale, workspace: as gqa_decode_attn (same workspace size).
 */
mxg_status gqa_decode_attn_paged(const void* q, int64_t ld_q, const void* k_pool, const void* v_pool,
                                 const int32_t* block_table, int64_t max_pages, int64_t page_size, int64_t num_pages,
                                 const int32_t* kv_len, int64_t bs, int64_t Hq, int64_t Hkv, int64_t D,
                                 int64_t max_kv_len, float scale, void* out, int32_t* err_flag, void* workspace,
                                 size_t ws_bytes, void* stream);

/*
 * kv_append_paged -- kv_append into paged pools: the row of position kv_len[b]-1 of sequence
 * b lives in page block_table[b*max_pages + (kv_len[b]-1) / page_size] at offset
 * (kv_len[b]-1) % page_size. Bit-exact copy. err_flag: MXG_EDEVICE for kv_len outside
 * [1, max_pages*page_size] or a page id outside [0, num_pages) (that row is skipped).
 */
mxg_status kv_append_paged(void* k_pool, void* v_pool, const int32_t* block_table, int64_t max_pages,
                           int64_t page_size, int64_t num_pages, const void* k_new, const void* v_new, int64_t ld_new,
                           const int32_t* kv_len, int64_t bs, int64_t Hkv, int64_t D, int32_t* err_flag,
                           void* stream);

/*
 * gqa_decode_attn_kv_mxfp8 -- gqa_decode_attn over an MXFP8 K/V cache ([S2.1] "What's Open
 * Source": MXFP8 FlashAttention, paged decode with native GQA; the MX format of [S2.1] "FP8
 * Quantization Strategy": 1x32 blocks, E4M3 elements, OCP UE8M0 shared exponents).
 *   k_codes, v_codes  E4M3 [bs, Hkv, cap, D] (one byte per element, D contiguous);
 *   k_scales, v_scales UE8M0 [bs, Hkv, cap, D/32]: element d of row t has the value
 *            E4M3(codes[.., t, d]) * 2^(scales[.., t, d/32] - 127), as written by
 *            kv_append_mxfp8 (or mxfp8_quantize of rows of D).
 *   cap a multiple of 16; other arguments, workspace size, errors and the result as
 *   gqa_decode_attn: o = softmax(scale q K^T) V over the dequantised prefix, bf16 out.
 *   Values are finite with block exponents up to 2^71 (scale bytes <= 198); scale bytes of 0
 *   (blocks whose values lie below 2^-118) contribute zero.
 */
mxg_status gqa_decode_attn_kv_mxfp8(const void* q, int64_t ld_q, const uint8_t* k_codes, const uint8_t* k_scales,
                                   const uint8_t* v_codes, const uint8_t* v_scales, const int32_t* kv_len, int64_t bs,
                                   int64_t Hq, int64_t Hkv, int64_t D, int64_t cap, int64_t max_kv_len, float scale,
                                   void* out, int32_t* err_flag, void* workspace, size_t ws_bytes, void* stream);

/*
 * gqa_decode_attn_kv_mxfp8_paged -- gqa_decode_attn_kv_mxfp8 over paged MXFP8 pools:
 * k_codes, v_codes E4M3 [num_pages, Hkv, page_size, D], k_scales, v_scales UE8M0
 * [num_pages, Hkv, page_size, D/32]; block_table, page_size, max_kv_len and err_flag as
 * gqa_decode_attn_paged.
 */
mxg_status gqa_decode_attn_kv_mxfp8_paged(const void* q, int64_t ld_q, const uint8_t* k_codes,
                                         const uint8_t* k_scales, const uint8_t* v_codes, const uint8_t* v_scales,
                                         const int32_t* block_table, int64_t max_pages, int64_t page_size,
                                         int64_t num_pages, const int32_t* kv_len, int64_t bs, int64_t Hq,
                                         int64_t Hkv, int64_t D, int64_t max_kv_len, float scale, void* out,
                                         int32_t* err_flag, void* workspace, size_t ws_bytes, void* stream);

/*
 * kv_append_mxfp8 -- kv_append into an MXFP8 cache: the bf16 rows k_new, v_new [bs, Hkv, D]
 * (row stride ld_new elements between sequences) are MX-quantised along D with the rule of
 * mxfp8_quantize (bit-identical to it) and written at position kv_len[b]-1 of the code and
 * scale arrays laid out as in gqa_decode_attn_kv_mxfp8. D a multiple of 32. err_flag:
 * MXG_EDEVICE for kv_len outside [1, cap] (that row is skipped).
 */
mxg_status kv_append_mxfp8(uint8_t* k_codes, uint8_t* k_scales, uint8_t* v_codes, uint8_t* v_scales,
                           const void* k_new, const void* v_new, int64_t ld_new, const int32_t* kv_len, int64_t bs,
                           int64_t Hkv, int64_t D, int64_t cap, int32_t* err_flag, void* stream);

/*
 * kv_append_mxfp8_paged -- kv_append_mxfp8 into paged MXFP8 pools (layout of
 * gqa_decode_attn_kv_mxfp8_paged, row lookup and errors of kv_append_paged).
 */
mxg_status kv_append_mxfp8_paged(uint8_t* k_codes, uint8_t* k_scales, uint8_t* v_codes, uint8_t* v_scales,
                                 const int32_t* block_table, int64_t max_pages, int64_t page_size, int64_t num_pages,
                                 const void* k_new, const void* v_new, int64_t ld_new, const int32_t* kv_len,
                                 int64_t bs, int64_t Hkv, int64_t D, int32_t* err_flag, void* stream);

/*
 * gqa_prefill_attn -- causal prefill / extend attention with native GQA ([S2.1] "What's Open
 * Source": contiguous prefill and paged prefill (extend); [FSKV] §5: the cache keeps its
 * capacity and only the filled prefix is read). Sequence b's new tokens are rows
 * q_start[b] .. q_start[b+1]-1 of q; their K/V rows are already in the cache (kv_append_extend),
 * so kv_len[b] counts them: new token i of b sits at position kv_len[b] - T_b + i
 * (T_b = q_start[b+1] - q_start[b]) and attends to positions 0 .. that position.
 *   q        bf16 [total_q, Hq, 128], ld_q elements between token rows (>= Hq*128, % 8 == 0).
 *   k_cache, v_cache bf16 [bs, Hkv, cap, 128] (contiguous).
 *   q_start  int32 [bs + 1] on the device, non-decreasing, q_start[bs] <= total_q;
 *   kv_len   int32 [bs] on the device; T_b <= max_q_len and T_b <= kv_len[b] <= cap.
 *   out      bf16 [total_q, Hq, 128] (rows of tokens that belong to no sequence are not written).
 *   D must be 128; Hq/Hkv must divide 128 and be <= 16.
 *   Computed with bf16 products and fp32 accumulation on the tensor cores; P = softmax weights
 *   enter the PV product in bf16 (|error| <= 2^-8 * max|V| + one bf16 step of the output).
 *   err_flag: MXG_EDEVICE for a sequence whose lengths break the rules above (it is skipped);
 *   MXG_ETIMEOUT if a bounded in-kernel wait ran out.
 */
mxg_status gqa_prefill_attn(const void* q, int64_t ld_q, const void* k_cache, const void* v_cache,
                            const int32_t* q_start, const int32_t* kv_len, int64_t bs, int64_t total_q, int64_t Hq,
                            int64_t Hkv, int64_t D, int64_t cap, int64_t max_q_len, float scale, void* out,
                            int32_t* err_flag, void* stream);

/*
 * gqa_prefill_attn_paged -- gqa_prefill_attn over paged pools bf16 [num_pages, Hkv,
 * page_size, 128] with block_table int32 [bs, max_pages] (layout, page_size rule and page-id
 * errors of gqa_decode_attn_paged; capacity max_pages * page_size).
 */
mxg_status gqa_prefill_attn_paged(const void* q, int64_t ld_q, const void* k_pool, const void* v_pool,
                                  const int32_t* block_table, int64_t max_pages, int64_t page_size, int64_t num_pages,
                                  const int32_t* q_start, const int32_t* kv_len, int64_t bs, int64_t total_q,
                                  int64_t Hq, int64_t Hkv, int64_t D, int64_t max_q_len, float scale, void* out,
                                  int32_t* err_flag, void* stream);

/*
 * kv_append_extend -- kv_append of a prefill / extend: row q_start[b] + i of k_new, v_new
 * (bf16 [total_q, Hkv, D], ld_new elements between token rows) goes to position
 * kv_len[b] - T_b + i of sequence b's cache [bs, Hkv, cap, D]. Bit-exact copy; D % 8 == 0.
 * err_flag: MXG_EDEVICE for a sequence with inconsistent lengths (skipped).
 */
mxg_status kv_append_extend(void* k_cache, void* v_cache, const void* k_new, const void* v_new, int64_t ld_new,
                            const int32_t* q_start, const int32_t* kv_len, int64_t bs, int64_t total_q, int64_t Hkv,
                            int64_t D, int64_t cap, int64_t max_q_len, int32_t* err_flag, void* stream);

/*
 * kv_append_extend_paged -- kv_append_extend into paged pools (row lookup and errors of
 * kv_append_paged).
 */
mxg_status kv_append_extend_paged(void* k_pool, void* v_pool, const int32_t* block_table, int64_t max_pages,
                                  int64_t page_size, int64_t num_pages, const void* k_new, const void* v_new,
                                  int64_t ld_new, const int32_t* q_start, const int32_t* kv_len, int64_t bs,
                                  int64_t total_q, int64_t Hkv, int64_t D, int64_t max_q_len, int32_t* err_flag,
                                  void* stream);

/*
 * Block-scaled FP8, the pages' "bsgemm" recipe ([S2.1] "FP8 Quantization Strategy": 128x128
 * block-scaled FP8; "What's Open Source": 1x128 activation x 128x128 weight blocks). Each block
 * has one fp32 scale s = amax / 448 (fp32 division) and E4M3 elements E4M3(x / s) (fp32
 * division, round to nearest even, saturating at +-448); a block with amax 0 has s = 0 and
 * signed-zero elements.
 *
 * bs_quantize_act -- x bf16 [M, K] (row stride ld_x) -> q E4M3 [M, K], s fp32 [M, K/128].
 * bs_quantize_weight -- w bf16 [N, K] (contiguous) -> q E4M3 [N, K], s fp32
 *   [ceil(N/128), K/128] (the last row block may be shorter than 128 rows).
 * Both bit-identical to the rule above; K % 128 == 0.
 */
mxg_status bs_quantize_act(const void* x, int64_t M, int64_t K, int64_t ld_x, uint8_t* q, float* s, void* stream);
mxg_status bs_quantize_weight(const void* w, int64_t N, int64_t K, uint8_t* q, float* s, void* stream);

/*
 * bs_gemm -- out[m][n] = sum over 128-wide K blocks kb of xs[m][kb] * ws[n/128][kb] *
 * (E4M3 xq[m, kb block] . E4M3 wq[n, kb block]), bf16 out [M, N] (contiguous). Operands as
 * produced by bs_quantize_act / bs_quantize_weight (xq [M, K], wq [N, K], contiguous).
 * Products of each block on the tensor cores in fp32, block scales applied in fp32.
 * workspace: bs_gemm_workspace(M, N, K) bytes (0 when K is not split), 16-byte aligned.
 * err_flag: MXG_ETIMEOUT if a bounded in-kernel wait ran out.
 */
size_t bs_gemm_workspace(int64_t M, int64_t N, int64_t K);
mxg_status bs_gemm(const uint8_t* xq, const float* xs, const uint8_t* wq, const float* ws, int64_t M, int64_t N,
                   int64_t K, void* out, void* workspace, size_t ws_bytes, int32_t* err_flag, void* stream);

/*
 * copy_bytes -- dst <- src, n bytes, by a kernel on `stream` (16-byte moves). Plumbing for a
 * decode step fed from the host (not an operation of the pages): either pointer may be
 * page-locked host memory (cudaHostAlloc / cudaMallocHost / registered), which the kernel
 * reads or writes through its device mapping, so a step's small host <-> device transfers run
 * as kernels chained to the step's own (graph-capturable, no copy engine). Device and managed
 * memory are used as they are. Ownership stays with the caller; the regions must not overlap.
 * Errors: MXG_EINVAL for a null pointer, n < 0, or memory the device cannot address (pageable
 * host memory is rejected on the host, never dereferenced); MXG_EALIGN unless both pointers
 * are 16-byte aligned and n % 16 == 0. n == 0 launches nothing.
 */
mxg_status copy_bytes(void* dst, const void* src, int64_t n, void* stream);

/*
 * prev_tokens_shift -- in-place slide of the Dual-AR previous-tokens window ([S2.1]
 * "DualAR: S2-Specific Batching Constraints": prev int32 [bs, W, cw], next_tokens int32
 * [bs, cw], strict shape/dtype contract). prev[b, w] <- prev[b, w+1] for w < W-1 and
 * prev[b, W-1] <- next[b]; frame 0 is the oldest. Bit-exact. W*cw <= 12288.
 */
mxg_status prev_tokens_shift(int32_t* prev, const int32_t* next_tokens, int64_t bs, int64_t W, int64_t cw,
                             void* stream);

#ifdef __cplusplus
}
#endif
#endif /* MXG_H */
