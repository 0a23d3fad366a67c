// CUDA-core MXFP8 GEMM: the portable path of C = A' B'^T for MX operands, used where the
// tensor-core kernel does not apply (and as its cross-check). Operands are decoded to fp32
// exactly (E4M3 * 2^s is representable in fp32) in shared memory, 64x64 output tile per CTA,
// 4x4 outputs per thread, fp32 accumulation.
//
// Two epilogues:
//  * kStore:  c = bf16(acc (+ residual))
//  * kSwiGLU: the B tile is 32 gate rows (j0..j0+31) and the matching 32 up rows
//    (d_ff+j0..), so each CTA holds g and u of one 32-wide d_ff block for 64 tokens and
//    emits h = silu(g) * u re-quantised to MXFP8 ([S2.1] "Kernel Benchmark Results": the
//    SwiGLU is fused into the down projection's activation quantisation; no bf16 h exists).
#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"

namespace mxg {

namespace {
constexpr int kBM = 64, kBN = 64, kBK = 32;

__device__ __forceinline__ float ue8m0_value(uint8_t s) {
  // 2^(s-127); s = 0 is the fp32 subnormal 2^-127
  return s == 0 ? __uint_as_float(0x00400000u) : __uint_as_float((uint32_t)s << 23);
}

// Decode 8 E4M3 bytes (little-endian in w) times the block scale into v[0..7].
__device__ __forceinline__ void decode8(uint2 w, float sc, float (&v)[8]) {
  const uint32_t x[2] = {w.x, w.y};
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float2 a = e4m3x2_to_f32x2((uint16_t)(x[i] & 0xFFFF));
    const float2 b = e4m3x2_to_f32x2((uint16_t)(x[i] >> 16));
    v[4 * i + 0] = a.x * sc;
    v[4 * i + 1] = a.y * sc;
    v[4 * i + 2] = b.x * sc;
    v[4 * i + 3] = b.y * sc;
  }
}
}  // namespace

enum { kStore = 0, kSwiGLU = 1 };

template <int EPI>
__global__ void __launch_bounds__(256) mx_gemm_simt_kernel(const uint8_t* __restrict__ aq,
                                                           const uint8_t* __restrict__ as,
                                                           const uint8_t* __restrict__ bq,
                                                           const uint8_t* __restrict__ bs, int M, int N, int K,
                                                           const uint16_t* __restrict__ res,
                                                           uint16_t* __restrict__ c, int d_ff,
                                                           uint8_t* __restrict__ hq, uint8_t* __restrict__ hs) {
  __shared__ float As[kBK][kBM + 4];
  __shared__ float Bs[kBK][kBN + 4];
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x;
  const int m0 = blockIdx.y * kBM;
  const int n0 = blockIdx.x * kBN;
  const int ty = tid >> 4, tx = tid & 15;
  const int KB = K >> 5;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

  // loader mapping: thread -> tile row (tid/4), 8 bytes of the 32-byte k-slice
  const int lr = tid >> 2, lk = (tid & 3) * 8;
  const int am = m0 + lr;
  int64_t brow;  // weight row feeding tile column lr
  if (EPI == kSwiGLU) {
    const int j0 = blockIdx.x * 32;
    brow = lr < 32 ? (int64_t)(j0 + lr) : (int64_t)(d_ff + j0 + lr - 32);
  } else {
    brow = n0 + lr;
  }
  const bool bvalid = EPI == kSwiGLU ? true : (n0 + lr < N);

  for (int k0 = 0; k0 < K; k0 += kBK) {
    float v[8];
    if (am < M) {
      const uint2 w = *reinterpret_cast<const uint2*>(aq + (int64_t)am * K + k0 + lk);
      decode8(w, ue8m0_value(as[(int64_t)am * KB + (k0 >> 5)]), v);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = 0.f;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) As[lk + i][lr] = v[i];
    if (bvalid) {
      const uint2 w = *reinterpret_cast<const uint2*>(bq + brow * K + k0 + lk);
      decode8(w, ue8m0_value(bs[brow * KB + (k0 >> 5)]), v);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = 0.f;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) Bs[lk + i][lr] = v[i];
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < kBK; ++kk) {
      const float4 a = *reinterpret_cast<const float4*>(&As[kk][ty * 4]);
      const float4 b = *reinterpret_cast<const float4*>(&Bs[kk][tx * 4]);
      const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }

  if (EPI == kStore) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int m = m0 + ty * 4 + i;
      if (m >= M) continue;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int n = n0 + tx * 4 + j;
        if (n >= N) continue;
        float y = acc[i][j];
        if (res) y += __bfloat162float(__ushort_as_bfloat16(res[(int64_t)m * N + n]));
        c[(int64_t)m * N + n] = __bfloat16_as_ushort(__float2bfloat16_rn(y));
      }
    }
  } else {
    // stage g | u for the 64 tokens in shared memory (reusing As/Bs), then one warp per row
    float* Cs = &As[0][0];  // needs 64 x 65 floats = 16.6 KB <= As + Bs (17.4 KB)
    static_assert(sizeof(As) + sizeof(Bs) >= 64 * 65 * sizeof(float), "staging does not fit");
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) Cs[(ty * 4 + i) * 65 + tx * 4 + j] = acc[i][j];
    __syncthreads();
    const int warp = tid >> 5, lane = tid & 31;
    const int j0 = blockIdx.x * 32;
    for (int r = warp; r < kBM; r += 8) {
      const int m = m0 + r;
      if (m >= M) break;
      const float g = Cs[r * 65 + lane], u = Cs[r * 65 + 32 + lane];
      const float h = silu_mul(g, u);
      float a = fabsf(h);
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) a = fmaxf(a, __shfl_xor_sync(MXG_FULL_MASK, a, off));
      const int s = mx_shared_exp(a);
      hq[(int64_t)m * d_ff + j0 + lane] = (uint8_t)(cvt_e4m3x2(h * mx_inv_scale(s), 0.f) & 0xFF);
      if (lane == 0) hs[(int64_t)m * (d_ff >> 5) + (j0 >> 5)] = (uint8_t)(s + 127);
    }
  }
}

cudaError_t launch_mx_gemm_simt(const uint8_t* aq, const uint8_t* as, const uint8_t* bq, const uint8_t* bs,
                                int64_t M, int64_t N, int64_t K, const uint16_t* res, uint16_t* c, cudaStream_t st) {
  dim3 grid((unsigned)((N + kBN - 1) / kBN), (unsigned)((M + kBM - 1) / kBM));
  return launch_k(mx_gemm_simt_kernel<kStore>, grid, dim3(256), 0, st, 1, aq, as, bq, bs, (int)M, (int)N, (int)K, res,
                  c, 0, static_cast<uint8_t*>(nullptr), static_cast<uint8_t*>(nullptr));
}

cudaError_t launch_gate_up_swiglu_simt(const uint8_t* xq, const uint8_t* xs, int64_t M, int64_t d_model,
                                       int64_t d_ff, const uint8_t* w13q, const uint8_t* w13s, uint8_t* hq,
                                       uint8_t* hs, cudaStream_t st) {
  dim3 grid((unsigned)(d_ff / 32), (unsigned)((M + kBM - 1) / kBM));
  return launch_k(mx_gemm_simt_kernel<kSwiGLU>, grid, dim3(256), 0, st, 1, xq, xs, w13q, w13s, (int)M, (int)(2 * d_ff),
                  (int)d_model, static_cast<const uint16_t*>(nullptr), static_cast<uint16_t*>(nullptr), (int)d_ff, hq, hs);
}

}  // namespace mxg
