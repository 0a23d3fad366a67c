// Block-scaled FP8 GEMM ("bsgemm" recipe) on the 5th-generation tensor cores.
//
// [S2.1] "FP8 Quantization Strategy" / "What's Open Source": 1x128 activation blocks and
// 128x128 weight blocks, each with its own scale, E4M3 elements. The scales here are fp32
// (s = amax / 448), so they cannot ride on the hardware's power-of-two block scaling: every
// 128-wide K group is its own tcgen05.mma (kind::f8f6f4, plain E4M3 x E4M3 -> fp32 in TMEM)
// and its partial is promoted in registers, acc += s_w * s_x * partial.
//
//  * swap-AB as in the MXFP8 decode GEMM: the 128 weight rows of a tile are the MMA's M
//    side, the tokens (16..128) its N side; the weight tile is exactly one 128-row scale block.
//  * warp 0: TMA ring (128-byte swizzle) of the weight tile and the token tile per K group;
//    warp 1: one thread issues 4 MMAs (K = 32 each) per group into one of two TMEM partial
//    buffers and commits; warps 2-5 (thread = weight row = TMEM lane) read each partial,
//    free its buffer and fold it into fp32 accumulators with the two block scales.
//  * split-K over grid.z when the tiles alone do not cover the SMs: fp32 partial tiles go to
//    a workspace and a second kernel sums them in a fixed order.
// Every wait is bounded (MXG_ETIMEOUT); TMEM is always released.
#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"
#include "tc.cuh"

namespace mxg {

namespace {

using namespace tc;

constexpr int kGK = 128;  // K per group (one activation / weight scale block)

template <int BN>
struct BsShape {
  static constexpr int kABytes = 128 * kGK;
  static constexpr int kBBytes = BN * kGK;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = BN <= 32 ? 6 : BN <= 64 ? 5 : 4;
  static constexpr int kRingBytes = kStages * kStageBytes;
  static constexpr uint32_t kTmemCols = 2 * BN <= 32 ? 32 : 2 * BN <= 64 ? 64 : 2 * BN <= 128 ? 128 : 256;
  // ring | barriers | weight-scale vector [ng] | token-scale table [BN][ng] (fp32)
  static constexpr int kBarOff = kRingBytes;
  static constexpr int kTabOff = kRingBytes + 8 * (2 * kStages + 5) + 16;
  static int smem(int ng) { return 1024 + kTabOff + 4 * ng * (1 + BN); }
};

// kind::f8f6f4 instruction descriptor: E4M3 A and B (format 0), fp32 D (bit 4), both K-major,
// N>>3 at bits 17-22, M>>4 at bits 24-28.
__host__ __device__ constexpr uint32_t idesc_e4m3(int m, int n) {
  return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void mma_e4m3(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

struct BsArgs {
  int M, N, K, groups, splits;
  const float* xs;   // [M][K/128]
  const float* ws;   // [ceil(N/128)][K/128]
  uint16_t* out;     // [M][N] bf16 (splits == 1)
  float* part;       // [splits][M][N] fp32 (splits > 1)
  int32_t* err;
};

__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  return cvt_e4m3x2(a, b) | (cvt_e4m3x2(c, d) << 16);
}

}  // namespace

// ------------------------------------------------------------------------- quantisers
// Activations: one warp per (row, 128-wide block); lane i holds elements 4i .. 4i+3.
__global__ void __launch_bounds__(256) bs_quantize_act_kernel(const uint16_t* __restrict__ x, int64_t M, int64_t K,
                                                              int64_t ld_x, uint8_t* __restrict__ q,
                                                              float* __restrict__ s) {
  pdl_wait();
  pdl_trigger();
  const int64_t gw = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t nb = K / kGK;
  if (gw >= M * nb) return;
  const int64_t m = gw / nb, b = gw - m * nb;
  const uint2 raw = *reinterpret_cast<const uint2*>(x + m * ld_x + b * kGK + 4 * lane);
  const float v0 = bf16_lo(raw.x), v1 = bf16_hi(raw.x), v2 = bf16_lo(raw.y), v3 = bf16_hi(raw.y);
  float am = fmaxf(fmaxf(fabsf(v0), fabsf(v1)), fmaxf(fabsf(v2), fabsf(v3)));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) am = fmaxf(am, __shfl_xor_sync(MXG_FULL_MASK, am, off));
  const float sc = __fdiv_rn(am, 448.f);
  const float d = sc == 0.f ? 1.f : sc;
  *reinterpret_cast<uint32_t*>(q + m * K + b * kGK + 4 * lane) =
      e4m3x4(__fdiv_rn(v0, d), __fdiv_rn(v1, d), __fdiv_rn(v2, d), __fdiv_rn(v3, d));
  if (lane == 0) s[m * nb + b] = sc;
}

// Weights: one CTA (256 threads) per 128 x 128 block; thread t covers row t/2, columns
// 64*(t%2) .. +63 (rows past N are skipped).
__global__ void __launch_bounds__(256) bs_quantize_weight_kernel(const uint16_t* __restrict__ w, int64_t N, int64_t K,
                                                                 uint8_t* __restrict__ q, float* __restrict__ s) {
  __shared__ float red[8];
  pdl_wait();
  pdl_trigger();
  const int64_t kb = blockIdx.x, nb = blockIdx.y;
  const int64_t row = nb * 128 + (threadIdx.x >> 1);
  const int64_t col = kb * kGK + 64 * (threadIdx.x & 1);
  const bool rv = row < N;
  float am = 0.f;
  if (rv) {
    const uint4* src = reinterpret_cast<const uint4*>(w + row * K + col);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint4 u = src[i];
      am = fmaxf(am, fmaxf(fmaxf(fabsf(bf16_lo(u.x)), fabsf(bf16_hi(u.x))), fmaxf(fabsf(bf16_lo(u.y)), fabsf(bf16_hi(u.y)))));
      am = fmaxf(am, fmaxf(fmaxf(fabsf(bf16_lo(u.z)), fabsf(bf16_hi(u.z))), fmaxf(fabsf(bf16_lo(u.w)), fabsf(bf16_hi(u.w)))));
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) am = fmaxf(am, __shfl_xor_sync(MXG_FULL_MASK, am, off));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = am;
  __syncthreads();
  am = red[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) am = fmaxf(am, red[i]);
  const float sc = __fdiv_rn(am, 448.f);
  const float d = sc == 0.f ? 1.f : sc;
  if (threadIdx.x == 0) s[nb * (K / kGK) + kb] = sc;
  if (!rv) return;
  const uint4* src = reinterpret_cast<const uint4*>(w + row * K + col);
  uint4* dst = reinterpret_cast<uint4*>(q + row * K + col);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 a = src[2 * i], b = src[2 * i + 1];
    uint4 o;
    o.x = e4m3x4(__fdiv_rn(bf16_lo(a.x), d), __fdiv_rn(bf16_hi(a.x), d), __fdiv_rn(bf16_lo(a.y), d),
                 __fdiv_rn(bf16_hi(a.y), d));
    o.y = e4m3x4(__fdiv_rn(bf16_lo(a.z), d), __fdiv_rn(bf16_hi(a.z), d), __fdiv_rn(bf16_lo(a.w), d),
                 __fdiv_rn(bf16_hi(a.w), d));
    o.z = e4m3x4(__fdiv_rn(bf16_lo(b.x), d), __fdiv_rn(bf16_hi(b.x), d), __fdiv_rn(bf16_lo(b.y), d),
                 __fdiv_rn(bf16_hi(b.y), d));
    o.w = e4m3x4(__fdiv_rn(bf16_lo(b.z), d), __fdiv_rn(bf16_hi(b.z), d), __fdiv_rn(bf16_lo(b.w), d),
                 __fdiv_rn(bf16_hi(b.w), d));
    dst[i] = o;
  }
}

// ------------------------------------------------------------------------- GEMM
template <int BN>
__global__ void __launch_bounds__(192, 1) bs_gemm_kernel(const __grid_constant__ CUtensorMap tmW,
                                                      const __grid_constant__ CUtensorMap tmX, const BsArgs a) {
  using S = BsShape<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::kBarOff);
  uint64_t* empty = full + S::kStages;
  uint64_t* dfull = empty + S::kStages;  // [2] partial buffer written
  uint64_t* dfree = dfull + 2;           // [2] partial buffer read
  uint64_t* drained = dfree + 2;         // every MMA of this CTA has completed
  uint32_t* tmem_sh = reinterpret_cast<uint32_t*>(drained + 1);
  float* sw = reinterpret_cast<float*>(smem + S::kTabOff);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ntile = blockIdx.x, mtile = blockIdx.y, split = blockIdx.z;
  const int n0 = ntile * 128, m0 = mtile * BN;
  const int g0 = (int)((int64_t)split * a.groups / a.splits);
  const int g1 = (int)((int64_t)(split + 1) * a.groups / a.splits);
  const int ng = g1 - g0;
  float* sx = sw + ng;  // [BN][ng]

  if (threadIdx.x == 0) {
    for (int s = 0; s < S::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&dfull[b], 1);
      mbar_init(&dfree[b], 128);
    }
    mbar_init(drained, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_sh, S::kTmemCols);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *tmem_sh;

  if (warp == 0) {
    // ------------------------------------------------------------------ producer (TMA)
    if (lane == 0) {
      prefetch_tensormap(&tmW);
      prefetch_tensormap(&tmX);
      constexpr uint32_t tx = S::kABytes + S::kBBytes;
      // weights are not produced upstream: the first ring-full goes out before the wait
      const int pre = ng < S::kStages ? ng : S::kStages;
      for (int i = 0; i < pre; ++i) {
        uint8_t* st = ring + i * S::kStageBytes;
        mbar_arrive_expect_tx(&full[i], tx);
        tma_load_2d(st, &tmW, &full[i], (g0 + i) * kGK, n0);
        tma_load_2d(st + 64 * kGK, &tmW, &full[i], (g0 + i) * kGK, n0 + 64);
      }
      pdl_wait();
      pdl_trigger();
      for (int i = 0; i < ng; ++i) {
        const int s = i % S::kStages;
        if (i >= S::kStages && !mbar_wait(&empty[s], ((i / S::kStages) - 1) & 1, a.err)) break;
        uint8_t* st = ring + s * S::kStageBytes;
        if (i >= pre) {
          mbar_arrive_expect_tx(&full[s], tx);
          tma_load_2d(st, &tmW, &full[s], (g0 + i) * kGK, n0);
          tma_load_2d(st + 64 * kGK, &tmW, &full[s], (g0 + i) * kGK, n0 + 64);
        }
        tma_load_2d(st + S::kABytes, &tmX, &full[s], (g0 + i) * kGK, m0);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issue (one thread)
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_e4m3(128, BN);
      bool issued = false;
      for (int i = 0; i < ng; ++i) {
        const int s = i % S::kStages, b = i & 1;
        if (!mbar_wait(&full[s], (i / S::kStages) & 1, a.err) ||
            (i >= 2 && !mbar_wait(&dfree[b], ((i >> 1) - 1) & 1, a.err)))
          break;
        fence_after_sync();
        const uint32_t sa = smem_u32(ring + s * S::kStageBytes), sb = sa + S::kABytes;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_e4m3(tmem + b * BN, desc_k128_sw128(sa + kk * 32), desc_k128_sw128(sb + kk * 32), idesc, kk > 0);
        commit(&empty[s]);
        commit(&dfull[b]);
        issued = true;
      }
      if (issued) {
        // every MMA has finished before TMEM is released, also when a wait above ran out
        commit(drained);
        mbar_wait(drained, 0, a.err);
      }
    }
  } else {
    // ------------------------------------------------------------------ promotion (thread = weight row)
    const int q = warp & 3;
    const int r = 32 * q + lane;
    const int tid = threadIdx.x - 64;
    pdl_wait();  // token scales and outputs belong to the previous kernel's world
    const int64_t KBs = a.K / kGK;
    for (int j = tid; j < ng; j += 128) sw[j] = a.ws[(int64_t)ntile * KBs + g0 + j];
    for (int e = tid; e < BN * ng; e += 128) {
      const int t = e / ng, j = e - t * ng;
      sx[e] = m0 + t < a.M ? a.xs[(int64_t)(m0 + t) * KBs + g0 + j] : 0.f;
    }
    asm volatile("bar.sync 1, 128;" ::: "memory");
    float acc[BN];
#pragma unroll
    for (int t = 0; t < BN; ++t) acc[t] = 0.f;
    const uint32_t trow = tmem + ((uint32_t)(32 * q) << 16);
    bool ok = true;
    for (int i = 0; i < ng; ++i) {
      const int b = i & 1;
      if (!__all_sync(MXG_FULL_MASK, mbar_wait(&dfull[b], (i >> 1) & 1, a.err))) {
        ok = false;
        break;
      }
      fence_after_sync();
      const float w = sw[i];
#pragma unroll
      for (int c = 0; c < BN; c += 16) {
        float v[16];
        ld16(trow + b * BN + c, v);
        wait_ld();
#pragma unroll
        for (int t = 0; t < 16; ++t) acc[c + t] = fmaf(w * sx[(c + t) * ng + i], v[t], acc[c + t]);
      }
      fence_before_sync();
      mbar_arrive(&dfree[b]);
    }
    const int n = n0 + r;
    if (ok && n < a.N) {
#pragma unroll
      for (int t = 0; t < BN; ++t) {
        const int m = m0 + t;
        if (m < a.M) {
          if (a.splits == 1)
            a.out[(int64_t)m * a.N + n] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[t]));
          else
            a.part[((int64_t)split * a.M + m) * a.N + n] = acc[t];
        }
      }
    }
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    fence_after_sync();
    tmem_dealloc(tmem, S::kTmemCols);
  }
}

// out[m][n] = bf16(sum_z part[z][m][n]), z in order.
__global__ void __launch_bounds__(256) bs_reduce_kernel(const float* __restrict__ part, int splits, int64_t MN,
                                                        uint16_t* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < MN; i += (int64_t)gridDim.x * blockDim.x) {
    float y = 0.f;
    for (int z = 0; z < splits; ++z) y += part[(int64_t)z * MN + i];
    out[i] = __bfloat16_as_ushort(__float2bfloat16_rn(y));
  }
}

// ------------------------------------------------------------------------- host
namespace {

int bs_pick_bn(int64_t M) { return M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : 128; }

struct BsPlan {
  int bn, ntiles, mtiles, splits;
};

BsPlan bs_plan(int64_t M, int64_t N, int64_t K) {
  BsPlan p;
  p.bn = bs_pick_bn(M);
  p.ntiles = (int)((N + 127) / 128);
  p.mtiles = (int)((M + p.bn - 1) / p.bn);
  const int groups = (int)(K / kGK);
  const int64_t ctas = (int64_t)p.ntiles * p.mtiles;
  // split K when the tiles alone cannot cover the 152 SMs (one wave, one CTA per SM)
  int s = ctas < 120 ? (int)(152 / ctas) : 1;
  if (s > groups) s = groups;
  p.splits = s < 1 ? 1 : s;
  return p;
}

template <int BN>
cudaError_t bs_launch(const CUtensorMap& tw, const CUtensorMap& tx, const BsArgs& a, dim3 grid, cudaStream_t st) {
  using S = BsShape<BN>;
  const int ng_max = (a.groups + a.splits - 1) / a.splits;
  const int smem = S::smem(ng_max);
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(bs_gemm_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_k(bs_gemm_kernel<BN>, grid, dim3(192), smem, st, 1, tw, tx, a);
}

}  // namespace

size_t bs_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  if (M <= 0 || N <= 0 || K <= 0 || K % kGK) return 0;
  const BsPlan p = bs_plan(M, N, K);
  return p.splits > 1 ? (size_t)p.splits * M * N * sizeof(float) : 0;
}

cudaError_t launch_bs_quantize_act(const uint16_t* x, int64_t M, int64_t K, int64_t ld_x, uint8_t* q, float* s,
                                   cudaStream_t st) {
  const int64_t warps = M * (K / kGK);
  return launch_k(bs_quantize_act_kernel, dim3((unsigned)((warps * 32 + 255) / 256)), dim3(256), 0, st, 1, x, M, K,
                  ld_x, q, s);
}

cudaError_t launch_bs_quantize_weight(const uint16_t* w, int64_t N, int64_t K, uint8_t* q, float* s, cudaStream_t st) {
  return launch_k(bs_quantize_weight_kernel, dim3((unsigned)(K / kGK), (unsigned)((N + 127) / 128)), dim3(256), 0, st,
                  1, w, N, K, q, s);
}

cudaError_t launch_bs_gemm(const uint8_t* xq, const float* xs, const uint8_t* wq, const float* ws, int64_t M,
                           int64_t N, int64_t K, uint16_t* out, void* workspace, int32_t* err, cudaStream_t st) {
  const BsPlan p = bs_plan(M, N, K);
  CUtensorMap tw, tx;
  if (!make_tensor_map_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, wq, (uint64_t)K, (uint64_t)N, (uint64_t)K, kGK, 64,
                          CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tensor_map_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_UINT8, xq, (uint64_t)K, (uint64_t)M, (uint64_t)K, kGK,
                          (uint32_t)p.bn, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  BsArgs a{};
  a.M = (int)M;
  a.N = (int)N;
  a.K = (int)K;
  a.groups = (int)(K / kGK);
  a.splits = p.splits;
  a.xs = xs;
  a.ws = ws;
  a.out = out;
  a.part = static_cast<float*>(workspace);
  a.err = err;
  const dim3 grid((unsigned)p.ntiles, (unsigned)p.mtiles, (unsigned)p.splits);
  cudaError_t e;
  switch (p.bn) {
    case 16: e = bs_launch<16>(tw, tx, a, grid, st); break;
    case 32: e = bs_launch<32>(tw, tx, a, grid, st); break;
    case 64: e = bs_launch<64>(tw, tx, a, grid, st); break;
    default: e = bs_launch<128>(tw, tx, a, grid, st); break;
  }
  if (e != cudaSuccess || p.splits == 1) return e;
  const int64_t MN = M * N;
  const int64_t blocks = (MN + 255) / 256 < 152 * 8 ? (MN + 255) / 256 : 152 * 8;
  return launch_k(bs_reduce_kernel, dim3((unsigned)blocks), dim3(256), 0, st, 1,
                  static_cast<const float*>(a.part), p.splits, MN, out);
}

}  // namespace mxg
