// MXFP8 activation quantisation (optionally fused with RMSNorm).
//
// [S2.1] "Kernel Benchmark Results": one launch quantises bf16 activations to E4M3 and packs
// the UE8M0 scales; "FP8 Quantization Strategy": 1x32 blocks along K, OCP UE8M0 exponents.
//
// Work split: one thread owns 8 consecutive elements (one 16-byte load), four adjacent lanes
// own one 32-element block and combine their |max| with two xor-shuffles. Loads are 128-bit
// and coalesced; each lane stores 8 E4M3 bytes, lane 0 of each quad stores the scale byte.
#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"

namespace mxg {

// Quantise the 8 values this lane holds as part of a 4-lane 32-element block.
// Every lane of the warp must call this (the shuffles use the full mask).
__device__ __forceinline__ void mx_quant8(const float (&v)[8], uint2& packed, uint8_t& sbyte) {
  float a = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(v[i]));
  a = fmaxf(a, __shfl_xor_sync(MXG_FULL_MASK, a, 1));
  a = fmaxf(a, __shfl_xor_sync(MXG_FULL_MASK, a, 2));
  const int s = mx_shared_exp(a);
  const float inv = mx_inv_scale(s);
  const uint32_t p0 = cvt_e4m3x2(v[0] * inv, v[1] * inv);
  const uint32_t p1 = cvt_e4m3x2(v[2] * inv, v[3] * inv);
  const uint32_t p2 = cvt_e4m3x2(v[4] * inv, v[5] * inv);
  const uint32_t p3 = cvt_e4m3x2(v[6] * inv, v[7] * inv);
  packed.x = p0 | (p1 << 16);
  packed.y = p2 | (p3 << 16);
  sbyte = (uint8_t)(s + 127);
}

__device__ __forceinline__ void unpack_bf16x8(const uint4& w, float (&v)[8]) {
  v[0] = bf16_lo(w.x); v[1] = bf16_hi(w.x);
  v[2] = bf16_lo(w.y); v[3] = bf16_hi(w.y);
  v[4] = bf16_lo(w.z); v[5] = bf16_hi(w.z);
  v[6] = bf16_lo(w.w); v[7] = bf16_hi(w.w);
}

__global__ void __launch_bounds__(256) mxfp8_quantize_kernel(const uint16_t* __restrict__ x, int64_t M, int64_t K,
                                                             int64_t ld_x, uint8_t* __restrict__ q,
                                                             uint8_t* __restrict__ s) {
  MXG_TL_SCOPE(kTlQuantize);
  pdl_wait();
  MXG_TL_WAITED();
  pdl_trigger();
  const int64_t cpr = K >> 3;  // 8-element chunks per row (a multiple of 4)
  const int64_t total = M * cpr;
  const int64_t step = (int64_t)gridDim.x * blockDim.x;
  // the trip count is uniform per block, so whole warps reach the shuffles together
  for (int64_t base = (int64_t)blockIdx.x * blockDim.x; base < total; base += step) {
    const int64_t c = base + threadIdx.x;
    const bool act = c < total;
    int64_t row = 0, col = 0;
    uint4 w = make_uint4(0, 0, 0, 0);
    if (act) {
      row = c / cpr;
      col = (c - row * cpr) << 3;
      w = __ldg(reinterpret_cast<const uint4*>(x + row * ld_x + col));
    }
    float v[8];
    unpack_bf16x8(w, v);
    uint2 packed;
    uint8_t sb;
    mx_quant8(v, packed, sb);
    if (act) {
      *reinterpret_cast<uint2*>(q + row * K + col) = packed;
      if ((threadIdx.x & 3) == 0) s[row * (K >> 5) + (col >> 5)] = sb;
    }
  }
}

// Error-free addition (Knuth two-sum): hi + lo carries the running sum with ~48 significant
// bits using fp32 arithmetic only (fp64 throughput on this part is a small fraction of fp32).
__device__ __forceinline__ void two_sum_acc(float& hi, float& lo, float x) {
  const float s = __fadd_rn(hi, x);
  const float bp = __fsub_rn(s, hi);
  const float e = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bp)), __fsub_rn(x, bp));
  hi = s;
  lo = __fadd_rn(lo, e);
}

constexpr int kRmsThreads = 320;  // = K/8 for K = 2560: one chunk per thread

// Error-free fp32 helpers for the RMSNorm factor (double-float arithmetic: a value is an
// unevaluated sum hi + lo of two fp32 numbers).
__device__ __forceinline__ void fast_two_sum(float a, float b, float& s, float& e) {  // |a| >= |b|
  s = __fadd_rn(a, b);
  e = __fsub_rn(b, __fsub_rn(s, a));
}
__device__ __forceinline__ void df_add(float& h, float& l, float ah, float al) {
  const float s = __fadd_rn(h, ah);
  const float bp = __fsub_rn(s, h);
  const float e = __fadd_rn(__fsub_rn(h, __fsub_rn(s, bp)), __fsub_rn(ah, bp));
  fast_two_sum(s, __fadd_rn(e, __fadd_rn(l, al)), h, l);
}

// r = fp32(1 / sqrt(T / K + eps)), T = sum over the warps of hi_w + lo_w, as the fp64 sequence
// fp64 mean -> + eps -> sqrt -> 1 / x -> round to fp32 gives it. fp64 arithmetic costs ~2400
// cycles on this part (measured), so the value is first estimated in double-float fp32
// arithmetic (the mean to ~2^-47, then one Newton step for 1/sqrt with its quadratic term,
// ~2^-44 overall). Unless that estimate lies within 2^-39 (relative) of a point halfway
// between two fp32 numbers -- then the fp64 result, within ~2^-51 of the exact value, rounds to
// the same fp32 number -- the estimate's rounding is the answer; otherwise (about one row in
// 2^14, and every out-of-range case) the fp64 sequence runs.
__device__ float rms_factor(const float (&wh)[kRmsThreads / 32], const float (&wl)[kRmsThreads / 32], int64_t K,
                            float eps) {
  float th = 0.f, tl = 0.f;
#pragma unroll
  for (int i = 0; i < kRmsThreads / 32; ++i) df_add(th, tl, wh[i], wl[i]);
  const float kf = (float)K;  // K < 2^24: exact
  const float mh = __fdiv_rn(th, kf);
  const float ph = __fmul_rn(mh, kf), pl = __fmaf_rn(mh, kf, -ph);
  const float ml = __fdiv_rn(__fadd_rn(__fsub_rn(__fsub_rn(th, ph), pl), tl), kf);
  float vh, vl;
  {
    const float s = __fadd_rn(mh, eps);
    const float bp = __fsub_rn(s, mh);
    const float e = __fadd_rn(__fsub_rn(mh, __fsub_rn(s, bp)), __fsub_rn(eps, bp));
    fast_two_sum(s, __fadd_rn(e, ml), vh, vl);
  }
  bool ok = isfinite(th) && vh > 0x1p-100f && vh < 0x1p100f;
  float r = 0.f;
  if (ok) {
    const float y0 = rsqrtf(vh);
    const float s2h = __fmul_rn(y0, y0), s2l = __fmaf_rn(y0, y0, -s2h);
    const float qh = __fmul_rn(vh, s2h);
    const float ql = __fadd_rn(__fmaf_rn(vh, s2h, -qh), __fadd_rn(__fmul_rn(vh, s2l), __fmul_rn(vl, s2h)));
    const float e = __fsub_rn(__fsub_rn(1.f, qh), ql);  // 1 - v y0^2, |e| ~ 2^-22
    const float c = __fmul_rn(y0, __fmaf_rn(0.375f * e, e, 0.5f * e));
    float yh, yl;
    fast_two_sum(y0, c, yh, yl);
    const uint32_t yb = __float_as_uint(yh);
    const int ex = (int)((yb >> 23) & 0xFFu);
    // half the fp32 spacing at yh (below a power of two the spacing halves)
    float half = __uint_as_float((uint32_t)(ex - 24) << 23);
    if ((yb & 0x7FFFFFu) == 0 && yl < 0.f) half *= 0.5f;
    ok = ex > 64 && ex < 190 && __fsub_rn(half, fabsf(yl)) > __fmul_rn(yh, 0x1p-39f);
    r = yh;
  }
  if (!ok) {
    double t = 0.0;
    for (int i = 0; i < kRmsThreads / 32; ++i) t += (double)wh[i] + (double)wl[i];
    const double ms = t / (double)K;
    r = (float)(1.0 / sqrt(ms + (double)eps));
  }
  return r;
}

// One CTA per row; each thread keeps its 8-element chunks of x (and gamma) in registers, so
// the row is read from memory once. Sum of squares: each square of a bf16 value is exact in
// fp32; they are summed as a two-sum pair (~48-bit), and the ten warp partials in fp64
// (rms_factor), so the fp64 mean agrees with an fp64 summation far below the fp32 rounding of
// r. Then y = bf16((x * r) * gamma) with r = fp32(1 / sqrt(mean + eps)), then the MX rule on y.
constexpr int kRmsChunks = 7;     // chunks per thread kept in registers: K <= 8 * 320 * 7 = 17920

__global__ void __launch_bounds__(kRmsThreads) rmsnorm_mxfp8_quantize_kernel(const uint16_t* __restrict__ x,
                                                                             const uint16_t* __restrict__ gamma,
                                                                             float eps, int64_t K, int64_t ld_x,
                                                                             uint8_t* __restrict__ q,
                                                                             uint8_t* __restrict__ s) {
  MXG_TL_SCOPE(kTlRmsQuant);
  const int64_t row = blockIdx.x;
  const uint16_t* xr = x + row * ld_x;
  const int cpr = (int)(K >> 3);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint4 gw[kRmsChunks];
#pragma unroll
  for (int i = 0; i < kRmsChunks; ++i) {  // gamma is a weight: read before waiting for upstream
    const int c = threadIdx.x + i * kRmsThreads;
    gw[i] = c < cpr ? __ldg(reinterpret_cast<const uint4*>(gamma + ((int64_t)c << 3))) : make_uint4(0, 0, 0, 0);
  }
  pdl_wait();
  MXG_TL_WAITED();
  pdl_trigger();
  uint4 xw[kRmsChunks];
#pragma unroll
  for (int i = 0; i < kRmsChunks; ++i) {
    const int c = threadIdx.x + i * kRmsThreads;
    xw[i] = c < cpr ? __ldg(reinterpret_cast<const uint4*>(xr + ((int64_t)c << 3))) : make_uint4(0, 0, 0, 0);
  }
  float hi = 0.f, lo = 0.f;
#pragma unroll
  for (int i = 0; i < kRmsChunks; ++i) {
    if (i * kRmsThreads >= cpr) break;  // uniform: no work on chunk slots past the row
    float v[8];
    unpack_bf16x8(xw[i], v);
#pragma unroll
    for (int j = 0; j < 8; ++j) two_sum_acc(hi, lo, __fmul_rn(v[j], v[j]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float h2 = __shfl_xor_sync(MXG_FULL_MASK, hi, o);
    const float l2 = __shfl_xor_sync(MXG_FULL_MASK, lo, o);
    two_sum_acc(hi, lo, h2);
    lo = __fadd_rn(lo, l2);
  }
  __shared__ float red_h[kRmsThreads / 32], red_l[kRmsThreads / 32];
  __shared__ float r_sh;
  if (lane == 0) {
    red_h[warp] = hi;
    red_l[warp] = lo;
  }
  __syncthreads();
  if (threadIdx.x == 0) r_sh = rms_factor(red_h, red_l, K, eps);
  __syncthreads();
  const float r = r_sh;
#pragma unroll
  for (int i = 0; i < kRmsChunks; ++i) {
    const int base = i * kRmsThreads;
    if (base >= cpr) break;  // uniform across the block
    const int c = base + threadIdx.x;
    const bool act = c < cpr;
    float xv[8], gv[8], v[8];
    unpack_bf16x8(xw[i], xv);
    unpack_bf16x8(gw[i], gv);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float y = __fmul_rn(__fmul_rn(xv[j], r), gv[j]);
      v[j] = act ? __bfloat162float(__float2bfloat16_rn(y)) : 0.f;
    }
    uint2 packed;
    uint8_t sb;
    mx_quant8(v, packed, sb);
    if (act) {
      *reinterpret_cast<uint2*>(q + row * K + ((int64_t)c << 3)) = packed;
      if ((lane & 3) == 0) s[row * (K >> 5) + (c >> 2)] = sb;
    }
  }
}

cudaError_t launch_mxfp8_quantize(const uint16_t* x, int64_t M, int64_t K, int64_t ld_x, uint8_t* q, uint8_t* s,
                                  cudaStream_t st) {
  const int64_t total = M * (K >> 3);
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (blocks < 1) blocks = 1;
  return launch_k(mxfp8_quantize_kernel, dim3((unsigned)blocks), dim3(threads), 0, st, 1, x, M, K, ld_x, q, s);
}

cudaError_t launch_rmsnorm_mxfp8_quantize(const uint16_t* x, const uint16_t* gamma, float eps, int64_t M, int64_t K,
                                          int64_t ld_x, uint8_t* q, uint8_t* s, cudaStream_t st) {
  return launch_k(rmsnorm_mxfp8_quantize_kernel, dim3((unsigned)M), dim3(kRmsThreads), 0, st, 1, x, gamma, eps, K, ld_x,
                  q, s);
}

}  // namespace mxg

MXG_TL_UNIT(quant)
