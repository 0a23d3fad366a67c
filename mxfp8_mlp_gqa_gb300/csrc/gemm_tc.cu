// MXFP8 block-scaled GEMM on the 5th-generation tensor cores (tcgen05, sm_103a).
//
// out[m][n] = sum_k X'[m][k] W'[n][k] for MX operands (E4M3 + one UE8M0 scale per 32 along
// K), [S2.1] "FP8 Quantization Strategy" / "Kernel Benchmark Results". Decode shapes have
// few tokens (M <= 128) and many output features, so the MMA runs "swapped": the weight
// tile is the 128-row MMA operand A, the tokens are the MMA N dimension (16..256), and the
// fp32 accumulator D^T[128 features][N tokens] lives in tensor memory.
//
// Per CTA (192 threads):
//   warp 0  producer: lane 0 issues TMA (128-byte swizzle) for the weight tile (two 64-row
//           boxes) and the token tile of each 128-wide K group; all 32 lanes cp.async the
//           UE8M0 words of that group (4 k-blocks per row) into the 32x4 atom layout
//           (byte 16*(r%32) + 4*(r/32) + kb) that tcgen05.cp 32x128b.warpx4 expects;
//   warp 1  TMEM owner; lane 0 issues per group: 2 scale copies to TMEM + 4 MMAs
//           (kind::mxf8f6f4.block_scale, K=32 each, scale byte kb selected in the
//           instruction descriptor), then tcgen05.commit frees the stage;
//   warps 2-5 epilogue: read D^T from TMEM (each warp its lane quadrant) and
//           * kEpiStore : write bf16 out (+ bf16 residual),
//           * kEpiSplit : split-K over a thread-block cluster of S CTAs (grid.z = S): every
//                         CTA stages its fp32 partial tile in shared memory, and after a
//                         cluster barrier CTA z sums rows [z*128/S, (z+1)*128/S) of all S
//                         partials through distributed shared memory in a fixed order
//                         (+ residual) and writes bf16 -- deterministic, no global scratch,
//           * kEpiSwiGLU: the weight tile is 64 gate rows + the matching 64 up rows; h =
//                         silu(g) * u in fp32, re-quantised to MXFP8 along d_ff in the
//                         epilogue (no bf16 h is ever written).
// Every wait is bounded (MXG_ETIMEOUT in the error flag); TMEM is always released.
#include "kernels.h"
#include "launch.cuh"
#include "tc.cuh"

namespace mxg {

namespace {

constexpr int kKG = 128;  // K elements per stage: one 4-block group of scales
enum { kEpiStore = 0, kEpiSplit = 1, kEpiSwiGLU = 2 };

template <int BN>
struct TcShape {
  static constexpr int kABytes = 128 * kKG;
  static constexpr int kBBytes = BN * kKG;
  static constexpr int kSfbAtoms = (BN + 127) / 128;
  static constexpr int kSfBytes = 1024 * ((512 * (1 + kSfbAtoms) + 1023) / 1024);  // keeps stages 1024-aligned
  static constexpr int kStageBytes = kABytes + kBBytes + kSfBytes;
  // At least 5 stages (>= 80 KB of weights in flight per SM: the weight stream is latency-
  // bound below that), otherwise as many as fit in ~96 KB so that small-BN kernels still fit
  // two CTAs per SM (the next kernel, launched early by PDL, can then stream alongside).
  static constexpr int kStagesRaw = (BN >= 256 ? 200 * 1024 : 96 * 1024) / kStageBytes;
  static constexpr int kStages = kStagesRaw > 8 ? 8 : (kStagesRaw < (BN >= 256 ? 2 : 5) ? (BN >= 256 ? 2 : 5)
                                                                                       : kStagesRaw);
  static constexpr int kRingBytes = kStages * kStageBytes;
  static constexpr int kRS = 128 + 4;  // split-K staging [BN][kRS] (column-major, 16-byte rows)
  static constexpr int kStagingBytes =
      128 * (BN + 1) * 4 > BN * kRS * 4 ? 128 * (BN + 1) * 4 : BN * kRS * 4;  // max(SwiGLU, split-K)
  static constexpr int kBodyBytes = kRingBytes > kStagingBytes ? kRingBytes : kStagingBytes;
  static constexpr int kSmemBytes = 1024 + kBodyBytes + 8 * (2 * kStages + 1) + 16;
  // scale atoms rotate through kSfSlots TMEM slots, so the copy for stage i+1 never
  // overwrites columns that MMAs of stage i may still be reading
  static constexpr int kSfSlots = 4;
  static constexpr int kSfCols = 4 * (1 + kSfbAtoms);
  static constexpr int kTmemNeed = BN + kSfSlots * kSfCols;
  static constexpr uint32_t kTmemCols = kTmemNeed <= 32    ? 32
                                        : kTmemNeed <= 64  ? 64
                                        : kTmemNeed <= 128 ? 128
                                        : kTmemNeed <= 256 ? 256
                                                           : 512;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

struct TcArgs {
  int M, N, K;          // out[M tokens][N features]; N = 2*d_ff weight rows for SwiGLU
  int groups, splits;   // K/128 groups, K splits (grid.z)
  const uint8_t* ws;    // weight scales  [N rows][K/32]
  const uint8_t* xs;    // token scales   [M][K/32]
  int d_ff;
  uint8_t* hq;
  uint8_t* hs;
  const uint16_t* residual;
  uint16_t* out;
  int32_t* err;
  KvScatter kv;         // fused KV append of a QKV projection (kv.kc == nullptr: off)
  // Pre-packed scales (large GEMMs): group-major 512-byte atoms [K/128][row tiles][512 B],
  // one 1-D bulk copy per stage instead of per-lane gathers. nullptr: gather from ws / xs.
  const uint32_t* wsp;
  const uint32_t* xsp;
  int rt_w, rt_x;       // 128-row tiles per group in wsp / xsp
  int tma_out;          // pair kernel: plain bf16 output written by TMA stores
};

// Scales [rows][K/32] (row-major) -> group-major atoms: word w of atom (g, rt) holds the four
// k-blocks of group g of row rt*128 + (w >> 2) + 32 * (w & 3); rows past `rows` are zero.
__global__ void __launch_bounds__(256) pack_scales_kernel(const uint8_t* __restrict__ s, int64_t rows, int64_t KB,
                                                          int rt_pad, int groups, uint32_t* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const int64_t total = (int64_t)groups * rt_pad * 128;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int w = (int)(idx & 127);
    const int64_t t = idx >> 7;
    const int rt = (int)(t % rt_pad), g = (int)(t / rt_pad);
    const int64_t row = (int64_t)rt * 128 + (w >> 2) + 32 * (w & 3);
    out[idx] = row < rows ? *reinterpret_cast<const uint32_t*>(s + row * KB + 4 * (int64_t)g) : 0u;
  }
}

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// Destination of output element (m, n): `out`, or -- for the K/V columns of a fused QKV
// projection -- row kv_len[m]-1 of KV head (c / D) in the K or V cache (nullptr, with the
// error flag set, when that row is outside the cache).
__device__ __forceinline__ uint16_t* out_ptr(const TcArgs& a, int m, int n) {
  if (a.kv.kc == nullptr || n < a.kv.q_cols) return a.out + (int64_t)m * a.N + n;
  const int kvd = a.kv.Hkv * a.kv.D;
  int c = n - a.kv.q_cols;
  uint16_t* base = a.kv.kc;
  if (c >= kvd) {
    c -= kvd;
    base = a.kv.vc;
  }
  const int pos = a.kv.kv_len[m] - 1;
  if (pos < 0 || (int64_t)pos >= a.kv.cap) {
    set_error(a.err, MXG_EDEVICE);
    return nullptr;
  }
  const int g = c / a.kv.D, d = c - g * a.kv.D;
  return base + (((int64_t)m * a.kv.Hkv + g) * a.kv.cap + pos) * a.kv.D + d;
}

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Shared::cluster address of the object at `local`'s offset in CTA `rank`'s shared memory.
__device__ __forceinline__ uint32_t mapa_shared(const void* local, uint32_t rank) {
  uint32_t raddr;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(raddr) : "r"(smem_u32(local)), "r"(rank));
  return raddr;
}

// 4 x fp32 from the shared memory of CTA `rank` of this cluster, at the offset that `local`
// (16-byte aligned) has in this CTA's shared memory. Only read between the two cluster
// barriers of the split-K reduction, where the staged partials do not change: volatile keeps
// the loads between those barriers, and without a memory clobber the compiler may issue the
// loads of several output groups before the global stores of the first.
__device__ __forceinline__ float4 ld_dsmem_f32x4(const float* local, uint32_t rank) {
  uint32_t raddr;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(raddr) : "r"(smem_u32(local)), "r"(rank));
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(raddr));
  return v;
}

}  // namespace

template <int BN, int EPI>
__global__ void __launch_bounds__(192, 1) mx_gemm_tc_kernel(const __grid_constant__ CUtensorMap tmW,
                                                            const __grid_constant__ CUtensorMap tmX, const TcArgs a) {
  MXG_TL_SCOPE(kTlGemmTc + EPI);
  using S = TcShape<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::kBodyBytes);
  uint64_t* empty = full + S::kStages;
  uint64_t* tmem_full = empty + S::kStages;
  uint32_t* tmem_sh = reinterpret_cast<uint32_t*>(tmem_full + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ntile = blockIdx.x, mtile = blockIdx.y, split = blockIdx.z;
  const int m0 = mtile * BN;
  const int n0 = EPI == kEpiSwiGLU ? ntile * 64 : ntile * 128;
  const int a_lo = n0;                                         // weight rows of tile rows 0..63
  const int a_hi = EPI == kEpiSwiGLU ? a.d_ff + n0 : n0 + 64;  // weight rows of tile rows 64..127
  const int wrows = EPI == kEpiSwiGLU ? 2 * a.d_ff : a.N;
  const int g0 = (int)((int64_t)split * a.groups / a.splits);
  const int g1 = (int)((int64_t)(split + 1) * a.groups / a.splits);
  const int ng = g1 - g0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S::kStages; ++s) {
      // TMA expect-tx arrive (+ one cp.async arrive per producer lane when scales are gathered)
      mbar_init(&full[s], a.wsp ? 1 : 1 + 32);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tmem_full, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_sh, S::kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_sh;
  const uint32_t t_d = tmem;
  // split-K reduction work of an epilogue thread (filled by the epilogue warps, see below)
  constexpr int kNJ = EPI == kEpiSplit && BN <= 128 ? (BN / 8 > 0 ? BN / 8 : 1) : 1;
  constexpr bool kBatched = EPI == kEpiSplit && BN <= 128;
  const int S_ = a.splits;
  const int rb = 4 * ((split * 32) / (S_ > 0 ? S_ : 1));
  const int nq = ((split + 1) * 32) / (S_ > 0 ? S_ : 1) - (split * 32) / (S_ > 0 ? S_ : 1);
  uint16_t* dst[kNJ];
  uint2 rv[kNJ];
  int sidx[kNJ];
#pragma unroll
  for (int j = 0; j < kNJ; ++j) {
    dst[j] = nullptr;
    rv[j] = make_uint2(0u, 0u);
    sidx[j] = 0;
  }

  if (warp == 0) {
    // ----------------------------------------------------------------- producer
    if (lane == 0) {
      prefetch_tensormap(&tmW);
      prefetch_tensormap(&tmX);
    }
    const int64_t KB = a.K >> 5;
    const uint32_t tx = S::kABytes + S::kBBytes + (a.wsp ? 512u * (1 + S::kSfbAtoms) : 0u);
    // weight tiles of the first ring-full read nothing produced upstream: issue them before
    // waiting for the previous kernel (programmatic dependent launch)
    const int pre = ng < S::kStages ? ng : S::kStages;
    if (lane == 0) {
      for (int i = 0; i < pre; ++i) {
        uint8_t* st = ring + i * S::kStageBytes;
        mbar_arrive_expect_tx(&full[i], tx);
        tma_load_2d(st, &tmW, &full[i], (g0 + i) * kKG, a_lo);
        tma_load_2d(st + 64 * kKG, &tmW, &full[i], (g0 + i) * kKG, a_hi);
      }
    }
    pdl_wait();
    MXG_TL_WAITED();
    // the next kernel may start its own weight prefetch only once the previous one is complete
    pdl_trigger();
    for (int i = 0; i < ng; ++i) {
      const int s = i % S::kStages;
      if (i >= S::kStages && !mbar_wait(&empty[s], ((i / S::kStages) - 1) & 1, a.err)) break;
      uint8_t* st = ring + s * S::kStageBytes;
      const int g = g0 + i;
      if (lane == 0) {
        if (i >= pre) {
          mbar_arrive_expect_tx(&full[s], tx);
          tma_load_2d(st, &tmW, &full[s], g * kKG, a_lo);
          tma_load_2d(st + 64 * kKG, &tmW, &full[s], g * kKG, a_hi);
        }
        if (BN > 128) {  // the token map's box is 128 rows for 256-token tiles
          tma_load_2d(st + S::kABytes, &tmX, &full[s], g * kKG, m0);
          tma_load_2d(st + S::kABytes + 128 * kKG, &tmX, &full[s], g * kKG, m0 + 128);
        } else {
          tma_load_2d(st + S::kABytes, &tmX, &full[s], g * kKG, m0);
        }
      }
      uint32_t* sfa = reinterpret_cast<uint32_t*>(st + S::kABytes + S::kBBytes);
      if (a.wsp) {
        if (lane == 0) {
          bulk_load(sfa, a.wsp + ((int64_t)g * a.rt_w + ntile) * 128, 512, &full[s]);
          bulk_load(sfa + 128, a.xsp + ((int64_t)g * a.rt_x + (m0 >> 7)) * 128, 512 * S::kSfbAtoms, &full[s]);
        }
        continue;
      }
#pragma unroll
      for (int r1 = 0; r1 < 4; ++r1) {
        const int r = lane + 32 * r1;
        const int grow = r < 64 ? a_lo + r : a_hi + (r - 64);
        if (grow < wrows) tc::cp_async4(&sfa[4 * lane + r1], a.ws + (int64_t)grow * KB + 4 * g);
      }
#pragma unroll
      for (int at = 0; at < S::kSfbAtoms; ++at) {
        uint32_t* sfb = sfa + 128 * (1 + at);
#pragma unroll
        for (int r1 = 0; r1 < 4; ++r1) {
          const int r = 128 * at + lane + 32 * r1;
          if (r < BN && m0 + r < a.M) tc::cp_async4(&sfb[4 * lane + r1], a.xs + (int64_t)(m0 + r) * KB + 4 * g);
        }
      }
      tc::cp_async_arrive(&full[s]);
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      for (int i = 0; i < ng; ++i) {
        const int s = i % S::kStages;
        if (!mbar_wait(&full[s], (i / S::kStages) & 1, a.err)) break;
        MXG_TL_MARK1();  // timeline: first stage landed
        if (!a.wsp) fence_proxy_async_smem();  // cp.async (generic proxy) scale words -> tcgen05.cp (async proxy)
        tc::fence_after_sync();
        const uint32_t t_sfa = tmem + BN + (uint32_t)((i % S::kSfSlots) * S::kSfCols), t_sfb = t_sfa + 4;
        uint8_t* st = ring + s * S::kStageBytes;
        const uint32_t sa = smem_u32(st), sb = smem_u32(st + S::kABytes);
        const uint32_t ssf = smem_u32(st + S::kABytes + S::kBBytes);
        tc::cp_sf_atom(t_sfa, tc::desc_sf_atom(ssf));
#pragma unroll
        for (int at = 0; at < S::kSfbAtoms; ++at) tc::cp_sf_atom(t_sfb + 4 * at, tc::desc_sf_atom(ssf + 512 * (1 + at)));
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc::mma_mxf8(t_d, tc::desc_k128_sw128(sa + kk * 32), tc::desc_k128_sw128(sb + kk * 32),
                       tc::idesc_mxf8(BN, kk, kk), t_sfa, t_sfb, (i > 0 || kk > 0) ? 1u : 0u);
        tc::commit(&empty[s]);
      }
      tc::commit(tmem_full);
      MXG_TL_MARK2();  // timeline: last MMA issued
    }
    __syncwarp();
  } else {
    // ----------------------------------------------------------------- epilogue
    const int q = warp & 3;  // the TMEM lane quadrant this warp may read
    const int r = 32 * q + lane;
    pdl_wait();  // outputs and the residual are touched only after the previous kernel is done
    MXG_TL_WAITED();
    // Split-K (BN <= 128): CTA z of the cluster owns the 4-row groups [z*32/S, (z+1)*32/S) of
    // the 128-row tile; an epilogue thread takes groups e = tid - 64 + 128 j of them (nq <= 16
    // groups per token for S >= 2, so j < BN/8). Their destinations (for the K/V columns of a
    // fused QKV projection a kv_len read) and residuals are inputs from upstream: they are read
    // here, right after the programmatic wait, while the MMAs still run.
    if (kBatched) {
      int mj[kNJ], nj[kNJ];
#pragma unroll
      for (int j = 0; j < kNJ; ++j) {
        const int e = threadIdx.x - 64 + 128 * j;
        const int c = e / nq, rr = rb + 4 * (e - c * nq);
        mj[j] = -1;
        nj[j] = n0 + rr;
        sidx[j] = c * S::kRS + rr;
        if (e < BN * nq && m0 + c < a.M && nj[j] < a.N) mj[j] = m0 + c;
      }
#pragma unroll
      for (int j = 0; j < kNJ; ++j)
        if (mj[j] >= 0 && a.residual) rv[j] = *reinterpret_cast<const uint2*>(a.residual + (int64_t)mj[j] * a.N + nj[j]);
#pragma unroll
      for (int j = 0; j < kNJ; ++j)
        if (mj[j] >= 0) dst[j] = out_ptr(a, mj[j], nj[j]);  // 4 consecutive columns never straddle a head
    }
    // warp-uniform outcome: the SwiGLU epilogue below shuffles with the full mask
    const bool ok = __all_sync(MXG_FULL_MASK, mbar_wait(tmem_full, 0, a.err));
    MXG_TL_MARK1();  // timeline: accumulator complete
    tc::fence_after_sync();
    const uint32_t trow = t_d + ((uint32_t)(32 * q) << 16);
    if (EPI == kEpiStore) {
      const int n = n0 + r;
      const bool nv = n < a.N;
      for (int c = 0; c < BN; c += 16) {
        float v[16];
        tc::ld16(trow + c, v);
        tc::wait_ld();
        if (!ok) continue;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int m = m0 + c + j;
          if (m < a.M && nv) {
            float y = v[j];
            if (a.residual) y += __bfloat162float(__ushort_as_bfloat16(a.residual[(int64_t)m * a.N + n]));
            uint16_t* dst = out_ptr(a, m, n);
            if (dst) *dst = __bfloat16_as_ushort(__float2bfloat16_rn(y));
          }
        }
      }
    } else if (EPI == kEpiSplit) {
      // stage this CTA's partial tile (column-major: rows contiguous); the cluster reduction
      // below reads it remotely
      float* stg = reinterpret_cast<float*>(ring);  // [BN tokens][kRS]
      for (int c = 0; c < BN; c += 16) {
        float v[16];
        tc::ld16(trow + c, v);
        tc::wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) stg[(c + j) * S::kRS + r] = v[j];
      }
    } else {
      // SwiGLU + MXFP8 re-quantisation along d_ff
      float* stg = reinterpret_cast<float*>(ring);  // [128 tile rows][BN + 1]
      for (int c = 0; c < BN; c += 16) {
        float v[16];
        tc::ld16(trow + c, v);
        tc::wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) stg[r * (BN + 1) + c + j] = v[j];
      }
      epi_bar();
      if (ok && BN <= 16) {
        // few tokens: the warp spreads one token's 32-value block over its lanes
        const int e = warp - 2, blk = e & 1, half = e >> 1;
        const int j0 = n0 + 32 * blk;
        for (int t = half * (BN / 2); t < (half + 1) * (BN / 2); ++t) {
          const int m = m0 + t;
          if (m >= a.M) break;
          const float g = stg[(32 * blk + lane) * (BN + 1) + t];
          const float u = stg[(64 + 32 * blk + lane) * (BN + 1) + t];
          const float h = silu_mul(g, u);
          mx_quant_warp_store(h, a.hq + (int64_t)m * a.d_ff + j0 + lane, a.hs + (int64_t)m * (a.d_ff >> 5) + (j0 >> 5));
        }
      } else if (ok) {
        // one lane per token: the lane holds all 32 d_ff values of its MX block, so the block
        // max needs no shuffles and the 32 codes leave in two 16-byte stores
        const int e = warp - 2, blk = e & 1, half = e >> 1;
        const int j0 = n0 + 32 * blk;  // first d_ff index of this warp's block
        const float* gs = stg + (32 * blk) * (BN + 1);
        const float* us = stg + (64 + 32 * blk) * (BN + 1);
        for (int t = half * (BN / 2) + lane; t < (half + 1) * (BN / 2); t += 32) {
          const int m = m0 + t;
          if (m >= a.M) continue;
          float h[32];
          float am = 0.f;
#pragma unroll
          for (int r = 0; r < 32; ++r) {
            const float g = gs[r * (BN + 1) + t], u = us[r * (BN + 1) + t];
            h[r] = silu_mul(g, u);
            am = fmaxf(am, fabsf(h[r]));
          }
          const int se = mx_shared_exp(am);
          const float inv = mx_inv_scale(se);
          uint32_t w[8];
#pragma unroll
          for (int k = 0; k < 8; ++k)
            w[k] = cvt_e4m3x2(h[4 * k] * inv, h[4 * k + 1] * inv) | (cvt_e4m3x2(h[4 * k + 2] * inv, h[4 * k + 3] * inv) << 16);
          uint4* dst = reinterpret_cast<uint4*>(a.hq + (int64_t)m * a.d_ff + j0);
          dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
          dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
          a.hs[(int64_t)m * (a.d_ff >> 5) + (j0 >> 5)] = (uint8_t)(se + 127);
        }
      }
    }
  }
  if (EPI == kEpiSplit) {
    cluster_sync_all();  // every CTA of the cluster has staged its partial tile
    MXG_TL_MARK2();      // timeline: partial tiles staged cluster-wide
    if (kBatched && warp >= 2) {
      // split by split: the partials of all of the thread's groups are loaded before they are
      // added, so the remote loads overlap (summation order per element: split 0, 1, ...)
      const float* stg = reinterpret_cast<const float*>(ring);
      float4 y[kNJ];
#pragma unroll
      for (int j = 0; j < kNJ; ++j) y[j] = dst[j] ? ld_dsmem_f32x4(&stg[sidx[j]], 0u) : make_float4(0.f, 0.f, 0.f, 0.f);
      if (S_ >= 4) {
        // nq <= 8: a thread has at most BN/16 groups (j < kNJ/2), so three splits' partials of
        // all of them are loaded per round
        constexpr int kNJ4 = kNJ / 2 > 0 ? kNJ / 2 : 1;
        for (int z = 1; z < S_; z += 3) {
          float4 p[kNJ4][3];
#pragma unroll
          for (int j = 0; j < kNJ4; ++j)
#pragma unroll
            for (int c = 0; c < 3; ++c)
              p[j][c] = dst[j] && z + c < S_ ? ld_dsmem_f32x4(&stg[sidx[j]], (uint32_t)(z + c))
                                             : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int j = 0; j < kNJ4; ++j)
#pragma unroll
            for (int c = 0; c < 3; ++c)
              if (z + c < S_) {
                y[j].x += p[j][c].x;
                y[j].y += p[j][c].y;
                y[j].z += p[j][c].z;
                y[j].w += p[j][c].w;
              }
        }
      } else {
        for (int z = 1; z < S_; ++z) {
          float4 p[kNJ];
#pragma unroll
          for (int j = 0; j < kNJ; ++j)
            p[j] = dst[j] ? ld_dsmem_f32x4(&stg[sidx[j]], (uint32_t)z) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int j = 0; j < kNJ; ++j) {
            y[j].x += p[j].x;
            y[j].y += p[j].y;
            y[j].z += p[j].z;
            y[j].w += p[j].w;
          }
        }
      }
#pragma unroll
      for (int j = 0; j < kNJ; ++j) {
        if (!dst[j]) continue;
        float4 v = y[j];
        if (a.residual) {
          v.x += bf16_lo(rv[j].x);
          v.y += bf16_hi(rv[j].x);
          v.z += bf16_lo(rv[j].y);
          v.w += bf16_hi(rv[j].y);
        }
        uint2 ov;
        ov.x = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v.x)) |
               ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v.y)) << 16);
        ov.y = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v.z)) |
               ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v.w)) << 16);
        *reinterpret_cast<uint2*>(dst[j]) = ov;
      }
    }
    if (!kBatched && warp >= 2) {
      const float* stg = reinterpret_cast<const float*>(ring);
      for (int e = threadIdx.x - 64; e < BN * nq; e += 128) {
        const int c = e / nq, rr = rb + 4 * (e - c * nq);
        const int m = m0 + c, n = n0 + rr;
        if (m >= a.M || n >= a.N) continue;
        float4 v = ld_dsmem_f32x4(&stg[c * S::kRS + rr], 0u);
        for (int z = 1; z < S_; ++z) {
          const float4 p = ld_dsmem_f32x4(&stg[c * S::kRS + rr], (uint32_t)z);
          v.x += p.x;
          v.y += p.y;
          v.z += p.z;
          v.w += p.w;
        }
        if (a.residual) {
          const uint2 r2 = *reinterpret_cast<const uint2*>(a.residual + (int64_t)m * a.N + n);
          v.x += bf16_lo(r2.x);
          v.y += bf16_hi(r2.x);
          v.z += bf16_lo(r2.y);
          v.w += bf16_hi(r2.y);
        }
        uint2 ov;
        ov.x = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v.x)) |
               ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v.y)) << 16);
        ov.y = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v.z)) |
               ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v.w)) << 16);
        uint16_t* d = out_ptr(a, m, n);
        if (d) *reinterpret_cast<uint2*>(d) = ov;
      }
    }
    cluster_sync_all();  // keep this CTA's shared memory alive until every reader is done
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(tmem, S::kTmemCols);
}

// Large GEMMs (M > 1024): one M=256 block-scaled MMA per CTA pair (cta_group::2). The pair
// (a 2-CTA cluster along x) owns 256 weight rows x 256 tokens; each CTA stages its own 128
// weight rows and one 128-token half of the token tile, so a stage is 32 KB per CTA and six
// stages are in flight. Scales arrive pre-packed: each CTA holds the atom of its own weight
// rows and both atoms of the 256 tokens. Every load of both CTAs completes on the even CTA's
// `full` barrier (TMA with cta_group::2), so the even CTA's MMA thread learns of the odd CTA's
// data from the copy engine itself; its commits arrive on the `empty` / `tmem_full` barriers
// of both CTAs. (A thread-level remote arrive with release semantics in this loop costs
// microseconds per stage and throttles the pipeline below a third of the copy rate.) Each
// CTA's epilogue writes its own 128 feature rows (bf16, + residual).
struct Tc2Shape {
  static constexpr int kABytes = 128 * kKG;  // this CTA's weight rows
  static constexpr int kBBytes = 128 * kKG;  // this CTA's token half
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = 6;
  static constexpr int kSfBytes = 3 * 512;  // weight atom + two token atoms
  static constexpr int kRingBytes = kStages * kStageBytes;
  static constexpr int kSfRingBytes = kStages * kSfBytes;
  static constexpr int kSmemBytes = 1024 + kRingBytes + kSfRingBytes + 8 * (2 * kStages + 1) + 16;
  static constexpr int kSfSlots = 4;
  static constexpr int kSfCols = 12;  // 4 (weight scales) + 8 (token scales)
  static constexpr uint32_t kTmemCols = 512;  // 256 accumulator columns + kSfSlots * kSfCols
  static_assert(256 + kSfSlots * kSfCols <= 512, "tensor memory budget");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__global__ void __launch_bounds__(192) mx_gemm_tc2_kernel(const __grid_constant__ CUtensorMap tmW,
                                                             const __grid_constant__ CUtensorMap tmX,
                                                             const __grid_constant__ CUtensorMap tmSW,
                                                             const __grid_constant__ CUtensorMap tmSX,
                                                             const __grid_constant__ CUtensorMap tmO, const TcArgs a) {
  using S = Tc2Shape;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  uint8_t* sfring = smem + S::kRingBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(sfring + S::kSfRingBytes);  // used in the even CTA
  uint64_t* empty = full + S::kStages;
  uint64_t* tmem_full = empty + S::kStages;
  uint32_t* tmem_sh = reinterpret_cast<uint32_t*>(tmem_full + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int ntile = blockIdx.x, m0 = blockIdx.y * 256;
  const int n0 = ntile * 128;
  const int ng = a.groups;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tmem_full, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc2(tmem_sh, S::kTmemCols);
    tc::tmem_relinquish2();
  }
  tc::fence_before_sync();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers and TMEM exist before any cross-CTA signal
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_sh;

  if (warp == 0) {
    // ----------------------------------------------------------------- producer (both CTAs)
    if (lane == 0) {
      prefetch_tensormap(&tmW);
      prefetch_tensormap(&tmX);
      prefetch_tensormap(&tmSW);
      prefetch_tensormap(&tmSX);
      // the even CTA expects the bytes of both CTAs; the odd CTA's copies complete there too
      constexpr uint32_t tx = 2 * (S::kStageBytes + S::kSfBytes);
      const int pre = ng < S::kStages ? ng : S::kStages;
      for (int i = 0; i < pre; ++i) {  // weights read nothing produced upstream
        uint8_t* st = ring + i * S::kStageBytes;
        const uint32_t fb = mapa_shared(&full[i], 0);
        if (rank == 0) mbar_arrive_expect_tx(&full[i], tx);
        tma_load_2d_pair(st, &tmW, fb, i * kKG, n0);  // the weight map's box is 128 rows here
      }
      pdl_wait();
      pdl_trigger();
      int i = 0;
      for (; i < ng; ++i) {
        const int s = i % S::kStages;
        if (i >= S::kStages && !mbar_wait(&empty[s], ((i / S::kStages) - 1) & 1, a.err)) break;
        uint8_t* st = ring + s * S::kStageBytes;
        const uint32_t fb = mapa_shared(&full[s], 0);
        if (i >= pre) {
          if (rank == 0) mbar_arrive_expect_tx(&full[s], tx);
          tma_load_2d_pair(st, &tmW, fb, i * kKG, n0);
        }
        tma_load_2d_pair(st + S::kABytes, &tmX, fb, i * kKG, m0 + 128 * (int)rank);
        uint8_t* sf = sfring + s * S::kSfBytes;
        tma_load_2d_pair(sf, &tmSW, fb, ntile * 128, i);
        tma_load_2d_pair(sf + 512, &tmSX, fb, (m0 >> 7) * 128, i);
      }
      // Before this CTA may exit, every MMA that reads its stages has signalled (the last phase
      // of each stage's `empty`); those MMAs were issued only after all copies had landed.
      for (int j = i - S::kStages < 0 ? 0 : i - S::kStages; j < i; ++j)
        if (!mbar_wait(&empty[j % S::kStages], (j / S::kStages) & 1, a.err)) break;
    }
    __syncwarp();
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA issuer (even CTA)
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc0 = tc::idesc_mxf8(256, 0, 0, 256);
      for (int i = 0; i < ng; ++i) {
        const int s = i % S::kStages;
        if (!mbar_wait(&full[s], (i / S::kStages) & 1, a.err)) break;
        tc::fence_after_sync();
        const uint32_t t_sfa = tmem + 256 + (uint32_t)((i % S::kSfSlots) * S::kSfCols), t_sfb = t_sfa + 4;
        const uint32_t sa = smem_u32(ring + s * S::kStageBytes), sb = sa + S::kABytes;
        const uint32_t ssf = smem_u32(sfring + s * S::kSfBytes);
        tc::cp_sf_atom2(t_sfa, tc::desc_sf_atom(ssf));
        tc::cp_sf_atom2(t_sfb, tc::desc_sf_atom(ssf + 512));
        tc::cp_sf_atom2(t_sfb + 4, tc::desc_sf_atom(ssf + 1024));
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc::mma_mxf8_2(tmem, tc::desc_k128_sw128(sa + kk * 32), tc::desc_k128_sw128(sb + kk * 32),
                         idesc0 | ((uint32_t)kk << 4) | ((uint32_t)kk << 29), t_sfa, t_sfb, (i > 0 || kk > 0) ? 1u : 0u);
        tc::commit2_mc(&empty[s], (uint16_t)0x3);
      }
      tc::commit2_mc(tmem_full, (uint16_t)0x3);
    }
    __syncwarp();
  } else {
    // ----------------------------------------------------------------- epilogue
    const int q = warp & 3;
    const int r = 32 * q + lane;
    pdl_wait();
    // one thread polls the accumulator barrier for the four epilogue warps
    __shared__ int ok_sh;
    if (threadIdx.x == 64) ok_sh = mbar_wait(tmem_full, 0, a.err) ? 1 : 0;
    epi_bar();
    const bool ok = ok_sh != 0;
    tc::fence_after_sync();
    const uint32_t trow = tmem + ((uint32_t)(32 * q) << 16);
    const int n = n0 + r;
    if (a.tma_out) {
      // plain store: the warp stages each 16-token chunk of its 32 features ([16][32] bf16, 1 KB,
      // conflict-free row writes) in the now idle operand ring and hands it to a TMA store
      uint16_t* stg = reinterpret_cast<uint16_t*>(ring) + (size_t)q * (256 * 32);
      for (int c = 0; c < 256 && ok; c += 16) {
        float v[16];
        tc::ld16(trow + c, v);
        tc::wait_ld();
        uint16_t* ch = stg + c * 32;
#pragma unroll
        for (int j = 0; j < 16; ++j) ch[j * 32 + lane] = __bfloat16_as_ushort(__float2bfloat16_rn(v[j]));
        fence_proxy_async_smem();  // generic-proxy writes -> the TMA engine's reads
        __syncwarp();
        if (lane == 0 && n0 + 32 * q < a.N && m0 + c < a.M) {  // boxes are clipped at the edges
          tma_store_2d(&tmO, ch, n0 + 32 * q, m0 + c);
          bulk_commit_group();
        }
      }
      if (lane == 0) bulk_wait_group0();
      __syncwarp();
    } else {
      const bool nv = n < a.N;
      for (int c = 0; c < 256; c += 16) {
        float v[16];
        tc::ld16(trow + c, v);
        tc::wait_ld();
        if (!ok) continue;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int m = m0 + c + j;
          if (m < a.M && nv) {
            float y = v[j];
            if (a.residual) y += __bfloat162float(__ushort_as_bfloat16(a.residual[(int64_t)m * a.N + n]));
            uint16_t* dst = out_ptr(a, m, n);
            if (dst) *dst = __bfloat16_as_ushort(__float2bfloat16_rn(y));
          }
        }
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  cluster_sync_all();  // neither CTA frees its TMEM or leaves while the pair may still use it
  tc::fence_after_sync();
  if (warp == 1) tc::tmem_dealloc2(tmem, S::kTmemCols);
}

// Persistent form of the CTA-pair kernel for plain bf16 stores (config-5 GEMMs). One cluster
// (CTA pair) per two SMs walks tiles pair, pair + P, ... of a grouped raster order: `group`
// token-tile rows at a time, weight-tile columns within a group, so that the tiles in flight
// together share their weight and token panels in L2. The operand ring streams across tile
// boundaries without draining. The MMA warp starts a tile once the epilogue warps of both CTAs
// have read the previous tile's accumulator out of TMEM (acc_empty, in the even CTA, 8
// arrivals); the epilogue then converts and stores from registers through a double-buffered
// staging area with TMA while the next tile accumulates. The scale atoms of a stage arrive with
// its operands; a seventh warp copies them to TMEM (slot stage % kSfStages) and commits to the
// stage's sf_ready barrier, which is what the MMA thread waits for: with the copies issued by
// the MMA thread itself, its per-stage issue work (~720 cycles) exceeded the MMAs' (~590).
struct Tc2pShape {
  static constexpr int kABytes = 128 * kKG;
  static constexpr int kBBytes = 128 * kKG;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = 6;
  static constexpr int kSfBytes = 3 * 512;
  static constexpr int kSfStages = 8;  // TMEM scale slots
  static constexpr int kRingBytes = kStages * kStageBytes;
  static constexpr int kSfRingBytes = kStages * kSfBytes;
  static constexpr int kChunkBytes = 16 * 32 * 2;          // [16 tokens][32 features] bf16
  static constexpr int kStgBytes = 4 * 2 * kChunkBytes;    // two chunks per epilogue warp
  static constexpr int kSmemBytes = 1024 + kRingBytes + kSfRingBytes + kStgBytes + 8 * (3 * kStages + 2) + 16;
  static constexpr int kThreads = 224;  // producer, MMA, 4 epilogue warps, scale copier
  static constexpr int kSfCols = 12;
  static constexpr uint32_t kTmemCols = 512;
  static_assert(256 + kSfStages * kSfCols <= 512, "tensor memory budget");
  // the copier fills TMEM scale slot x % kSfStages after stage x's operands landed, which the
  // producer could load only once the MMAs of stage x - kStages completed
  static_assert(kSfStages >= kStages, "TMEM scale slot reuse");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

__device__ __forceinline__ void bulk_wait_group_read1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}

// arrive on an mbarrier given by its shared::cluster address (this CTA's or a peer's)
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cl) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(bar_cl) : "memory");
}

__device__ __forceinline__ void tc2p_tile(int t, int tiles_m, int tiles_n, int group, int& tm, int& tn) {
  const int gsz = group * tiles_n;
  const int g = t / gsz, r = t - g * gsz;
  const int rows = min(group, tiles_m - g * group);
  tm = g * group + r % rows;
  tn = r / rows;
}

__global__ void __launch_bounds__(Tc2pShape::kThreads, 1) mx_gemm_tc2p_kernel(const __grid_constant__ CUtensorMap tmW,
                                                                const __grid_constant__ CUtensorMap tmX,
                                                                const __grid_constant__ CUtensorMap tmSW,
                                                                const __grid_constant__ CUtensorMap tmSX,
                                                                const __grid_constant__ CUtensorMap tmO,
                                                                const TcArgs a, int tiles_m, int tiles_n, int group) {
  using S = Tc2pShape;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  uint8_t* sfring = smem + S::kRingBytes;
  uint8_t* stg_base = sfring + S::kSfRingBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(stg_base + S::kStgBytes);  // used in the even CTA
  uint64_t* empty = full + S::kStages;
  uint64_t* sf_ready = empty + S::kStages;  // used in the even CTA
  uint64_t* tmem_full = sf_ready + S::kStages;
  uint64_t* acc_empty = tmem_full + 1;  // used in the even CTA
  uint32_t* tmem_sh = reinterpret_cast<uint32_t*>(acc_empty + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int P = (int)(gridDim.x >> 1), pair = (int)(blockIdx.x >> 1);
  const int T = tiles_m * tiles_n;
  const int ng = a.groups;
  const int my_tiles = pair < T ? (T - 1 - pair) / P + 1 : 0;
  const int nstages = my_tiles * ng;  // operand stages this pair runs

  if (threadIdx.x == 0) {
    for (int s = 0; s < S::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&sf_ready[s], 1);
    }
    mbar_init(tmem_full, 1);
    mbar_init(acc_empty, 8);  // four epilogue warps of each CTA
    fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc2(tmem_sh, S::kTmemCols);
    tc::tmem_relinquish2();
  }
  tc::fence_before_sync();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers and TMEM exist before any cross-CTA signal
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_sh;

  if (warp == 0) {
    // ----------------------------------------------------------------- producer (both CTAs)
    if (lane == 0) {
      prefetch_tensormap(&tmW);
      prefetch_tensormap(&tmX);
      prefetch_tensormap(&tmSW);
      prefetch_tensormap(&tmSX);
      // the even CTA expects the bytes of both CTAs; the odd CTA's copies complete there too
      constexpr uint32_t tx = 2 * (S::kStageBytes + S::kSfBytes);
      int pre = 0;
      if (pair < T) {  // the first tile's weights read nothing produced upstream
        int tm, tn;
        tc2p_tile(pair, tiles_m, tiles_n, group, tm, tn);
        pre = ng < S::kStages ? ng : S::kStages;
        for (int i = 0; i < pre; ++i) {
          const uint32_t fb = mapa_shared(&full[i], 0);
          if (rank == 0) mbar_arrive_expect_tx(&full[i], tx);
          tma_load_2d_pair(ring + i * S::kStageBytes, &tmW, fb, i * kKG, (2 * tn + (int)rank) * 128);
        }
      }
      pdl_wait();
      pdl_trigger();
      int it = 0;
      bool live = true;
      for (int t = pair; t < T && live; t += P) {
        int tm, tn;
        tc2p_tile(t, tiles_m, tiles_n, group, tm, tn);
        const int wrow = (2 * tn + (int)rank) * 128;  // this CTA's 128 weight rows
        const int xrow = tm * 256 + 128 * (int)rank;  // this CTA's 128-token half
        for (int k = 0; k < ng; ++k, ++it) {
          const int s = it % S::kStages;
          if (it >= S::kStages && !mbar_wait(&empty[s], ((it / S::kStages) - 1) & 1, a.err)) {
            live = false;
            break;
          }
          uint8_t* st = ring + s * S::kStageBytes;
          const uint32_t fb = mapa_shared(&full[s], 0);
          if (it >= pre) {
            if (rank == 0) mbar_arrive_expect_tx(&full[s], tx);
            tma_load_2d_pair(st, &tmW, fb, k * kKG, wrow);
          }
          tma_load_2d_pair(st + S::kABytes, &tmX, fb, k * kKG, xrow);
          uint8_t* sf = sfring + s * S::kSfBytes;
          tma_load_2d_pair(sf, &tmSW, fb, (2 * tn + (int)rank) * 128, k);
          tma_load_2d_pair(sf + 512, &tmSX, fb, tm * 256, k);
        }
      }
      // Before this CTA may exit, every MMA that reads its stages has signalled (the last phase
      // of each stage's `empty`); those MMAs were issued only after all copies had landed.
      for (int j = it - S::kStages < 0 ? 0 : it - S::kStages; j < it; ++j)
        if (!mbar_wait(&empty[j % S::kStages], (j / S::kStages) & 1, a.err)) break;
    }
    __syncwarp();
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA issuer (even CTA)
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc0 = tc::idesc_mxf8(256, 0, 0, 256);
      int it = 0, tl = 0;
      bool live = true;
      for (int t = pair; t < T && live; t += P, ++tl) {
        if (tl > 0) {  // both CTAs' epilogues have read the previous tile's accumulator
          if (!mbar_wait(acc_empty, (tl - 1) & 1, a.err)) break;
          tc::fence_after_sync();
        }
        for (int k = 0; k < ng; ++k, ++it) {
          const int s = it % S::kStages;
          // the stage's operands have landed and its scales are in TMEM (the copier's commit)
          if (!mbar_wait(&sf_ready[s], (it / S::kStages) & 1, a.err)) {
            live = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t t_sfa = tmem + 256 + (uint32_t)((it % S::kSfStages) * S::kSfCols), t_sfb = t_sfa + 4;
          const uint32_t sa = smem_u32(ring + s * S::kStageBytes), sb = sa + S::kABytes;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc::mma_mxf8_2(tmem, tc::desc_k128_sw128(sa + kk * 32), tc::desc_k128_sw128(sb + kk * 32),
                           idesc0 | ((uint32_t)kk << 4) | ((uint32_t)kk << 29), t_sfa, t_sfb, (k > 0 || kk > 0) ? 1u : 0u);
          tc::commit2_mc(&empty[s], (uint16_t)0x3);
        }
        if (live) tc::commit2_mc(tmem_full, (uint16_t)0x3);
      }
    }
    __syncwarp();
  } else if (warp == 6) {
    // ----------------------------------------------------------------- scale copier (even CTA)
    if (lane == 0 && rank == 0) {
      for (int it = 0; it < nstages; ++it) {
        const int s = it % S::kStages, j = it % S::kSfStages;
        if (!mbar_wait(&full[s], (it / S::kStages) & 1, a.err)) break;
        tc::fence_after_sync();
        const uint32_t t_sfa = tmem + 256 + (uint32_t)(j * S::kSfCols), t_sfb = t_sfa + 4;
        const uint32_t ssf = smem_u32(sfring + s * S::kSfBytes);
        tc::cp_sf_atom2(t_sfa, tc::desc_sf_atom(ssf));
        tc::cp_sf_atom2(t_sfb, tc::desc_sf_atom(ssf + 512));
        tc::cp_sf_atom2(t_sfb + 4, tc::desc_sf_atom(ssf + 1024));
        tc::commit2_mc(&sf_ready[s], (uint16_t)0x1);  // arrives once the copies are done
      }
    }
    __syncwarp();
  } else {
    // ----------------------------------------------------------------- epilogue (both CTAs)
    const int q = warp & 3;
    pdl_wait();
    __shared__ int ok_sh[2];  // one thread polls the accumulator barrier for the four warps
    uint16_t* stg = reinterpret_cast<uint16_t*>(stg_base + q * 2 * S::kChunkBytes);
    const uint32_t ae = mapa_shared(acc_empty, 0);  // the even CTA's barrier
    const uint32_t trow = tmem + ((uint32_t)(32 * q) << 16);
    int tl = 0, nchunk = 0;
    for (int t = pair; t < T; t += P, ++tl) {
      int tm, tn;
      tc2p_tile(t, tiles_m, tiles_n, group, tm, tn);
      const int n0 = (2 * tn + (int)rank) * 128, m0 = tm * 256;
      if (threadIdx.x == 64) ok_sh[tl & 1] = mbar_wait(tmem_full, tl & 1, a.err) ? 1 : 0;
      epi_bar();
      if (!ok_sh[tl & 1]) break;
      tc::fence_after_sync();
      // the row's 256 accumulators, as bf16 pairs (token 2i low, 2i + 1 high)
      uint32_t pk[128];
#pragma unroll
      for (int c = 0; c < 256; c += 32) {
        float v[32];
        tc::ld16(trow + c, *reinterpret_cast<float(*)[16]>(v));
        tc::ld16(trow + c + 16, *reinterpret_cast<float(*)[16]>(v + 16));
        tc::wait_ld();
#pragma unroll
        for (int j = 0; j < 32; j += 2)
          pk[(c + j) >> 1] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[j])) |
                             ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v[j + 1])) << 16);
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(ae);  // the accumulator may take the next tile
      // each warp owns features n0 + 32q .. + 31 (its lanes) of all 256 tokens: 16 chunks of 16
      // tokens, staged [token][feature] and written by TMA (clipped at the edges)
#pragma unroll
      for (int c = 0; c < 256; c += 16, ++nchunk) {
        uint16_t* ch = stg + (nchunk & 1) * (16 * 32);
        if (nchunk >= 2) {
          if (lane == 0) bulk_wait_group_read1();  // the store that last read this buffer is done
          __syncwarp();
        }
#pragma unroll
        for (int j = 0; j < 16; j += 2) {
          ch[j * 32 + lane] = (uint16_t)(pk[(c + j) >> 1] & 0xFFFFu);
          ch[(j + 1) * 32 + lane] = (uint16_t)(pk[(c + j) >> 1] >> 16);
        }
        fence_proxy_async_smem();  // generic-proxy writes -> the TMA engine's reads
        __syncwarp();
        if (lane == 0) {
          if (n0 + 32 * q < a.N && m0 + c < a.M) tma_store_2d(&tmO, ch, n0 + 32 * q, m0 + c);
          bulk_commit_group();
        }
      }
    }
    if (lane == 0) bulk_wait_group0();
    __syncwarp();
  }
  tc::fence_before_sync();
  __syncthreads();
  cluster_sync_all();  // neither CTA frees its TMEM or leaves while the pair may still use it
  tc::fence_after_sync();
  if (warp == 1) tc::tmem_dealloc2(tmem, S::kTmemCols);
}

// ---------------------------------------------------------------------------------- host
namespace {

int pick_bn(int64_t M) { return M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : 128; }

struct Plan {
  int bn, ntiles, mtiles, splits;
};

template <int BN>
int max_clusters(int cs) {
  // how many clusters of `cs` CTAs of the split-K kernel can be resident at once (1 CTA/SM)
  static int cache[9] = {0, 0, 0, 0, 0, 0, 0, 0, 0};
  if (cache[cs]) return cache[cs];
  using S = TcShape<BN>;
  cudaFuncSetAttribute(mx_gemm_tc_kernel<BN, kEpiSplit>, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmemBytes);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1, 1, cs);
  cfg.blockDim = dim3(192);
  cfg.dynamicSmemBytes = S::kSmemBytes;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 1;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = cs;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, mx_gemm_tc_kernel<BN, kEpiSplit>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 152 / cs;
  }
  cache[cs] = n > 0 ? n : 1;
  return cache[cs];
}

int max_clusters_bn(int bn, int cs) {
  switch (bn) {
    case 16: return max_clusters<16>(cs);
    case 32: return max_clusters<32>(cs);
    case 64: return max_clusters<64>(cs);
    case 128: return max_clusters<128>(cs);
    default: return max_clusters<256>(cs);
  }
}

Plan plan_gemm(int64_t M, int64_t N, int64_t K) {
  Plan p;
  p.bn = M > 1024 ? 256 : pick_bn(M);
  p.ntiles = (int)((N + 127) / 128);
  if (p.bn == 256) p.ntiles = (p.ntiles + 1) & ~1;  // CTA pairs along x (one M=256 MMA per pair)
  p.mtiles = (int)((M + p.bn - 1) / p.bn);
  const int groups = (int)(K / kKG);
  const int64_t ctas = (int64_t)p.ntiles * p.mtiles;
  // split K over a cluster of S <= 8 CTAs (the portable cluster size) when the tiles alone
  // cannot cover the 152 SMs, keeping the launch within one wave (one CTA per SM);
  // N % 4 == 0 keeps the 4-wide reduction stores aligned
  // (the largest S whose clusters are all resident together: no second wave)
  p.splits = 1;
  if (ctas < 120 && N % 4 == 0) {
    int s = (int)(152 / ctas);
    if (s > 8) s = 8;
    if (s > groups) s = groups;
    while (s > 1 && (int64_t)max_clusters_bn(p.bn, s) < ctas) --s;
    p.splits = s < 1 ? 1 : s;
  }
  return p;
}

template <int BN, int EPI>
cudaError_t launch_tc(const CUtensorMap& tw, const CUtensorMap& tx, const TcArgs& a, dim3 grid, cudaStream_t st) {
  using S = TcShape<BN>;
  cudaError_t e = cudaFuncSetAttribute(mx_gemm_tc_kernel<BN, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       S::kSmemBytes);
  if (e != cudaSuccess) return e;
  const dim3 cluster = EPI == kEpiSplit ? dim3(1, 1, grid.z) : dim3(1, 1, 1);
  return launch_kc(mx_gemm_tc_kernel<BN, EPI>, grid, dim3(192), S::kSmemBytes, st, cluster, tw, tx, a);
}

// token-tile rows per raster group of the persistent pair kernel
constexpr int kRasterGroup = 8;

// CTA pairs of the persistent kernel that are resident at once (queried once)
int tc2p_pairs() {
  static int cache = 0;
  if (cache) return cache;
  using P2 = Tc2pShape;
  cudaFuncSetAttribute(mx_gemm_tc2p_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, P2::kSmemBytes);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * 76, 1, 1);
  cfg.blockDim = dim3(P2::kThreads);
  cfg.dynamicSmemBytes = P2::kSmemBytes;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, mx_gemm_tc2p_kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 76;
  }
  cache = n > 0 ? n : 1;
  return cache;
}

cudaError_t launch_tc2(const CUtensorMap& tw, const CUtensorMap& tx, const TcArgs& a, dim3 grid, cudaStream_t st) {
  using S = Tc2Shape;
  if (!a.wsp || (grid.x & 1) || grid.z != 1) return cudaErrorInvalidValue;
  // packed scale atoms as 2-D u32 tensors [K/128][row tiles * 128]: one 512-byte atom (weights)
  // or two adjacent atoms (the 256 tokens) per load
  CUtensorMap tsw, tsx;
  if (!make_tensor_map_2d(&tsw, CU_TENSOR_MAP_DATA_TYPE_UINT32, a.wsp, (uint64_t)a.rt_w * 128, (uint64_t)a.groups,
                          (uint64_t)a.rt_w * 512, 128, 1, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !make_tensor_map_2d(&tsx, CU_TENSOR_MAP_DATA_TYPE_UINT32, a.xsp, (uint64_t)a.rt_x * 128, (uint64_t)a.groups,
                          (uint64_t)a.rt_x * 512, 256, 1, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  // bf16 output [M][N] for the staged epilogue (boxes of 32 features x 16 tokens); a residual,
  // a KV scatter or an output the copy engine cannot address keeps the per-element stores
  CUtensorMap tso{};
  TcArgs b = a;
  b.tma_out = a.residual == nullptr && a.kv.kc == nullptr &&
              make_tensor_map_2d(&tso, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.out, (uint64_t)a.N, (uint64_t)a.M,
                                 (uint64_t)a.N * 2, 32, 16, CU_TENSOR_MAP_SWIZZLE_NONE);
  cudaError_t e;
  if (b.tma_out) {
    // plain stores: the persistent kernel, one CTA pair per two SMs (all resident at once)
    using P2 = Tc2pShape;
    e = cudaFuncSetAttribute(mx_gemm_tc2p_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, P2::kSmemBytes);
    if (e != cudaSuccess) return e;
    const int tiles_n = (int)(grid.x / 2), tiles_m = (int)grid.y;
    const int T = tiles_n * tiles_m;
    int pairs = tc2p_pairs();
    if (pairs > T) pairs = T;
    return launch_kc(mx_gemm_tc2p_kernel, dim3(2u * (unsigned)pairs), dim3(P2::kThreads), P2::kSmemBytes, st, dim3(2, 1, 1),
                     tw, tx, tsw, tsx, tso, b, tiles_m, tiles_n, kRasterGroup);
  }
  e = cudaFuncSetAttribute(mx_gemm_tc2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmemBytes);
  if (e != cudaSuccess) return e;
  return launch_kc(mx_gemm_tc2_kernel, grid, dim3(192), S::kSmemBytes, st, dim3(2, 1, 1), tw, tx, tsw, tsx, tso, b);
}

template <int EPI>
cudaError_t launch_tc_bn(int bn, const CUtensorMap& tw, const CUtensorMap& tx, const TcArgs& a, dim3 grid,
                         cudaStream_t st) {
  switch (bn) {
    case 16: return launch_tc<16, EPI>(tw, tx, a, grid, st);
    case 32: return launch_tc<32, EPI>(tw, tx, a, grid, st);
    case 64: return launch_tc<64, EPI>(tw, tx, a, grid, st);
    case 128: return launch_tc<128, EPI>(tw, tx, a, grid, st);
    default:
      if constexpr (EPI == kEpiStore) return launch_tc2(tw, tx, a, grid, st);
      else if constexpr (EPI == kEpiSplit) return launch_tc<256, kEpiSplit>(tw, tx, a, grid, st);
      else return cudaErrorInvalidValue;  // the SwiGLU epilogue tiles at most 128 tokens
  }
}

bool maps(CUtensorMap* tw, CUtensorMap* tx, const uint8_t* wq, int64_t wrows, const uint8_t* xq, int64_t M, int64_t K,
          int bn, uint32_t wbox = 64) {
  if (bn > 128) bn /= 2;  // 256-token tiles are loaded as two 128-row halves
  return make_tensor_map_2d(tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, wq, (uint64_t)K, (uint64_t)wrows, (uint64_t)K, kKG, wbox,
                            CU_TENSOR_MAP_SWIZZLE_128B) &&
         make_tensor_map_2d(tx, CU_TENSOR_MAP_DATA_TYPE_UINT8, xq, (uint64_t)K, (uint64_t)M, (uint64_t)K, kKG,
                            (uint32_t)bn, CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace

bool tc_gemm_supported(int64_t M, int64_t N, int64_t K) {
  return M > 0 && K % kKG == 0 && N % 8 == 0 && K / kKG >= 1 && M < (1ll << 31) && N < (1ll << 31);
}

namespace {
// Large GEMMs (256-token tiles) read pre-packed scale atoms: [K/128][rt_w][512 B] for the
// weight operand, then [K/128][rt_x][512 B] for the token operand (rt_x padded to whole tiles).
struct PackPlan {
  int rt_w = 0, rt_x = 0, groups = 0;
  size_t w_bytes = 0, bytes = 0;
};
PackPlan pack_plan(const Plan& p, int64_t M, int64_t N, int64_t K) {
  PackPlan q;
  if (p.bn != 256) return q;
  q.groups = (int)(K / kKG);
  q.rt_w = p.ntiles;  // even: the CTA pairs of the M=256 MMA read whole pairs of weight tiles
  (void)N;
  q.rt_x = p.mtiles * (p.bn / 128);
  (void)M;
  q.w_bytes = (size_t)q.groups * q.rt_w * 512;
  q.bytes = q.w_bytes + (size_t)q.groups * q.rt_x * 512;
  return q;
}
}  // namespace

size_t tc_gemm_workspace(int64_t M, int64_t N, int64_t K) {
  // split-K partials are reduced inside a cluster through distributed shared memory (no
  // scratch); only large GEMMs need scratch, for their pre-packed scales
  if (!tc_gemm_supported(M, N, K)) return 0;
  return pack_plan(plan_gemm(M, N, K), M, N, K).bytes;
}

cudaError_t launch_mx_gemm_tc(const uint8_t* xq, const uint8_t* xs, const uint8_t* wq, const uint8_t* ws, int64_t M,
                              int64_t N, int64_t K, const uint16_t* residual, uint16_t* out, void* workspace,
                              int32_t* err, cudaStream_t st, bool* unsupported, const KvScatter* kv) {
  const Plan p = plan_gemm(M, N, K);
  CUtensorMap tw, tx;
  *unsupported = false;
  // the CTA-pair kernel (256-token tiles, no split) loads its 128 weight rows as one box
  if (!maps(&tw, &tx, wq, N, xq, M, K, p.bn, p.bn == 256 && p.splits == 1 ? 128 : 64)) {
    *unsupported = true;
    return cudaSuccess;
  }
  TcArgs a{};
  a.M = (int)M;
  a.N = (int)N;
  a.K = (int)K;
  a.groups = (int)(K / kKG);
  a.splits = p.splits;
  a.ws = ws;
  a.xs = xs;
  a.residual = residual;
  a.out = out;
  a.err = err;
  if (kv) a.kv = *kv;
  dim3 grid((unsigned)p.ntiles, (unsigned)p.mtiles, (unsigned)p.splits);
  const PackPlan q = pack_plan(p, M, N, K);
  if (q.bytes) {
    uint32_t* pw = static_cast<uint32_t*>(workspace);
    uint32_t* px = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(workspace) + q.w_bytes);
    const int64_t KB = K / 32;
    cudaError_t e = launch_k(pack_scales_kernel, dim3(1024), dim3(256), 0, st, 1, ws, N, KB, q.rt_w, q.groups, pw);
    if (e != cudaSuccess) return e;
    e = launch_k(pack_scales_kernel, dim3(1024), dim3(256), 0, st, 1, xs, M, KB, q.rt_x, q.groups, px);
    if (e != cudaSuccess) return e;
    a.wsp = pw;
    a.xsp = px;
    a.rt_w = q.rt_w;
    a.rt_x = q.rt_x;
  }
  if (p.splits > 1) return launch_tc_bn<kEpiSplit>(p.bn, tw, tx, a, grid, st);
  return launch_tc_bn<kEpiStore>(p.bn, tw, tx, a, grid, st);
}

cudaError_t launch_gate_up_swiglu_tc(const uint8_t* xq, const uint8_t* xs, int64_t M, int64_t d_model, int64_t d_ff,
                                     const uint8_t* w13q, const uint8_t* w13s, uint8_t* hq, uint8_t* hs, int32_t* err,
                                     cudaStream_t st, bool* unsupported) {
  const int bn = pick_bn(M);
  CUtensorMap tw, tx;
  *unsupported = false;
  if (d_model % kKG || d_ff % 64 || !maps(&tw, &tx, w13q, 2 * d_ff, xq, M, d_model, bn)) {
    *unsupported = true;
    return cudaSuccess;
  }
  TcArgs a{};
  a.M = (int)M;
  a.N = (int)(2 * d_ff);
  a.K = (int)d_model;
  a.groups = (int)(d_model / kKG);
  a.splits = 1;
  a.ws = w13s;
  a.xs = xs;
  a.d_ff = (int)d_ff;
  a.hq = hq;
  a.hs = hs;
  a.err = err;
  dim3 grid((unsigned)(d_ff / 64), (unsigned)((M + bn - 1) / bn), 1);
  return launch_tc_bn<kEpiSwiGLU>(bn, tw, tx, a, grid, st);
}

}  // namespace mxg

MXG_TL_UNIT(gemm_tc)
