// The whole decode-size MXFP8 SwiGLU MLP in one persistent tcgen05 kernel (sm_103a).
//
// [S2.1] "Kernel Benchmark Results" / "FP8 Quantization Strategy": quantise -> gate/up ->
// SwiGLU -> quantise -> down, MX (1x32, E4M3 + UE8M0) operands, no bf16 intermediate. At
// decode sizes (M <= 128 tokens) the MLP is a weight stream: 2*d_ff*d_model + d_model*d_ff
// E4M3 bytes plus scales. Split into a gate/up launch and a down launch, each launch pays its
// own ramp (first bytes ~2 us after the start) and drain, and W2 cannot start streaming
// until gate/up has left the SMs. Here one CTA per SM streams its share of W13 and then, with
// no break, its share of W2:
//
//   phase 1  CTA j owns d_ff columns [64j, 64j + 64): the weight tile is 64 gate rows + the
//            matching 64 up rows (the MMA's 128 rows; tokens are the MMA N), accumulated in
//            TMEM. The epilogue forms h = silu(g) * u in fp32, MX-quantises it along d_ff and
//            writes (hq, hs); then the CTA counts itself in a global counter.
//   phase 2  CTA c < T2*S2 owns (row tile t = c / S2, split z = c % S2) of the down GEMM:
//            W2 rows [128t, 128t + 128) over the K-groups [z*NG2/S2, (z+1)*NG2/S2) of d_ff.
//            Its W2 tiles enter the ring as soon as phase-1 slots free up -- ahead of h -- so
//            the HBM stream does not stop while phase 1 drains; the h tiles (the MMA's B
//            operand) are loaded once every phase-1 tile has been counted.
//   reduce   each CTA stores its fp32 partial tile, counts itself in its row tile's counter,
//            waits for the tile's S2 partials and sums one slice of the tile over the splits
//            in split order (deterministic), adds the residual and writes bf16 y.
//
// The split boundaries, the per-split accumulation order and the split order of the sum are
// those of the two-launch path (gate/up kernel + split-K down kernel), so both give the same
// bits. Two rings: weight tiles (16 KB + their scale atom) run as far ahead as the ring
// allows; token tiles (x in phase 1, h in phase 2) follow just in time.
//
// Every wait is bounded (MXG_ETIMEOUT in the status word); TMEM is always released; all CTAs
// reach the exit, and the last one returns the counters to zero for the next call.
#include "kernels.h"
#include "launch.cuh"
#include "tc.cuh"

namespace mxg {

namespace {

constexpr int kKG = 128;         // K elements per stage (one 4-block group of UE8M0 scales)
constexpr int kWBytes = 128 * kKG;  // one weight tile: 128 rows x 128 K
constexpr int kTokStages = 4;    // token-tile ring depth
constexpr int kChunk = 16;       // tokens per SwiGLU staging chunk
constexpr int kLine = 32;        // int32 words per control word (one 128-byte line each)
constexpr int kMaxSplit = 8;     // splits per down-projection row tile

template <int BN>
struct FuseShape {
  static constexpr int kTBytes = BN * kKG;                       // one token tile
  static constexpr int kStgBytes = 128 * (kChunk + 1) * 4;       // SwiGLU staging [128 rows][17]
  static constexpr int kFixed = 1024 + kTokStages * (kTBytes + 512) + kStgBytes + 1024;
  static constexpr int kWStagesRaw = (227 * 1024 - kFixed) / (kWBytes + 512);
  static constexpr int kWStages = kWStagesRaw > 12 ? 12 : kWStagesRaw;
  static constexpr int kWRing = kWStages * kWBytes;
  static constexpr int kTRing = kTokStages * kTBytes;
  static constexpr int kSfW = kWRing + kTRing;                   // weight scale atoms [kWStages][512]
  static constexpr int kSfT = kSfW + kWStages * 512;             // token scale atoms [kTokStages][512]
  static constexpr int kStg = kSfT + kTokStages * 512;
  static constexpr int kBars = kStg + kStgBytes;
  static constexpr int kNumBars = 2 * kWStages + 2 * kTokStages + 2;
  static constexpr int kSmemBytes = 1024 + kBars + 8 * kNumBars + 16;
  // TMEM: phase-1 accumulator [0, BN), phase-2 accumulator [BN, 2BN), then 4 rotating slots of
  // 8 scale columns (weight atom, token atom)
  static constexpr int kSfSlots = 4;
  static constexpr int kTmemNeed = 2 * BN + kSfSlots * 8;
  static constexpr uint32_t kTmemCols = kTmemNeed <= 64 ? 64 : kTmemNeed <= 128 ? 128 : kTmemNeed <= 256 ? 256 : 512;
  static_assert(kWStages >= 6, "weight ring depth");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

struct FuseArgs {
  int M, d_model, d_ff;
  int T1, T2, S2, NG1, NG2;
  const uint8_t* xs;    // [M][d_model/32]
  const uint8_t* w13s;  // [2*d_ff][d_model/32]
  const uint8_t* w2s;   // [d_model][d_ff/32]
  uint8_t* hq;          // [M][d_ff]
  uint8_t* hs;          // [M][d_ff/32]
  float* part;          // [T2*S2][M][128] split partials
  int* ctrl;            // control words, one per 128-byte line: [0] phase-1 tiles done,
                        // [1 .. T2] partials of row tile t, [T2+1] CTAs done, [T2+2] status
  const uint16_t* residual;
  uint16_t* y;
};

__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void red_release_gpu_add(int* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int atom_acq_rel_gpu_add(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Bounded spin until *p >= target (acquire); every lane of the calling warp polls, the outcome
// is warp-uniform. Records MXG_ETIMEOUT and returns false after kWaitLimitNs.
__device__ __forceinline__ bool wait_count(const int* p, int target, int32_t* status) {
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (__all_sync(MXG_FULL_MASK, ld_acquire_gpu(p) >= target)) return true;
    if (__any_sync(MXG_FULL_MASK, globaltimer_ns() - t0 > kWaitLimitNs)) {
      if ((threadIdx.x & 31) == 0) set_error(status, MXG_ETIMEOUT);
      return false;
    }
    __nanosleep(64);
  }
}

}  // namespace

template <int BN>
__global__ void __launch_bounds__(192, 1) mlp_fused_kernel(const __grid_constant__ CUtensorMap tmW13,
                                                            const __grid_constant__ CUtensorMap tmX,
                                                            const __grid_constant__ CUtensorMap tmW2,
                                                            const __grid_constant__ CUtensorMap tmH, const FuseArgs a) {
  using S = FuseShape<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* wring = smem;
  uint8_t* tring = smem + S::kWRing;
  uint32_t* sfw = reinterpret_cast<uint32_t*>(smem + S::kSfW);
  uint32_t* sft = reinterpret_cast<uint32_t*>(smem + S::kSfT);
  float* stg = reinterpret_cast<float*>(smem + S::kStg);
  uint64_t* wfull = reinterpret_cast<uint64_t*>(smem + S::kBars);
  uint64_t* wempty = wfull + S::kWStages;
  uint64_t* tfull = wempty + S::kWStages;
  uint64_t* tempty = tfull + kTokStages;
  uint64_t* acc1_full = tempty + kTokStages;
  uint64_t* acc2_full = acc1_full + 1;
  uint32_t* tmem_sh = reinterpret_cast<uint32_t*>(acc2_full + 1);
  __shared__ int sh_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x, G = gridDim.x;
  int* const cnt1 = a.ctrl;
  int* const done = a.ctrl + (a.T2 + 1) * kLine;
  int32_t* const status = a.ctrl + (a.T2 + 2) * kLine;
  // phase 1: tile c; phase 2: (row tile t2, split z2) = (c / S2, c % S2)
  const int n1 = c < a.T1 ? a.NG1 : 0;
  const bool has2 = c < a.T2 * a.S2;
  const int t2 = has2 ? c / a.S2 : 0, z2 = has2 ? c % a.S2 : 0;
  const int g2a = (int)((int64_t)z2 * a.NG2 / a.S2);
  const int n2 = has2 ? (int)((int64_t)(z2 + 1) * a.NG2 / a.S2) - g2a : 0;
  const int total = n1 + n2;
  const int64_t KB1 = a.d_model >> 5, KB2 = a.d_ff >> 5;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S::kWStages; ++s) {
      mbar_init(&wfull[s], 1 + 32);  // TMA expect-tx arrive + one cp.async arrive per producer lane
      mbar_init(&wempty[s], 1);
    }
    for (int s = 0; s < kTokStages; ++s) {
      mbar_init(&tfull[s], 1 + 32);
      mbar_init(&tempty[s], 1);
    }
    mbar_init(acc1_full, 1);
    mbar_init(acc2_full, 1);
    sh_flag = 0;
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
  const uint32_t t_acc1 = tmem, t_acc2 = tmem + BN, t_sf = tmem + 2 * BN;

  if (warp == 0) {
    // ----------------------------------------------------------------- producer
    if (lane == 0) {
      prefetch_tensormap(&tmW13);
      prefetch_tensormap(&tmX);
      prefetch_tensormap(&tmW2);
      prefetch_tensormap(&tmH);
    }
    // weight stage i: TMA of the 128-row tile (two 64-row boxes) + the 128 rows' scale words
    // of the stage's K-group, gathered by the 32 lanes into the 32x4 atom layout
    auto issue_w = [&](int i) {
      const int s = i % S::kWStages;
      uint8_t* st = wring + s * kWBytes;
      uint32_t* atom = sfw + s * 128;
      if (i < n1) {
        const int g = i;
        if (lane == 0) {
          mbar_arrive_expect_tx(&wfull[s], kWBytes);
          tma_load_2d(st, &tmW13, &wfull[s], g * kKG, c * 64);                      // gate rows
          tma_load_2d(st + 64 * kKG, &tmW13, &wfull[s], g * kKG, a.d_ff + c * 64);  // up rows
        }
#pragma unroll
        for (int r1 = 0; r1 < 4; ++r1) {
          const int r = lane + 32 * r1;
          const int64_t grow = r < 64 ? (int64_t)c * 64 + r : (int64_t)a.d_ff + c * 64 + (r - 64);
          tc::cp_async4(&atom[4 * lane + r1], a.w13s + grow * KB1 + 4 * g);
        }
      } else {
        const int g = g2a + (i - n1);
        if (lane == 0) {
          mbar_arrive_expect_tx(&wfull[s], kWBytes);
          tma_load_2d(st, &tmW2, &wfull[s], g * kKG, t2 * 128);
          tma_load_2d(st + 64 * kKG, &tmW2, &wfull[s], g * kKG, t2 * 128 + 64);
        }
#pragma unroll
        for (int r1 = 0; r1 < 4; ++r1) {
          const int r = lane + 32 * r1;
          tc::cp_async4(&atom[4 * lane + r1], a.w2s + (int64_t)(t2 * 128 + r) * KB2 + 4 * g);
        }
      }
      tc::cp_async_arrive(&wfull[s]);
    };
    // token stage i: TMA of the token tile (x or h; rows >= M are zero-filled) + token scales
    auto issue_t = [&](int i) {
      const int s = i % kTokStages;
      uint8_t* st = tring + s * S::kTBytes;
      uint32_t* atom = sft + s * 128;
      const bool p1 = i < n1;
      const int g = p1 ? i : g2a + (i - n1);
      if (lane == 0) {
        mbar_arrive_expect_tx(&tfull[s], S::kTBytes);
        tma_load_2d(st, p1 ? &tmX : &tmH, &tfull[s], g * kKG, 0);
      }
      const uint8_t* sc = p1 ? a.xs : a.hs;
      const int64_t kb = p1 ? KB1 : KB2;
#pragma unroll
      for (int r1 = 0; r1 < 4; ++r1) {
        const int r = lane + 32 * r1;
        if (r < BN && r < a.M) tc::cp_async4(&atom[4 * lane + r1], sc + (int64_t)r * kb + 4 * g);
      }
      tc::cp_async_arrive(&tfull[s]);
    };
    // weights read nothing produced upstream: the first ring-full goes out before the wait
    int wi = 0;
    for (; wi < total && wi < S::kWStages; ++wi) issue_w(wi);
    pdl_wait();
    pdl_trigger();
    bool ok = true;
    bool h_ready = false;
    int ti = 0;  // token stages issued
    for (int i = 0; i < total && ok; ++i) {
      // keep the weight ring full: issue every weight stage whose slot is free, without
      // blocking on slots the MMAs still hold
      while (wi < total) {
        const int s = wi % S::kWStages;
        const uint32_t par = ((wi / S::kWStages) - 1) & 1;
        bool freed = __shfl_sync(MXG_FULL_MASK, lane == 0 ? mbar_test(&wempty[s], par) : false, 0);
        if (!freed) {
          if (wi > i) break;  // stage i's weights are already on their way; come back later
          freed = __all_sync(MXG_FULL_MASK, mbar_wait(&wempty[s], par, status));
          if (!freed) {
            ok = false;
            break;
          }
        }
        issue_w(wi);
        ++wi;
      }
      if (!ok) break;
      if (i == n1 && !h_ready) {
        // phase 2 needs h from every phase-1 tile; weight slots that free up meanwhile keep
        // receiving W2
        const uint64_t t0 = globaltimer_ns();
        while (!h_ready) {
          h_ready = __all_sync(MXG_FULL_MASK, ld_acquire_gpu(cnt1) >= a.T1);
          if (h_ready) break;
          if (wi < total) {
            const int s = wi % S::kWStages;
            const uint32_t par = ((wi / S::kWStages) - 1) & 1;
            if (__shfl_sync(MXG_FULL_MASK, lane == 0 ? mbar_test(&wempty[s], par) : false, 0)) {
              issue_w(wi);
              ++wi;
              continue;
            }
          }
          if (__any_sync(MXG_FULL_MASK, globaltimer_ns() - t0 > kWaitLimitNs)) {
            if (lane == 0) set_error(status, MXG_ETIMEOUT);
            ok = false;
            break;
          }
          __nanosleep(32);
        }
        if (!ok) break;
        fence_proxy_async_global();  // h was written through the generic proxy; TMA reads it
      }
      const int s = i % kTokStages;
      if (i >= kTokStages &&
          !__all_sync(MXG_FULL_MASK, mbar_wait(&tempty[s], ((i / kTokStages) - 1) & 1, status))) {
        ok = false;
        break;
      }
      issue_t(i);
      ti = i + 1;
    }
    // Before the CTA may leave, every copy it issued has landed (on the normal path the MMA
    // thread has already waited for each of them, and these waits return at once).
    if (lane == 0) {
      for (int j = wi - S::kWStages < 0 ? 0 : wi - S::kWStages; j < wi; ++j)
        if (!mbar_wait(&wfull[j % S::kWStages], (j / S::kWStages) & 1, status)) break;
      for (int j = ti - kTokStages < 0 ? 0 : ti - kTokStages; j < ti; ++j)
        if (!mbar_wait(&tfull[j % kTokStages], (j / kTokStages) & 1, status)) break;
    }
    __syncwarp();
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      for (int i = 0; i < total; ++i) {
        const int sw = i % S::kWStages, st = i % kTokStages;
        if (!mbar_wait(&wfull[sw], (i / S::kWStages) & 1, status)) break;
        if (!mbar_wait(&tfull[st], (i / kTokStages) & 1, status)) break;
        fence_proxy_async_smem();  // cp.async (generic proxy) scale words -> tcgen05.cp (async proxy)
        tc::fence_after_sync();
        const bool p1 = i < n1;
        const int gi = p1 ? i : i - n1;
        const uint32_t t_d = p1 ? t_acc1 : t_acc2;
        const uint32_t t_sfa = t_sf + (uint32_t)((i % S::kSfSlots) * 8), t_sfb = t_sfa + 4;
        tc::cp_sf_atom(t_sfa, tc::desc_sf_atom(smem_u32(sfw + sw * 128)));
        tc::cp_sf_atom(t_sfb, tc::desc_sf_atom(smem_u32(sft + st * 128)));
        const uint32_t sa = smem_u32(wring + sw * kWBytes), sb = smem_u32(tring + st * S::kTBytes);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc::mma_mxf8(t_d, tc::desc_k128_sw128(sa + kk * 32), tc::desc_k128_sw128(sb + kk * 32),
                       tc::idesc_mxf8(BN, kk, kk), t_sfa, t_sfb, (gi > 0 || kk > 0) ? 1u : 0u);
        tc::commit(&wempty[sw]);
        tc::commit(&tempty[st]);
        if (p1 && i == n1 - 1) tc::commit(acc1_full);
      }
      if (n2 > 0) tc::commit(acc2_full);
    }
    __syncwarp();
  } else {
    // ----------------------------------------------------------------- epilogue (warps 2-5)
    const int q = warp & 3;  // the TMEM lane quadrant this warp may read
    const int r = 32 * q + lane;
    const int e = warp - 2, blk = e & 1, half = e >> 1;
    pdl_wait();  // outputs, h and the residual are touched only after the previous kernel is done
    bool ok = true;
    if (n1 > 0) {
      ok = __all_sync(MXG_FULL_MASK, mbar_wait(acc1_full, 0, status));
      tc::fence_after_sync();
      const uint32_t trow = t_acc1 + ((uint32_t)(32 * q) << 16);
      const int j0 = c * 64 + 32 * blk;  // first d_ff index of this warp's MX block
      for (int c0 = 0; c0 < BN && c0 < a.M; c0 += kChunk) {
        float v[16];
        tc::ld16(trow + c0, v);
        tc::wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) stg[r * (kChunk + 1) + j] = v[j];
        epi_bar();
        if (ok) {
          // warp (blk, half): MX block blk of tokens c0 + half*8 .. +7, one d_ff value per lane
          for (int tt = half * 8; tt < half * 8 + 8; ++tt) {
            const int m = c0 + tt;
            if (m >= a.M) break;
            const float g = stg[(32 * blk + lane) * (kChunk + 1) + tt];
            const float u = stg[(64 + 32 * blk + lane) * (kChunk + 1) + tt];
            mx_quant_warp_store(silu_mul(g, u), a.hq + (int64_t)m * a.d_ff + j0 + lane,
                                a.hs + (int64_t)m * (a.d_ff >> 5) + (j0 >> 5));
          }
        }
        epi_bar();  // the staging buffer is read before the next chunk overwrites it
      }
      // every thread's h stores are ordered before the count (phase-2 producers read h through TMA)
      __threadfence();
      fence_proxy_async_global();
      epi_bar();
      if (threadIdx.x == 64) red_release_gpu_add(cnt1, 1);
    }
    if (n2 > 0) {
      const bool ok2 = __all_sync(MXG_FULL_MASK, mbar_wait(acc2_full, 0, status));
      tc::fence_after_sync();
      const uint32_t trow = t_acc2 + ((uint32_t)(32 * q) << 16);
      float* pt = a.part + (int64_t)c * a.M * 128;  // this CTA's partial [M][128]
      for (int c0 = 0; c0 < BN && c0 < a.M; c0 += 16) {
        float v[16];
        tc::ld16(trow + c0, v);
        tc::wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (c0 + j < a.M) pt[(int64_t)(c0 + j) * 128 + r] = ok2 ? v[j] : 0.f;
      }
      __threadfence();
      epi_bar();
      int* cnt2 = a.ctrl + (1 + t2) * kLine;
      if (threadIdx.x == 64) red_release_gpu_add(cnt2, 1);
      if (warp == 2) {
        const bool all = wait_count(cnt2, a.S2, status);
        if (lane == 0) sh_flag = all ? 1 : 0;
      }
      epi_bar();
      if (sh_flag) {
        // slice z2 of the tile's M*32 float4 outputs, summed over the splits in split order
        const int E4 = a.M * 32;
        const int e0 = (int)((int64_t)z2 * E4 / a.S2), e1 = (int)((int64_t)(z2 + 1) * E4 / a.S2);
        const float* tp = a.part + (int64_t)(t2 * a.S2) * a.M * 128;
        for (int idx = e0 + (threadIdx.x - 64); idx < e1; idx += 128) {
          const int m = idx >> 5, rr = (idx & 31) * 4;
          float4 y = __ldcg(reinterpret_cast<const float4*>(tp + (int64_t)m * 128 + rr));
          for (int z = 1; z < a.S2; ++z) {
            const float4 p = __ldcg(reinterpret_cast<const float4*>(tp + ((int64_t)z * a.M + m) * 128 + rr));
            y.x += p.x;
            y.y += p.y;
            y.z += p.z;
            y.w += p.w;
          }
          const int64_t o = (int64_t)m * a.d_model + t2 * 128 + rr;
          if (a.residual) {
            const uint2 rv = *reinterpret_cast<const uint2*>(a.residual + o);
            y.x += bf16_lo(rv.x);
            y.y += bf16_hi(rv.x);
            y.z += bf16_lo(rv.y);
            y.w += bf16_hi(rv.y);
          }
          uint2 ov;
          ov.x = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(y.x)) |
                 ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(y.y)) << 16);
          ov.y = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(y.z)) |
                 ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(y.w)) << 16);
          *reinterpret_cast<uint2*>(a.y + o) = ov;
        }
      }
    }
    (void)ok;
  }
  // every CTA reaches this point whatever its waits returned
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(tmem, S::kTmemCols);
  if (threadIdx.x == 64) {
    // the last CTA out returns the counters to zero for the next call (every CTA has passed
    // all of its waits on them by the time it counts itself here)
    if (atom_acq_rel_gpu_add(done, 1) == G - 1) {
      *cnt1 = 0;
      for (int t = 0; t < a.T2; ++t) a.ctrl[(1 + t) * kLine] = 0;
      *done = 0;
      __threadfence();
    }
  }
}

// ---------------------------------------------------------------------------------- host
namespace {

struct FusePlan {
  int bn = 0, grid = 0, T1 = 0, T2 = 0, S2 = 0, NG1 = 0, NG2 = 0;
};

int sm_count() {
  static int n = -1;
  if (n < 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
  }
  return n;
}

FusePlan fuse_plan(int64_t M, int64_t d_model, int64_t d_ff) {
  FusePlan p;
  if (M < 1 || M > 128 || d_model % 128 || d_ff % 128 || d_model > (1 << 20) || d_ff > (1 << 20)) return p;
  const int G = sm_count();
  p.T1 = (int)(d_ff / 64);
  p.T2 = (int)(d_model / 128);
  p.NG1 = (int)(d_model / 128);
  p.NG2 = (int)(d_ff / 128);
  if (G <= 0 || p.T1 > G || p.T2 > G) return p;
  // the down projection's split count, as the split-K down GEMM of the two-launch path picks
  // it for the same shape (at most 8 splits, all of them resident with the row tiles)
  int s = G / p.T2;
  if (s > kMaxSplit) s = kMaxSplit;
  if (s > p.NG2) s = p.NG2;
  p.S2 = s;
  p.grid = p.T1 > p.T2 * p.S2 ? p.T1 : p.T2 * p.S2;
  p.bn = M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : 128;
  return p;
}

template <int BN>
cudaError_t launch_fused(const CUtensorMap& m13, const CUtensorMap& mx, const CUtensorMap& m2, const CUtensorMap& mh,
                         const FuseArgs& a, int grid, cudaStream_t st) {
  using S = FuseShape<BN>;
  cudaError_t e = cudaFuncSetAttribute(mlp_fused_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kSmemBytes);
  if (e != cudaSuccess) return e;
  return launch_k(mlp_fused_kernel<BN>, dim3((unsigned)grid), dim3(192), S::kSmemBytes, st, 1, m13, mx, m2, mh, a);
}

}  // namespace

size_t mlp_fused_part_bytes(int64_t M, int64_t d_model, int64_t d_ff) {
  const FusePlan p = fuse_plan(M, d_model, d_ff);
  if (!p.bn) return 0;
  return (size_t)p.T2 * p.S2 * (size_t)M * 128 * sizeof(float);
}

size_t mlp_fused_ctrl_bytes(int64_t d_model) { return (size_t)((d_model + 127) / 128 + 3) * kLine * 4; }

bool mlp_fused_supported(int64_t M, int64_t d_model, int64_t d_ff) { return fuse_plan(M, d_model, d_ff).bn != 0; }

cudaError_t launch_mlp_fused(const uint8_t* xq, const uint8_t* xs, int64_t M, int64_t d_model, int64_t d_ff,
                             const uint8_t* w13q, const uint8_t* w13s, const uint8_t* w2q, const uint8_t* w2s,
                             const uint16_t* residual, uint16_t* y, uint8_t* hq, uint8_t* hs, float* part, int* ctrl,
                             cudaStream_t st, bool* unsupported) {
  *unsupported = true;
  const FusePlan p = fuse_plan(M, d_model, d_ff);
  if (!p.bn) return cudaSuccess;
  CUtensorMap m13, mx, m2, mh;
  if (!make_tensor_map_2d(&m13, CU_TENSOR_MAP_DATA_TYPE_UINT8, w13q, (uint64_t)d_model, (uint64_t)(2 * d_ff),
                          (uint64_t)d_model, kKG, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tensor_map_2d(&mx, CU_TENSOR_MAP_DATA_TYPE_UINT8, xq, (uint64_t)d_model, (uint64_t)M, (uint64_t)d_model,
                          kKG, (uint32_t)p.bn, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tensor_map_2d(&m2, CU_TENSOR_MAP_DATA_TYPE_UINT8, w2q, (uint64_t)d_ff, (uint64_t)d_model, (uint64_t)d_ff,
                          kKG, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tensor_map_2d(&mh, CU_TENSOR_MAP_DATA_TYPE_UINT8, hq, (uint64_t)d_ff, (uint64_t)M, (uint64_t)d_ff, kKG,
                          (uint32_t)p.bn, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaSuccess;
  *unsupported = false;
  FuseArgs a{};
  a.M = (int)M;
  a.d_model = (int)d_model;
  a.d_ff = (int)d_ff;
  a.T1 = p.T1;
  a.T2 = p.T2;
  a.S2 = p.S2;
  a.NG1 = p.NG1;
  a.NG2 = p.NG2;
  a.xs = xs;
  a.w13s = w13s;
  a.w2s = w2s;
  a.hq = hq;
  a.hs = hs;
  a.part = part;
  a.ctrl = ctrl;
  a.residual = residual;
  a.y = y;
  switch (p.bn) {
    case 16: return launch_fused<16>(m13, mx, m2, mh, a, p.grid, st);
    case 32: return launch_fused<32>(m13, mx, m2, mh, a, p.grid, st);
    case 64: return launch_fused<64>(m13, mx, m2, mh, a, p.grid, st);
    default: return launch_fused<128>(m13, mx, m2, mh, a, p.grid, st);
  }
}

}  // namespace mxg
