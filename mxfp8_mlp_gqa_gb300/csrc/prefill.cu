// Causal prefill / extend attention with native GQA on the 5th-generation tensor cores.
//
// [S2.1] "What's Open Source": the pages' attention library covers contiguous prefill and paged
// prefill (extend) besides paged decode, with GQA by a stride-0 K/V broadcast. Sequence b holds
// kv_len[b] rows in its cache, the last T_b of which are its new tokens (already appended);
// new token i sits at position kv_len[b] - T_b + i and attends to positions 0 .. that position
// (T_b = kv_len[b]: a prefill from scratch). Its query row is q[q_start[b] + i].
//
// Two kernels share this design; the launcher picks by prompt length (see launch_gqa_prefill_attn).
// Design (tensor-bound: S = Q K^T and O = P V are dense 128 x 128 x 128 contractions):
//  * CTA = 128 query rows of one (sequence b, kv head g): 128/G consecutive new tokens x the G
//    query heads of the group (row r = token r/G, head g*G + r%G), so every K/V tile is read
//    once for all G heads (no head expansion). Tiles are scheduled heaviest (latest) first.
//  * warp 0 drives TMA: the Q tile once (a 3-D box over [tokens, heads, D]), then 128-key K
//    and V tiles (128-byte swizzle) into a 2-stage ring; with a page table each 64-key half
//    is looked up separately.
//  * warp 1 (one thread) issues tcgen05.mma kind::f16 (bf16 in, fp32 accumulate in TMEM):
//    S_j = Q K_j^T into one of two S buffers, then O += P_{j-1} V_{j-1}, so S_j overlaps the
//    softmax of tile j-1. V is read as an MN-major operand straight from its [key][D] tile.
//  * warps 2..5 (thread = query row = TMEM lane) run the online softmax: S row from TMEM,
//    causal mask, base-2 exponentials, P written in bf16 to a K-major swizzled tile for the
//    PV product. The reference maximum moves only when the row maximum exceeds it by more
//    than 2^8 (P stays <= 256, exact in the final O / l); O in TMEM is rescaled then.
//  * the same warps normalise O / l and write bf16 rows.
// All waits are bounded; a timeout sets MXG_ETIMEOUT and every role winds down before TMEM is
// released.
#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"
#include "tc.cuh"

namespace mxg {

namespace {

using namespace tc;

constexpr int kRows = 128;                      // query rows per CTA (tokens x group heads)
constexpr int kKeys = 128;                      // keys per tile
constexpr int kHd = 128;                        // head dim
constexpr int kTile = kRows * kHd * 2;          // one bf16 [128, 128] tile (two 64-column boxes)
constexpr int kBox = kTile / 2;                 // one [128 rows, 64 columns] box: 16 KB
constexpr int kStages = 2;
constexpr int kThreads = 6 * 32;                // producer, MMA, four softmax warps (2..5)
constexpr float kRescaleLog2 = 8.f;             // move the reference max only past 2^8 growth

// Shared memory: Q | K[2] | V[2] | P | barriers.
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kTile;
constexpr int kOffV = kOffK + kStages * kTile;
constexpr int kOffP = kOffV + kStages * kTile;
constexpr int kOffBar = kOffP + kTile;
// q full, k/v full, k/v empty, s full/free, p full, pv done, mma drained
constexpr int kNumBars = 1 + 4 * kStages + 2 * 2 + 3;
constexpr int kSmemBytes = 1024 + kOffBar + kNumBars * 8 + 16;

// TMEM columns: S buffers at 0 and 128, O at 256.
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 256;

// Instruction descriptor of kind::f16: bf16 A and B (format 1 at bits 7-9 / 10-12), fp32 D
// (bit 4), A K-major, B K-major or MN-major (bit 16), N>>3 at bits 17-22, M>>4 at bits 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16_tc(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]), "f"(v[8]), "f"(v[9]),
      "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]), "f"(v[15]), "f"(v[16]), "f"(v[17]), "f"(v[18]),
      "f"(v[19]), "f"(v[20]), "f"(v[21]), "f"(v[22]), "f"(v[23]), "f"(v[24]), "f"(v[25]), "f"(v[26]), "f"(v[27]),
      "f"(v[28]), "f"(v[29]), "f"(v[30]), "f"(v[31])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int32_t x,
                                            int32_t y, int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
          smem_u32(smem_dst)),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

// K-major bf16 tile [128 rows][64-column box] x 2 with the 128-byte swizzle: 16-element step
// ks of the contraction starts at box ks/4, byte 32*(ks%4) of each 128-byte row.
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t tile, int ks) {
  return smem_desc(tile + (ks >> 2) * kBox + (ks & 3) * 32, 0, 1024, 2);
}

// V tile [128 keys][64-column box] x 2 read as the MN-major B operand (N = head dim, K = keys):
// 8-key groups 1024 bytes apart (SBO), the second 64-column half one box away (LBO); the
// 16-key step ks starts 2048 bytes further.
__device__ __forceinline__ uint64_t desc_v_mn(uint32_t tile, int ks) {
  return smem_desc(tile + ks * 2048, kBox, 1024, 2);
}

struct PrefillParams {
  const int32_t* q_start;  // [bs + 1]
  const int32_t* kv_len;   // [bs]
  uint16_t* out;           // [total_q, Hq, D]
  int32_t* err;
  int Hq, Hkv, group, bs;
  int64_t cap, total_q;
  int max_q_len;
  float scale_log2;
  // paged caches (table != nullptr): as the paged decode attention
  const int32_t* table;
  int max_pages, page_size;
  int64_t num_pages;
};

}  // namespace

using namespace tc;

// Bounded wait whose outcome is the same for every lane of the warp (the softmax warps run
// warp-collective TMEM loads after it).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int32_t* err) {
  return __all_sync(MXG_FULL_MASK, mbar_wait(bar, parity, err));
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packed fp32 pairs (sm_100 family): each lane rounds exactly as the scalar instruction does.
__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void upk2(uint64_t r, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// max of three (exact, order-free)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__global__ void __launch_bounds__(kThreads, 1) gqa_prefill_kernel(const __grid_constant__ CUtensorMap tmQ,
                                                                  const __grid_constant__ CUtensorMap tmK,
                                                                  const __grid_constant__ CUtensorMap tmV,
                                                                  const PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* v_full = k_full + kStages;
  uint64_t* k_empty = v_full + kStages;  // K_j's stage is free once S_j has completed,
  uint64_t* v_empty = k_empty + kStages;  // V_j's once PV_j has
  uint64_t* s_full = v_empty + kStages;
  uint64_t* s_free = s_full + 2;
  uint64_t* p_full = s_free + 2;
  uint64_t* pv_done = p_full + 1;
  uint64_t* drained = pv_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars);

  pdl_wait();
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bg = blockIdx.y;
  const int b = bg / p.Hkv, g = bg - b * p.Hkv;
  const int G = p.group, tpt = kRows / G;
  const int tile = (int)gridDim.x - 1 - (int)blockIdx.x;  // latest (heaviest) tiles first
  const int qs = p.q_start[b];
  const int T = p.q_start[b + 1] - qs;
  const int n = p.kv_len[b];
  if (T < 0 || T > p.max_q_len || T > n || (int64_t)n > p.cap || qs < 0 || (int64_t)qs + T > p.total_q) {
    if (tile == 0 && g == 0 && threadIdx.x == 0) set_error(p.err, MXG_EDEVICE);
    return;
  }
  const int tok0 = tile * tpt;
  if (tok0 >= T) return;
  const int P0 = n - T;  // cached positions before the new tokens
  const int pos_hi = P0 + min(T, tok0 + tpt) - 1;
  const int nk = pos_hi / kKeys + 1;  // key tiles this query tile sees
  const int64_t row0 = ((int64_t)b * p.Hkv + g) * p.cap;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&s_free[s], 128);
    }
    mbar_init(p_full, 128);
    mbar_init(pv_done, 1);
    mbar_init(drained, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;

  if (warp == 0) {
    // ------------------------------------------------------------------ producer (TMA)
    if (lane == 0) {
      prefetch_tensormap(&tmQ);
      prefetch_tensormap(&tmK);
      prefetch_tensormap(&tmV);
      mbar_arrive_expect_tx(q_full, kTile);
      tma_load_3d(smem + kOffQ, &tmQ, q_full, 0, g * G, qs + tok0);
      tma_load_3d(smem + kOffQ + kBox, &tmQ, q_full, 64, g * G, qs + tok0);
      const int64_t past = p.table ? p.num_pages * p.Hkv * p.page_size : 0;
      for (int j = 0; j < nk && ok; ++j) {
        const int s = j & 1;
        if (j >= kStages && !mbar_wait(&k_empty[s], ((j >> 1) - 1) & 1, p.err)) {
          ok = false;
          break;
        }
        int rows[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int key = j * kKeys + 64 * h;
          if (!p.table) {
            rows[h] = (int)(row0 + key);
          } else if (key >= n) {
            rows[h] = (int)past;  // nothing visible there: the copy engine reads zeros
          } else {
            const int page = p.table[(int64_t)b * p.max_pages + key / p.page_size];
            if (page < 0 || page >= p.num_pages) {
              set_error(p.err, MXG_EDEVICE);
              rows[h] = (int)past;
            } else {
              rows[h] = (int)(((int64_t)page * p.Hkv + g) * p.page_size + key % p.page_size);
            }
          }
        }
        uint8_t* kt = smem + kOffK + s * kTile;
        uint8_t* vt = smem + kOffV + s * kTile;
        mbar_arrive_expect_tx(&k_full[s], kTile);
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int h = 0; h < 2; ++h) tma_load_2d(kt + c * kBox + h * (kBox / 2), &tmK, &k_full[s], 64 * c, rows[h]);
        // the K load above goes out a softmax period before this one: V_{j-2} is read later
        if (j >= kStages && !mbar_wait(&v_empty[s], ((j >> 1) - 1) & 1, p.err)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&v_full[s], kTile);
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int h = 0; h < 2; ++h) tma_load_2d(vt + c * kBox + h * (kBox / 2), &tmV, &v_full[s], 64 * c, rows[h]);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issue (one thread)
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16(kRows, kKeys, false);
      constexpr uint32_t kIdPV = idesc_bf16(kRows, kHd, true);
      const uint32_t qa = smem_u32(smem + kOffQ), pa = smem_u32(smem + kOffP);
      bool issued = false;
      ok = mbar_wait(q_full, 0, p.err);
      for (int j = 0; j <= nk && ok; ++j) {
        if (j < nk) {
          const int s = j & 1;
          if (!mbar_wait(&k_full[s], (j >> 1) & 1, p.err) ||
              (j >= 2 && !mbar_wait(&s_free[s], ((j >> 1) - 1) & 1, p.err))) {
            ok = false;
            break;
          }
          fence_after_sync();
          const uint32_t ka = smem_u32(smem + kOffK + s * kTile);
#pragma unroll
          for (int ks = 0; ks < kHd / 16; ++ks)
            mma_bf16_tc(tmem + s * kKeys, desc_kmajor(qa, ks), desc_kmajor(ka, ks), kIdS, ks > 0);
          commit(&s_full[s]);
          commit(&k_empty[s]);
          issued = true;
        }
        if (j >= 1) {
          const int jj = j - 1, s2 = jj & 1;
          if (!mbar_wait(p_full, jj & 1, p.err) || !mbar_wait(&v_full[s2], (jj >> 1) & 1, p.err)) {
            ok = false;
            break;
          }
          fence_after_sync();
          const uint32_t va = smem_u32(smem + kOffV + s2 * kTile);
#pragma unroll
          for (int ks = 0; ks < kKeys / 16; ++ks)
            mma_bf16_tc(tmem + kColO, desc_kmajor(pa, ks), desc_v_mn(va, ks), kIdPV, (jj > 0 || ks > 0) ? 1u : 0u);
          commit(pv_done);
          commit(&v_empty[s2]);
        }
      }
      // every MMA this thread issued has finished before TMEM can be released
      if (issued) {
        commit(drained);
        mbar_wait(drained, 0, p.err);
      }
    }
  } else {
    // ------------------------------------------------------------------ softmax + epilogue (thread = row)
    const int quad = warp & 3;  // TMEM lane quadrant this warp may access
    const int r = quad * 32 + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(quad * 32) << 16);
    const int tl = r / G, hh = r - tl * G;
    const int tok = tok0 + tl;
    const bool valid = tok < T;
    const int pos = valid ? P0 + tok : -1;  // rows past the sequence see no key
    float m_ref = -INFINITY, l = 0.f;
    for (int j = 0; j < nk; ++j) {
      const int s = j & 1;
      const int key0 = j * kKeys;
      if (!warp_wait(&s_full[s], (j >> 1) & 1, p.err)) {
        ok = false;
        break;
      }
      fence_after_sync();
      float x[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(lane_addr + s * kKeys + 32 * c, x[c]);
      wait_ld();
      fence_before_sync();
      mbar_arrive(&s_free[s]);
      // causal mask (column c is key key0 + c), needed only on tiles that reach the diagonal
      const int lim = pos - key0;
      if (!__all_sync(MXG_FULL_MASK, lim >= kKeys - 1)) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (32 * c + i > lim) x[c][i] = -INFINITY;
      }
      // row maximum over eight independent partials (three-input max); the scale is positive
      // (host-checked) and rounding is monotonic, so max(x) * scale is the maximum of the scaled
      // products
      float mp[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mp[k] = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int i = 0; i < 32; i += 2) mp[(i >> 1) & 7] = fmax3(mp[(i >> 1) & 7], x[c][i], x[c][i + 1]);
      const float mx = fmax3(fmax3(mp[0], mp[1], mp[2]), fmax3(mp[3], mp[4], mp[5]), fmaxf(mp[6], mp[7])) *
                       p.scale_log2;
      const float m_new = mx > m_ref + kRescaleLog2 ? mx : m_ref;
      const bool moved = m_new != m_ref;
      const float alpha = moved ? fast_exp2(m_ref - m_new) : 1.f;
      const float nmu = m_new == -INFINITY ? 0.f : -m_new;
      // p = 2^(x * scale - m) with one rounding in the exponent's argument (packed pairs); the
      // row sum runs over eight partials (four packed pairs: partial k holds the elements
      // i = k mod 8) so that no 128-long chain of dependent adds forms
      const uint64_t sc2 = pk2(p.scale_log2, p.scale_log2), nm2 = pk2(nmu, nmu);
      uint64_t sp2[4] = {0, 0, 0, 0};
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          float t0, t1;
          upk2(fma_f32x2(pk2(x[c][i], x[c][i + 1]), sc2, nm2), t0, t1);
          x[c][i] = fast_exp2(t0);
          x[c][i + 1] = fast_exp2(t1);
          sp2[(i >> 1) & 3] = add_f32x2(sp2[(i >> 1) & 3], pk2(x[c][i], x[c][i + 1]));
        }
      float sp[8];
#pragma unroll
      for (int k = 0; k < 4; ++k) upk2(sp2[k], sp[2 * k], sp[2 * k + 1]);
      l = l * alpha + (((sp[0] + sp[1]) + (sp[2] + sp[3])) + ((sp[4] + sp[5]) + (sp[6] + sp[7])));
      m_ref = m_new;
      // the P tile and O are free once the previous PV product has completed
      if (j >= 1 && !warp_wait(pv_done, (j - 1) & 1, p.err)) {
        ok = false;
        break;
      }
      fence_after_sync();
      if (key0 + kKeys > n) {
        // V rows past kv_len may hold anything (P is 0 there): zero them so 0 * V stays 0
        if (!warp_wait(&v_full[s], (j >> 1) & 1, p.err)) {
          ok = false;
          break;
        }
        if (key0 + r >= n) {
          uint8_t* vt = smem + kOffV + s * kTile + r * 128;
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            *reinterpret_cast<uint4*>(vt + 16 * q) = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(vt + kBox + 16 * q) = make_uint4(0, 0, 0, 0);
          }
        }
      }
      if (j >= 1 && __any_sync(MXG_FULL_MASK, moved)) {
        // rows whose reference maximum moved: O (tiles < j) *= 2^(old - new)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float o[32];
          tmem_ld32(lane_addr + kColO + 32 * c, o);
          wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= alpha;
          tmem_st32(lane_addr + kColO + 32 * c, o);
        }
        tmem_wait_st();
      }
      // P row in bf16: 16-byte chunk cc holds keys 8cc .. 8cc+7 (128-byte swizzle)
#pragma unroll
      for (int cc = 0; cc < 16; ++cc) {
        const float* v = &x[cc >> 2][(cc & 3) * 8];
        uint4 w;
        w.x = pack_bf16x2(v[0], v[1]);
        w.y = pack_bf16x2(v[2], v[3]);
        w.z = pack_bf16x2(v[4], v[5]);
        w.w = pack_bf16x2(v[6], v[7]);
        *reinterpret_cast<uint4*>(smem + kOffP + (cc >> 3) * kBox + r * 128 + (((cc & 7) ^ (r & 7)) << 4)) = w;
      }
      fence_proxy_async_smem();
      fence_before_sync();
      mbar_arrive(p_full);
    }
    if (ok && warp_wait(pv_done, (nk - 1) & 1, p.err)) {
      fence_after_sync();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint16_t* orow = p.out + ((int64_t)(qs + (valid ? tok : 0)) * p.Hq + g * G + hh) * kHd;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float o[32];
        tmem_ld32(lane_addr + kColO + 32 * c, o);
        wait_ld();
        if (valid) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 w;
            w.x = pack_bf16x2(o[8 * q] * inv, o[8 * q + 1] * inv);
            w.y = pack_bf16x2(o[8 * q + 2] * inv, o[8 * q + 3] * inv);
            w.z = pack_bf16x2(o[8 * q + 4] * inv, o[8 * q + 5] * inv);
            w.w = pack_bf16x2(o[8 * q + 6] * inv, o[8 * q + 7] * inv);
            *reinterpret_cast<uint4*>(orow + 32 * c + 8 * q) = w;
          }
        }
      }
    }
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------------------------------
// Ping-pong variant: two 128-row query tiles (A, B) per CTA share every K/V tile. P of a tile is
// written in bf16 into TMEM over that tile's own S (the columns already read) and the PV MMA
// takes it from tensor memory, so shared memory holds only Q_A, Q_B and the K/V ring. The MMA
// thread issues S_A(0), S_B(0), then per key tile j: PV_A(j), S_A(j+1), PV_B(j), S_B(j+1): while
// one softmax warpgroup works on its tile, the tensor cores serve the other.
constexpr int kPPThreads = 10 * 32;  // producer, MMA, softmax A (warps 2..5), softmax B (6..9)
constexpr int kPPOffQ = 0;                        // Q_A, Q_B
constexpr int kPPOffK = kPPOffQ + 2 * kTile;
constexpr int kPPOffV = kPPOffK + kStages * kTile;
constexpr int kPPOffBar = kPPOffV + kStages * kTile;
// q full, k/v full, k/v empty, s full[2], p full[2], o done[2], mma drained
constexpr int kPPNumBars = 1 + 4 * kStages + 2 + 2 + 2 + 1;
constexpr int kPPSmemBytes = 1024 + kPPOffBar + kPPNumBars * 8 + 16;

__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

__global__ void __launch_bounds__(kPPThreads) gqa_prefill_pp_kernel(const __grid_constant__ CUtensorMap tmQ,
                                                                      const __grid_constant__ CUtensorMap tmK,
                                                                      const __grid_constant__ CUtensorMap tmV,
                                                                      const PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kPPOffBar);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* v_full = k_full + kStages;
  uint64_t* k_empty = v_full + kStages;  // K_j's stage is free once both S products of tile j are,
  uint64_t* v_empty = k_empty + kStages;  // V_j's once both PV products are
  uint64_t* s_full = v_empty + kStages;   // [tile]
  uint64_t* p_full = s_full + 2;          // [tile]
  uint64_t* o_done = p_full + 2;          // [tile]
  uint64_t* drained = o_done + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kPPNumBars);

  pdl_wait();
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bg = blockIdx.y;
  const int b = bg / p.Hkv, g = bg - b * p.Hkv;
  const int G = p.group, tpt = kRows / G;  // tokens per 128-row tile
  const int tile = (int)gridDim.x - 1 - (int)blockIdx.x;  // latest (heaviest) tiles first
  const int qs = p.q_start[b];
  const int T = p.q_start[b + 1] - qs;
  const int n = p.kv_len[b];
  if (T < 0 || T > p.max_q_len || T > n || (int64_t)n > p.cap || qs < 0 || (int64_t)qs + T > p.total_q) {
    if (tile == 0 && g == 0 && threadIdx.x == 0) set_error(p.err, MXG_EDEVICE);
    return;
  }
  const int tok0 = tile * 2 * tpt;  // tile A: tok0 .., tile B: tok0 + tpt ..
  if (tok0 >= T) return;
  const int P0 = n - T;
  const int pos_hi = P0 + min(T, tok0 + 2 * tpt) - 1;
  const int nk = pos_hi / kKeys + 1;
  const int64_t row0 = ((int64_t)b * p.Hkv + g) * p.cap;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&s_full[x], 1);
      mbar_init(&p_full[x], 128);
      mbar_init(&o_done[x], 1);
    }
    mbar_init(drained, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *tmem_slot;  // S/P_A at 0, S/P_B at 128, O_A at 256, O_B at 384
  bool ok = true;


  if (warp == 0) {
    // ------------------------------------------------------------------ producer (TMA)
    if (lane == 0) {
      prefetch_tensormap(&tmQ);
      prefetch_tensormap(&tmK);
      prefetch_tensormap(&tmV);
      mbar_arrive_expect_tx(q_full, 2 * kTile);
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        tma_load_3d(smem + kPPOffQ + x * kTile, &tmQ, q_full, 0, g * G, qs + tok0 + x * tpt);
        tma_load_3d(smem + kPPOffQ + x * kTile + kBox, &tmQ, q_full, 64, g * G, qs + tok0 + x * tpt);
      }
      const int64_t past = p.table ? p.num_pages * p.Hkv * p.page_size : 0;
      for (int j = 0; j < nk; ++j) {
        const int s = j & 1;
        if (j >= kStages && !mbar_wait(&k_empty[s], ((j >> 1) - 1) & 1, p.err)) break;
        int rows[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int key = j * kKeys + 64 * h;
          if (!p.table) {
            rows[h] = (int)(row0 + key);
          } else if (key >= n) {
            rows[h] = (int)past;  // nothing visible there: the copy engine reads zeros
          } else {
            const int page = p.table[(int64_t)b * p.max_pages + key / p.page_size];
            if (page < 0 || page >= p.num_pages) {
              set_error(p.err, MXG_EDEVICE);
              rows[h] = (int)past;
            } else {
              rows[h] = (int)(((int64_t)page * p.Hkv + g) * p.page_size + key % p.page_size);
            }
          }
        }
        uint8_t* kt = smem + kPPOffK + s * kTile;
        uint8_t* vt = smem + kPPOffV + s * kTile;
        mbar_arrive_expect_tx(&k_full[s], kTile);
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int h = 0; h < 2; ++h) tma_load_2d(kt + c * kBox + h * (kBox / 2), &tmK, &k_full[s], 64 * c, rows[h]);
        if (j >= kStages && !mbar_wait(&v_empty[s], ((j >> 1) - 1) & 1, p.err)) break;
        mbar_arrive_expect_tx(&v_full[s], kTile);
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int h = 0; h < 2; ++h) tma_load_2d(vt + c * kBox + h * (kBox / 2), &tmV, &v_full[s], 64 * c, rows[h]);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issue (one thread)
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16(kRows, kKeys, false);
      constexpr uint32_t kIdPV = idesc_bf16(kRows, kHd, true);
      const uint32_t qa = smem_u32(smem + kPPOffQ);
      bool issued = false;
      // S_x(j) = Q_x K_j^T into the S/P buffer of tile x
      auto issue_s = [&](int x, int j) {
        const uint32_t ka = smem_u32(smem + kPPOffK + (j & 1) * kTile);
#pragma unroll
        for (int ks = 0; ks < kHd / 16; ++ks)
          mma_bf16_tc(tmem + x * kKeys, desc_kmajor(qa + x * kTile, ks), desc_kmajor(ka, ks), kIdS, ks > 0);
        commit(&s_full[x]);
        issued = true;
      };
      // O_x += P_x(j) V_j, P from tensor memory (16-key step ks = 8 columns of bf16 pairs)
      auto issue_pv = [&](int x, int j) {
        const uint32_t va = smem_u32(smem + kPPOffV + (j & 1) * kTile);
#pragma unroll
        for (int ks = 0; ks < kKeys / 16; ++ks)
          mma_bf16_ts(tmem + kColO + x * kKeys, tmem + x * kKeys + 8 * ks, desc_v_mn(va, ks), kIdPV,
                      (j > 0 || ks > 0) ? 1u : 0u);
      };
      ok = mbar_wait(q_full, 0, p.err) && mbar_wait(&k_full[0], 0, p.err);
      if (ok) {
        fence_after_sync();
        issue_s(0, 0);
        issue_s(1, 0);
        commit(&k_empty[0]);
      }
      for (int j = 0; j < nk && ok; ++j) {
        const int s = j & 1;
        const bool more = j + 1 < nk;
        if (!mbar_wait(&p_full[0], j & 1, p.err) || !mbar_wait(&v_full[s], (j >> 1) & 1, p.err)) {
          ok = false;
          break;
        }
        fence_after_sync();
        issue_pv(0, j);
        if (!more) {
          commit(&o_done[0]);
        } else {
          if (!mbar_wait(&k_full[(j + 1) & 1], ((j + 1) >> 1) & 1, p.err)) {
            ok = false;
            break;
          }
          fence_after_sync();
          issue_s(0, j + 1);
        }
        if (!mbar_wait(&p_full[1], j & 1, p.err)) {
          ok = false;
          break;
        }
        fence_after_sync();
        issue_pv(1, j);
        commit(&v_empty[s]);
        if (!more) {
          commit(&o_done[1]);
        } else {
          issue_s(1, j + 1);
          commit(&k_empty[(j + 1) & 1]);
        }
      }
      if (issued) {
        // every MMA has finished before TMEM is released, also when a wait above ran out
        commit(drained);
        mbar_wait(drained, 0, p.err);
      }
    }
  } else {
    // ------------------------------------------------ softmax of tile x (thread = row = TMEM lane)
    const int x = (warp - 2) >> 2;
    const int quad = warp & 3;  // TMEM lane quadrant this warp may access
    const int r = quad * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t sbuf = tmem + lane_off + x * kKeys;          // S, then P (bf16 pairs) of tile x
    const uint32_t obuf = tmem + lane_off + kColO + x * kKeys;  // O of tile x
    const int tl = r / G, hh = r - tl * G;
    const int tok = tok0 + x * tpt + tl;
    const bool valid = tok < T;
    const int pos = valid ? P0 + tok : -1;  // rows past the sequence see no key
    float m_ref = -INFINITY, l = 0.f;
    for (int j = 0; j < nk; ++j) {
      const int key0 = j * kKeys;
      if (!warp_wait(&s_full[x], j & 1, p.err)) {
        ok = false;
        break;
      }
      fence_after_sync();
      const int lim = pos - key0;  // columns <= lim are visible to this row
      const bool masked = !__all_sync(MXG_FULL_MASK, lim >= kKeys - 1);
      // pass 1: the row maximum of the raw products; the scale is positive (host-checked) and
      // rounding is monotonic, so max(s) * scale is the maximum of the scaled products (base 2)
      float mp[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float v[32];
        tmem_ld32(sbuf + 32 * c, v);
        wait_ld();
#pragma unroll
        for (int i = 0; i < 32; i += 2)
          mp[(i >> 1) & 3] = fmax3(mp[(i >> 1) & 3], (masked && 32 * c + i > lim) ? -INFINITY : v[i],
                                   (masked && 32 * c + i + 1 > lim) ? -INFINITY : v[i + 1]);
      }
      const float mx = fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])) * p.scale_log2;
      const float m_new = mx > m_ref + kRescaleLog2 ? mx : m_ref;
      const bool moved = m_new != m_ref;
      const float alpha = moved ? fast_exp2(m_ref - m_new) : 1.f;
      const float nmu = m_new == -INFINITY ? 0.f : -m_new;
      if (j >= 1 && __any_sync(MXG_FULL_MASK, moved)) {
        // O holds tiles < j (PV_x(j-1) completed before S_x(j) was committed): rescale moved rows
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float o[32];
          tmem_ld32(obuf + 32 * c, o);
          wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= alpha;
          tmem_st32(obuf + 32 * c, o);
        }
      }
      bool zeroed = false;
      if (x == 0 && key0 + kKeys > n) {
        // V rows past kv_len may hold anything (P is 0 there): zero them for both tiles
        if (!warp_wait(&v_full[j & 1], (j >> 1) & 1, p.err)) {
          ok = false;
          break;
        }
        if (key0 + r >= n) {
          uint8_t* vt = smem + kPPOffV + (j & 1) * kTile + r * 128;
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            *reinterpret_cast<uint4*>(vt + 16 * q) = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(vt + kBox + 16 * q) = make_uint4(0, 0, 0, 0);
          }
        }
        zeroed = true;
      }
      // pass 2: P = 2^(s * scale - m) in bf16 pairs (column c: keys 2c, 2c+1) over S columns already read
      const uint64_t sc2 = pk2(p.scale_log2, p.scale_log2), nm2 = pk2(nmu, nmu);
      uint64_t sp2[2] = {0, 0};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float v[32];
        tmem_ld32(sbuf + 32 * c, v);
        wait_ld();
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float t0, t1;
          upk2(fma_f32x2(pk2(v[2 * i], v[2 * i + 1]), sc2, nm2), t0, t1);
          if (masked && 32 * c + 2 * i > lim) t0 = -INFINITY;
          if (masked && 32 * c + 2 * i + 1 > lim) t1 = -INFINITY;
          const float e0 = fast_exp2(t0), e1 = fast_exp2(t1);
          sp2[i & 1] = add_f32x2(sp2[i & 1], pk2(e0, e1));
          w[i] = pack_bf16x2(e0, e1);
        }
        tmem_st16(sbuf + 16 * c, w);
      }
      float sp[4];
      upk2(sp2[0], sp[0], sp[1]);
      upk2(sp2[1], sp[2], sp[3]);
      l = l * alpha + ((sp[0] + sp[1]) + (sp[2] + sp[3]));
      m_ref = m_new;
      tmem_wait_st();
      if (zeroed) fence_proxy_async_smem();
      fence_before_sync();
      mbar_arrive(&p_full[x]);
    }
    if (ok && warp_wait(&o_done[x], 0, p.err)) {
      fence_after_sync();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint16_t* orow = p.out + ((int64_t)(qs + (valid ? tok : 0)) * p.Hq + g * G + hh) * kHd;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float o[32];
        tmem_ld32(obuf + 32 * c, o);
        wait_ld();
        if (valid) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 wv;
            wv.x = pack_bf16x2(o[8 * q] * inv, o[8 * q + 1] * inv);
            wv.y = pack_bf16x2(o[8 * q + 2] * inv, o[8 * q + 3] * inv);
            wv.z = pack_bf16x2(o[8 * q + 4] * inv, o[8 * q + 5] * inv);
            wv.w = pack_bf16x2(o[8 * q + 6] * inv, o[8 * q + 7] * inv);
            *reinterpret_cast<uint4*>(orow + 32 * c + 8 * q) = wv;
          }
        }
      }
    }
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// kv_append for a prefill / extend: token i of sequence b (row q_start[b] + i of k_new / v_new,
// [total_q, Hkv, D] with ld_new elements between token rows) lands at position
// kv_len[b] - T_b + i. One warp per (token, sequence); 16-byte moves.
__global__ void __launch_bounds__(256) kv_append_extend_kernel(uint16_t* __restrict__ kc, uint16_t* __restrict__ vc,
                                                               const uint16_t* __restrict__ kn,
                                                               const uint16_t* __restrict__ vn, int64_t ld_new,
                                                               const int32_t* __restrict__ q_start,
                                                               const int32_t* __restrict__ kv_len, int Hkv, int D,
                                                               int64_t cap, int64_t total_q, int max_q_len,
                                                               int32_t* err, KvPages pg) {
  pdl_wait();
  // no early trigger: decode attention reads the cache rows below kv_len - 1 before its own
  // wait, and these rows are among them, so the successor starts only once this one completes
  const int b = blockIdx.y;
  const int i = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int qs = q_start[b], T = q_start[b + 1] - qs, n = kv_len[b];
  if (T < 0 || T > max_q_len || T > n || (int64_t)n > cap || qs < 0 || (int64_t)qs + T > total_q) {
    if (blockIdx.x == 0 && threadIdx.x == 0) set_error(err, MXG_EDEVICE);
    return;
  }
  if (i >= T) return;
  const int pos = n - T + i;
  int64_t base;  // cache row of head 0 (heads are cap / page_size rows apart)
  int64_t hstride;
  if (pg.table) {
    const int page = pg.table[(int64_t)b * pg.max_pages + pos / pg.page_size];
    if (page < 0 || page >= pg.num_pages) {
      if (lane == 0) set_error(err, MXG_EDEVICE);
      return;
    }
    base = (int64_t)page * Hkv * pg.page_size + pos % pg.page_size;
    hstride = pg.page_size;
  } else {
    base = (int64_t)b * Hkv * cap + pos;
    hstride = cap;
  }
  const int64_t src = (int64_t)(qs + i) * ld_new;
  const int chunks = D / 8;  // 16-byte pieces per row
  for (int e = lane; e < Hkv * chunks; e += 32) {
    const int h = e / chunks, c = e - h * chunks;
    const int64_t dst = (base + h * hstride) * D + c * 8;
    *reinterpret_cast<uint4*>(kc + dst) = *reinterpret_cast<const uint4*>(kn + src + h * D + c * 8);
    *reinterpret_cast<uint4*>(vc + dst) = *reinterpret_cast<const uint4*>(vn + src + h * D + c * 8);
  }
}

cudaError_t launch_gqa_prefill_attn(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                                    const int32_t* q_start, const int32_t* kv_len, int64_t bs, int64_t Hq,
                                    int64_t Hkv, int64_t cap, int64_t total_q, int64_t max_q_len, float scale,
                                    uint16_t* out, int32_t* err, cudaStream_t st, const KvPages* pages) {
  PrefillParams p;
  p.q_start = q_start;
  p.kv_len = kv_len;
  p.out = out;
  p.err = err;
  p.Hq = (int)Hq;
  p.Hkv = (int)Hkv;
  p.group = (int)(Hq / Hkv);
  p.bs = (int)bs;
  p.cap = cap;
  p.total_q = total_q;
  p.max_q_len = (int)max_q_len;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.table = pages ? pages->table : nullptr;
  p.max_pages = pages ? pages->max_pages : 0;
  p.page_size = pages ? pages->page_size : 0;
  p.num_pages = pages ? pages->num_pages : 0;
  const int tpt = kRows / p.group;
  if (max_q_len * p.group <= 8 * kRows) {
    // short prompts (at most 8 query tiles per head group): two tiles per CTA share each K/V tile
    // and the per-CTA fixed costs (measured faster: 64 x 234 tokens 162 vs 187 us)
    dim3 grid((unsigned)((max_q_len + 2 * tpt - 1) / (2 * tpt)), (unsigned)(bs * Hkv));
    cudaError_t e =
        cudaFuncSetAttribute(gqa_prefill_pp_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPPSmemBytes);
    if (e != cudaSuccess) return e;
    return launch_k(gqa_prefill_pp_kernel, grid, dim3(kPPThreads), kPPSmemBytes, st, 1, tmQ, tmK, tmV, p);
  }
  // long prompts: one tile per CTA (measured faster: 4096 tokens 231 vs 309 us)
  dim3 grid((unsigned)((max_q_len + tpt - 1) / tpt), (unsigned)(bs * Hkv));
  cudaError_t e = cudaFuncSetAttribute(gqa_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  return launch_k(gqa_prefill_kernel, grid, dim3(kThreads), kSmemBytes, st, 1, tmQ, tmK, tmV, p);
}

cudaError_t launch_kv_append_extend(uint16_t* kc, uint16_t* vc, const uint16_t* kn, const uint16_t* vn,
                                    int64_t ld_new, const int32_t* q_start, const int32_t* kv_len, int64_t bs,
                                    int64_t Hkv, int64_t D, int64_t cap, int64_t total_q, int64_t max_q_len,
                                    int32_t* err, cudaStream_t st, const KvPages* pages) {
  const KvPages pg = pages ? *pages : KvPages{};
  dim3 grid((unsigned)((max_q_len + 7) / 8), (unsigned)bs);
  return launch_k(kv_append_extend_kernel, grid, dim3(256), 0, st, 1, kc, vc, kn, vn, ld_new, q_start, kv_len,
                  (int)Hkv, (int)D, cap, total_q, (int)max_q_len, err, pg);
}

}  // namespace mxg
