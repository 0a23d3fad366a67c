// GQA decode attention over the active prefix of a preallocated KV cache.
//
// [FSKV] §5: the cache keeps its full capacity and attention reads only the filled prefix
// K[:, :, :kv_len], V[:, :, :kv_len]; §4: expanding the KV heads (repeat_interleave) before
// attention multiplies the bytes touched. [S2.1] "What's Open Source": decode with native
// GQA (a stride-0 broadcast of K/V over the query heads of a group).
//
// Design (HBM-bound: 4 flop per byte of K/V at group 4):
//  * split-KV ("flash-decoding"): CTA = (kv split, sequence b, kv head g). Each CTA streams
//    its slice of K and V exactly once and serves all Hq/Hkv query heads of the group, so
//    K/V bytes are read once per KV head, never per query head.
//  * one producer warp drives TMA (2-D tiled, 128-byte swizzle) into a 3-4 stage ring of
//    64-token K and V tiles, with mbarrier full/empty handshakes (bounded waits);
//  * four consumer warps, 16 tokens each per tile, compute S^T = K Q^T and O^T += V^T P^T
//    with m16n8k16 bf16 tensor-core tiles (tokens x heads, heads padded to 8), fp32
//    online softmax in base 2; P enters the PV product as a bf16 pair hi + lo (two MMAs on
//    the same V fragments), so the weights keep ~16 significant bits instead of 8;
//  * the CTA merges its 4 warps and writes (O/l, log2-sum-exp) per head; a small combine
//    kernel merges the splits of each (b, h). With a single split the CTA writes bf16 out.
// Grid size is fixed by a host bound on kv_len, so the call is graph-capturable; CTAs whose
// split starts past kv_len exit at once.
#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"

namespace mxg {

namespace {

constexpr int kTileTok = 64;        // tokens per pipeline stage
constexpr int kMaxSplitTiles = 16;  // a split covers at most 1024 tokens (attn_chunk)
constexpr int kSplitTok = 768;      // split length (attn_chunk)
constexpr int kSplitTokFew = 512;   // split length with at most kFewPairs (b, g) pairs (attn_chunk)
constexpr int kFewPairs = 32;
constexpr int kMinSplitItems = 128; // fewest (split, b, g) items at the kv_len bound (attn_chunk)
constexpr int kConsumers = 4;       // consumer warps (16 tokens each per tile)
constexpr int kThreads = (kConsumers + 1) * 32;

// Shared-memory plan of the split kernel. kMx: K and V are MXFP8 (E4M3 codes [64, D] per tile,
// plus their UE8M0 scales [64, D/32]); otherwise bf16 [64, D] per tile.
template <int D, bool kMx>
struct AttnShape {
  static constexpr int kTileBytes = kTileTok * D * (kMx ? 1 : 2);      // one K (or V) tile
  static constexpr int kScaleTileBytes = kMx ? kTileTok * D / 32 : 0;  // its scale bytes
  static constexpr int kCodeStageBytes = 2 * kTileBytes;
  static constexpr int kStageBytes = kCodeStageBytes + 2 * kScaleTileBytes;  // bytes landing per stage
  // MXFP8: 3 stages of 16.5 KB keep 4 CTAs (16 consumer warps) on an SM; the consumer's
  // conversion work, not the bytes in flight, limits that variant
  static constexpr int kStages = kMx ? (D == 128 ? 3 : 6) : (D == 128 ? 3 : 4);
  static constexpr int kScaleRingOff = kStages * kCodeStageBytes;  // scales after all code stages
  static constexpr int kRingBytes = kStages * kStageBytes;
  static constexpr int kMergeBytes = kConsumers * 8 * D * 4 + kConsumers * 8 * 2 * 4;
  static constexpr int kBodyBytes = kRingBytes > kMergeBytes ? kRingBytes : kMergeBytes;
  static constexpr int kPBytes = kConsumers * 2 * 8 * 16 * 2;  // per-warp P^T staging, hi and lo (bf16 [8][16])
  static constexpr int kSmemBytes = 1024 + kBodyBytes + kPBytes + 2 * kStages * 8;
};

// Byte address (shared space) of element (row, col) of a [64, D] bf16 tile stored as D/64
// column boxes of 64 rows x 128 bytes with the 128-byte swizzle (16-byte chunk ^= row % 8).
__device__ __forceinline__ uint32_t tile_addr(uint32_t base, int row, int col) {
  const int half = col >> 6;
  const int chunk = (col & 63) >> 3;
  return base + half * (kTileTok * 128) + row * 128 + ((chunk ^ (row & 7)) << 4);
}

// Byte address of code byte `col` of row `row` in a [64, D] E4M3 tile loaded by TMA with a
// D-byte swizzle: 128-byte rows, 16-byte chunk ^= row % 8 (D = 128); 64-byte rows, chunk ^=
// (row / 2) % 4 (D = 64).
template <int D>
__device__ __forceinline__ uint32_t code_addr(uint32_t base, int row, int col) {
  if constexpr (D == 128)
    return base + row * 128 + (((col >> 4) ^ (row & 7)) << 4) + (col & 15);
  else
    return base + row * 64 + (((col >> 4) ^ ((row >> 1) & 3)) << 4) + (col & 15);
}

// Shared-memory loads that the compiler may schedule freely between memory barriers (not
// volatile; the "memory" clobber keeps them after the mbarrier wait that publishes the stage).
__device__ __forceinline__ uint32_t lds_u32(uint32_t addr) {
  uint32_t v;
  asm("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ uint2 lds_u32x2(uint32_t addr) {
  uint2 v;
  asm("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t lds_u16(uint32_t addr) {
  uint16_t v;
  asm("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr) : "memory");
  return v;
}

// Four E4M3 codes (the bytes of w) -> two f16 pairs, exactly: lo = codes 0, 1; hi = codes 2, 3.
__device__ __forceinline__ void e4m3x4_to_f16(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// Byte X of a and byte X of b, each an E4M3 code, as a bf16 pair (value * 2^-120 each). The
// code's sign goes to bf16's sign bit and its 4 exponent + 3 mantissa bits to bf16 bits 10..4;
// read with bf16's exponent bias (127 instead of 7) every code -- zero and subnormals included
// -- is its E4M3 value times 2^-120 exactly, and none is Inf or NaN. (prmt with the selector's
// high bit set replicates the selected byte's sign into the byte above it.)
template <int X>
__device__ __forceinline__ uint32_t e4m3_pair_bf16(uint32_t a, uint32_t b) {
  constexpr uint32_t sel = ((8u | (4u + X)) << 12) | ((4u + X) << 8) | ((8u | X) << 4) | X;
  uint32_t t;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(t) : "r"(a), "r"(b), "n"(sel));
  return (t << 4) & 0x87F087F0u;
}

// UE8M0 byte e -> 2^(e - 127) in fp32. e = 0 (2^-127, blocks whose values are all below
// 2^-118) is read as 0.
__device__ __forceinline__ float ue8m0_f32(uint32_t e) { return __uint_as_float(e << 23); }

// Scale bytes e0 (bits 0..7) and e1 (bits 16..23) of v -> the bf16 pair (2^(e0-71), 2^(e1-71)),
// i.e. 2^(s + 56) for s = e - 127: bf16 exponent field e + 56 (exact for e <= 198).
__device__ __forceinline__ uint32_t pscale_pair(uint32_t v) { return (v & 0x00FF00FFu) * 128u + 0x1C001C00u; }

__device__ __forceinline__ uint32_t bmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

struct SplitParams {
  const uint16_t* q;
  int64_t ld_q;
  const int32_t* kv_len;
  int Hq, Hkv, group;
  int64_t cap;
  int chunk, max_splits, max_kv_len;
  float scale_log2;  // softmax scale * log2(e)
  float* o_part;     // [bs, Hq, max_splits, D]
  float* lse;        // [bs, Hq, max_splits]
  uint16_t* out;     // written directly when max_splits == 1
  uint8_t* oq;       // optional MXFP8 copy of out ([bs, Hq*D] E4M3 + [bs, Hq*D/32] UE8M0)
  uint8_t* os;
  int32_t* err;
  // Paged caches (table != nullptr): K/V rows of position t of sequence b, head g live at row
  // (page * Hkv + g) * page_size + t % page_size of a [num_pages, Hkv, page_size, D] pool, with
  // page = table[b * max_pages + t / page_size]. Otherwise [bs, Hkv, cap, D] (row bg * cap + t).
  const int32_t* table;
  int max_pages, page_size;
  int64_t num_pages;
};

// Failure-detection test hook (mxg_debug_stall_attn_loads): while it is nonzero the copy warp
// of the split kernel issues no loads, so the consumer warps wait on stages that nothing will
// fill; their bounded waits run out and the kernel winds down with MXG_ETIMEOUT. No copy is
// in flight when the CTA leaves, and nothing faults.
__device__ int g_stall_attn_loads = 0;

}  // namespace

// B fragments of Q^T (k = dim, n = head); lane holds head r4.
//  bf16 cache: k-step ks, dims ks*16 + 2*c4 (+1) and +8 (+9).
//  MXFP8 cache: k-steps 2j, 2j+1 cover MX block j; the thread's k slots of step 2j+e hold
//  dims 32j + 8*c4 + 4e + {0, 1} and + {2, 3} (the K fragments below use the same order, so
//  the dot product is unchanged), as f16 after scaling q by 2^qa.
template <int D, bool kMx>
__device__ __forceinline__ void load_q_frags(const uint16_t* __restrict__ q, int64_t ld_q, int b, int h0, int group,
                                             float scale_log2, int lane, uint32_t (&qb)[D / 16][2], float& sl2) {
  constexpr int KS = D / 16;
  constexpr int NB = D / 32;
  const int c4 = lane & 3, r4 = lane >> 2;
  sl2 = scale_log2;
  const bool hv = r4 < group;
  const uint16_t* qh = q + (int64_t)b * ld_q + (int64_t)(h0 + (hv ? r4 : 0)) * D;
  if constexpr (!kMx) {
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      qb[ks][0] = hv ? *reinterpret_cast<const uint32_t*>(qh + ks * 16 + 2 * c4) : 0u;
      qb[ks][1] = hv ? *reinterpret_cast<const uint32_t*>(qh + ks * 16 + 8 + 2 * c4) : 0u;
    }
  } else {
    uint4 qw[NB];
    float am = 0.f;
#pragma unroll
    for (int j = 0; j < NB; ++j) {
      qw[j] = hv ? *reinterpret_cast<const uint4*>(qh + 32 * j + 8 * c4) : make_uint4(0, 0, 0, 0);
      const uint32_t w[4] = {qw[j].x, qw[j].y, qw[j].z, qw[j].w};
#pragma unroll
      for (int k = 0; k < 4; ++k) am = fmaxf(am, fmaxf(fabsf(bf16_lo(w[k])), fabsf(bf16_hi(w[k]))));
    }
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) am = fmaxf(am, __shfl_xor_sync(MXG_FULL_MASK, am, off));
    // 2^qa brings the group's largest |q| into [2^14, 2^15): every bf16 q is then an f16 exactly
    // unless it sits 2^38 below that maximum
    int qa = 0;
    if (am > 0.f) qa = min(100, max(-100, 14 - ((int)((__float_as_uint(am) >> 23) & 0xFF) - 127)));
    const float f = __uint_as_float((uint32_t)(qa + 127) << 23);
#pragma unroll
    for (int j = 0; j < NB; ++j) {
      const uint32_t w[4] = {qw[j].x, qw[j].y, qw[j].z, qw[j].w};
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        qb[2 * j + e][0] = pack_f16x2(bf16_lo(w[2 * e]) * f, bf16_hi(w[2 * e]) * f);
        qb[2 * j + e][1] = pack_f16x2(bf16_lo(w[2 * e + 1]) * f, bf16_hi(w[2 * e + 1]) * f);
      }
    }
    sl2 = scale_log2 * __uint_as_float((uint32_t)(127 - qa) << 23);
  }
}

// Copy the K and V tile starting at cache row `row` (and, for an MXFP8 cache, their scales)
// into ring stage s; the stage's full barrier expects all of its bytes.
template <int D, bool kMx>
__device__ __forceinline__ void issue_tile(uint8_t* ring, int s, int row, uint64_t* full_s, const CUtensorMap* tmK,
                                           const CUtensorMap* tmV, const CUtensorMap* tmKS, const CUtensorMap* tmVS,
                                           uint64_t pol) {
  using S = AttnShape<D, kMx>;
  mbar_arrive_expect_tx(full_s, S::kStageBytes);
  uint8_t* kt = ring + s * S::kCodeStageBytes;
  uint8_t* vt = kt + S::kTileBytes;
  if constexpr (kMx) {
    uint8_t* kst = ring + S::kScaleRingOff + s * 2 * S::kScaleTileBytes;
    tma_load_2d_hint(kt, tmK, full_s, 0, row, pol);
    tma_load_2d_hint(vt, tmV, full_s, 0, row, pol);
    // row is a multiple of 64, so its scales start on a 16-byte line
    const int line = row / (16 / (D / 32));
    tma_load_2d_hint(kst, tmKS, full_s, 0, line, pol);
    tma_load_2d_hint(kst + S::kScaleTileBytes, tmVS, full_s, 0, line, pol);
  } else {
#pragma unroll
    for (int h = 0; h < D / 64; ++h) {  // 128-byte boxes (64 bf16) across the row
      tma_load_2d_hint(kt + h * kTileTok * 128, tmK, full_s, h * 64, row, pol);
      tma_load_2d_hint(vt + h * kTileTok * 128, tmV, full_s, h * 64, row, pol);
    }
  }
}

// One consumer warp's share of a 64-token K/V tile in ring stage s: its 16 tokens tb .. tb+15
// (tokens at or past t1 are masked), S^T = K Q^T, the online-softmax update of (m, l) per head
// and O^T += V^T P^T.
template <int D, bool kMx>
__device__ __forceinline__ void consume_tile(uint8_t* ring, int s, int tb, int t1, int r0, int lane,
                                             const uint32_t (&qb)[D / 16][2], float sl2, float& m_a, float& m_b,
                                             float& l_a, float& l_b, float (&o)[D / 16][4], uint16_t* ps,
                                             uint16_t* pl) {
  using S = AttnShape<D, kMx>;
  constexpr int KS = D / 16;
  constexpr int NB = D / 32;
  const int c4 = lane & 3, r4 = lane >> 2;
  const uint32_t kbase = smem_u32(ring + s * S::kCodeStageBytes);
  const uint32_t vbase = kbase + S::kTileBytes;
  const uint32_t ksbase = smem_u32(ring + S::kScaleRingOff + s * 2 * S::kScaleTileBytes);
  const uint32_t vsbase = ksbase + S::kScaleTileBytes;

  // S^T[16 tok x 8 heads] = K[16 x D] Q^T[D x 8]
  float sc[4] = {0.f, 0.f, 0.f, 0.f};
  if constexpr (!kMx) {
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      uint32_t a0, a1, a2, a3;
      ldmatrix_x4(tile_addr(kbase, r0 + (lane & 7) + 8 * ((lane >> 3) & 1), ks * 16 + 8 * (lane >> 4)), a0, a1,
                  a2, a3);
      mma_bf16_16816(sc, a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
    }
  } else {
    float acc[NB][4];
#pragma unroll
    for (int j = 0; j < NB; ++j) {
      acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
      const uint2 ka = lds_u32x2(code_addr<D>(kbase, r0 + r4, 32 * j + 8 * c4));
      const uint2 kb = lds_u32x2(code_addr<D>(kbase, r0 + r4 + 8, 32 * j + 8 * c4));
      uint32_t a0, a1, a2, a3;
      e4m3x4_to_f16(ka.x, a0, a2);
      e4m3x4_to_f16(kb.x, a1, a3);
      mma_f16_16816(acc[j], a0, a1, a2, a3, qb[2 * j][0], qb[2 * j][1]);
      e4m3x4_to_f16(ka.y, a0, a2);
      e4m3x4_to_f16(kb.y, a1, a3);
      mma_f16_16816(acc[j], a0, a1, a2, a3, qb[2 * j + 1][0], qb[2 * j + 1][1]);
    }
    // per-block exponents of tokens r4 and r4+8
    uint32_t ska, skb;
    if constexpr (D == 128) {
      ska = lds_u32(ksbase + (r0 + r4) * NB);
      skb = lds_u32(ksbase + (r0 + r4 + 8) * NB);
    } else {
      ska = lds_u16(ksbase + (r0 + r4) * NB);
      skb = lds_u16(ksbase + (r0 + r4 + 8) * NB);
    }
#pragma unroll
    for (int j = 0; j < NB; ++j) {
      const float fa = ue8m0_f32((ska >> (8 * j)) & 0xFF), fb = ue8m0_f32((skb >> (8 * j)) & 0xFF);
      sc[0] = fmaf(acc[j][0], fa, sc[0]);
      sc[1] = fmaf(acc[j][1], fa, sc[1]);
      sc[2] = fmaf(acc[j][2], fb, sc[2]);
      sc[3] = fmaf(acc[j][3], fb, sc[3]);
    }
  }
  const bool va = tb + r4 < t1, vb = tb + r4 + 8 < t1;
  const float x0 = va ? sc[0] * sl2 : -INFINITY;  // token r4,   head 2c4
  const float x1 = va ? sc[1] * sl2 : -INFINITY;  // token r4,   head 2c4+1
  const float x2 = vb ? sc[2] * sl2 : -INFINITY;  // token r4+8, head 2c4
  const float x3 = vb ? sc[3] * sl2 : -INFINITY;  // token r4+8, head 2c4+1
  float ma = fmaxf(x0, x2), mb = fmaxf(x1, x3);
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    ma = fmaxf(ma, __shfl_xor_sync(MXG_FULL_MASK, ma, off));
    mb = fmaxf(mb, __shfl_xor_sync(MXG_FULL_MASK, mb, off));
  }
  const float na = fmaxf(m_a, ma), nb = fmaxf(m_b, mb);
  const float ua = na == -INFINITY ? 0.f : na, ub = nb == -INFINITY ? 0.f : nb;
  const float alpha_a = exp2f(m_a - ua), alpha_b = exp2f(m_b - ub);
  m_a = na;
  m_b = nb;
  const float f0 = exp2f(x0 - ua), f1 = exp2f(x1 - ub), f2 = exp2f(x2 - ua), f3 = exp2f(x3 - ub);
  const __nv_bfloat16 p0 = __float2bfloat16_rn(f0), p1 = __float2bfloat16_rn(f1);
  const __nv_bfloat16 p2 = __float2bfloat16_rn(f2), p3 = __float2bfloat16_rn(f3);
  const __nv_bfloat16 q0 = __float2bfloat16_rn(f0 - __bfloat162float(p0));
  const __nv_bfloat16 q1 = __float2bfloat16_rn(f1 - __bfloat162float(p1));
  const __nv_bfloat16 q2 = __float2bfloat16_rn(f2 - __bfloat162float(p2));
  const __nv_bfloat16 q3 = __float2bfloat16_rn(f3 - __bfloat162float(p3));
  l_a = l_a * alpha_a + (f0 + f2);
  l_b = l_b * alpha_b + (f1 + f3);
#pragma unroll
  for (int mt = 0; mt < KS; ++mt) {
    o[mt][0] *= alpha_a;
    o[mt][1] *= alpha_b;
    o[mt][2] *= alpha_a;
    o[mt][3] *= alpha_b;
  }
  ps[(2 * c4) * 16 + r4] = __bfloat16_as_ushort(p0);
  ps[(2 * c4 + 1) * 16 + r4] = __bfloat16_as_ushort(p1);
  ps[(2 * c4) * 16 + r4 + 8] = __bfloat16_as_ushort(p2);
  ps[(2 * c4 + 1) * 16 + r4 + 8] = __bfloat16_as_ushort(p3);
  pl[(2 * c4) * 16 + r4] = __bfloat16_as_ushort(q0);
  pl[(2 * c4 + 1) * 16 + r4] = __bfloat16_as_ushort(q1);
  pl[(2 * c4) * 16 + r4 + 8] = __bfloat16_as_ushort(q2);
  pl[(2 * c4 + 1) * 16 + r4 + 8] = __bfloat16_as_ushort(q3);
  // rows past the split end may hold anything; P is 0 there, and V (codes and scales) is
  // zeroed so that a non-finite value cannot turn 0 * V into NaN
  if (tb + 16 > t1) {
    uint8_t* vt = ring + s * S::kCodeStageBytes + S::kTileBytes;
    if constexpr (!kMx) {
      for (int rr = lane >> 4; rr < 16; rr += 2) {
        if (tb + rr >= t1) {
          const int row = r0 + rr;
          const int cb = (lane & 15) * 16;  // 16 lanes x 16 bytes cover 256 bytes (two 128-byte halves)
          if (cb < D * 2) {
            const int half = cb >> 7;
            *reinterpret_cast<uint4*>(vt + half * (kTileTok * 128) + row * 128 + (cb & 127)) = make_uint4(0, 0, 0, 0);
          }
        }
      }
    } else {
      // a row's D code bytes stay inside its own D-byte span under the swizzle
      for (int idx = lane; idx < 16 * (D / 16); idx += 32) {
        const int rr = idx / (D / 16);
        if (tb + rr >= t1) *reinterpret_cast<uint4*>(vt + (r0 + rr) * D + (idx % (D / 16)) * 16) = make_uint4(0, 0, 0, 0);
      }
      uint8_t* vst = ring + S::kScaleRingOff + s * 2 * S::kScaleTileBytes + S::kScaleTileBytes;
      if (lane < 16 && tb + lane >= t1) {
#pragma unroll
        for (int j = 0; j < NB; ++j) vst[(r0 + lane) * NB + j] = 0;
      }
    }
    fence_proxy_async_smem();
  }
  __syncwarp();
  const uint32_t b0 = *reinterpret_cast<const uint32_t*>(ps + r4 * 16 + 2 * c4);
  const uint32_t b1 = *reinterpret_cast<const uint32_t*>(ps + r4 * 16 + 8 + 2 * c4);
  const uint32_t l0 = *reinterpret_cast<const uint32_t*>(pl + r4 * 16 + 2 * c4);
  const uint32_t l1 = *reinterpret_cast<const uint32_t*>(pl + r4 * 16 + 8 + 2 * c4);
  // O^T[D x 8] += V^T[D x 16 tok] P^T[16 tok x 8]
  if constexpr (!kMx) {
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
      uint32_t a0, a1, a2, a3;
      ldmatrix_x4_trans(tile_addr(vbase, r0 + (lane & 7) + 8 * (lane >> 4), mt * 16 + 8 * ((lane >> 3) & 1)), a0,
                        a1, a2, a3);
      mma_bf16_16816(o[mt], a0, a1, a2, a3, b0, b1);
      mma_bf16_16816(o[mt], a0, a1, a2, a3, l0, l1);
    }
  } else {
    // m-tile 2j+f of block j: A row r4 is dim 32j + 4*r4 + 2f, row r4+8 is that dim + 1; the
    // k slots are tokens 2*c4 (+1) and 2*c4 + 8 (+9), as in P^T.
    uint32_t s01[NB], s89[NB];  // (token 2c4, 2c4+1) / (2c4+8, 2c4+9) exponent bytes of block j at bits 0 / 16
    if constexpr (D == 128) {
      const uint2 x01 = lds_u32x2(vsbase + (r0 + 2 * c4) * NB);
      const uint2 x89 = lds_u32x2(vsbase + (r0 + 2 * c4 + 8) * NB);
#pragma unroll
      for (int j = 0; j < NB; ++j) {
        s01[j] = __byte_perm(x01.x, x01.y, 0x0400 + j * 0x0101);
        s89[j] = __byte_perm(x89.x, x89.y, 0x0400 + j * 0x0101);
      }
    } else {
      const uint32_t x01 = lds_u32(vsbase + (r0 + 2 * c4) * NB);
      const uint32_t x89 = lds_u32(vsbase + (r0 + 2 * c4 + 8) * NB);
#pragma unroll
      for (int j = 0; j < NB; ++j) {
        s01[j] = __byte_perm(x01, 0, 0x0200 + j * 0x0101);
        s89[j] = __byte_perm(x89, 0, 0x0200 + j * 0x0101);
      }
    }
#pragma unroll
    for (int j = 0; j < NB; ++j) {
      const uint32_t f01 = pscale_pair(s01[j]), f89 = pscale_pair(s89[j]);
      const uint32_t bh0 = bmul2(b0, f01), bh1 = bmul2(b1, f89), bl0 = bmul2(l0, f01), bl1 = bmul2(l1, f89);
      const uint32_t w0 = lds_u32(code_addr<D>(vbase, r0 + 2 * c4, 32 * j + 4 * r4));
      const uint32_t w1 = lds_u32(code_addr<D>(vbase, r0 + 2 * c4 + 1, 32 * j + 4 * r4));
      const uint32_t w8 = lds_u32(code_addr<D>(vbase, r0 + 2 * c4 + 8, 32 * j + 4 * r4));
      const uint32_t w9 = lds_u32(code_addr<D>(vbase, r0 + 2 * c4 + 9, 32 * j + 4 * r4));
      {
        const uint32_t a0 = e4m3_pair_bf16<0>(w0, w1), a1 = e4m3_pair_bf16<1>(w0, w1);
        const uint32_t a2 = e4m3_pair_bf16<0>(w8, w9), a3 = e4m3_pair_bf16<1>(w8, w9);
        mma_bf16_16816(o[2 * j], a0, a1, a2, a3, bh0, bh1);
        mma_bf16_16816(o[2 * j], a0, a1, a2, a3, bl0, bl1);
      }
      {
        const uint32_t a0 = e4m3_pair_bf16<2>(w0, w1), a1 = e4m3_pair_bf16<3>(w0, w1);
        const uint32_t a2 = e4m3_pair_bf16<2>(w8, w9), a3 = e4m3_pair_bf16<3>(w8, w9);
        mma_bf16_16816(o[2 * j + 1], a0, a1, a2, a3, bh0, bh1);
        mma_bf16_16816(o[2 * j + 1], a0, a1, a2, a3, bl0, bl1);
      }
    }
  }
}

// Stage a consumer warp's (m, l) of its 8 (padded) heads into ml [warp][8][2] and its O of
// heads h_lo .. h_lo + HR - 1 into os [warp][HR][D] (fp32; an MXFP8 cache's O loses its 2^-64).
template <int D, bool kMx, int HR>
__device__ __forceinline__ void stage_warp(float* os, float* ml, int warp, int lane, const float (&o)[D / 16][4],
                                           float m_a, float l_a, float m_b, float l_b, int h_lo) {
  constexpr int KS = D / 16;
  const int c4 = lane & 3, r4 = lane >> 2;
  const float oscale = kMx ? 0x1p64f : 1.f;
  const int ha = 2 * c4 - h_lo, hb = ha + 1;  // this thread's two heads, relative to the round
#pragma unroll
  for (int mt = 0; mt < KS; ++mt) {
    const int d = kMx ? 32 * (mt >> 1) + 4 * r4 + 2 * (mt & 1) : mt * 16 + r4;
    const int d2 = kMx ? d + 1 : d + 8;
    if (ha >= 0 && ha < HR) {
      os[(warp * HR + ha) * D + d] = o[mt][0] * oscale;
      os[(warp * HR + ha) * D + d2] = o[mt][2] * oscale;
    }
    if (hb >= 0 && hb < HR) {
      os[(warp * HR + hb) * D + d] = o[mt][1] * oscale;
      os[(warp * HR + hb) * D + d2] = o[mt][3] * oscale;
    }
  }
  if (r4 == 0) {
    ml[(warp * 8 + 2 * c4) * 2] = m_a;
    ml[(warp * 8 + 2 * c4) * 2 + 1] = l_a;
    ml[(warp * 8 + 2 * c4 + 1) * 2] = m_b;
    ml[(warp * 8 + 2 * c4 + 1) * 2 + 1] = l_b;
  }
}

// Merge the consumer warps' staged state for head h (round-relative hr) and dimension d: the
// running maximum M, the softmax denominator L and the unnormalised output O.
template <int D, int HR>
__device__ __forceinline__ void merge_warps(const float* os, const float* ml, int h, int hr, int d, float& M,
                                            float& L, float& O) {
  M = -INFINITY;
#pragma unroll
  for (int w = 0; w < kConsumers; ++w) M = fmaxf(M, ml[(w * 8 + h) * 2]);
  L = 0.f;
  O = 0.f;
#pragma unroll
  for (int w = 0; w < kConsumers; ++w) {
    const float mw = ml[(w * 8 + h) * 2];
    const float f = mw == -INFINITY ? 0.f : exp2f(mw - M);
    L += ml[(w * 8 + h) * 2 + 1] * f;
    O += os[(w * HR + hr) * D + d] * f;
  }
}

// One CTA = one (split, b, g). tmK/tmV map the K/V rows (bf16 [rows, D], or E4M3 codes
// [rows, D] when kMx); tmKS/tmVS map the UE8M0 scales of an MXFP8 cache as 16-byte lines
// ([rows * D/32 / 16, 16]) and are unused for bf16.
//
// MXFP8 K/V: a cached value is c * 2^s (c an E4M3 value, s the shared exponent of its 32-wide
// block along D). S = K q^T is taken per block: the codes enter an f16 MMA exactly (hardware
// E4M3 -> f16 conversion) against q prescaled by a power of two into f16's range, and each
// block's partial dot product is multiplied by 2^s in fp32. In O^T += V^T P^T the exponent
// varies along the contraction (tokens), so it moves to P: a code enters as the bf16 c * 2^-120
// (bit placement, exact) and P as P * 2^(s + 56) (exact bf16 multiply); O then carries 2^-64,
// removed in the merge.
template <int D, bool kMx>
__global__ void __launch_bounds__(kThreads) gqa_split_kernel(const __grid_constant__ CUtensorMap tmK,
                                                             const __grid_constant__ CUtensorMap tmV,
                                                             const __grid_constant__ CUtensorMap tmKS,
                                                             const __grid_constant__ CUtensorMap tmVS,
                                                             const SplitParams p) {
  using S = AttnShape<D, kMx>;
  constexpr int KS = D / 16;  // k-steps of the QK^T product / m-tiles of O^T
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  uint16_t* pstage = reinterpret_cast<uint16_t*>(smem + S::kBodyBytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::kBodyBytes + S::kPBytes);
  uint64_t* empty = full + S::kStages;

  // Read before the programmatic wait, while the previous kernel may still run: the test hook
  // (written by the host alone), kv_len, and -- contiguous caches -- the first ring-full of
  // tiles lying wholly below row kv_len - 1. The previous kernel of a decode step is the KV
  // append, which writes only that row; the library's kernels that write other cache rows or
  // kv_len (kv_append_extend*, copy_bytes) let their successor start only after they complete.
  MXG_TL_SCOPE(kTlSplitAttn);
  const int stall = *reinterpret_cast<volatile int*>(&g_stall_attn_loads);
  const int split = blockIdx.x;
  const int bg = blockIdx.y;
  const int b = bg / p.Hkv, g = bg - b * p.Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = p.kv_len[b];
  const bool bad_len = n < 1 || (int64_t)n > p.cap || n > p.max_kv_len;

  // set by a consumer warp whose wait ran out; read by all consumers after the merge barrier
  __shared__ volatile int merge_abort;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumers);
    }
    merge_abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  int npre = 0;  // tiles the copy warp issues before the wait
  if (!bad_len && split * p.chunk < n && !p.table && !stall) {
    const int t0p = split * p.chunk;
    const int ntp = (min(n, t0p + p.chunk) - t0p + kTileTok - 1) / kTileTok;
    npre = min(min(S::kStages, ntp), (n - 1 - t0p) / kTileTok);
    if (warp == kConsumers && lane == 0 && npre > 0) {
      prefetch_tensormap(&tmK);
      prefetch_tensormap(&tmV);
      if constexpr (kMx) {
        prefetch_tensormap(&tmKS);
        prefetch_tensormap(&tmVS);
      }
      const uint64_t pol = l2_policy_evict_first();
      const int row0p = (int)((int64_t)bg * p.cap + t0p);
      for (int i = 0; i < npre; ++i)
        issue_tile<D, kMx>(ring, i, row0p + i * kTileTok, &full[i], &tmK, &tmV, &tmKS, &tmVS, pol);
    }
  }
  pdl_wait();
  MXG_TL_WAITED();
  pdl_trigger();
  if (bad_len) {  // (nothing was issued before the wait)
    if (split == 0 && g == 0 && threadIdx.x == 0) set_error(p.err, MXG_EDEVICE);
    // several splits: weight zero for every split of the sequence, so the combine writes zeros
    if (p.max_splits > 1 && threadIdx.x < p.group)
      p.lse[((int64_t)b * p.Hq + g * p.group + threadIdx.x) * p.max_splits + split] = -INFINITY;
    if (p.max_splits == 1 && warp < kConsumers) {  // single-split mode: no combine pass, zero here
      for (int i = threadIdx.x; i < p.group * D; i += kConsumers * 32) {
        const int64_t o = ((int64_t)b * p.Hq + g * p.group) * D + i;
        p.out[o] = 0;
        if (p.oq) {
          p.oq[o] = 0;
          if ((i & 31) == 0) p.os[o >> 5] = 0;
        }
      }
    }
    return;
  }
  const int t0 = split * p.chunk;
  if (t0 >= n) {  // a split past the prefix: weight zero, so the combine needs no kv_len
    if (p.max_splits > 1 && threadIdx.x < p.group)
      p.lse[((int64_t)b * p.Hq + g * p.group + threadIdx.x) * p.max_splits + split] = -INFINITY;
    return;
  }
  const int t1 = min(n, t0 + p.chunk);
  const int ntiles = (t1 - t0 + kTileTok - 1) / kTileTok;
  const int row0 = (int)((int64_t)bg * p.cap + t0);  // host guarantees bs*Hkv*cap < 2^31 (contiguous)


  if (warp == kConsumers) {
    // ------------------------------------------------------------- producer
    // Paged caches: the warp looks up the page of every tile of the split at once (one round
    // trip for the table instead of one per tile on the copy issue path). A 64-token tile never
    // straddles a page (page_size % 64 == 0 and tile starts are multiples of 64).
    __shared__ int tile_row[kMaxSplitTiles];
    if (p.table) {
      for (int i = lane; i < ntiles; i += 32) {
        const int t = t0 + i * kTileTok;
        const int page = p.table[(int64_t)b * p.max_pages + t / p.page_size];
        int row;
        if (page < 0 || page >= p.num_pages) {
          set_error(p.err, MXG_EDEVICE);
          row = (int)(p.num_pages * p.Hkv * p.page_size);  // past the pool: the copy engine reads zeros
        } else {
          row = (int)(((int64_t)page * p.Hkv + g) * p.page_size + t % p.page_size);
        }
        tile_row[i] = row;
      }
      __syncwarp();
    }
    if (lane == 0) {
      prefetch_tensormap(&tmK);
      prefetch_tensormap(&tmV);
      if constexpr (kMx) {
        prefetch_tensormap(&tmKS);
        prefetch_tensormap(&tmVS);
      }
      const uint64_t pol = l2_policy_evict_first();
      const int nissue = stall ? 0 : ntiles;
      for (int i = npre; i < nissue; ++i) {  // npre = 0 when the hook stalls the loads
        const int s = i % S::kStages;
        if (i >= S::kStages && !mbar_wait(&empty[s], ((i / S::kStages) - 1) & 1, p.err)) break;
        issue_tile<D, kMx>(ring, s, p.table ? tile_row[i] : row0 + i * kTileTok, &full[s], &tmK, &tmV, &tmKS, &tmVS,
                           pol);
      }
    }
    return;
  }

  // --------------------------------------------------------------- consumers
  const int h0 = g * p.group;
  uint32_t qb[KS][2];
  float sl2;
  load_q_frags<D, kMx>(p.q, p.ld_q, b, h0, p.group, p.scale_log2, lane, qb, sl2);
  float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;
  float o[KS][4];
#pragma unroll
  for (int i = 0; i < KS; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

  uint16_t* ps = pstage + warp * (2 * 8 * 16);  // P^T staging: hi [8 heads][16 tokens], then lo
  uint16_t* pl = ps + 8 * 16;
  const int r0 = warp * 16;
  bool ok = true;
  for (int i = 0; i < ntiles; ++i) {
    const int s = i % S::kStages;
    if (!__all_sync(MXG_FULL_MASK, mbar_wait(&full[s], (i / S::kStages) & 1, p.err))) {
      ok = false;
      break;
    }
    MXG_TL_MARK1();  // timeline: first tile landed
    consume_tile<D, kMx>(ring, s, t0 + i * kTileTok + r0, t1, r0, lane, qb, sl2, m_a, m_b, l_a, l_b, o, ps, pl);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
  MXG_TL_MARK2();  // timeline: last tile consumed
  // A warp whose wait ran out still meets the other consumer warps at the named barrier below
  // (leaving would hold them there for good): it publishes the failure before the barrier, and
  // all consumer warps leave together after it.
  if (!ok) merge_abort = 1;

  // l partial sums: reduce over the 8 lanes that share a head pair
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    l_a += __shfl_xor_sync(MXG_FULL_MASK, l_a, off);
    l_b += __shfl_xor_sync(MXG_FULL_MASK, l_b, off);
  }
  // merge the consumer warps through shared memory (the ring is idle now: every issued tile
  // was consumed before the named barrier below)
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumers * 32) : "memory");
  if (merge_abort) {
    // the error flag holds MXG_ETIMEOUT; leave nothing stale behind: zeros for a single
    // split, otherwise a split of weight zero (lse = -inf), which the combine pass skips
    for (int idx = threadIdx.x; idx < p.group * D; idx += kConsumers * 32) {
      const int h = idx / D, d = idx - h * D;
      const int64_t bh = (int64_t)b * p.Hq + h0 + h;
      if (p.max_splits == 1) {
        p.out[bh * D + d] = 0;
        if (p.oq) {
          p.oq[bh * D + d] = 0;
          if ((d & 31) == 0) p.os[(bh * D + d) >> 5] = 0;
        }
      } else {
        p.o_part[(bh * p.max_splits + split) * D + d] = 0.f;
        if (d == 0) p.lse[bh * p.max_splits + split] = -INFINITY;
      }
    }
    return;
  }
  float* os = reinterpret_cast<float*>(ring);  // [warp][8 heads][D]
  float* ml = os + kConsumers * 8 * D;         // [warp][8 heads][m, l]
  stage_warp<D, kMx, 8>(os, ml, warp, lane, o, m_a, l_a, m_b, l_b, 0);
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumers * 32) : "memory");
  for (int idx = threadIdx.x; idx < p.group * D; idx += kConsumers * 32) {
    const int h = idx / D, d = idx - h * D;
    float M, L, O;
    merge_warps<D, 8>(os, ml, h, h, d, M, L, O);
    const int64_t bh = (int64_t)b * p.Hq + h0 + h;
    if (p.max_splits == 1) {
      const __nv_bfloat16 ob = __float2bfloat16_rn(O / L);
      p.out[bh * D + d] = __bfloat16_as_ushort(ob);
      // idx runs over whole warps of consecutive d (D is a multiple of 32): one MX block per warp
      if (p.oq) mx_quant_warp_store(__bfloat162float(ob), p.oq + bh * D + d, p.os + ((bh * D + d) >> 5));
    } else {
      p.o_part[(bh * p.max_splits + split) * D + d] = O / L;
      if (d == 0) p.lse[bh * p.max_splits + split] = M + log2f(L);
    }
  }
}

// Merge the splits of each (b, h): weights 2^(lse_i - max lse). Every split writes its lse each
// call (-inf for a split past the prefix or a sequence whose kv_len is out of range, or one
// that gave up on a bounded wait), so the kernel reads no kv_len: it loads the lse values and
// the partial outputs of up to kSplits splits at once, skips splits of weight zero, and writes
// zeros when every split has weight zero. One D-thread CTA serves the `group` query heads of
// one (b, kv head) -- thread d takes dimension d of each head, up to kHeads heads' loads in
// flight together. (Capping it at 64 registers, so that the O projection's CTAs become resident
// and prefetch during the combine, measured no faster: the prefetch then competes with the
// combine's own loads.)
template <int D>
__global__ void __launch_bounds__(D) gqa_combine_kernel(const float* __restrict__ o_part,
                                                        const float* __restrict__ lse, int max_splits, int group,
                                                        uint16_t* __restrict__ out, uint8_t* __restrict__ oq,
                                                        uint8_t* __restrict__ os) {
  MXG_TL_SCOPE(kTlCombine);
  pdl_wait();
  MXG_TL_WAITED();
  pdl_trigger();
  constexpr int kSplits = 8, kHeads = 4;
  const int d = threadIdx.x;
  for (int hb = 0; hb < group; hb += kHeads) {
    float M[kHeads], W[kHeads], acc[kHeads];
#pragma unroll
    for (int j = 0; j < kHeads; ++j) {
      M[j] = -INFINITY;
      W[j] = 0.f;
      acc[j] = 0.f;
    }
    for (int i0 = 0; i0 < max_splits; i0 += kSplits) {
      float lv[kHeads][kSplits], ov[kHeads][kSplits];
#pragma unroll
      for (int j = 0; j < kHeads; ++j) {
        const int64_t bh = (int64_t)blockIdx.x * group + hb + j;
        const bool hv = hb + j < group;
#pragma unroll
        for (int i = 0; i < kSplits; ++i) {
          const bool v = hv && i0 + i < max_splits;
          lv[j][i] = v ? lse[bh * max_splits + i0 + i] : -INFINITY;
          ov[j][i] = v ? o_part[(bh * max_splits + i0 + i) * D + d] : 0.f;
        }
      }
#pragma unroll
      for (int j = 0; j < kHeads; ++j) {
        float Mb = M[j];
#pragma unroll
        for (int i = 0; i < kSplits; ++i) Mb = fmaxf(Mb, lv[j][i]);
        if (Mb == -INFINITY) continue;
        const float r = M[j] == -INFINITY ? 0.f : exp2f(M[j] - Mb);  // rescale the earlier batches' sums
        W[j] *= r;
        acc[j] *= r;
#pragma unroll
        for (int i = 0; i < kSplits; ++i)
          if (lv[j][i] != -INFINITY) {
            const float w = exp2f(lv[j][i] - Mb);
            W[j] += w;
            acc[j] += w * ov[j][i];
          }
        M[j] = Mb;
      }
    }
#pragma unroll
    for (int j = 0; j < kHeads; ++j) {
      if (hb + j >= group) break;
      const int64_t o = ((int64_t)blockIdx.x * group + hb + j) * D + d;
      const __nv_bfloat16 ob = __float2bfloat16_rn(M[j] == -INFINITY ? 0.f : acc[j] / W[j]);
      MXG_TL_MARK1();  // timeline: merged
      out[o] = __bfloat16_as_ushort(ob);
      if (oq) mx_quant_warp_store(__bfloat162float(ob), oq + o, os + (o >> 5));
    }
  }
  MXG_TL_MARK2();  // timeline: stores issued
}

// ---------------------------------------------------------------------------------- host
cudaError_t set_attn_load_stall(int on) {
  const int v = on ? 1 : 0;
  return cudaMemcpyToSymbol(g_stall_attn_loads, &v, sizeof(v));
}

int attn_chunk(int64_t bs, int64_t Hkv, int64_t max_kv_len) {
  // Splits of 768 tokens (12 tiles), 512 with at most 32 (b, g) pairs; below ~128 (split, b,
  // g) items at the bound (a few sequences), shorter splits so that at least that many CTAs
  // stream. Measured on GB300 at 32/8 heads, kv_len ~ U[234, 4096], splits of 128..1024
  // tokens: 768 the fastest (or within 1 %) for bs = 8..64, 512 for bs = 2..4 (bs = 4: 19.0
  // against 20.6 us at 768, MXFP8 cache 19.1 against 23.0), 256..640 alike for bs = 1.
  const int64_t cmax = bs * Hkv <= kFewPairs ? kSplitTokFew : kSplitTok;
  int64_t c = (bs * Hkv * max_kv_len + kMinSplitItems - 1) / kMinSplitItems;
  c = (c + kTileTok - 1) / kTileTok * kTileTok;
  if (c < kTileTok) c = kTileTok;
  if (c > cmax) c = cmax;
  return (int)c;
}

size_t attn_workspace_bytes(int64_t bs, int64_t Hq, int64_t Hkv, int64_t D, int64_t max_kv_len) {
  const int chunk = attn_chunk(bs, Hkv, max_kv_len);
  const int64_t ms = (max_kv_len + chunk - 1) / chunk;
  if (ms <= 1) return 0;
  return (size_t)(bs * Hq * ms * (D + 1)) * sizeof(float);
}

namespace {

template <bool kMx>
cudaError_t launch_split(const CUtensorMap& tmK, const CUtensorMap& tmV, const CUtensorMap& tmKS,
                         const CUtensorMap& tmVS, const uint16_t* q, int64_t ld_q, const int32_t* kv_len, int64_t bs,
                         int64_t Hq, int64_t Hkv, int64_t D, int64_t cap, int64_t max_kv_len, float scale,
                         uint16_t* out, int32_t* err, void* ws, cudaStream_t st, uint8_t* oq, uint8_t* os,
                         const KvPages* pages) {
  const int chunk = attn_chunk(bs, Hkv, max_kv_len);
  const int ms = (int)((max_kv_len + chunk - 1) / chunk);
  SplitParams p;
  p.q = q;
  p.ld_q = ld_q;
  p.kv_len = kv_len;
  p.Hq = (int)Hq;
  p.Hkv = (int)Hkv;
  p.group = (int)(Hq / Hkv);
  p.cap = cap;
  p.chunk = chunk;
  p.max_splits = ms;
  p.max_kv_len = (int)max_kv_len;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.o_part = reinterpret_cast<float*>(ws);
  p.lse = ms > 1 ? p.o_part + bs * Hq * ms * D : nullptr;
  p.out = out;
  p.oq = oq;
  p.os = os;
  p.err = err;
  p.table = pages ? pages->table : nullptr;
  p.max_pages = pages ? pages->max_pages : 0;
  p.page_size = pages ? pages->page_size : 0;
  p.num_pages = pages ? pages->num_pages : 0;
  dim3 grid((unsigned)ms, (unsigned)(bs * Hkv));
  cudaError_t e;
  if (D == 128) {
    const int smem = AttnShape<128, kMx>::kSmemBytes;
    e = cudaFuncSetAttribute(gqa_split_kernel<128, kMx>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    e = launch_k(gqa_split_kernel<128, kMx>, grid, dim3(kThreads), smem, st, 1, tmK, tmV, tmKS, tmVS, p);
  } else {
    const int smem = AttnShape<64, kMx>::kSmemBytes;
    e = cudaFuncSetAttribute(gqa_split_kernel<64, kMx>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    e = launch_k(gqa_split_kernel<64, kMx>, grid, dim3(kThreads), smem, st, 1, tmK, tmV, tmKS, tmVS, p);
  }
  if (e != cudaSuccess || ms == 1) return e;
  // one D-thread CTA per (b, kv head)
  const dim3 cgrid((unsigned)(bs * Hkv));
  if (D == 128)
    return launch_k(gqa_combine_kernel<128>, cgrid, dim3(128), 0, st, 1, static_cast<const float*>(p.o_part),
                    static_cast<const float*>(p.lse), ms, p.group, out, oq, os);
  return launch_k(gqa_combine_kernel<64>, cgrid, dim3(64), 0, st, 1, static_cast<const float*>(p.o_part),
                  static_cast<const float*>(p.lse), ms, p.group, out, oq, os);
}

}  // namespace

cudaError_t launch_gqa_decode_attn(const CUtensorMap& tmK, const CUtensorMap& tmV, const uint16_t* q, int64_t ld_q,
                                   const int32_t* kv_len, int64_t bs, int64_t Hq, int64_t Hkv, int64_t D, int64_t cap,
                                   int64_t max_kv_len, float scale, uint16_t* out, int32_t* err, void* ws,
                                   cudaStream_t st, uint8_t* oq, uint8_t* os, const KvPages* pages) {
  return launch_split<false>(tmK, tmV, tmK, tmV, q, ld_q, kv_len, bs, Hq, Hkv, D, cap, max_kv_len, scale, out, err, ws,
                             st, oq, os, pages);
}

cudaError_t launch_gqa_decode_attn_kv_mx(const CUtensorMap& tmK, const CUtensorMap& tmV, const CUtensorMap& tmKS,
                                         const CUtensorMap& tmVS, const uint16_t* q, int64_t ld_q,
                                         const int32_t* kv_len, int64_t bs, int64_t Hq, int64_t Hkv, int64_t D,
                                         int64_t cap, int64_t max_kv_len, float scale, uint16_t* out, int32_t* err,
                                         void* ws, cudaStream_t st, const KvPages* pages) {
  return launch_split<true>(tmK, tmV, tmKS, tmVS, q, ld_q, kv_len, bs, Hq, Hkv, D, cap, max_kv_len, scale, out, err,
                            ws, st, nullptr, nullptr, pages);
}

}  // namespace mxg

MXG_TL_UNIT(attn)
