// Shared device helpers for the sm_103a kernels of libmxg.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mxg.h"

#define MXG_FULL_MASK 0xffffffffu

namespace mxg {

// ------------------------------------------------------------------ error flag
// First device-side error wins (atomicCAS from 0); the host reads it when it wants.
__device__ __forceinline__ void set_error(int32_t* err, int32_t code) {
  if (err) atomicCAS(err, 0, code);
}

// ------------------------------------------------------------------ MX element/scale
// UE8M0 shared exponent of a block whose max |v| is `amax` (fp32): s = floor(log2 amax) - 8,
// clamped to [-127, 127]; zero and fp32-subnormal amax give the clamp value -127
// (their exponent field is 0, i.e. "below range").
__device__ __forceinline__ int mx_shared_exp(float amax) {
  int e = (int)((__float_as_uint(amax) >> 23) & 0xFFu) - 127;
  int s = e - 8;
  return s < -127 ? -127 : (s > 127 ? 127 : s);
}

// 2^-s as an fp32 (exact, normal for s in [-127, 119], which covers every finite fp32 amax).
__device__ __forceinline__ float mx_inv_scale(int s) { return __uint_as_float((uint32_t)(127 - s) << 23); }

// Two fp32 -> packed E4M3 pair (round to nearest even, saturating to +-448); `lo` lands in
// the low byte, i.e. at the lower address when stored little-endian.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return (uint32_t)r;
}

// Packed E4M3 pair -> two fp32 (exact).
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint16_t v) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(v));
  __half2 hh = *reinterpret_cast<__half2*>(&h);
  return __half22float2(hh);
}

// One 32-element MX block held one value per lane of a full warp: lane i stores the E4M3
// byte of its value to q_dst, lane 0 stores the block's UE8M0 scale byte to s_dst.
__device__ __forceinline__ void mx_quant_warp_store(float v, uint8_t* q_dst, uint8_t* s_dst) {
  float am = fabsf(v);
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) am = fmaxf(am, __shfl_xor_sync(MXG_FULL_MASK, am, off));
  const int s = mx_shared_exp(am);
  *q_dst = (uint8_t)(cvt_e4m3x2(v * mx_inv_scale(s), 0.f) & 0xFF);
  if ((threadIdx.x & 31) == 0) *s_dst = (uint8_t)(s + 127);
}

// SwiGLU activation in fp32, silu(g) * u = g / (1 + e^-g) * u, with the hardware exp and
// divide intrinsics (a few fp32 ulp); every SwiGLU epilogue of the library uses this one
// definition, so all kernel paths produce the same bits.
__device__ __forceinline__ float silu_mul(float g, float u) { return __fdividef(g, 1.f + __expf(-g)) * u; }

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// ------------------------------------------------------------------ programmatic dependent launch
// Let the next kernel on the stream be scheduled (it still waits for this one to finish).
// Executed only after this kernel's own pdl_wait(), so the next kernel's pre-wait prologue
// can never overlap anything but this kernel.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
// Wait until the previous kernel on the stream has completed and its writes are visible.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ------------------------------------------------------------------ timers / bounded waits
__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Upper bound on any in-kernel wait (mbarrier phase flips). A healthy wait is microseconds;
// after this the waiting thread records MXG_ETIMEOUT and the kernel winds down.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// ------------------------------------------------------------------ optional device timeline
// Compiled in only with -DMXG_TIMELINE (a separate, instrumented build of the library; the
// production library holds none of it). Lane 0 of every warp of an instrumented kernel appends
// one record {kernel id << 48 | linear block << 16 | warp, entry, return from the programmatic
// wait (0 if the warp does not wait), exit, mark 1, mark 2} in globaltimer ns to the buffer
// attached through
// the translation unit's mxg_tl_attach_<unit> entry point. The buffer has one region of `cap`
// records per SM, each with its own counter (one shared counter would serialise thousands of
// warps leaving at once); records past a region's end are dropped.
#ifdef MXG_TIMELINE
namespace tl {
static __device__ unsigned long long* g_buf;
static __device__ unsigned int* g_cnt;
static __device__ unsigned int g_cap;
constexpr unsigned kRec = 6;  // u64 per record
struct Scope {
  unsigned long long t0, tw, m1, m2;
  unsigned id;
  __device__ explicit Scope(unsigned kid) : t0(globaltimer_ns()), tw(0), m1(0), m2(0), id(kid) {}
  __device__ void waited() { tw = globaltimer_ns(); }
  // kernel-specific phase points: mark 1 keeps its first time, mark 2 its last
  __device__ void mark1() {
    if (!m1) m1 = globaltimer_ns();
  }
  __device__ void mark2() { m2 = globaltimer_ns(); }
  __device__ ~Scope() {
    if ((threadIdx.x & 31) || !g_buf) return;
    unsigned sm;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
    const unsigned i = atomicAdd(g_cnt + sm, 1u);
    if (i >= g_cap) return;
    const unsigned long long blk = ((unsigned long long)blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
    unsigned long long* r = g_buf + kRec * ((unsigned long long)sm * g_cap + i);
    r[0] = ((unsigned long long)id << 48) | (blk << 16) | (threadIdx.x >> 5);
    r[1] = t0;
    r[2] = tw;
    r[3] = globaltimer_ns();
    r[4] = m1;
    r[5] = m2;
  }
};
}  // namespace tl
#define MXG_TL_SCOPE(id) ::mxg::tl::Scope mxg_tl_scope_(id)
#define MXG_TL_WAITED() mxg_tl_scope_.waited()
#define MXG_TL_MARK1() mxg_tl_scope_.mark1()
#define MXG_TL_MARK2() mxg_tl_scope_.mark2()
#define MXG_TL_UNIT(name)                                                                            \
  extern "C" cudaError_t mxg_tl_attach_##name(void* buf, void* cnt, unsigned cap) {                  \
    cudaError_t e = cudaMemcpyToSymbol(::mxg::tl::g_buf, &buf, sizeof(buf));                         \
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(::mxg::tl::g_cnt, &cnt, sizeof(cnt));               \
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(::mxg::tl::g_cap, &cap, sizeof(cap));               \
    return e;                                                                                        \
  }
#else
#define MXG_TL_SCOPE(id) \
  do {                   \
  } while (0)
#define MXG_TL_WAITED() \
  do {                  \
  } while (0)
#define MXG_TL_MARK1() \
  do {                 \
  } while (0)
#define MXG_TL_MARK2() \
  do {                 \
  } while (0)
#define MXG_TL_UNIT(name)
#endif
// kernel ids of the timeline records
constexpr unsigned kTlMaxSm = 256;  // regions (and counters) of the timeline buffer
enum TlKernel : unsigned {
  kTlQuantize = 1,
  kTlRmsQuant = 2,
  kTlShift = 3,
  kTlCopy16 = 4,
  kTlKvAppend = 5,
  kTlSplitAttn = 6,
  kTlCombine = 7,
  kTlGemmTc = 16,  // + epilogue kind
  kTlGemmTc2 = 24,
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// Expect `bytes` more on the barrier's current phase without arriving on it.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity to complete. Returns false (and records
// MXG_ETIMEOUT in *err) if it did not complete within kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int32_t* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      set_error(err, MXG_ETIMEOUT);
      return false;
    }
  }
}

// ------------------------------------------------------------------ TMA
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int32_t x,
                                            int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(smem_dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_load_2d_hint(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int32_t x,
                                                 int32_t y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, %3}], "
      "[%4], %5;" ::"r"(smem_u32(smem_dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// 2-D TMA load into this CTA's shared memory whose completion is signalled on the mbarrier at
// shared::cluster address `bar_cl`, which may belong to the peer CTA of a tcgen05 CTA pair.
__device__ __forceinline__ void tma_load_2d_pair(void* smem_dst, const CUtensorMap* map, uint32_t bar_cl, int32_t x,
                                                 int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(smem_u32(smem_dst)),
      "l"(map), "r"(x), "r"(y), "r"(bar_cl)
      : "memory");
}

// 2-D TMA store of a shared-memory box (bulk-group completion); coordinates must be >= 0, the
// box is clipped at the tensor's edges.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* smem_src, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(map), "r"(x),
               "r"(y), "r"(smem_u32(smem_src))
               : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until every committed bulk store of this thread has completed.
__device__ __forceinline__ void bulk_wait_group0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------ tensor-core (legacy mma.sync) helpers
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, "
      "%2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                                  uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D(16x8, f32) += A(16x16, bf16, row) * B(16x8, bf16, col)
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, "
      "%2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

}  // namespace mxg
