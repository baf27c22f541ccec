// csa2_dev.cuh -- device helpers shared by the CSA2 kernels (sm_103a only).
//
// Inline-PTX wrappers for the Blackwell tensor-core path (tcgen05 MMA, TMEM,
// tcgen05.cp), bulk async copies with mbarrier completion, bounded waits, the
// E2M1/E4M3 block codec and the cache-page layouts.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/csa2.h"

namespace csa2 {

// ----------------------------------------------------------------- error word
// Workspace header: ws[0] = first error status, ws[1] = info code.
enum ErrInfo : int32_t {
  kInfoPage = 1,      // page id outside [0, n_pages)
  kInfoPos = 2,       // position beyond the request's pages
  kInfoTopkIdx = 3,   // a selected index outside [0, n_visible)
  kInfoGroup = 4,     // queries of one indexer group belong to different requests
  kInfoWait = 5,      // a bounded pipeline wait ran out
  kInfoPool = 6,      // a candidate pool that is not ascending blocks of 8 visible positions
};

__device__ __forceinline__ void report(int32_t* err, int32_t status, int32_t info) {
  if (err != nullptr && atomicCAS(err, 0, status) == 0) atomicExch(err + 1, info);
}

// Default bound of a pipeline wait, and the fixed bound of every wait that drains work
// already in flight before a CTA exits: about 2 s of wall time (globaltimer, ns).
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ----------------------------------------------------------------- smem / mbarrier
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// Expect `bytes` more transaction bytes on the current phase without arriving.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

// Order-preserving 32-bit key of an fp32 score (larger score -> larger key; -0 and +0
// share one key; a real score never has key 0).
__device__ __forceinline__ uint32_t order_key(float v) {
  uint32_t u = __float_as_uint(v);
  if ((u << 1) == 0u) u = 0u;  // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Maximum of v over the full warp (every lane must take part).
__device__ __forceinline__ float redux_max(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

// The smallest fp32 value whose order key is at least `key` (key 0x80000000 gives +0;
// keys at or below the key of -inf give -inf).  v >= key_floor(k) exactly when
// order_key(v) >= k, for every non-NaN v.
__device__ __forceinline__ float key_floor(uint32_t key) {
  if (key & 0x80000000u) return __uint_as_float(key & 0x7FFFFFFFu);
  const float f = __uint_as_float(~key);
  return f != f ? -INFINITY : f;  // below -inf's key lie only negative NaN patterns
}

// Programmatic dependent launch.  pdl_wait() returns once the previous kernel on the
// stream has completed and its memory is visible (immediately when the launch did not
// overlap it); every kernel calls it before touching that kernel's outputs or anything
// that kernel reads.  pdl_trigger() lets the next kernel's CTAs be scheduled early.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Named barrier over `count` threads (warps park in hardware, no polling).
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
// Arrival at named barrier `id` without waiting (producer side of a producer/consumer
// hand-off; the consumers wait with named_bar_sync on the same id and count).
__device__ __forceinline__ void named_bar_arrive(uint32_t id, uint32_t count) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Bounded wait on an mbarrier phase.  A waiting thread is parked by the hardware
// (suspend-time hint) instead of spinning, so waiting warps leave the issue slots to
// the warps that work; the wall-clock bound is checked every 16 polls.  Returns false
// (after at most about limit_ns) when the phase did not complete or *abort became
// non-zero.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int32_t* abort,
                                          uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  // a bound below the default (failure-path tests) shortens the suspend hint and is checked
  // after every poll, so that a wait longer than the bound reliably gives up
  const bool short_bound = limit_ns < kWaitLimitNs;
  const uint32_t hint = limit_ns < 20000ull ? static_cast<uint32_t>(limit_ns) : 20000u;
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_sleep(bar, parity, hint)) return true;
    if (abort != nullptr && *abort) return false;
    if ((short_bound || (it & 15u) == 0) && global_ns() - t0 > limit_ns) return false;
  }
}

// Wait for work this CTA already has in flight (copies, MMAs) before it exits: the fixed
// bound, whatever the pipeline limit, and no abort flag.
__device__ __forceinline__ bool mbar_drain_wait(uint64_t* bar, uint32_t parity) {
  return mbar_wait(bar, parity, nullptr, kWaitLimitNs);
}

// 1-D bulk copy global -> shared, completion counted on `bar` (bytes % 16 == 0,
// both addresses 16-byte aligned).
__device__ __forceinline__ void bulk_g2s(void* sdst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(sdst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void bulk_g2s_hint(void* sdst, const void* gsrc, uint32_t bytes, uint64_t* bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
      "%4;" ::"r"(smem_u32(sdst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// Generic-proxy shared-memory writes become visible to the async proxy (tensor core).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ----------------------------------------------------------------- TMEM / tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_dst, uint32_t ncols) {  // whole warp
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {  // whole warp
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {  // whole warp
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor, no swizzle ("interleaved" core matrices of
// 8 rows x 16 bytes).  lbo: byte stride between core matrices along K (K-major) /
// along K (MN-major); sbo: byte stride between core matrices along M/N.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;  // descriptor version for tcgen05
  return d;                             // base offset 0, swizzle none
}

// Instruction descriptor, kind::f16 with f16 operands (A and B of the same type) and an
// fp32 accumulator; a_mn_major / b_mn_major select the MN-major operand layouts.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, int a_mn_major, int b_mn_major) {
  return (1u << 4) | (static_cast<uint32_t>(a_mn_major) << 15) | (static_cast<uint32_t>(b_mn_major) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// Instruction descriptor, kind::mxf4nvf4: E2M1 x E2M1, UE4M3 scale per 16 elements.
__host__ __device__ constexpr uint32_t idesc_nvf4(int M, int N) {
  return (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) | (0u << 23) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// Instruction descriptor, MX block scaling (scale_vec::2X): E2M1 x E2M1, UE8M0 scale per
// 32 elements (bit 23).  One 32-bit TMEM scale column holds four block scales of a row;
// sf_id (bits 29-30 for A, 4-5 for B) names the byte of the first of the two blocks this
// K = 64 MMA uses: 0 for channels 0-63, 2 for 64-127.
__host__ __device__ constexpr uint32_t idesc_mxf4(int M, int N, uint32_t sf_id) {
  return (sf_id << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) | (1u << 23) |
         (static_cast<uint32_t>(M >> 4) << 24) | (sf_id << 29);
}

// D (+)= A x B, kind::f16 (operand types in the instruction descriptor).
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_nvf4(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], "
      "p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_mxf4(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], "
      "p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once all previously issued tcgen05 operations of this thread finish.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// Copy a 32-row x 16-byte scale-factor atom from shared memory to TMEM, replicated
// into the four 32-lane quarters.
__device__ __forceinline__ void tmem_cp_sf(uint32_t taddr, uint64_t sdesc_src) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc_src) : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns -> 32 registers per thread.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

// acc += w * x on two fp32 lanes with one packed FMA (round to nearest per lane).
__device__ __forceinline__ void fma2(float2& acc, float2 w, float2 x) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;"
      : "=l"(d)
      : "l"(*reinterpret_cast<unsigned long long*>(&w)), "l"(*reinterpret_cast<unsigned long long*>(&x)),
        "l"(*reinterpret_cast<unsigned long long*>(&acc)));
  acc = *reinterpret_cast<float2*>(&d);
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ----------------------------------------------------------------- codec
// E4M3 (bias 7, subnormals, max 448) and E2M1 (magnitudes 0,.5,1,1.5,2,3,4,6) with
// round-to-nearest-even and saturation, through the hardware conversions.
__device__ __forceinline__ uint32_t cvt_e4m3(float x) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(x));
  return r & 0xFFu;  // second source lands in the low byte
}

// Two values -> one byte: `lo` in bits 0-3, `hi` in bits 4-7.
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
  uint16_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u16.u8 %0, t;\n\t}"
      : "=h"(r)
      : "f"(hi), "f"(lo));
  return r & 0xFFu;
}

__device__ __forceinline__ float e4m3_value(uint32_t c) {
  const uint32_t e = (c >> 3) & 15u, m = c & 7u;
  const float v = e ? ldexpf(1.0f + 0.125f * static_cast<float>(m), static_cast<int>(e) - 7)
                    : ldexpf(static_cast<float>(m), -9);
  return (c & 0x80u) ? -v : v;
}

// FP8 window block scale: the smallest e with amax <= 448 * 2^e, clamped to
// [-127, 127] (amax == 0: -127).  amax lies in [2^(E-1), 2^E), so e is E - 9 or E - 8;
// one exact comparison decides.
__device__ __forceinline__ int e8m0_exponent(float amax) {
  if (!(amax > 0.0f)) return -127;
  int E;
  frexpf(amax, &E);
  const int e = amax <= ldexpf(448.0f, E - 9) ? E - 9 : E - 8;
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// MXFP4 block scale: the smallest e with amax <= 6 * 2^e, clamped to [-127, 127]
// (amax == 0: -127).  amax lies in [2^(E-1), 2^E), so e is E - 3 or E - 2; one exact
// comparison decides (6 * 2^(E-3) is a normal fp32 wherever the clamp does not apply).
__device__ __forceinline__ int mx_exponent(float amax) {
  if (!(amax > 0.0f)) return -127;
  int E;
  frexpf(amax, &E);
  const int e = amax <= ldexpf(6.0f, E - 3) ? E - 3 : E - 2;
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// Quantise 32 fp32 values to MXFP4: returns the E8M0 code e + 127; writes 16 bytes of
// nibbles (value 2i in the low nibble of byte i) as four words.
__device__ __forceinline__ uint32_t quant_block32_mx(const float (&x)[32], uint32_t (&nib)[4]) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(x[i]));
  const int e = mx_exponent(amax);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint32_t v = 0;
#pragma unroll
    for (int m = 0; m < 4; ++m)
      v |= cvt_e2m1x2(ldexpf(x[8 * k + 2 * m], -e), ldexpf(x[8 * k + 2 * m + 1], -e)) << (8 * m);  // exact quotients
    nib[k] = v;
  }
  return static_cast<uint32_t>(e + 127);
}

// Two E4M3 codes (low byte first) -> f16x2, exactly (hardware conversion).
__device__ __forceinline__ __half2 e4m3x2_f16x2(uint32_t two) {
  uint32_t r;
  asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(r) : "r"(two));
  return *reinterpret_cast<__half2*>(&r);
}

// Quantise 16 fp32 values: returns the scale code; writes 8 bytes of nibbles
// (value 2i in the low nibble of byte i).
__device__ __forceinline__ uint32_t quant_block16(const float (&x)[16], uint32_t& nib_lo, uint32_t& nib_hi) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
  const uint32_t sc = cvt_e4m3(__fdiv_rn(amax, 6.0f));
  const float s = e4m3_value(sc);
  uint32_t b[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if (s == 0.0f)
      b[i] = 0u;
    else
      b[i] = cvt_e2m1x2(__fdiv_rn(x[2 * i], s), __fdiv_rn(x[2 * i + 1], s));
  }
  nib_lo = b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24);
  nib_hi = b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24);
  return sc;
}

// 8 packed E2M1 codes (one 32-bit word: code 2i in the low nibble, 2i+1 in the high
// nibble of byte i) times an f16x2 scale -> 4 f16x2 words, exactly: a product has at
// most 6 significant bits and lies in [2^-10, 2688], inside f16's normal range.  The f16
// patterns of the magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6 have a zero low byte, so one byte
// lookup (PRMT) per four codes gives the high bytes; the sign comes from each code's bit 3.
__device__ __forceinline__ void dequant8_f16(uint32_t w, uint32_t scale2, uint32_t (&out)[4]) {
  const uint32_t kHiA = 0x3E3C3800u, kHiB = 0x46444240u;  // high bytes of 0,.5,1,1.5 | 2,3,4,6
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const uint32_t c = (w >> (16 * half)) & 0xFFFFu;  // 4 codes e0..e3 in nibbles
    uint32_t hi, sg, w0, w1;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(hi) : "r"(kHiA), "r"(kHiB), "r"(c & 0x7777u));
    // byte k of sg: 0xFF when code k is negative (sign-replicating selectors)
    asm("prmt.b32 %0, %1, %2, 0xD9C8;" : "=r"(sg) : "r"(c << 4), "r"(c));
    hi |= sg & 0x80808080u;
    // f16 k = high byte k over a zero low byte
    asm("prmt.b32 %0, %1, %2, 0x1404;" : "=r"(w0) : "r"(hi), "r"(0u));
    asm("prmt.b32 %0, %1, %2, 0x3424;" : "=r"(w1) : "r"(hi), "r"(0u));
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(out[2 * half]) : "r"(w0), "r"(scale2));
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(out[2 * half + 1]) : "r"(w1), "r"(scale2));
  }
}

// Two E4M3 codes (low byte first) -> f16x2 bits, exactly.
__device__ __forceinline__ uint32_t e4m3x2_f16x2_bits(uint32_t two) {
  uint32_t r;
  asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(r) : "r"(two));
  return r;
}

// Two fp32 values -> f16x2 bits (lo in the low half), round to nearest, saturated to the
// finite f16 range.
__device__ __forceinline__ uint32_t f16x2_sat(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// ----------------------------------------------------------------- cache layout
constexpr int kD = CSA2_D, kDI = CSA2_DI, kPage = CSA2_PAGE;
constexpr int kKvBytes = CSA2_KV_BYTES, kKvPageBytes = CSA2_KV_PAGE_BYTES;
constexpr int kIdxPageBytes = CSA2_IDX_PAGE_BYTES;
constexpr int kIdxNibBytes = 8192;  // nibble region of an indexer page
constexpr int kIdxMxPageBytes = CSA2_IDX_MX_PAGE_BYTES;

__device__ __forceinline__ int64_t page_id(const csa2_cache& c, int32_t r, int64_t s) {
  const int64_t j = s / kPage;
  return c.block_table ? static_cast<int64_t>(c.block_table[static_cast<int64_t>(r) * c.max_pages + j])
                       : static_cast<int64_t>(r) * c.max_pages + j;
}

// Indexer operand layout (also used for the packed indexer query): row n, channel
// block b (16 channels) -> 8-byte slot of its nibbles, and its scale byte.
__device__ __forceinline__ uint32_t idx_nib_off(uint32_t n, uint32_t b) {
  return (n >> 3) * 512u + (b >> 1) * 128u + (n & 7u) * 16u + (b & 1u) * 8u;
}
__device__ __forceinline__ uint32_t idx_sf_off(uint32_t nib_bytes, uint32_t n, uint32_t b) {
  return nib_bytes + (b >> 2) * 512u + (n & 31u) * 16u + (n >> 5) * 4u + (b & 3u);
}

// MXFP4 scale byte of row n, 32-channel block b (one 512-byte atom holds all four).
__device__ __forceinline__ uint32_t idx_mx_sf_off(uint32_t nib_bytes, uint32_t n, uint32_t b) {
  return nib_bytes + (n & 31u) * 16u + (n >> 5) * 4u + b;
}

}  // namespace csa2
