// pulse_device.cuh -- device-side building blocks shared by the sm_103a
// kernels: the BF16 cast, look-back status words, bounded waits, and inline
// PTX for mbarriers and bulk (TMA) copies.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace pulse {

// Bits of the device error word.
constexpr uint32_t kErrTimeout = 1u;   // a bounded wait gave up
constexpr uint32_t kErrIndex = 2u;     // a checked apply met idx >= n

// ---------------------------------------------------------------- the cast
//
// FP32 -> BF16, round to nearest, ties to even, on the bit pattern (the
// rollout-visible view of "Taking Reinforcement Learning Cross Datacenter",
// talk 07:24-08:20; the absorption threshold of the PULSE summary, section
// "Osservazione Centrale"). Adding 0x7FFF plus the lowest kept bit carries
// into the kept half exactly when the dropped half is above one half, or
// equal to one half with an odd kept half; the carry also moves the exponent
// at a binade edge and reaches infinity past the largest finite value. No
// finite or infinite input wraps (the largest sum is 0xFF807FFF). NaN inputs
// are replaced by the quiet NaN 0x7FC0 explicitly, independent of how the
// hardware convert treats NaN.
__device__ __forceinline__ uint32_t bf16_rne_bits(uint32_t u) {
  const uint32_t rounded = (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;
  return ((u & 0x7FFFFFFFu) > 0x7F800000u) ? 0x7FC0u : rounded;
}

// Two FP32 values -> one packed BF16 pair with the hardware convert, round to
// nearest even: low half from `lo`, high half from `hi`. Finite and infinite
// inputs match bf16_rne_bits exactly; NaN inputs are not canonicalised here
// (see canon_nan_pair).
__device__ __forceinline__ uint32_t cvt_bf16x2_rn(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// True if either input is NaN (one compare for two elements).
__device__ __forceinline__ bool any_nan2(float a, float b) {
  uint32_t r;
  asm("{\n\t.reg .pred p;\n\tsetp.nan.f32 p, %1, %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "f"(a), "f"(b));
  return r != 0u;
}

// True if any of four inputs is NaN (two chained compares).
__device__ __forceinline__ uint32_t any_nan4(float a, float b, float c, float d) {
  uint32_t r;
  asm("{\n\t.reg .pred p;\n\tsetp.nan.f32 p, %1, %2;\n\tsetp.nan.or.f32 p, %3, %4, p;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "f"(a), "f"(b), "f"(c), "f"(d));
  return r;
}

// Replace the half of a packed BF16 pair whose FP32 source is NaN by the
// canonical quiet NaN 0x7FC0 (rare path).
__device__ __forceinline__ uint32_t canon_nan_pair(uint32_t b, float lo, float hi) {
  if (lo != lo) b = (b & 0xFFFF0000u) | 0x7FC0u;
  if (hi != hi) b = (b & 0x0000FFFFu) | 0x7FC00000u;
  return b;
}

// ------------------------------------------------------------ time / errors

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t ld_volatile_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.volatile.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void record_error(uint32_t* error_word, uint32_t bit) {
  atomicOr(error_word, bit);
}

// ------------------------------------------------------- look-back status
//
// One 64-bit word per tile: [63:62] flag (1 = tile aggregate published,
// 2 = inclusive prefix published), [61:32] launch epoch (30 bits), [31:0]
// value. A word whose epoch differs from the running launch's is treated as
// "not yet published", so the status array needs no clearing between
// launches. Each word is self-contained (readers use only its value), so
// relaxed single-copy-atomic 64-bit accesses suffice.
constexpr uint32_t kFlagAggregate = 1u;
constexpr uint32_t kFlagPrefix = 2u;
constexpr uint32_t kEpochMask = 0x3FFFFFFFu;

__device__ __forceinline__ uint64_t make_status(uint32_t flag, uint32_t epoch, uint32_t value) {
  return (static_cast<uint64_t>(flag) << 62) |
         (static_cast<uint64_t>(epoch & kEpochMask) << 32) | value;
}
__device__ __forceinline__ uint32_t status_flag(uint64_t w, uint32_t epoch) {
  return (static_cast<uint32_t>(w >> 32) & kEpochMask) == (epoch & kEpochMask)
             ? static_cast<uint32_t>(w >> 62)
             : 0u;
}
__device__ __forceinline__ uint32_t status_value(uint64_t w) {
  return static_cast<uint32_t>(w);
}
__device__ __forceinline__ void st_relaxed_u64(uint64_t* p, uint64_t v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// ------------------------------------------------------ mbarrier + bulk copy

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Non-blocking test of phase `parity` of `bar`.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// As mbar_try_wait, but lets the hardware suspend the waiting thread for up
// to `hint_ns` nanoseconds (or until the phase completes) instead of
// returning at once, so waiting warps do not take issue slots.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity,
                                                    uint32_t hint_ns) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return done != 0;
}

// Bounded wait for phase `parity` of `bar`. Returns false if it gave up.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0; it < (1u << 30); ++it) {
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
  return false;
}

// L2 policy: read-once streams are marked evict-first.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Bulk copy global -> shared (TMA, untiled). dst/src 16-byte aligned, bytes a
// multiple of 16; completion is signalled on `bar` as transaction bytes.
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gmem_src, uint32_t bytes,
                                         uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// Bulk prefetch of the whole 16-byte units inside [p, p + bytes) into L2 (no
// byte outside the range is touched; the ragged ends are left to the loads).
__device__ __forceinline__ void l2_prefetch_range(const void* p, uint64_t bytes) {
  const uint64_t a = reinterpret_cast<uint64_t>(p);
  const uint64_t lo = (a + 15u) & ~uint64_t(15);
  const uint64_t hi = (a + bytes) & ~uint64_t(15);
  if (hi > lo)
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(lo), "r"(uint32_t(hi - lo))
                 : "memory");
}

// Streaming 128/64/32-bit global loads that do not allocate in L1. The `_ro`
// forms use the read-only path and are only for buffers nothing writes
// during the kernel; the others are for in/out buffers.
__device__ __forceinline__ uint4 ld_stream_u4_ro(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ uint2 ld_stream_u2_ro(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
               : "=r"(v.x), "=r"(v.y)
               : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ld_stream_u1_ro(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ uint2 ld_u2_no_l1(const void* p) {
  uint2 v;
  asm volatile("ld.global.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
               : "=r"(v.x), "=r"(v.y)
               : "l"(p)
               : "memory");
  return v;
}

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

}  // namespace pulse
