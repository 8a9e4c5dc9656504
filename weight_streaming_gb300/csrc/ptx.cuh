// Thin inline-PTX wrappers for sm_103a used by the streaming executor: mbarriers, 1-D bulk (TMA)
// copies, acquire/release accesses for the grid barrier, the warp-level f16 MMA, and the FP4/FP8 ->
// f16 conversions.
#pragma once
#include <cstdint>
#include <cuda_fp16.h>

namespace vp {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
// Makes mbarrier initialisation visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("{ .reg .b64 st; mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1; }" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}
// try_wait with a suspend-time hint: the thread sleeps in hardware until the phase completes (or
// the hint, in ns, expires), so a waiting warp wakes as soon as its data has landed.
__device__ __forceinline__ bool mbar_try_wait_hint(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}
// Poll limits of the bounded waits: the mbarrier waits of the weight rings (suspended polls of <= 20
// us each) and the grid barrier (polls of about 1 us).  The wait-test build makes both tiny, so that
// a test can make a wait run out in milliseconds; normal waits take microseconds.
#ifdef VP_WAIT_TEST
constexpr uint32_t kMbarPolls = 1u << 8;
constexpr uint32_t kBarrierPolls = 1u << 13;
#else
constexpr uint32_t kMbarPolls = 1u << 16;
constexpr uint32_t kBarrierPolls = 1u << 22;
#endif

// Bounded wait for the phase with the given parity: at most kMbarPolls suspended polls of <= 20 us
// each (about 1.3 s), after which it returns false and the caller records a timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  for (uint32_t i = 0; i < kMbarPolls; ++i)
    if (mbar_try_wait_hint(bar, parity, 20000u)) return true;
  return false;
}

// ---------------------------------------------------------------- bulk copy global -> shared
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
// 1-D bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned) completing on `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(pol)
      : "memory");
}
// Orders this thread's earlier generic-proxy shared-memory accesses before later async-proxy ones.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- global acquire / release
__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Atomic add with acquire-release semantics at GPU scope; returns the old value.
__device__ __forceinline__ unsigned atom_add_acq_rel_gpu(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
// Shared-memory atomic add with acquire-release semantics at CTA scope; returns the old value.  It
// orders the warp's earlier global stores for the other warps of the CTA without waiting for the
// SM's outstanding bulk copies (a GPU-scope release waits for them).
__device__ __forceinline__ unsigned atom_add_acq_rel_cta_smem(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(smem_addr(p)), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ void st_release_cta_smem(int* p, int v) {
  asm volatile("st.release.cta.shared::cta.s32 [%0], %1;" ::"r"(smem_addr(p)), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_acquire_cta_smem(const int* p) {
  int v;
  asm volatile("ld.acquire.cta.shared::cta.s32 %0, [%1];" : "=r"(v) : "r"(smem_addr(p)) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// ---------------------------------------------------------------- tensor memory
// Tensor memory: allocation by one whole warp (cols a power of two, 32..512; the address lands in
// shared memory), the fences around a thread synchronisation, and 32-bit columns of the warp's own
// lane (lanes 32 (warp % 4) .. + 31 of the address's lane field).
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t cols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst)), "r"(cols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t cols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols) : "memory");
}
__device__ __forceinline__ void tmem_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tmem_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Four 32-bit columns of the warp's lane: store (then wait for it) / load (waited for).
__device__ __forceinline__ void tmem_st4(uint32_t taddr, const float (&v)[4]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(__float_as_uint(v[0])),
               "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3]))
               : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_ld4(uint32_t taddr, float (&v)[4]) {
  uint32_t a, b, c, d;
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(a), "=r"(b), "=r"(c), "=r"(d)
      : "r"(taddr)
      : "memory");
  v[0] = __uint_as_float(a);
  v[1] = __uint_as_float(b);
  v[2] = __uint_as_float(c);
  v[3] = __uint_as_float(d);
}
// ---------------------------------------------------------------- loads and stores
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ void sts64(uint32_t a, uint32_t x, uint32_t y) {
  asm volatile("st.shared.v2.u32 [%0], {%1,%2};" ::"r"(a), "r"(x), "r"(y) : "memory");
}
__device__ __forceinline__ void sts128(uint32_t a, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}
// 16-byte load through L2 only (data written by other CTAs of this grid or by earlier kernels).
__device__ __forceinline__ uint4 ldcg128(const void* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}
__device__ __forceinline__ float4 ldcg_f4(const float* p) {
  float4 v;
  asm volatile("ld.global.cg.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
  return v;
}

// ---------------------------------------------------------------- conversions
// Four bytes of packed E2M1 pairs -> four f16x2 (byte i -> o[i]; low nibble -> low half).  Exact.
__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t w, uint32_t (&o)[4]) {
  asm("{ .reg .b8 b0, b1, b2, b3;\n"
      " mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n"
      " cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n"
      " cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
      : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
      : "r"(w));
}
// Two E4M3 bytes (low byte -> low half) -> f16x2.  Exact: every E4M3 value is an f16 value.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
  uint32_t r;
  const uint16_t h = static_cast<uint16_t>(two_bytes);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(h));
  return r;
}
// Four E4M3 bytes -> (bytes 0,1) and (bytes 2,3) as f16x2.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{ .reg .b16 h0, h1;\n mov.b32 {h0, h1}, %2;\n cvt.rn.f16x2.e4m3x2 %0, h0;\n cvt.rn.f16x2.e4m3x2 %1, h1;\n}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}
// One Q4 word (eight 4-bit codes) -> four f16x2 of the exact integers 0..15: o[0] = nibbles 0 / 4,
// o[1] = 2 / 6, o[2] = 1 / 5, o[3] = 3 / 7 (first named -> low half).  Each pair is masked into the
// mantissa of 1024 = 0x6400 (the odd nibbles land 4 bits higher, as 1024 + 16 q), then the offset is
// removed: q = v - 1024, or q = v / 16 - 64, both exact in f16.
__device__ __forceinline__ void q4x8_to_f16x2x4(uint32_t w, uint32_t (&o)[4]) {
  const uint32_t w8 = w >> 8, lo = 0x000F000Fu, hi = 0x00F000F0u, k1024 = 0x64006400u;
  const uint32_t k16th = 0x2C002C00u, km64 = 0xD400D400u;
  uint32_t e0, e1, e2, e3;  // (a & b) | c
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(e0) : "r"(w), "r"(lo), "r"(k1024));
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(e1) : "r"(w), "r"(hi), "r"(k1024));
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(e2) : "r"(w8), "r"(lo), "r"(k1024));
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(e3) : "r"(w8), "r"(hi), "r"(k1024));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(o[0]) : "r"(e0), "r"(k1024));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(o[1]) : "r"(e2), "r"(k1024));
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(o[2]) : "r"(e1), "r"(k16th), "r"(km64));
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(o[3]) : "r"(e3), "r"(k16th), "r"(km64));
}
__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t dup_lo16(uint32_t x) { return __byte_perm(x, 0, 0x1010); }
__device__ __forceinline__ uint32_t dup_hi16(uint32_t x) { return __byte_perm(x, 0, 0x3232); }

// ---------------------------------------------------------------- tensor core (warp MMA)
// D(16x8, f32) += A(16x16, f16, row) * B(16x8, f16, col).
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------- exact powers of two
// 2^e as a float for e in [-149, 127] (subnormal below -126).
__device__ __forceinline__ float pow2f(int e) {
  return e >= -126 ? __int_as_float((e + 127) << 23) : __int_as_float(1 << (e + 149));
}
// x * 2^e for e in [-252, 254], in two exact steps (no intermediate over/underflow for the ranges
// the kernels use).
__device__ __forceinline__ float mul_pow2(float x, int e) {
  if (e > 127) return x * pow2f(127) * pow2f(e - 127);
  if (e < -126) return x * pow2f(-126) * pow2f(e + 126);
  return x * pow2f(e);
}

}  // namespace vp
