// tcgen05 / TMEM helpers shared by the tensor-core kernels: allocation,
// MMA issue and commit, TMEM loads and stores, shared-memory matrix
// descriptors (128-byte swizzle) and instruction descriptors.  sm_103a only.
#pragma once

#include "pkv_device.cuh"

namespace pkv {

constexpr int kHalf = 128 * 128;  // one 64-column (128-byte) half of a 128-row tile (16 KB)

// ---------------------------------------------------------------------------
// tcgen05 / TMEM wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem], bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// The same with A (M x 16 bf16, K-major) read from TMEM: row i in lane i of
// the accumulator's lane range, two consecutive k packed per 32-bit column
// (the lower k in the low half), 8 columns per MMA.
__device__ __forceinline__ void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on `bar` once every MMA issued so far by this thread has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

#define PKV_R32(i) "=r"(v[i])
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* v) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : PKV_R32(0), PKV_R32(1), PKV_R32(2), PKV_R32(3), PKV_R32(4), PKV_R32(5), PKV_R32(6), PKV_R32(7), PKV_R32(8),
        PKV_R32(9), PKV_R32(10), PKV_R32(11), PKV_R32(12), PKV_R32(13), PKV_R32(14), PKV_R32(15), PKV_R32(16),
        PKV_R32(17), PKV_R32(18), PKV_R32(19), PKV_R32(20), PKV_R32(21), PKV_R32(22), PKV_R32(23), PKV_R32(24),
        PKV_R32(25), PKV_R32(26), PKV_R32(27), PKV_R32(28), PKV_R32(29), PKV_R32(30), PKV_R32(31)
      : "r"(taddr));
}
#undef PKV_R32
#define PKV_W32(i) "r"(v[i])
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      PKV_W32(0), PKV_W32(1), PKV_W32(2), PKV_W32(3), PKV_W32(4), PKV_W32(5), PKV_W32(6), PKV_W32(7), PKV_W32(8),
      PKV_W32(9), PKV_W32(10), PKV_W32(11), PKV_W32(12), PKV_W32(13), PKV_W32(14), PKV_W32(15), PKV_W32(16),
      PKV_W32(17), PKV_W32(18), PKV_W32(19), PKV_W32(20), PKV_W32(21), PKV_W32(22), PKV_W32(23), PKV_W32(24),
      PKV_W32(25), PKV_W32(26), PKV_W32(27), PKV_W32(28), PKV_W32(29), PKV_W32(30), PKV_W32(31)
      : "memory");
}
#undef PKV_W32
__device__ __forceinline__ void tmem_ld4(uint32_t taddr, uint32_t* v) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t* v) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_st4(uint32_t taddr, const uint32_t* v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(v[0]), "r"(v[1]),
               "r"(v[2]), "r"(v[3])
               : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t* v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
               "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}
#define PKV_R16(i) "=r"(v[i])
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* v) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];"
      : PKV_R16(0), PKV_R16(1), PKV_R16(2), PKV_R16(3), PKV_R16(4), PKV_R16(5), PKV_R16(6), PKV_R16(7), PKV_R16(8),
        PKV_R16(9), PKV_R16(10), PKV_R16(11), PKV_R16(12), PKV_R16(13), PKV_R16(14), PKV_R16(15)
      : "r"(taddr));
}
#undef PKV_R16
#define PKV_W16(i) "r"(v[i])
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};" ::"r"(taddr),
      PKV_W16(0), PKV_W16(1), PKV_W16(2), PKV_W16(3), PKV_W16(4), PKV_W16(5), PKV_W16(6), PKV_W16(7), PKV_W16(8),
      PKV_W16(9), PKV_W16(10), PKV_W16(11), PKV_W16(12), PKV_W16(13), PKV_W16(14), PKV_W16(15)
      : "memory");
}
#undef PKV_W16
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptors (sm_100 format: start>>4 in [0,14), leading
// byte offset>>4 in [16,30), stride byte offset>>4 in [32,46), version 1 at
// [46,48), layout type at [61,64) with 2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}
// A descriptor moved by `bytes` within its swizzle atom or to another tile:
// only the start-address field changes (addresses stay below 256 KB, so the
// 14-bit field never carries).
__device__ __forceinline__ uint64_t desc_add(uint64_t desc, uint32_t bytes) { return desc + (uint64_t)(bytes >> 4); }

// K-major operand, 128-byte rows swizzled, 8-row groups 1024 bytes apart
// (Q, K, P).  The leading byte offset is not used by this layout.
__device__ __forceinline__ uint64_t desc_k(uint32_t saddr) { return smem_desc(saddr, 16, 1024); }
// MN-major operand (V, whose rows are keys): 64-element halves 16 KB apart
// (leading byte offset), 8-key groups 1024 bytes apart (stride byte offset).
__device__ __forceinline__ uint64_t desc_mn(uint32_t saddr) { return smem_desc(saddr, kHalf, 1024); }

// Instruction descriptor, kind::f16: D f32 (bits 4-5 = 1), A and B bf16
// (bits 7-9 and 10-12 = 1), A / B major-ness at bits 15 / 16 (1 = MN-major),
// N>>3 at 17-22, M>>4 at 24-28.
constexpr uint32_t idesc_bf16(int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}


}  // namespace pkv
