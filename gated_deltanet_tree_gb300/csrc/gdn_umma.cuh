// Tensor memory and the fifth-generation tensor cores (tcgen05) as the verify
// kernels use them, in inline PTX for sm_103a.
//
// Tensor memory (TMEM) is 128 lanes x 512 columns of 32-bit cells per SM.  A
// warp reaches the 32 lanes of its quarter (warp % 4); with the 32x32b access
// shape thread t of the warp reads or writes lane 32 (warp % 4) + t, one column
// per register.
//
// The MMA helpers issue kind::tf32 products with fp32 accumulation in tensor
// memory, D[M][N] (+)= A[M][K] B[N][K]^T, M = 128:
//   - A either from tensor memory (lane m = row m, column k = element k) or,
//     like B, from shared memory;
//   - shared-memory operands in the K-major layout without swizzle: 8 rows x
//     16 bytes (4 tf32) form a contiguous 128-byte core matrix; core matrices
//     adjacent along K are `lbo` bytes apart, those adjacent along M/N `sbo`
//     bytes apart;
//   - one instruction covers K = 8 (two core matrices along K).
// A tf32 operand keeps 10 of fp32's 23 mantissa bits.  Products that need fp32
// accuracy split each operand as x = hi + lo (tf32_hi / tf32_lo below) and
// accumulate hi*hi + hi*lo + lo*hi (the lo*lo term is below fp32 rounding).
#pragma once
#include <cstdint>

#include "gdn_tile.cuh"

namespace gdn {

#ifdef __CUDACC__
// ---- tensor memory (tcgen05) as a stash for register tiles: the 32x32b access shape gives each
// thread of a warp its own lane, so a tile held in registers moves in and out without crossing lanes.
__host__ __device__ constexpr uint32_t tmem_columns(int words) {   // allocation: a power of two >= 32, or none
  return words <= 0 ? 0u : words <= 32 ? 32u : words <= 64 ? 64u : words <= 128 ? 128u : words <= 256 ? 256u : 512u;
}
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t cols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst)), "r"(cols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t cols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols) : "memory");
}
__device__ __forceinline__ void tmem_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tmem_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Loads 32 words of this thread's lane into 16 packed pairs; the wait is inside, so the
// outputs are defined when the statement ends.
__device__ __forceinline__ void tmem_get32(uint32_t ta, u64 (&v)[16]) {
  asm volatile(
      "{\n"
      " .reg .b32 t<32>;\n"
      " tcgen05.ld.sync.aligned.32x32b.x16.b32 {t0, t1, t2, t3, t4, t5, t6, t7, t8, t9, t10, t11, t12, t13, t14, t15}, [%16];\n"
      " tcgen05.ld.sync.aligned.32x32b.x16.b32 {t16, t17, t18, t19, t20, t21, t22, t23, t24, t25, t26, t27, t28, t29, t30, t31}, [%17];\n"
      " tcgen05.wait::ld.sync.aligned;\n"
      " mov.b64 %0, {t0, t1};\n"
      " mov.b64 %1, {t2, t3};\n"
      " mov.b64 %2, {t4, t5};\n"
      " mov.b64 %3, {t6, t7};\n"
      " mov.b64 %4, {t8, t9};\n"
      " mov.b64 %5, {t10, t11};\n"
      " mov.b64 %6, {t12, t13};\n"
      " mov.b64 %7, {t14, t15};\n"
      " mov.b64 %8, {t16, t17};\n"
      " mov.b64 %9, {t18, t19};\n"
      " mov.b64 %10, {t20, t21};\n"
      " mov.b64 %11, {t22, t23};\n"
      " mov.b64 %12, {t24, t25};\n"
      " mov.b64 %13, {t26, t27};\n"
      " mov.b64 %14, {t28, t29};\n"
      " mov.b64 %15, {t30, t31};\n"
      "}"
      : "=l"(v[0]), "=l"(v[1]), "=l"(v[2]), "=l"(v[3]), "=l"(v[4]), "=l"(v[5]), "=l"(v[6]), "=l"(v[7]), "=l"(v[8]), "=l"(v[9]), "=l"(v[10]), "=l"(v[11]), "=l"(v[12]), "=l"(v[13]), "=l"(v[14]), "=l"(v[15])
      : "r"(ta + 0u), "r"(ta + 16u)
      : "memory");
}
// Stores 16 packed pairs as 32 words of this thread's lane and waits for the stores.
__device__ __forceinline__ void tmem_put32(uint32_t ta, const u64 (&v)[16]) {
  asm volatile(
      "{\n"
      " .reg .b32 t<32>;\n"
      " mov.b64 {t0, t1}, %0;\n"
      " mov.b64 {t2, t3}, %1;\n"
      " mov.b64 {t4, t5}, %2;\n"
      " mov.b64 {t6, t7}, %3;\n"
      " mov.b64 {t8, t9}, %4;\n"
      " mov.b64 {t10, t11}, %5;\n"
      " mov.b64 {t12, t13}, %6;\n"
      " mov.b64 {t14, t15}, %7;\n"
      " mov.b64 {t16, t17}, %8;\n"
      " mov.b64 {t18, t19}, %9;\n"
      " mov.b64 {t20, t21}, %10;\n"
      " mov.b64 {t22, t23}, %11;\n"
      " mov.b64 {t24, t25}, %12;\n"
      " mov.b64 {t26, t27}, %13;\n"
      " mov.b64 {t28, t29}, %14;\n"
      " mov.b64 {t30, t31}, %15;\n"
      " tcgen05.st.sync.aligned.32x32b.x16.b32 [%16], {t0, t1, t2, t3, t4, t5, t6, t7, t8, t9, t10, t11, t12, t13, t14, t15};\n"
      " tcgen05.st.sync.aligned.32x32b.x16.b32 [%17], {t16, t17, t18, t19, t20, t21, t22, t23, t24, t25, t26, t27, t28, t29, t30, t31};\n"
      " tcgen05.wait::st.sync.aligned;\n"
      "}"
      :
      : "l"(v[0]), "l"(v[1]), "l"(v[2]), "l"(v[3]), "l"(v[4]), "l"(v[5]), "l"(v[6]), "l"(v[7]), "l"(v[8]), "l"(v[9]), "l"(v[10]), "l"(v[11]), "l"(v[12]), "l"(v[13]), "l"(v[14]), "l"(v[15]), "r"(ta + 0u), "r"(ta + 16u)
      : "memory");
}


// ---- MMA operands and issue
// Shared-memory matrix descriptor: start address, leading (K-direction) and stride (M/N-direction)
// byte offsets, the fixed version bits of this architecture, no swizzle.
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(lbo >> 4) << 16) |
         (static_cast<uint64_t>(sbo >> 4) << 32) | (1ull << 46);
}
// Instruction descriptor of kind::tf32: fp32 accumulator, tf32 A and B, both K-major, M x N.
__host__ __device__ constexpr uint32_t umma_idesc_tf32(int m, int n) {
  return (1u << 4) | (2u << 7) | (2u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}
// The two-term tf32 split x = hi + lo: hi keeps the sign, the exponent and the top 10 fraction bits of x
// (the low 13 fraction bits cleared, so it is a tf32 value exactly), lo = x - hi is exact in fp32 and holds
// at most the remaining 13 bits; read as tf32 by the tensor cores it loses at most its lowest bits, an error
// below 2^-21 |x|.  Two integer/fp ops instead of two conversions and a subtraction.
__device__ __forceinline__ float tf32_hi(float x) { return __uint_as_float(__float_as_uint(x) & 0xFFFFE000u); }
__device__ __forceinline__ float tf32_lo(float x) { return x - tf32_hi(x); }
// D (+)= A B^T with A in tensor memory.
__device__ __forceinline__ void umma_tf32_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, int accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n}" ::"r"(d),
      "r"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D (+)= A B^T with A in shared memory.
__device__ __forceinline__ void umma_tf32_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, int accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on `bar` once every MMA this thread issued so far has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}
// Hint: bring `bytes` (a multiple of 16, 16-byte aligned) of global memory into L2.
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
// Generic-proxy shared-memory writes made visible to the tensor cores (async proxy).
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// ---- 32x32b accesses of 16 and 4 columns; stores complete at tmem_wait_st(), loads at tmem_wait_ld()
__device__ __forceinline__ void tmem_st16(uint32_t ta, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16};" ::"r"(ta),
      "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]), "f"(v[8]), "f"(v[9]),
      "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]), "f"(v[15])
      : "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t ta, float (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, "
      "[%16];"
      : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]), "=f"(v[7]), "=f"(v[8]),
        "=f"(v[9]), "=f"(v[10]), "=f"(v[11]), "=f"(v[12]), "=f"(v[13]), "=f"(v[14]), "=f"(v[15])
      : "r"(ta)
      : "memory");
}
__device__ __forceinline__ void tmem_ld4(uint32_t ta, float (&v)[4]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3])
               : "r"(ta)
               : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
#endif

}  // namespace gdn
