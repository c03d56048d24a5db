// tc.cuh -- tcgen05 glue shared by the tensor-core kernels: shared-memory
// matrix and instruction descriptors, MMA issue with A in tensor memory,
// tensor-memory loads and stores, and the int4 -> bf16 / fp16 decodes that
// feed A.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "ptx.cuh"

namespace moe {

static __device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
static __device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, 8-row
// groups 1024 bytes apart (stride byte offset), start address in 16-byte units.
static __device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFF) >> 4);          // start address
  d |= (uint64_t)1 << 16;                            // leading byte offset (unused: 16 B)
  d |= (uint64_t)(1024 >> 4) << 32;                  // stride byte offset
  d |= (uint64_t)1 << 46;                            // descriptor version
  d |= (uint64_t)2 << 61;                            // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: bf16 A and B (K-major), f32 accumulator.
static __device__ __forceinline__ uint32_t idesc_bf16(int M, int N) {
  return (1u << 4)                          // D format f32
         | (1u << 7)                        // A format bf16
         | (1u << 10)                       // B format bf16
         | ((uint32_t)(N >> 3) << 17)       // N / 8
         | ((uint32_t)(M >> 4) << 24);      // M / 16
}

// Instruction descriptor, kind::f16: fp16 A and B (K-major), f32 accumulator
// (format fields 0 = f16; A and B of one MMA always share a type).
static __device__ __forceinline__ uint32_t idesc_f16(int M, int N) {
  return (1u << 4)                          // D format f32
         | ((uint32_t)(N >> 3) << 17)       // N / 8
         | ((uint32_t)(M >> 4) << 24);      // M / 16
}

static __device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t da, uint64_t db,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(da), "l"(db), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] . B[smem]^T: A in tensor memory, 128 lanes = 128 rows,
// two bf16 per 32-bit column in K order.
// One 64-K block: four K=16 MMAs, A columns a0 + 8 kk, B descriptor db + 2 kk
// (32 bytes further along the swizzled row); the first accumulates only if
// `accumulate`, the other three always.
static __device__ __forceinline__ void mma_kblock_ta(uint32_t tmem_d, uint32_t a0, uint64_t db,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.eq.b32 q, %3, %3;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%5], %6, %3, q;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%7], %8, %3, q;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%9], %10, %3, q;\n\t}" ::"r"(tmem_d),
      "r"(a0), "l"(db), "r"(idesc), "r"(accumulate), "r"(a0 + 8), "l"(db + 2), "r"(a0 + 16),
      "l"(db + 4), "r"(a0 + 24), "l"(db + 6)
      : "memory");
}

// Thread i of the warp writes 16 consecutive 32-bit columns of TMEM lane
// (quadrant base + i), and waits for the store.  The store and its wait are
// one asm statement: tcgen05.st may read its source registers after it issues,
// so they must not be reused before tcgen05.wait::st, and a separate statement
// would let the compiler reallocate them in between.
static __device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t v[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15])
      : "memory");
}

// Two 16-column stores (columns a0.. and a1..) and one wait, in one statement.
static __device__ __forceinline__ void tmem_st16x2(uint32_t a0, const uint32_t v[16], uint32_t a1,
                                                   const uint32_t u[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17};\n\t"
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%1], "
      "{%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(a0), "r"(a1),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15]), "r"(u[0]), "r"(u[1]), "r"(u[2]), "r"(u[3]), "r"(u[4]), "r"(u[5]), "r"(u[6]),
      "r"(u[7]), "r"(u[8]), "r"(u[9]), "r"(u[10]), "r"(u[11]), "r"(u[12]), "r"(u[13]),
      "r"(u[14]), "r"(u[15])
      : "memory");
}

static __device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

static __device__ __forceinline__ void mma_commit(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// 32 lanes x 32 consecutive columns: thread i gets lane (quadrant base + i).
// The load and its wait are one asm statement: tcgen05.ld writes its
// destination registers asynchronously, so nothing may read them before
// tcgen05.wait::ld, and a separate statement would let the compiler schedule
// uses in between.
static __device__ __forceinline__ void tmem_ld32(uint32_t taddr, float v[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 lanes x 16 consecutive columns (load and wait in one statement).
static __device__ __forceinline__ void tmem_ld16(uint32_t taddr, float v[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// ------------------------------------------------------------- dequant --

// bf16x2 arithmetic on raw 32-bit registers.
static __device__ __forceinline__ uint32_t hsub2_bf16(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
static __device__ __forceinline__ uint32_t lop_nib(uint32_t w) {
  uint32_t d;
  // (w & 0x000F000F) | 0x43004300: two offset-binary nibbles into bf16 128 + n.
  asm("lop3.b32 %0, %1, 0x000F000F, 0x43004300, 0xEA;" : "=r"(d) : "r"(w));
  return d;
}

// 8 weights of one library-layout word -> 4 bf16x2 words of the exact codes q.
static __device__ __forceinline__ void dequant_word_q(uint32_t w, uint32_t out[4]) {
  const uint32_t c136 = 0x43084308u;   // bf16x2 (136, 136)
#pragma unroll
  for (int i = 0; i < 4; ++i) out[i] = hsub2_bf16(lop_nib(w >> (4 * i)), c136);
}

// fp16x2 arithmetic on raw 32-bit registers.
static __device__ __forceinline__ uint32_t hsub2_f16(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
static __device__ __forceinline__ uint32_t hmul2_f16(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// (w & mask) | 0x64006400 with mask 0x000F000F: two offset-binary nibbles n in
// bits 0-3 / 16-19 into fp16 1024 + n (the unit in the last place of 1024 is
// 1); with mask 0x00F000F0 the nibbles in bits 4-7 / 20-23 become 1024 + 16 n.
static __device__ __forceinline__ uint32_t lop_nib16_lo(uint32_t w) {
  uint32_t d;
  asm("lop3.b32 %0, %1, 0x000F000F, 0x64006400, 0xEA;" : "=r"(d) : "r"(w));
  return d;
}
static __device__ __forceinline__ uint32_t lop_nib16_hi(uint32_t w) {
  uint32_t d;
  asm("lop3.b32 %0, %1, 0x00F000F0, 0x64006400, 0xEA;" : "=r"(d) : "r"(w));
  return d;
}

// 8 weights of one library-layout word -> 4 fp16x2 words of fp16(q * s), s
// given as fp16 (s2) and as fp16 s / 16 (s16_2, exact).  The pairs in nibble
// positions 0 and 2 decode as q = (1024 + n) - 1032, those in positions 1 and 3
// in place as 16 q = (1024 + 16 n) - 1152 (both exact), so one shift serves
// the word; 16 q * (s / 16) is the same product as q * s.  13 instructions
// per 8 weights.
static __device__ __forceinline__ void dequant_word_f16(uint32_t w, uint32_t s2, uint32_t s16_2,
                                                        uint32_t out[4]) {
  const uint32_t c1032 = 0x64086408u;   // fp16x2 (1032, 1032)
  const uint32_t c1152 = 0x64806480u;   // fp16x2 (1152, 1152)
  const uint32_t w8 = w >> 8;
  out[0] = hmul2_f16(hsub2_f16(lop_nib16_lo(w), c1032), s2);
  out[1] = hmul2_f16(hsub2_f16(lop_nib16_hi(w), c1152), s16_2);
  out[2] = hmul2_f16(hsub2_f16(lop_nib16_lo(w8), c1032), s2);
  out[3] = hmul2_f16(hsub2_f16(lop_nib16_hi(w8), c1152), s16_2);
}

static __device__ __forceinline__ uint32_t f16x2_splat(__half v) {
  const uint16_t b = __half_as_ushort(v);
  return (uint32_t)b | ((uint32_t)b << 16);
}

// 2^e as an f32, e in [-126, 127].
static __device__ __forceinline__ float pow2f(int e) { return __int_as_float((e + 127) << 23); }

// The exponent e of a power of two with |v| < 2^e for a finite v >= 0 (v = 0
// and subnormals give -125).
static __device__ __forceinline__ int pow2_above(float v) {
  const int eb = (__float_as_int(v) >> 23) & 0xFF;
  return (eb > 0 ? eb : 1) - 126;
}



// Thread i of the warp writes 32 consecutive 32-bit columns of TMEM lane
// (quadrant base + i), and waits for the store (one asm statement, as
// tmem_st16).
static __device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t v[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]),
      "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]),
      "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

// 32 lanes x N consecutive columns, N in {1, 2, 4, 8} (load and wait in one
// statement).
template <int N>
static __device__ __forceinline__ void tmem_ld_n(uint32_t taddr, float *v) {
  uint32_t r[N];
  if constexpr (N == 1) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0])
        : "r"(taddr)
        : "memory");
  } else if constexpr (N == 2) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x2.b32 {%0,%1}, [%2];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1])
        : "r"(taddr)
        : "memory");
  } else if constexpr (N == 4) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
        : "r"(taddr)
        : "memory");
  } else {
    static_assert(N == 8, "tmem_ld_n: 1, 2, 4 or 8 columns");
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7])
        : "r"(taddr)
        : "memory");
  }
#pragma unroll
  for (int i = 0; i < N; ++i) v[i] = __uint_as_float(r[i]);
}

}  // namespace moe
