// tcgen05 building blocks of the tensor-memory GEMM (prefill MMQ): UMMA
// shared-memory descriptors and instruction descriptors, MMA with A in tensor
// memory, TMEM loads and stores, 2-D TMA loads, the bounded barrier wait, and the
// unpacking of Q4_K quants into fp16 q * scale.
#pragma once
#include <cuda.h>

#include "common.cuh"

namespace q4k {
namespace {

// Position of element i (0..7) of an aligned group of 8 k in the order the nibble
// unpacking produces (0,2,1,3,4,6,5,7); both MMA operands use it.
__device__ __forceinline__ int perm8(int i) { return (i == 1 || i == 5) ? i + 1 : (i == 2 || i == 6) ? i - 1 : i; }

__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  // K-major, 128-byte swizzle, 8-row atoms 1024 bytes apart (SBO), version 1 (sm_100 family)
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// kind::f16: fp16 A and B, fp32 D, both K-major, M x N
constexpr uint32_t idesc_f16(int m, int n) {
  return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// D (+)= A . B with A read from tensor memory (128 lanes = rows, K along the
// columns) and B from a shared-memory descriptor
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                           uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float v[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float v[8]) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// Each lane stores 8 consecutive 32-bit columns of its own TMEM lane (16 with tmem_st16 below).
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&v)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(v[0]),
               "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* tm, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Bounded wait that also gives up when another role has already aborted.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag, uint32_t* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
      set_error(err, ERRBIT_TIMEOUT);
      *abort_flag = 1;
      return false;
    }
  }
}

// One 64-k chunk of a Q4_K row is 32 fp16x2 TMEM columns (k = 2j, 2j + 1 in column j): 32
// low-nibble k of sub-block 2c in columns 0-15, then 32 high-nibble k of sub-block 2c + 1 in
// columns 16-31. unpack_half<false> gives the first 16 columns, unpack_half<true> the other
// 16, so that a chunk is stored in two halves with half the registers live. ga, gb: the
// chunk's 32 quant bytes; sc: the sub-block's 6-bit scale. Each quant becomes q * scale
// exactly: the 0x6400-exponent trick gives 1024 + q (or 1024 + 16 q) and one fp16 fma scales
// it and removes the offset; the multipliers come straight from the integer (exact in fp16).
template <bool HI>
__device__ __forceinline__ void unpack_half(uint4 ga, uint4 gb, uint32_t sc, uint32_t (&a)[16]) {
  const __half hs = __uint2half_rn(sc);
  const __half2 m = __half2half2(HI ? __hmul(hs, __float2half(0.0625f)) : hs);
  const __half2 o = __half2half2(__hmul(hs, __float2half(HI ? -64.f : -1024.f)));
  const uint32_t mask = HI ? 0x00F000F0u : 0x000F000Fu;
  const uint32_t wds[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const uint32_t w0 = wds[2 * p], w1 = wds[2 * p + 1];
    a[4 * p + 0] = h2_as_u32(__hfma2(u32_as_h2(lop3_and_or(w0, mask, 0x64006400u)), m, o));
    a[4 * p + 1] = h2_as_u32(__hfma2(u32_as_h2(lop3_and_or(w0 >> 8, mask, 0x64006400u)), m, o));
    a[4 * p + 2] = h2_as_u32(__hfma2(u32_as_h2(lop3_and_or(w1, mask, 0x64006400u)), m, o));
    a[4 * p + 3] = h2_as_u32(__hfma2(u32_as_h2(lop3_and_or(w1 >> 8, mask, 0x64006400u)), m, o));
  }
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

// The 8 mins of a superblock as A of the K = 16 min MMA: twice (k 0-7 against the
// hi sums, k 8-15 against the lo sums).
__device__ __forceinline__ void min_operand(const uint32_t (&mns)[8], uint32_t (&v)[8]) {
  v[0] = v[4] = h2_as_u32(__halves2half2(__uint2half_rn(mns[0]), __uint2half_rn(mns[1])));
  v[1] = v[5] = h2_as_u32(__halves2half2(__uint2half_rn(mns[2]), __uint2half_rn(mns[3])));
  v[2] = v[6] = h2_as_u32(__halves2half2(__uint2half_rn(mns[4]), __uint2half_rn(mns[5])));
  v[3] = v[7] = h2_as_u32(__halves2half2(__uint2half_rn(mns[6]), __uint2half_rn(mns[7])));
}

}  // namespace
}  // namespace q4k
