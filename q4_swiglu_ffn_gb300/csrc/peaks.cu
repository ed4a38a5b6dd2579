// Benchmark hooks.
// - The int8 tensor-core rate of this part, measured in the same run as the kernels
//   it is compared with. tcgen05.mma has no integer kind on sm_103a, so the int8
//   tensor path is mma.sync.m16n8k32 (s8 x s8 -> s32); this kernel issues nothing
//   else. Each warp runs CHAINS independent accumulator chains; each step of a chain
//   is one m16n8k32 MMA, 2*16*8*32 = 8192 integer operations.
// - The issue rate of tcgen05.mma kind::f16 from one or more issuing threads per CTA
//   (the measurement behind the prefill MMQ's one N = 256 MMA per K step).
#include <cstdint>

#include "api_internal.h"
#include "common.cuh"
#include "q4kffn.h"
#include "tc05.cuh"

namespace {

constexpr int CHAINS = 8;
constexpr int WARPS = 8;

static __device__ int g_mma_sink;  // keeps the accumulators live; written only if they reach an impossible sum

__global__ void __launch_bounds__(WARPS * 32) mma_s8_rate_kernel(int64_t iters) {
  const uint32_t t = threadIdx.x;
  // small operands (|v| <= 3) so that no sum over any iteration count overflows int32
  const uint32_t a0 = 0x01FF0102u ^ (t & 1), a1 = 0x02010301u, a2 = 0xFF010201u, a3 = 0x0102FF01u ^ (t & 2);
  const uint32_t b0 = 0x0101FF01u ^ (t & 1), b1 = 0x010201FFu;
  int c[CHAINS][4];
#pragma unroll
  for (int k = 0; k < CHAINS; ++k) c[k][0] = c[k][1] = c[k][2] = c[k][3] = 0;
#pragma unroll 1
  for (int64_t i = 0; i < iters; ++i) {
#pragma unroll
    for (int k = 0; k < CHAINS; ++k)
      asm volatile(
          "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
          "{%0,%1,%2,%3};"
          : "+r"(c[k][0]), "+r"(c[k][1]), "+r"(c[k][2]), "+r"(c[k][3])
          : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
  int s = 0;
#pragma unroll
  for (int k = 0; k < CHAINS; ++k) s += c[k][0] + c[k][1] + c[k][2] + c[k][3];
  if (s == 0x7FFFFFF3) g_mma_sink = s;
}

// One CTA per SM; warps 0 .. issuers-1 each issue `iters` rounds of 4 MMAs (M = 128, N = n,
// K = 16; A from tensor memory, B from zeroed shared memory, K-major 128-byte swizzle) into
// their own accumulator columns, committing each round to an mbarrier, then wait (bounded)
// for all of them. Lane 0 of warp 0 records its cycles from the first issue to completion.
constexpr int ISSUE_SMEM = 32768 + 1024 + 64;  // B (up to 256 rows x 64 fp16), alignment, barriers
static __device__ unsigned long long g_issue_cycles[1024];

__global__ void __launch_bounds__(128, 1) mma_issue_kernel(int n, int issuers, int64_t iters, uint32_t* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + 32768);  // [2 * warp]: rounds, [2 * warp + 1]: the end
  uint32_t* slot = reinterpret_cast<uint32_t*>(bar + 8);
  const int warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < 32768 / 16; i += blockDim.x) reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
  if (threadIdx.x == 0) {
    for (int i = 0; i < 8; ++i) q4k::mbar_init(&bar[i], 1);
    q4k::fence_mbar_init();
  }
  q4k::fence_proxy_async_smem();  // the zeroed operand before the tensor core reads it
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(q4k::smem_u32(slot)),
                 "r"(512)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  q4k::tc_fence_before();
  __syncthreads();
  q4k::tc_fence_after();
  const uint32_t tmem = *slot;
  if ((threadIdx.x & 31) == 0 && warp < issuers) {
    uint64_t* wb = bar + 2 * warp;
    const uint32_t idesc = (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);  // f16 -> f32
    const uint64_t bdesc = q4k::sw128_desc(q4k::smem_u32(smem));
    const uint32_t d = tmem + (uint32_t)(warp * n), a = tmem + 256;  // A: columns 256-287
    const long long t0 = clock64();
    for (int64_t it = 0; it < iters; ++it) {
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) q4k::mma_f16_ts(d, a + ks * 8, bdesc + (uint64_t)((ks * 32) >> 4), idesc, 1u);
      q4k::mma_commit(&wb[0]);
    }
    q4k::mma_commit(&wb[1]);  // its first phase completes when every MMA above has
    q4k::mbar_wait(&wb[1], 0u, err);
    if (warp == 0 && blockIdx.x < 1024) g_issue_cycles[blockIdx.x] = (unsigned long long)(clock64() - t0);
  }
  q4k::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    q4k::tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512) : "memory");
  }
}

}  // namespace

extern "C" q4k_status q4k_bench_tcgen05_issue(int n, int issuers, int64_t iters, double* cycles_per_mma,
                                              q4k_stream_t stream) {
  if (!cycles_per_mma) return q4k::record_failure(Q4K_ERR_NULL);
  if ((n != 64 && n != 128 && n != 256) || (issuers != 1 && issuers != 2 && issuers != 4) || n * issuers > 256 ||
      iters < 1 || iters > (int64_t(1) << 20))
    return q4k::record_failure(Q4K_ERR_SHAPE);
  int sms = 0;
  uint32_t* err = nullptr;
  const q4k_status st = q4k::current_device(&sms, &err);
  if (st != Q4K_OK) return q4k::record_failure(st);
  const int grid = sms < 1024 ? sms : 1024;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaFuncSetAttribute(mma_issue_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 120 * 1024) != cudaSuccess)
    return q4k::record_failure(Q4K_ERR_CUDA);
  // 120 KB of shared memory keeps one CTA per SM (the tensor memory is allocated whole)
  mma_issue_kernel<<<grid, 128, 120 * 1024, s>>>(n, issuers, iters, err);
  static unsigned long long cyc[1024];
  if (cudaGetLastError() != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess ||
      cudaMemcpyFromSymbol(cyc, g_issue_cycles, sizeof(unsigned long long) * grid) != cudaSuccess)
    return q4k::record_failure(Q4K_ERR_CUDA);
  double sum = 0;
  for (int i = 0; i < grid; ++i) sum += (double)cyc[i];
  *cycles_per_mma = sum / grid / (4.0 * (double)iters);
  return Q4K_OK;
}

extern "C" q4k_status q4k_bench_int8_mma(int64_t iters, double* ops_per_launch, q4k_stream_t stream) {
  if (!ops_per_launch) return q4k::record_failure(Q4K_ERR_NULL);
  if (iters < 1 || iters > (int64_t(1) << 24)) return q4k::record_failure(Q4K_ERR_SHAPE);
  int sms = 0;
  uint32_t* err = nullptr;
  const q4k_status st = q4k::current_device(&sms, &err);
  if (st != Q4K_OK) return q4k::record_failure(st);
  const int grid = 4 * sms;  // 32 warps per SM
  mma_s8_rate_kernel<<<grid, WARPS * 32, 0, static_cast<cudaStream_t>(stream)>>>(iters);
  if (cudaGetLastError() != cudaSuccess) return q4k::record_failure(Q4K_ERR_CUDA);
  *ops_per_launch = (double)grid * WARPS * (double)iters * CHAINS * (2.0 * 16 * 8 * 32);
  return Q4K_OK;
}
