// Benchmark hook: the int8 tensor-core rate of this part, measured in the same
// run as the kernels it is compared with. tcgen05.mma has no integer kind on
// sm_103a, so the int8 tensor path is mma.sync.m16n8k32 (s8 x s8 -> s32); this
// kernel issues nothing else. Each warp runs CHAINS independent accumulator
// chains; each step of a chain is one m16n8k32 MMA, 2*16*8*32 = 8192 integer
// operations.
#include <cstdint>

#include "api_internal.h"
#include "common.cuh"
#include "q4kffn.h"

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

}  // namespace

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
