// Q4_K x Q8_1 GEMM on tcgen05 with FP8 operands (kind::f8f6f4, E4M3 x E4M3):
//
//   out[t][r] = sum_k deq(W)[r][k] * deq(xq)[t][k]        t < m tokens, r < n rows
//
// the product of spark_model/layers/ops/q4k_mmq.rs, q4k_mmq_gemm (C[m, n] =
// A_q8[m, k] x W_q4k[n, k]^T), with every integer product formed exactly on the
// 8-bit tensor path:
//   A (weights):     the 4-bit quant q itself as an E4M3 code. A byte whose top
//                    four bits are zero encodes q * 2^-9 exactly: q < 8 is a
//                    subnormal (q/8 * 2^-6), q >= 8 has exponent field 1 and
//                    mantissa q - 8 ((1 + (q-8)/8) * 2^-6). So one AND per four
//                    weights turns a quant word into four A bytes, and the low
//                    (high) nibbles of a 32-byte quant group are the 32 k of
//                    sub-block 2g (2g+1) in order.
//   B (activations): q8 = 16 h + l with h = q8 >> 4 in -8..7 and l = q8 & 15 in
//                    0..15; 16 h and l are exact in E4M3 (two planes, written by
//                    expand_fp8_kernel).
// One MMA of K = 32 is one sub-block: D_j = A_j B_hi_j + A_j B_lo_j = 2^-9 *
// sum_i q_i q8_i, exact in float32 (|sum| <= 60960). Neither the 6-bit
// sub-block scale (q * scale reaches 945) nor the Q8_1 scale d8 fits in an E4M3
// operand, so every sub-block's accumulator is read back from tensor memory and
// scaled in float32:
//   acc[t][r] += D_j * d8_tj * (d * scale_j * 2^9)  -  dmin * min_j * s8_tj
// (the closed form d * sum_j scale_j * d8_j * I_j - dmin * sum_j min_j * s8_j).
// That read-back and its two to three float operations per (row, token,
// sub-block) are what this kernel exists to measure against the fp16 path,
// which carries q * scale in its operands and reads its accumulator once per
// superblock.
//
// CTA: one 128-row x 128-token tile over the whole of K. Warp 0 loads the B planes
// and the (d8, s8) pairs by TMA, warp 1 allocates tensor memory and issues the MMAs,
// warps 2-5 write A (one row per thread) into 128-byte-swizzled shared memory,
// warps 6-21 are the epilogue (four per TMEM lane quarter, 32 tokens each). A stage
// holds 128 k (four sub-blocks); four accumulator buffers let the MMAs run up to
// four sub-blocks ahead of the epilogue.
#include <cuda.h>
#include <cuda_fp8.h>

#include <cstdint>

#include "api_internal.h"
#include "common.cuh"
#include "gemv_stream.cuh"
#include "kernels.h"
#include "q4kffn.h"
#include "tc05.cuh"
#include "tmap.h"

namespace q4k {
namespace {

constexpr int F8_TM = 128, F8_TN = 128;
constexpr int F8_KST = 128;                        // k per stage: four sub-blocks, one swizzle atom of bytes
constexpr int F8_STAGES = 4;
constexpr int F8_ATILE = F8_TM * F8_KST;           // 16 KB
constexpr int F8_BTILE = F8_TN * F8_KST;           // 16 KB per B plane
constexpr int F8_DS = F8_TN * 8 * 4;               // (d8, s8) of four sub-blocks for 128 tokens
constexpr int F8_STAGE = F8_ATILE + 2 * F8_BTILE + F8_DS;
constexpr int F8_NDB = 4;                          // accumulator buffers
constexpr int F8_N_EPI = 16;                       // epilogue warps: four per TMEM lane quarter, 32 tokens each
constexpr int F8_W_TMA = 0, F8_W_MMA = 1, F8_W_EPI = 6, F8_WARPS = F8_W_EPI + F8_N_EPI;
constexpr int F8_EPI_TOK = F8_TN / (F8_N_EPI / 4);  // tokens per epilogue thread
constexpr uint32_t F8_TMEM_COLS = F8_NDB * F8_TN;  // 512
constexpr int F8_SMEM = F8_STAGES * F8_STAGE + 1024 /*align*/ + 256 /*barriers*/;
constexpr uint32_t F8_IDESC = idesc_f16(F8_TM, F8_TN);  // E4M3 x E4M3 -> F32 has the same field values

__device__ __forceinline__ void mma_f8_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

// Q8_1 quants -> the E4M3 planes of 16 h and l (q8 = 16 h + l), 16 quants per thread.
__global__ void expand_fp8_kernel(const int8_t* __restrict__ qs, int64_t n16, uint8_t* __restrict__ bh,
                                  uint8_t* __restrict__ bl) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n16) return;
  const uint4 raw = reinterpret_cast<const uint4*>(qs)[i];
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
  uint32_t oh[4], ol[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t vh = 0, vl = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int q8 = (int)(int8_t)((w[j] >> (8 * b)) & 0xFFu);
      const int l = q8 & 15, h = (q8 - l) / 16;  // q8 = 16 h + l, h in -8..7
      vh |= (uint32_t)__nv_cvt_float_to_fp8((float)(16 * h), __NV_SATFINITE, __NV_E4M3) << (8 * b);
      vl |= (uint32_t)__nv_cvt_float_to_fp8((float)l, __NV_SATFINITE, __NV_E4M3) << (8 * b);
    }
    oh[j] = vh;
    ol[j] = vl;
  }
  reinterpret_cast<uint4*>(bh)[i] = make_uint4(oh[0], oh[1], oh[2], oh[3]);
  reinterpret_cast<uint4*>(bl)[i] = make_uint4(ol[0], ol[1], ol[2], ol[3]);
}

struct Fp8Params {
  const uint8_t* w;  // Q4_K rows [n][k / 256]
  int nsb;           // superblocks along k
  int m, n;
  int nmt;           // row tiles (n / 128)
  float* out;        // [m][n]
  uint32_t* err;
};

__global__ void __launch_bounds__(F8_WARPS * 32, 1)
    mmq_fp8_kernel(const __grid_constant__ CUtensorMap tm_bh, const __grid_constant__ CUtensorMap tm_bl,
                   const __grid_constant__ CUtensorMap tm_ds, const Fp8Params P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + F8_STAGES * F8_STAGE);
  uint64_t* empty = full + F8_STAGES;
  uint64_t* accf = empty + F8_STAGES;
  uint64_t* acce = accf + F8_NDB;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acce + F8_NDB);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mt = blockIdx.x % P.nmt, nt = blockIdx.x / P.nmt;
  const int nst = P.nsb * 2;  // stages: two per superblock
  const int64_t rowbytes = (int64_t)P.nsb * BLK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < F8_STAGES; ++s) {
      mbar_init(&full[s], 5);               // the TMA producer + 4 transform warps
      mbar_init(&empty[s], 1 + F8_N_EPI);   // the MMAs' commit + the epilogue warps (done with d8, s8)
    }
    for (int b = 0; b < F8_NDB; ++b) {
      mbar_init(&accf[b], 1);
      mbar_init(&acce[b], F8_N_EPI);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == F8_W_MMA) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(F8_TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncwarp();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == F8_W_TMA) {
    // ------------------------------------------------------------ TMA: B planes and (d8, s8)
    if (lane == 0) {
      for (int q = 0; q < nst; ++q) {
        const int s = q % F8_STAGES, u = q / F8_STAGES;
        if (u > 0 && !wait_bar(&empty[s], (u - 1) & 1, abort_flag, P.err)) break;
        uint8_t* st = smem + s * F8_STAGE;
        mbar_arrive_expect_tx(&full[s], 2 * F8_BTILE + F8_DS);
        tma_load_2d(st + F8_ATILE, &tm_bh, q * F8_KST, nt * F8_TN, &full[s]);
        tma_load_2d(st + F8_ATILE + F8_BTILE, &tm_bl, q * F8_KST, nt * F8_TN, &full[s]);
        tma_load_2d(st + F8_ATILE + 2 * F8_BTILE, &tm_ds, q * 8, nt * F8_TN, &full[s]);
      }
    }
  } else if (warp == F8_W_MMA) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = true;
      for (int q = 0; q < nst && ok; ++q) {
        const int s = q % F8_STAGES, u = q / F8_STAGES;
        if (!wait_bar(&full[s], u & 1, abort_flag, P.err)) break;
        tc_fence_after();
        const uint32_t st = smem_u32(smem + s * F8_STAGE);
        const uint64_t a0 = sw128_desc(st), bh0 = sw128_desc(st + F8_ATILE),
                       bl0 = sw128_desc(st + F8_ATILE + F8_BTILE);
        for (int j = 0; j < 4; ++j) {
          const int jj = q * 4 + j, b = jj % F8_NDB;
          if (jj >= F8_NDB && !wait_bar(&acce[b], ((jj / F8_NDB) - 1) & 1, abort_flag, P.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t off = (uint64_t)((j * 32) >> 4);  // 32 bytes of k along the swizzled row
          const uint32_t d = tmem + b * F8_TN;
          mma_f8_ss(d, a0 + off, bh0 + off, F8_IDESC, 0u);
          mma_f8_ss(d, a0 + off, bl0 + off, F8_IDESC, 1u);
          mma_commit(&accf[b]);
        }
        mma_commit(&empty[s]);
      }
    }
  } else if (warp < F8_W_EPI) {
    // ------------------------------------------------------------ transform: quants -> E4M3 A rows
    const int r = (warp & 3) * 32 + lane;
    const uint8_t* row = P.w + (int64_t)(mt * F8_TM + r) * rowbytes;
    uint8_t* rowoff_base = smem + (r >> 3) * 1024 + (r & 7) * 128;
    for (int q = 0; q < nst; ++q) {
      const int s = q % F8_STAGES, u = q / F8_STAGES;
      // this stage: quant groups 2(q & 1) and 2(q & 1) + 1 of superblock q / 2
      const uint4* src = reinterpret_cast<const uint4*>(row + (int64_t)(q >> 1) * BLK + 16 + 64 * (q & 1));
      uint4 g[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) g[i] = __ldg(src + i);
      if (u > 0 && !wait_bar(&empty[s], (u - 1) & 1, abort_flag, P.err)) break;
      uint8_t* dst = rowoff_base + s * F8_STAGE;
      // 16-byte chunks of the 128-byte row: lo(group a) lo(group a) hi(a) hi(a) lo(b) lo(b) hi(b) hi(b)
#pragma unroll
      for (int grp = 0; grp < 2; ++grp) {
        const uint4 x0 = g[2 * grp], x1 = g[2 * grp + 1];
        const uint4 lo0 = make_uint4(x0.x & 0x0F0F0F0Fu, x0.y & 0x0F0F0F0Fu, x0.z & 0x0F0F0F0Fu, x0.w & 0x0F0F0F0Fu);
        const uint4 lo1 = make_uint4(x1.x & 0x0F0F0F0Fu, x1.y & 0x0F0F0F0Fu, x1.z & 0x0F0F0F0Fu, x1.w & 0x0F0F0F0Fu);
        const uint4 hi0 = make_uint4((x0.x >> 4) & 0x0F0F0F0Fu, (x0.y >> 4) & 0x0F0F0F0Fu, (x0.z >> 4) & 0x0F0F0F0Fu,
                                     (x0.w >> 4) & 0x0F0F0F0Fu);
        const uint4 hi1 = make_uint4((x1.x >> 4) & 0x0F0F0F0Fu, (x1.y >> 4) & 0x0F0F0F0Fu, (x1.z >> 4) & 0x0F0F0F0Fu,
                                     (x1.w >> 4) & 0x0F0F0F0Fu);
        const int c = 4 * grp;
        *reinterpret_cast<uint4*>(dst + (((c + 0) ^ (r & 7)) << 4)) = lo0;
        *reinterpret_cast<uint4*>(dst + (((c + 1) ^ (r & 7)) << 4)) = lo1;
        *reinterpret_cast<uint4*>(dst + (((c + 2) ^ (r & 7)) << 4)) = hi0;
        *reinterpret_cast<uint4*>(dst + (((c + 3) ^ (r & 7)) << 4)) = hi1;
      }
      fence_proxy_async_smem();  // the MMAs read A through the async proxy
      __syncwarp();
      if (lane == 0) mbar_arrive(&full[s]);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3, part = (warp - F8_W_EPI) >> 2;
    const int r = quarter * 32 + lane, c0 = part * F8_EPI_TOK;
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    const uint8_t* row = P.w + (int64_t)(mt * F8_TM + r) * rowbytes;
    float acc[F8_EPI_TOK];
#pragma unroll
    for (int i = 0; i < F8_EPI_TOK; ++i) acc[i] = 0.f;
    float fj[8], nj[8];  // per sub-block of the current superblock: d * scale * 2^9 and -dmin * min
    bool ok = true;
    for (int q = 0; q < nst && ok; ++q) {
      const int s = q % F8_STAGES, u = q / F8_STAGES;
      if ((q & 1) == 0) {
        const uint4 hd = __ldg(reinterpret_cast<const uint4*>(row + (int64_t)(q >> 1) * BLK));
        const float d = fp16_bits_to_f32(hd.x), dmin = fp16_bits_to_f32(hd.x >> 16);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          uint32_t sc, mn;
          scale_min(hd.y, hd.z, hd.w, j, sc, mn);
          fj[j] = d * (float)sc * 512.f;
          nj[j] = -dmin * (float)mn;
        }
      }
      ok = __all_sync(0xffffffffu, wait_bar(&full[s], u & 1, abort_flag, P.err));  // (d8, s8) of this stage
      if (!ok) break;
      const float* ds = reinterpret_cast<const float*>(smem + s * F8_STAGE + F8_ATILE + 2 * F8_BTILE);
      for (int j = 0; j < 4; ++j) {
        const int jj = q * 4 + j, b = jj % F8_NDB;
        ok = __all_sync(0xffffffffu, wait_bar(&accf[b], (jj / F8_NDB) & 1, abort_flag, P.err));
        if (!ok) break;
        tc_fence_after();
        const float f = fj[4 * (q & 1) + j], nm = nj[4 * (q & 1) + j];
#pragma unroll
        for (int cc = 0; cc < F8_EPI_TOK; cc += 16) {
          float v[16];
          tmem_ld16(tmem + lane_addr + b * F8_TN + c0 + cc, v);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float2 e = reinterpret_cast<const float2*>(ds + (c0 + cc + i) * 8)[j];  // (d8, s8), all lanes alike
            acc[cc + i] = fmaf(nm, e.y, fmaf(v[i] * e.x, f, acc[cc + i]));
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acce[b]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    if (!ok) *abort_flag = 1;
    if (!*abort_flag) {
#pragma unroll
      for (int i = 0; i < F8_EPI_TOK; ++i) {
        const int t = nt * F8_TN + c0 + i;
        if (t < P.m) P.out[(int64_t)t * P.n + mt * F8_TM + r] = acc[i];
      }
    }
  }
  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncwarp();
  __syncthreads();
  if (*abort_flag) {  // let copies and MMAs in flight land before the shared memory and TMEM go away
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 1000000ull) {
    }
  }
  if (warp == F8_W_MMA) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(F8_TMEM_COLS) : "memory");
  }
}

bool fp8_shape_ok(int64_t m, int64_t k, int64_t n) {
  return m >= 1 && m <= (int64_t(1) << 20) && k >= 256 && k % 256 == 0 && k <= 65536 && n >= 128 && n % 128 == 0 &&
         n <= (int64_t(1) << 20);
}

}  // namespace
}  // namespace q4k

extern "C" size_t q4k_mmq_fp8_workspace_bytes(int64_t m, int64_t k) {
  if (!q4k::fp8_shape_ok(m, k, 128)) return 0;
  return (size_t)2 * (size_t)m * (size_t)k;  // the two E4M3 planes
}

extern "C" q4k_status q4k_mmq_fp8(const void* xq8, int64_t m, int64_t k, const void* W, int64_t n, float* out,
                                  void* workspace, size_t ws_bytes, q4k_stream_t stream) {
  using namespace q4k;
  if (!xq8 || !W || !out || !workspace) return record_failure(Q4K_ERR_NULL);
  if (!fp8_shape_ok(m, k, n)) return record_failure(Q4K_ERR_SHAPE);
  if (((reinterpret_cast<uintptr_t>(xq8) | reinterpret_cast<uintptr_t>(W) | reinterpret_cast<uintptr_t>(out)) & 15u) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return record_failure(Q4K_ERR_ALIGN);
  if (ws_bytes < q4k_mmq_fp8_workspace_bytes(m, k)) return record_failure(Q4K_ERR_NOMEM);
  int sms = 0;
  uint32_t* err = nullptr;
  q4k_status st = current_device(&sms, &err);
  if (st != Q4K_OK) return record_failure(st);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* bh = static_cast<uint8_t*>(workspace);
  uint8_t* bl = bh + (size_t)m * k;
  const int64_t n16 = m * k / 16;
  expand_fp8_kernel<<<(unsigned)((n16 + 255) / 256), 256, 0, s>>>(static_cast<const int8_t*>(xq8), n16, bh, bl);
  if (cudaGetLastError() != cudaSuccess) return record_failure(Q4K_ERR_CUDA);
  CUtensorMap mh, ml, md;
  const float* ds = reinterpret_cast<const float*>(static_cast<const uint8_t*>(xq8) + (size_t)m * k);
  if (!tmap_2d(&mh, CU_TENSOR_MAP_DATA_TYPE_UINT8, bh, (uint64_t)m, (uint64_t)k, (uint64_t)k, F8_KST, F8_TN,
               CU_TENSOR_MAP_SWIZZLE_128B) ||
      !tmap_2d(&ml, CU_TENSOR_MAP_DATA_TYPE_UINT8, bl, (uint64_t)m, (uint64_t)k, (uint64_t)k, F8_KST, F8_TN,
               CU_TENSOR_MAP_SWIZZLE_128B) ||
      !tmap_2d(&md, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, ds, (uint64_t)m, (uint64_t)(k / 16), (uint64_t)(k / 16) * 4, 8,
               F8_TN, CU_TENSOR_MAP_SWIZZLE_NONE))
    return record_failure(Q4K_ERR_CUDA);
  static uint64_t attr_set = 0;
  if (set_smem_once(reinterpret_cast<const void*>(mmq_fp8_kernel), F8_SMEM, &attr_set) != cudaSuccess)
    return record_failure(Q4K_ERR_CUDA);
  Fp8Params P{static_cast<const uint8_t*>(W), (int)(k / QK), (int)m, (int)n, (int)(n / F8_TM), out, err};
  const unsigned grid = (unsigned)((n / F8_TM) * ((m + F8_TN - 1) / F8_TN));
  mmq_fp8_kernel<<<grid, F8_WARPS * 32, F8_SMEM, s>>>(mh, ml, md, P);
  if (cudaGetLastError() != cudaSuccess) return record_failure(Q4K_ERR_CUDA);
  record_kernels(2);
  return Q4K_OK;
}
