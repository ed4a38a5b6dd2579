// Q6_K GEMV (the LM head): y[t][n] = sum_k W[n][k] x[t][k] for 1..8 tokens, on sm_103a.
// Source: realizar src/cuda/executor/q4k_gemv_cached_uses.rs, q6k_gemv_cached_async
// (the Q4_K GEMV's contract -- float32 input, float32 output, k a multiple of
// 256, enqueued without synchronisation -- for Q6_K weights, used for the LM head).
//
// Block (GGML block_q6_K, 210 bytes): ql[128] low 4 bits, qh[64] high 2 bits,
// 16 signed 8-bit sub-block scales, fp16 d. Weight i belongs to sub-block
// i / 16 and is d * scale[i / 16] * (q_i - 32); in half h, weight
// 128h + 32s + l takes its low bits from nibble (s >= 2) of ql[64h + l + 32(s % 2)]
// and its high bits from bits 2s..2s+1 of qh[32h + l].
//
//   K0 prep_q6k_x: x -> mma.sync B fragments per token and superblock (fp16 hi + lo
//                  of x * 2^-e, e per token and superblock, as in the Q4_K decode)
//   K1 q6k_gemv:   the GEMV, with programmatic dependent launch after K0
//
// Arithmetic. A 16-row tile is multiplied on the tensor cores with
// mma.sync.m16n8k16: one k16 step is exactly one 16-weight sub-block. The A
// operand is q - 32, exact in fp16 (one byte permute puts q under the fp16
// exponent of 1024, one fp16 add removes 1056). (q - 32) * scale needs up to 13
// significant bits, more than fp16 holds, so the signed scale is applied to the
// fp32 result of each sub-block's MMA instead; per superblock the sum is scaled
// by d * 2^e.
//
// Streaming. Rows of a Q6_K matrix are 210 * nsb bytes, so a 3-D TMA box (whose
// inner extent must be a multiple of 16 bytes) cannot address one block; but 16
// whole rows are 3360 * nsb contiguous bytes starting at a multiple of 16, so a
// CTA streams 16-row tiles over the full K with one 1-D bulk copy per stage. The
// 8 warps of a CTA split a tile's superblocks (warp w takes superblocks w, w+8,
// ...) and keep those superblocks' B fragments in registers; at the end of a tile
// an owner warp sums the 8 warps' partial dot products and stores y. Blocks
// start at 2-byte boundaries, so 32-bit fields are read from shared memory as
// two aligned words joined by a funnel shift when the block is not 4-byte aligned.
#include <algorithm>

#include "common.cuh"
#include "gemv_stream.cuh"
#include "kernels.h"

namespace q4k {

namespace {

constexpr int Q6_BLK = 210;

struct Q6Frags {
  uint2* fx;  // [nsb][16 sub-blocks][nt][32 lanes] B fragments (hi and lo parts in adjacent columns)
  float* sc;  // [nsb][8] 2^e per token slot
};

// K0: one CTA per superblock of x, one warp per token slot. Lane L holds
// inputs 8L..8L+7: sub-block L/2, positions 8(L%2)..8(L%2)+7, i.e. the
// fragment positions of quad threads tig = 2(L%2) and 2(L%2)+1.
template <typename T>
__global__ void prep_q6k_x_kernel(const T* __restrict__ x, int k, int m, int nt, Q6Frags f) {
  pdl_launch_dependents();
  const int t = threadIdx.x >> 5, sb = blockIdx.x, lane = threadIdx.x & 31;
  const int ntile = t >> 2, gcol = 2 * (t & 3);  // columns gcol (hi) and gcol + 1 (lo)
  const int j = lane >> 1;
  uint2* fx = f.fx + (((int64_t)sb * 16 + j) * nt + ntile) * 32;
  float v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = 0.f;
  if (t < m) {
    const T* p = x + (int64_t)t * k + (int64_t)sb * QK + lane * 8;
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = static_cast<float>(p[i]);
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
  amax = warp_max(amax);
  int e = 0;
  if (amax > 0.f) e = max((int)((__float_as_uint(amax) >> 23) & 0xFF) - 127 - 14, -100);
  const float s = __uint_as_float((uint32_t)(127 - e) << 23);  // 2^-e
  __half hi[8], lo[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float y = v[i] * s;
    hi[i] = __float2half_rn(y);
    lo[i] = __float2half_rn(y - __half2float(hi[i]));
  }
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int tig = 2 * (lane & 1) + q;
#pragma unroll
    for (int part = 0; part < 2; ++part) {
      const __half* h = part ? lo : hi;
      uint2 fr;  // b0: positions 4tig, 4tig+1; b1: positions 4tig+2, 4tig+3
      fr.x = h2_as_u32(__halves2half2(h[4 * q + 0], h[4 * q + 1]));
      fr.y = h2_as_u32(__halves2half2(h[4 * q + 2], h[4 * q + 3]));
      fx[(gcol + part) * 4 + tig] = fr;
    }
  }
  if (lane == 0) f.sc[(int64_t)sb * 8 + t] = __uint_as_float((uint32_t)(127 + e) << 23);
}

__device__ __forceinline__ void mma16816(float c[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 32-bit little-endian field at a 2-byte aligned shared-memory address.
__device__ __forceinline__ uint32_t ld_u32_2(const uint8_t* p) {
  const uint32_t a = smem_u32(p);
  const uint32_t* w = reinterpret_cast<const uint32_t*>(p - (a & 3u));
  return (a & 2u) ? __funnelshift_r(w[0], w[1], 16) : w[0];
}

// The signed byte b (0..3) of w as a float: 1.5 * 2^23 + v holds v in its mantissa.
__device__ __forceinline__ float sbyte_f(uint32_t w, int b) {
  const uint32_t sel = (uint32_t)b | (uint32_t)(b | 8) << 4 | (uint32_t)(b | 8) << 8 | (uint32_t)(b | 8) << 12;
  return __int_as_float((int)prmt(w, 0u, sel) + 0x4B400000) - 12582912.f;
}

// A 32-bit field of a block in shared memory. AL = 0: the field is 4-byte
// aligned; AL = 1: it sits 2 bytes past a 4-byte boundary; AL = 2: either.
template <int AL>
__device__ __forceinline__ uint32_t ld_field(const uint8_t* p) {
  if constexpr (AL == 0) {
    return *reinterpret_cast<const uint32_t*>(p);
  } else if constexpr (AL == 1) {
    const uint32_t* w = reinterpret_cast<const uint32_t*>(p - 2);
    return __funnelshift_r(w[0], w[1], 16);
  } else {
    return ld_u32_2(p);
  }
}

// One superblock of a 16-row tile: rows g and g+8 start at r0 and r1. Adds to
// acc[n][r] this superblock's dot products of rows g + 8r with the tokens of
// token tile n (B: the superblock's B fragments, xsc: 2^e of this lane's token).
template <int AL, int NT>
__device__ __forceinline__ void q6k_superblock(const uint8_t* r0, const uint8_t* r1, int tig,
                                               const uint2 (&B)[16][NT], const float (&xsc)[NT], float (&acc)[NT][2]) {
  const uint8_t* blk[2] = {r0, r1};
  float dd[2];
  uint32_t scw[2][4];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    dd[r] = __half2float(__ushort_as_half(*reinterpret_cast<const unsigned short*>(blk[r] + 208)));
#pragma unroll
    for (int q = 0; q < 4; ++q) scw[r][q] = ld_field<AL>(blk[r] + 192 + 4 * q);
  }
  float sacc[NT][4];
#pragma unroll
  for (int n = 0; n < NT; ++n)
#pragma unroll
    for (int c = 0; c < 4; ++c) sacc[n][c] = 0.f;
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int bb = 0; bb < 2; ++bb) {
      uint32_t qhw[2], qlw[2][2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        qhw[r] = ld_field<AL>(blk[r] + 128 + 32 * h + 16 * bb + 4 * tig);
#pragma unroll
        for (int s1 = 0; s1 < 2; ++s1) qlw[r][s1] = ld_field<AL>(blk[r] + 64 * h + 32 * s1 + 16 * bb + 4 * tig);
      }
#pragma unroll
      for (int sp = 0; sp < 4; ++sp) {
        const int j = 8 * h + 2 * sp + bb;  // sub-block: weights 16j .. 16j+15
        uint32_t A[2][2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const uint32_t qw = qlw[r][sp & 1];
          const uint32_t nib = sp < 2 ? (qw & 0x0F0F0F0Fu) : ((qw >> 4) & 0x0F0F0F0Fu);
          const uint32_t top = sp < 2 ? ((qhw[r] << (4 - 2 * sp)) & 0x30303030u)
                                      : ((qhw[r] >> (2 * sp - 4)) & 0x30303030u);
          const uint32_t q4 = nib | top;  // bytes: the 6-bit q of positions 4tig .. 4tig+3
          // fp16 1024 + q, then - 1056: q - 32 exactly
          A[r][0] = h2_as_u32(__hadd2(u32_as_h2(prmt(q4, 0x64646464u, 0x5140u)), u32_as_h2(0xE420E420u)));
          A[r][1] = h2_as_u32(__hadd2(u32_as_h2(prmt(q4, 0x64646464u, 0x7362u)), u32_as_h2(0xE420E420u)));
        }
        const float s0 = sbyte_f(scw[0][j >> 2], j & 3), s1 = sbyte_f(scw[1][j >> 2], j & 3);
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          float d4[4] = {0.f, 0.f, 0.f, 0.f};
          mma16816(d4, A[0][0], A[1][0], A[0][1], A[1][1], B[j][n].x, B[j][n].y);
          sacc[n][0] = fmaf(d4[0], s0, sacc[n][0]);
          sacc[n][1] = fmaf(d4[1], s0, sacc[n][1]);
          sacc[n][2] = fmaf(d4[2], s1, sacc[n][2]);
          sacc[n][3] = fmaf(d4[3], s1, sacc[n][3]);
        }
      }
    }
#pragma unroll
  for (int n = 0; n < NT; ++n) {
    acc[n][0] = fmaf(sacc[n][0] + sacc[n][1], dd[0] * xsc[n], acc[n][0]);
    acc[n][1] = fmaf(sacc[n][2] + sacc[n][3], dd[1] * xsc[n], acc[n][1]);
  }
}

struct Q6Params {
  const uint8_t* w;  // [n][nsb][210]
  int n, nsb, m, nt;
  Q6Frags in;
  float* y;          // [m][n]
  uint32_t* err;
};

constexpr int Q6_WARPS = 8;
constexpr int Q6_STAGES = 2;

// Superblocks a warp holds B fragments for in registers: SBW (nsb <= 8 * SBW);
// SBW = 0 reads them from global memory per tile instead.
template <int NT, int SBW, int CPS>
__global__ void __launch_bounds__(Q6_WARPS * 32, CPS) q6k_gemv_kernel(const Q6Params P) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int RB = P.nsb * Q6_BLK;           // bytes per row
  const int TILE = 16 * RB;                // bytes per 16-row tile (a multiple of 16)
  const int SSTR = (TILE + 16 + 127) & ~127;  // stage stride (16 bytes of slack for the funnel reads)
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Q6_STAGES * SSTR);
  uint64_t* empty = full + Q6_STAGES;
  float* red = reinterpret_cast<float*>(empty + Q6_STAGES);  // [Q6_WARPS][32][NT][2]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(red + Q6_WARPS * 32 * NT * 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, tig = lane & 3;
  const int ntiles = P.n / 16;
  const int t0 = (int)((int64_t)ntiles * blockIdx.x / gridDim.x), t1 = (int)((int64_t)ntiles * (blockIdx.x + 1) / gridDim.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < Q6_STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], Q6_WARPS);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  const bool producer = (warp == 0 && lane == 0);
  const uint64_t pol = policy_evict_first();
  int ptile = t0;
  auto produce = [&]() -> bool {
    const int i = ptile - t0, s = i % Q6_STAGES;
    if (i >= Q6_STAGES && !mbar_wait(&empty[s], (uint32_t)((i / Q6_STAGES) - 1) & 1u, P.err)) return false;
    mbar_arrive_expect_tx(&full[s], (uint32_t)TILE);
    bulk_g2s_hint(smem + (size_t)s * SSTR, P.w + (int64_t)ptile * TILE, (uint32_t)TILE, &full[s], pol);
    ++ptile;
    return true;
  };
  bool failed = false;
  if (producer) {
    for (int i = 0; i < Q6_STAGES - 1 && ptile < t1; ++i)
      if (!produce()) {
        failed = true;
        *abort_flag = 1;
        break;
      }
  }
  failed = __any_sync(0xffffffffu, failed);
  pdl_launch_dependents();
  pdl_wait();  // B fragments come from K0

  // B fragment lane per token tile: this lane when its token is real, else the
  // same position of token 4n (always real); padding columns are never stored.
  int flane[NT];
#pragma unroll
  for (int n = 0; n < NT; ++n) flane[n] = ((lane >> 3) < P.m - 4 * n) ? lane : (lane & 7);
  constexpr int SBC = SBW > 0 ? SBW : 1;
  uint2 bq[SBC][16][NT];
  float xs[SBC][NT];
  if (SBW > 0) {
#pragma unroll
    for (int i = 0; i < SBC; ++i) {
      const int sb = warp + Q6_WARPS * i;
      if (sb < P.nsb) {
#pragma unroll
        for (int j = 0; j < 16; ++j)
#pragma unroll
          for (int n = 0; n < NT; ++n) bq[i][j][n] = P.in.fx[(((int64_t)sb * 16 + j) * NT + n) * 32 + flane[n]];
#pragma unroll
        for (int n = 0; n < NT; ++n) xs[i][n] = P.in.sc[(int64_t)sb * 8 + 4 * n + tig];
      }
    }
  }

  int cstep = 0;
#pragma unroll 1
  for (int tile = t0; tile < t1; ++tile, ++cstep) {
    bool pf = false;
    if (producer && !failed && ptile < t1) pf = !produce();
    if (__any_sync(0xffffffffu, pf)) {
      failed = true;
      *abort_flag = 1;
    }
    const int s = cstep % Q6_STAGES;
    if (!failed) {
      if (*abort_flag) {
        failed = true;
      } else {
        const bool ok = mbar_wait(&full[s], (uint32_t)(cstep / Q6_STAGES) & 1u, P.err);
        if (__any_sync(0xffffffffu, !ok)) failed = true;
      }
      if (failed) *abort_flag = 1;
    }
    float acc[NT][2];
#pragma unroll
    for (int n = 0; n < NT; ++n) acc[n][0] = acc[n][1] = 0.f;
    if (!failed) {
      const uint8_t* st = smem + (size_t)s * SSTR;
#pragma unroll
      for (int i = 0; i < (SBW > 0 ? SBW : 1); ++i) {
        // SBW = 0: a runtime loop over this warp's superblocks
        for (int sb = warp + Q6_WARPS * i; sb < P.nsb; sb += (SBW > 0 ? P.nsb : Q6_WARPS)) {
          uint2 bl[16][NT];
          float xl[NT];
          if (SBW == 0) {
#pragma unroll
            for (int j = 0; j < 16; ++j)
#pragma unroll
              for (int n = 0; n < NT; ++n) bl[j][n] = P.in.fx[(((int64_t)sb * 16 + j) * NT + n) * 32 + flane[n]];
#pragma unroll
            for (int n = 0; n < NT; ++n) xl[n] = P.in.sc[(int64_t)sb * 8 + 4 * n + tig];
          }
          const uint8_t* r0 = st + (size_t)g * RB + (size_t)sb * Q6_BLK;
          const uint8_t* r1 = r0 + (size_t)8 * RB;
          // With an even number of blocks per row, a block's 2-byte offset from a 4-byte
          // boundary depends only on its index, so it is the same for the whole warp.
          const int mode = (RB & 3) ? 2 : (sb & 1);
          if constexpr (SBW > 0) {
            if (mode == 0) q6k_superblock<0, NT>(r0, r1, tig, bq[i], xs[i], acc);
            else if (mode == 1) q6k_superblock<1, NT>(r0, r1, tig, bq[i], xs[i], acc);
            else q6k_superblock<2, NT>(r0, r1, tig, bq[i], xs[i], acc);
          } else {
            if (mode == 0) q6k_superblock<0, NT>(r0, r1, tig, bl, xl, acc);
            else if (mode == 1) q6k_superblock<1, NT>(r0, r1, tig, bl, xl, acc);
            else q6k_superblock<2, NT>(r0, r1, tig, bl, xl, acc);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0 && !failed) mbar_arrive(&empty[s]);
    // ------------------------------------------------ end of a tile: sum the warps' parts
    float* slot = red + ((size_t)warp * 32 + lane) * NT * 2;
#pragma unroll
    for (int n = 0; n < NT; ++n) slot[2 * n] = acc[n][0], slot[2 * n + 1] = acc[n][1];
    __syncwarp();
    __syncthreads();
    if (warp == (tile & (Q6_WARPS - 1)) && !*abort_flag) {
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int w = 0; w < Q6_WARPS; ++w) {
          const float* q = red + ((size_t)w * 32 + lane) * NT * 2 + 2 * n;
          s0 += q[0];
          s1 += q[1];
        }
        const int tok = 4 * n + tig;
        if (tok < P.m) {
          float* o = P.y + (int64_t)tok * P.n + tile * 16;
          o[g] = s0;
          o[g + 8] = s1;
        }
      }
    }
    __syncthreads();
  }
  if (producer && *abort_flag) {
    for (int t = max(0, (ptile - t0) - Q6_STAGES); t < ptile - t0; ++t)
      (void)mbar_wait(&full[t % Q6_STAGES], (uint32_t)(t / Q6_STAGES) & 1u, nullptr);
  }
}

size_t q6k_smem(int nsb, int nt) {
  const size_t tile = (size_t)16 * nsb * Q6_BLK;
  const size_t sstr = (tile + 16 + 127) & ~(size_t)127;
  return Q6_STAGES * sstr + 2 * Q6_STAGES * 8 + (size_t)Q6_WARPS * 32 * nt * 2 * 4 + 16;
}

template <int NT, int SBW, int CPS>
cudaError_t launch_q6k_kernel(const Q6Params& P, int grid, size_t smem, cudaStream_t s) {
  auto kern = q6k_gemv_kernel<NT, SBW, CPS>;
  static uint64_t attr_set = 0;  // one bit per device
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), Q6_STAGES * 110592 + 8192, &attr_set);
  if (e != cudaSuccess) return e;
  void* args[] = {const_cast<Q6Params*>(&P)};
  return launch_pdl(reinterpret_cast<const void*>(kern), dim3(grid), dim3(Q6_WARPS * 32), smem, s, args);
}

__global__ void q6k_dequant_kernel(const uint8_t* __restrict__ w, float* __restrict__ out, int64_t nblocks) {
  // one thread per weight; exact: d * scale * (q - 32) has at most 24 significant bits
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= nblocks * QK) return;
  const int64_t b = i / QK;
  const int k = (int)(i % QK), h = k >> 7, s = (k >> 5) & 3, l = k & 31;
  const uint8_t* blk = w + b * Q6_BLK;
  const uint32_t qlb = blk[64 * h + l + 32 * (s & 1)];
  const uint32_t q = (s < 2 ? (qlb & 15u) : (qlb >> 4)) | (((uint32_t)blk[128 + 32 * h + l] >> (2 * s)) & 3u) << 4;
  const float d = __half2float(__ushort_as_half((unsigned short)(blk[208] | blk[209] << 8)));
  const int sc = (int)(int8_t)blk[192 + k / 16];
  out[i] = d * (float)(sc * ((int)q - 32));
}

}  // namespace

bool q6k_plan(int64_t m, int64_t n, int64_t k, int num_sms, Q6Plan* p) {
  if (m < 1 || m > 8 || n < 16 || n % 16 != 0 || k < QK || k % QK != 0 || k > 8192) return false;
  p->m = (int)m;
  p->n = (int)n;
  p->k = (int)k;
  p->nt = (int)((m + 3) / 4);
  const int nsb = (int)(k / QK);
  p->smem = q6k_smem(nsb, p->nt);
  p->cps = 2 * p->smem + 2048 <= 232448 ? 2 : 1;  // two CTAs per SM when two fit
  p->grid = (int)std::min<int64_t>((int64_t)num_sms * p->cps, n / 16);
  size_t o = 0;
  p->off_fx = o;
  o = align256(o + (size_t)nsb * 16 * p->nt * 32 * 8);
  p->off_sc = o;
  o = align256(o + (size_t)nsb * 8 * 4);
  p->ws_bytes = o;
  return true;
}

cudaError_t launch_q6k_gemv(const Q6Plan& p, const void* x, int bf16, const void* w, float* y, void* ws,
                            uint32_t* err, cudaStream_t s, const ProfileEvents& prof) {
  uint8_t* W = (uint8_t*)ws;
  Q6Frags f{(uint2*)(W + p.off_fx), (float*)(W + p.off_sc)};
  const int nsb = p.k / QK;
  prof.before(0, s);
  if (bf16)
    prep_q6k_x_kernel<__nv_bfloat16><<<nsb, 128 * p.nt, 0, s>>>((const __nv_bfloat16*)x, p.k, p.m, p.nt, f);
  else
    prep_q6k_x_kernel<float><<<nsb, 128 * p.nt, 0, s>>>((const float*)x, p.k, p.m, p.nt, f);
  prof.after(0, s);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  Q6Params P{(const uint8_t*)w, p.n, nsb, p.m, p.nt, f, y, err};
  prof.before(1, s);
  const bool cache = nsb <= 16;
  if (p.nt == 1) {
    if (cache)
      e = p.cps == 2 ? launch_q6k_kernel<1, 2, 2>(P, p.grid, p.smem, s) : launch_q6k_kernel<1, 2, 1>(P, p.grid, p.smem, s);
    else
      e = launch_q6k_kernel<1, 0, 1>(P, p.grid, p.smem, s);
  } else {
    e = p.cps == 2 ? launch_q6k_kernel<2, 0, 2>(P, p.grid, p.smem, s) : launch_q6k_kernel<2, 0, 1>(P, p.grid, p.smem, s);
  }
  prof.after(1, s);
  return e;
}

cudaError_t launch_q6k_dequant(const void* w, float* out, int64_t rows, int64_t cols, cudaStream_t s) {
  const int64_t nb = rows * (cols / QK);
  const int64_t threads = nb * QK;
  q6k_dequant_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, s>>>((const uint8_t*)w, out, nb);
  return cudaGetLastError();
}

}  // namespace q4k
