// Decode regime (m = 1..8 tokens) of the Q4_K SwiGLU FFN on sm_103a.
//
//   K0 prep_x:       x [m][hidden] fp32 -> B fragments (below)
//   K1 gemv<2>:      g = Wg.x, u = Wu.x in one pass over both weight rows,
//                    h = silu(g) * u, then h -> B fragments for K2
//   K2 gemv<1>:      y = Wd.h
// K1 and K2 are launched with programmatic dependent launch, so each starts
// streaming its weights while the previous kernel drains.
// Source: realizar src/cuda/executor/layers/ffn.rs, fused_ffn_swiglu_gpu
// (gate and up GEMVs of the same input, fused SwiGLU, down GEMV, chained on
// one stream without synchronisation); realizar q4k_gemv_cached_uses.rs,
// TiledQ4KGemv / ChunkedTiledQ4KGemv (activations staged once and reused by
// several output rows; K chunked when it is large) as prior art.
//
// Arithmetic. The weights are multiplied on the tensor cores with
// mma.sync.m16n8k16 (fp16 inputs, fp32 accumulation). A weight tile (16 rows
// x 16 k) is the A operand: each 4-bit quant q is widened with the
// 0x6400-exponent trick and multiplied by its 6-bit sub-block scale in one
// fp16 fma, giving q*scale exactly (<= 945). The activations are the B
// operand: column n = (token 4*tile + n/2, part n%2), part 0 the fp16 value of
// x*2^-e and part 1 the fp16 remainder, so hi + lo carries about 22 bits of x.
// e is chosen per token and superblock so that the largest |x| maps into
// [2^14, 2^15). Per superblock the MMA result is scaled by d * 2^e and the
// min term dmin * sum_j min_j * X_j (X_j = sum of x over sub-block j) is
// subtracted; that term comes from one extra MMA whose A holds the 6-bit
// mins and whose B holds X_j * 2^-(e+6) split into hi and lo.
//
// Work split. Each warp streams its own weight rows through a ring of shared
// memory stages filled by 144-byte bulk copies (one per row per superblock),
// so every warp keeps several KB of weights in flight without using
// registers. A unit of work is (K-split, 16-row tile); each CTA takes a
// contiguous range of units and its warps take units round-robin. When K is
// split, partial sums go to the workspace and the last warp to finish a tile
// (per-tile semaphore) adds them in a fixed order, so results are
// deterministic. The last warp to finish the 16 tiles of a 256-row block of h
// converts that block to B fragments for K2.
#include <algorithm>
#include <cmath>

#include "common.cuh"
#include "kernels.h"
#include "tmap.h"

namespace q4k {

namespace {

struct FragPtrs {
  uint2* fx;     // [nsb][16 k-steps][nt][32 lanes] main B fragments
  uint32_t* fm;  // [nsb][nt][32 lanes] min-term B fragments (b0b1; b2b3 are zero)
  float* sc;     // [nsb][8] 2^e per token
};

// Loads the 8 inputs of this lane for one token (float32 or bf16, widened exactly).
__device__ __forceinline__ void load_inputs8(const float* p, bool coherent, float v[8]) {
  const float4* q = reinterpret_cast<const float4*>(p);
  const float4 a = coherent ? __ldcg(q) : q[0];
  const float4 b = coherent ? __ldcg(q + 1) : q[1];
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void load_inputs8(const __nv_bfloat16* p, bool, float v[8]) {
  const uint4 a = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// One warp converts token t of superblock `sb` (256 consecutive inputs starting
// at `row`) into B fragments; `zero` writes the zeros of a padding token.
template <typename T>
__device__ __forceinline__ void prep_token(const T* row, bool coherent, bool zero, int t, int nt, int sb,
                                           FragPtrs f) {
  const int lane = threadIdx.x & 31;
  const int sbk = lane >> 2;              // sub-block of this lane's 8 inputs
  const int tgp = sbk >> 1, p = sbk & 1;  // quad thread owning that sub-block and its nibble half
  const int ntile = t >> 2, gbase = 2 * (t & 3);
  uint2* fx = f.fx + ((int64_t)sb * 16 * nt + ntile) * 32 + tgp;
  uint32_t* fm = f.fm + ((int64_t)sb * nt + ntile) * 32 + (lane >> 3);
  if (zero) {
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int step = 2 * ((lane & 3) * 2 + hh) + p;
      fx[(int64_t)step * nt * 32 + gbase * 4] = make_uint2(0u, 0u);
      fx[(int64_t)step * nt * 32 + (gbase + 1) * 4] = make_uint2(0u, 0u);
    }
    if ((lane & 7) == 0) fm[gbase * 4] = fm[(gbase + 1) * 4] = 0u;
    if (lane == 0) f.sc[(int64_t)sb * 8 + t] = 1.f;
    return;
  }
  float v[8];
  load_inputs8(row + lane * 8, coherent, v);
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
  amax = warp_max(amax);
  int e = 0;
  if (amax > 0.f) e = max((int)((__float_as_uint(amax) >> 23) & 0xFF) - 127 - 14, -100);
  const float s = __uint_as_float((uint32_t)(127 - e) << 23);  // 2^-e
  __half hi[8], lo[8];
  float xsum = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float y = v[i] * s;
    hi[i] = __float2half_rn(y);
    lo[i] = __float2half_rn(y - __half2float(hi[i]));
    xsum += y;
  }
  xsum += __shfl_xor_sync(0xffffffffu, xsum, 1);
  xsum += __shfl_xor_sync(0xffffffffu, xsum, 2);
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int step = 2 * ((lane & 3) * 2 + hh) + p;
#pragma unroll
    for (int part = 0; part < 2; ++part) {
      const __half* h8 = part ? lo : hi;
      uint2 fr;
      fr.x = h2_as_u32(__halves2half2(h8[4 * hh + 0], h8[4 * hh + 2]));
      fr.y = h2_as_u32(__halves2half2(h8[4 * hh + 1], h8[4 * hh + 3]));
      fx[(int64_t)step * nt * 32 + (gbase + part) * 4] = fr;
    }
  }
  // X_j * 2^-6 keeps the sub-block sums inside the fp16 range
  const float xl = __shfl_sync(0xffffffffu, xsum, lane & ~7) * 0.015625f;
  const float xh = __shfl_sync(0xffffffffu, xsum, (lane & ~7) + 4) * 0.015625f;
  if ((lane & 7) == 0) {
    const __half xlh = __float2half_rn(xl), xhh = __float2half_rn(xh);
    const __half xll = __float2half_rn(xl - __half2float(xlh)), xhl = __float2half_rn(xh - __half2float(xhh));
    fm[gbase * 4] = h2_as_u32(__halves2half2(xlh, xhh));
    fm[(gbase + 1) * 4] = h2_as_u32(__halves2half2(xll, xhl));
  }
  if (lane == 0) f.sc[(int64_t)sb * 8 + t] = __uint_as_float((uint32_t)(127 + e) << 23);
}

// One warp converts all 4*nt token slots of superblock `sb` of src [m][ld].
template <typename T>
__device__ void prep_superblock(const T* src, int64_t ld, int m, int nt, int sb, FragPtrs f, bool coherent) {
  for (int t = 0; t < 4 * nt; ++t)
    prep_token<T>(src + (int64_t)min(t, m - 1) * ld + (int64_t)sb * QK, coherent, t >= m, t, nt, sb, f);
}

// K0: one CTA per superblock of x, one warp per token slot. It also zeroes the
// split-K semaphores and h-block counters of this call; K1 and K2 touch them
// only after their dependent-launch wait on K0.
template <typename T>
__global__ void prep_x_kernel(const T* __restrict__ x, int hidden, int m, int nt, FragPtrs f,
                              uint32_t* __restrict__ counters, int ncounters) {
  pdl_launch_dependents();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < ncounters; i += gridDim.x * blockDim.x) counters[i] = 0u;
  const int t = threadIdx.x >> 5, sb = blockIdx.x;
  prep_token<T>(x + (int64_t)min(t, m - 1) * hidden + (int64_t)sb * QK, false, t >= m, t, nt, sb, f);
}

struct GemvParams {
  const uint8_t* w0;  // gate (K1) or down (K2)
  const uint8_t* w1;  // up (K1)
  int rows, nsb, m, kc, nks;
  FragPtrs in;        // B fragments of the input
  float* part;        // [nks][nmat][m][rows] partial sums when nks > 1
  uint32_t* sem;      // [rows/16] per-tile semaphores (zero between calls)
  float* out;         // h (K1) or y (K2), [m][rows]
  FragPtrs next;      // K1: fragments of h for K2
  uint32_t* cnt_next; // K1: [rows/256] counters (zero between calls)
  uint32_t* err;
};

__device__ __forceinline__ void mma16816(float c[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }

// Per-thread constants for reading the two sub-blocks (2*tig, 2*tig+1) a quad
// thread owns out of the 12 packed scale/min bytes (s0, s1, s2 = bytes 0-3, 4-7,
// 8-11): their bytes sit at positions bp, bp+1 (bp = 2*(tig&1)); sub-blocks
// 4-7 (tig >= 2) take the low/high nibbles of bytes 8-11 plus the top two bits
// of bytes 0-7.
struct ScaleSel {
  uint32_t shift;  // 8 * bp
  bool high;       // tig >= 2
};
__device__ __forceinline__ void owned_scales(const ScaleSel& S, uint32_t s0, uint32_t s1, uint32_t s2,
                                             uint32_t& sc_a, uint32_t& sc_b, uint32_t& m_a, uint32_t& m_b) {
  const uint32_t w0 = s0 >> S.shift, w1 = s1 >> S.shift, w2 = s2 >> S.shift;
  if (!S.high) {
    sc_a = w0 & 63u;
    sc_b = (w0 >> 8) & 63u;
    m_a = w1 & 63u;
    m_b = (w1 >> 8) & 63u;
  } else {
    sc_a = (w2 & 15u) | ((w0 >> 2) & 0x30u);
    sc_b = ((w2 >> 8) & 15u) | ((w0 >> 10) & 0x30u);
    m_a = ((w2 >> 4) & 15u) | ((w1 >> 2) & 0x30u);
    m_b = ((w2 >> 12) & 15u) | ((w1 >> 10) & 0x30u);
  }
}
// half2(v, v) for an integer 0 <= v < 1024, exactly: (1024 + v) - 1024 in fp16
__device__ __forceinline__ __half2 small_int_h2(uint32_t v) {
  return __hsub2(u32_as_h2(0x64006400u | (v * 0x00010001u)), u32_as_h2(0x64006400u));
}
__device__ __forceinline__ __half2 small_int_pair_h2(uint32_t a, uint32_t b) {
  return __hsub2(u32_as_h2(0x64006400u | a | (b << 16)), u32_as_h2(0x64006400u));
}

__device__ __forceinline__ void tma_tile(void* dst, const CUtensorMap* tm, int x, int y, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

template <int NMAT, int NT, int STAGES, int WARPS>
__global__ void __launch_bounds__(WARPS * 32, 1)
    gemv_kernel(const __grid_constant__ CUtensorMap tm0, const __grid_constant__ CUtensorMap tm1,
                const GemvParams P) {
  constexpr int ROWS = 16;
  constexpr int TILE = ROWS * BLK;        // one 16-row x 1-superblock tile of one matrix
  constexpr int STREAMS = WARPS / NMAT;   // units are walked by warp pairs (gate, up) when NMAT == 2
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, tig = lane & 3;
  const int mat = (NMAT == 2) ? (warp & 1) : 0;
  const int strm = (NMAT == 2) ? (warp >> 1) : warp;
  uint8_t* ring = smem + warp * STAGES * TILE;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + WARPS * STAGES * TILE) + warp * STAGES;
  // gate/up exchange slots: [stream][2][32 lanes][NT][2]
  float* xch = reinterpret_cast<float*>(smem + WARPS * STAGES * TILE + WARPS * STAGES * 8);
  const CUtensorMap* tm = mat ? &tm1 : &tm0;

  const int nrt = P.rows / ROWS;
  const int64_t U = (int64_t)P.nks * nrt;
  const int64_t u0 = U * blockIdx.x / gridDim.x, u1 = U * (blockIdx.x + 1) / gridDim.x;

  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < STAGES; ++s) mbar_init(&bar[s], 1);
    fence_mbar_init();
  }
  __syncwarp();

  // issue cursor (which step the next tile load fetches)
  int64_t iu = u0 + strm;
  int isb = 0, isb_end = 0, irt = 0;
  if (iu < u1) {
    irt = (int)(iu % nrt);
    isb = (int)(iu / nrt) * P.kc;
    isb_end = min(P.nsb, isb + P.kc);
  }
  const uint64_t pol = policy_evict_first();
  auto issue = [&](int stage) {
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      mbar_arrive_expect_tx(&bar[stage], TILE);
      tma_tile(ring + stage * TILE, tm, isb * (BLK / 8), irt * ROWS, &bar[stage], pol);
    }
    if (++isb == isb_end) {
      iu += STREAMS;
      if (iu < u1) {
        irt = (int)(iu % nrt);
        isb = (int)(iu / nrt) * P.kc;
        isb_end = min(P.nsb, isb + P.kc);
      }
    }
  };

  int issued = 0;
  for (; issued < STAGES - 1 && iu < u1; ++issued) issue(issued % STAGES);
  pdl_launch_dependents();
  pdl_wait();  // input fragments come from the previous kernel

  const uint32_t sshift = 16u * (uint32_t)(tig & 1);  // byte pair of the owned sub-blocks
  const bool shigh = tig >= 2;                       // owned sub-blocks are 4..7
  bool live[NT];                                     // B lanes that hold a real token
#pragma unroll
  for (int n = 0; n < NT; ++n) live[n] = (lane >> 3) < P.m - 4 * n;

  // consume cursor
  int64_t cu = u0 + strm;
  int csb = 0, csb_end = 0, crt = 0, cks = 0, nunit = 0;
  if (cu < u1) {
    crt = (int)(cu % nrt);
    cks = (int)(cu / nrt);
    csb = cks * P.kc;
    csb_end = min(P.nsb, csb + P.kc);
  }
  float acc[NT][2];
#pragma unroll
  for (int n = 0; n < NT; ++n) acc[n][0] = acc[n][1] = 0.f;

  int step = 0;
  bool failed = false;
#pragma unroll 1
  while (cu < u1) {
    const int stage = step % STAGES;
    if (iu < u1) {
      issue((step + STAGES - 1) % STAGES);
      ++issued;
    }
    if (!mbar_wait(&bar[stage], (uint32_t)(step / STAGES) & 1u, P.err)) {
      failed = true;
      break;
    }
    // ------------------------------------------------ one superblock of 16 rows
    const uint8_t* st = ring + stage * TILE;
    uint4 q0[2], q1[2];
    uint32_t A_min[2];
    __half2 mlo[2], alo[2], mhi[2], ahi[2];
    float dd[2], dm[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const uint8_t* rb = st + (g + 8 * r) * BLK;
      const uint4 hd = *reinterpret_cast<const uint4*>(rb);
      q0[r] = *reinterpret_cast<const uint4*>(rb + 16 + 32 * tig);
      q1[r] = *reinterpret_cast<const uint4*>(rb + 32 + 32 * tig);
      const float2 dpair = __half22float2(u32_as_h2(hd.x));
      dd[r] = dpair.x;
      dm[r] = dpair.y;
      // 6-bit scale and min of the two owned sub-blocks (2*tig, 2*tig+1)
      const uint32_t w0 = hd.y >> sshift, w1 = hd.z >> sshift, w2 = hd.w >> sshift;
      const uint32_t sa = shigh ? ((w2 & 15u) | ((w0 >> 2) & 0x30u)) : (w0 & 63u);
      const uint32_t sb = shigh ? (((w2 >> 8) & 15u) | ((w0 >> 10) & 0x30u)) : ((w0 >> 8) & 63u);
      const uint32_t ma = shigh ? (((w2 >> 4) & 15u) | ((w1 >> 2) & 0x30u)) : (w1 & 63u);
      const uint32_t mb = shigh ? (((w2 >> 12) & 15u) | ((w1 >> 10) & 0x30u)) : ((w1 >> 8) & 63u);
      mlo[r] = small_int_h2(sa);
      alo[r] = __hmul2(mlo[r], u32_as_h2(0xE400E400u));  // * -1024
      const __half2 shb = small_int_h2(sb);
      mhi[r] = __hmul2(shb, u32_as_h2(0x2C002C00u));     // * 1/16
      ahi[r] = __hmul2(shb, u32_as_h2(0xD400D400u));     // * -64
      A_min[r] = h2_as_u32(small_int_pair_h2(ma, mb));
    }
    float c[NT][2][4], cm[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int i = 0; i < 4; ++i) c[n][0][i] = c[n][1][i] = cm[n][i] = 0.f;

    const uint2* fx = P.in.fx + (int64_t)csb * 16 * NT * 32 + lane;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      uint2 b0[NT], b1[NT];
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        b0[n] = live[n] ? fx[((2 * w) * NT + n) * 32] : make_uint2(0u, 0u);
        b1[n] = live[n] ? fx[((2 * w + 1) * NT + n) * 32] : make_uint2(0u, 0u);
      }
      uint32_t L0[2], L1[2], H0[2], H1[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const uint4& qq = (w < 4) ? q0[r] : q1[r];
        const uint32_t wd = (w & 3) == 0 ? qq.x : (w & 3) == 1 ? qq.y : (w & 3) == 2 ? qq.z : qq.w;
        const uint32_t t8 = wd >> 8;
        L0[r] = h2_as_u32(__hfma2(u32_as_h2(lop3_and_or(wd, 0x000F000Fu, 0x64006400u)), mlo[r], alo[r]));
        L1[r] = h2_as_u32(__hfma2(u32_as_h2(lop3_and_or(t8, 0x000F000Fu, 0x64006400u)), mlo[r], alo[r]));
        H0[r] = h2_as_u32(__hfma2(u32_as_h2(lop3_and_or(wd, 0x00F000F0u, 0x64006400u)), mhi[r], ahi[r]));
        H1[r] = h2_as_u32(__hfma2(u32_as_h2(lop3_and_or(t8, 0x00F000F0u, 0x64006400u)), mhi[r], ahi[r]));
      }
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        mma16816(c[n][0], L0[0], L0[1], L1[0], L1[1], b0[n].x, b0[n].y);
        mma16816(c[n][1], H0[0], H0[1], H1[0], H1[1], b1[n].x, b1[n].y);
      }
    }
    {
      const uint32_t* fm = P.in.fm + (int64_t)csb * NT * 32 + lane;
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        const uint32_t bm = live[n] ? fm[n * 32] : 0u;
        mma16816(cm[n], A_min[0], A_min[1], 0u, 0u, bm, 0u);
      }
    }
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      const float xs = P.in.sc[(int64_t)csb * 8 + n * 4 + tig];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const float main = (c[n][0][2 * r] + c[n][1][2 * r]) + (c[n][0][2 * r + 1] + c[n][1][2 * r + 1]);
        const float mins = cm[n][2 * r] + cm[n][2 * r + 1];
        acc[n][r] = fmaf(main, dd[r] * xs, acc[n][r]);
        acc[n][r] = fmaf(-mins, dm[r] * (64.f * xs), acc[n][r]);
      }
    }
    ++step;
    // ------------------------------------------------ end of a unit
    if (++csb == csb_end) {
      const int row0 = crt * ROWS;
      float fin[NMAT][NT][2];
      bool owner = true;  // the warp that finishes the unit (gate warp of a pair)
      if (NMAT == 2) {
        float* slot = xch + (((strm * 2 + (nunit & 1)) * 32 + lane) * NT) * 2;
        if (mat == 1) {
#pragma unroll
          for (int n = 0; n < NT; ++n) slot[2 * n] = acc[n][0], slot[2 * n + 1] = acc[n][1];
        }
        asm volatile("bar.sync %0, 64;" ::"r"(1 + strm) : "memory");
        owner = (mat == 0);
        if (owner) {
#pragma unroll
          for (int n = 0; n < NT; ++n) {
            fin[0][n][0] = acc[n][0];
            fin[0][n][1] = acc[n][1];
            fin[NMAT - 1][n][0] = slot[2 * n];
            fin[NMAT - 1][n][1] = slot[2 * n + 1];
          }
        }
      } else {
#pragma unroll
        for (int n = 0; n < NT; ++n) fin[0][n][0] = acc[n][0], fin[0][n][1] = acc[n][1];
      }
      if (owner) {
        bool last = true;
        if (P.nks > 1) {
#pragma unroll
          for (int n = 0; n < NT; ++n) {
            const int tok = n * 4 + tig;
            if (tok < P.m) {
#pragma unroll
              for (int a = 0; a < NMAT; ++a)
#pragma unroll
                for (int r = 0; r < 2; ++r)
                  P.part[(((int64_t)cks * NMAT + a) * P.m + tok) * P.rows + row0 + g + 8 * r] = fin[a][n][r];
            }
          }
          __threadfence();
          __syncwarp();
          uint32_t old = 0;
          if (lane == 0) old = atomicAdd(&P.sem[crt], 1u);
          old = __shfl_sync(0xffffffffu, old, 0);
          last = (old == (uint32_t)(P.nks - 1));
          if (last) {
            __threadfence();
#pragma unroll
            for (int n = 0; n < NT; ++n) {
              const int tok = n * 4 + tig;
              if (tok < P.m) {
#pragma unroll
                for (int a = 0; a < NMAT; ++a)
#pragma unroll
                  for (int r = 0; r < 2; ++r) {
                    float sum = 0.f;
                    for (int k = 0; k < P.nks; ++k)
                      sum += __ldcg(&P.part[(((int64_t)k * NMAT + a) * P.m + tok) * P.rows + row0 + g + 8 * r]);
                    fin[a][n][r] = sum;
                  }
              }
            }
            if (lane == 0) P.sem[crt] = 0u;
          }
        }
        if (last) {
#pragma unroll
          for (int n = 0; n < NT; ++n) {
            const int tok = n * 4 + tig;
            if (tok < P.m) {
#pragma unroll
              for (int r = 0; r < 2; ++r) {
                const float v = (NMAT == 2) ? silu_f(fin[0][n][r]) * fin[NMAT - 1][n][r] : fin[0][n][r];
                P.out[(int64_t)tok * P.rows + row0 + g + 8 * r] = v;
              }
            }
          }
          if (NMAT == 2) {
            // the last of the 16 tiles of a 256-row block of h converts it for the down projection
            __threadfence();
            __syncwarp();
            const int sbh = row0 / QK;
            uint32_t old = 0;
            if (lane == 0) old = atomicAdd(&P.cnt_next[sbh], 1u);
            old = __shfl_sync(0xffffffffu, old, 0);
            if (old == (uint32_t)(QK / ROWS - 1)) {
              __threadfence();
              prep_superblock<float>(P.out, P.rows, P.m, NT, sbh, P.next, true);
              if (lane == 0) P.cnt_next[sbh] = 0u;
            }
          }
        }
      }
#pragma unroll
      for (int n = 0; n < NT; ++n) acc[n][0] = acc[n][1] = 0.f;
      ++nunit;
      cu += STREAMS;
      if (cu < u1) {
        crt = (int)(cu % nrt);
        cks = (int)(cu / nrt);
        csb = cks * P.kc;
        csb_end = min(P.nsb, csb + P.kc);
      }
    }
  }
  if (failed) {
    // let copies already in flight land before the CTA's shared memory goes away
    for (int s = step; s < issued; ++s) (void)mbar_wait(&bar[s % STAGES], (uint32_t)(s / STAGES) & 1u, nullptr);
  }
}

// Warps per CTA and ring stages per warp: 16 warps for up to 4 tokens (128
// registers per thread), 10 warps for 5-8 tokens, whose fragments need more.
template <int NT> struct Shape;
template <> struct Shape<1> { static constexpr int WARPS = 16, STAGES = 4; };
template <> struct Shape<2> { static constexpr int WARPS = 10, STAGES = 6; };

template <int NMAT, int NT>
cudaError_t launch_gemv(const CUtensorMap& t0, const CUtensorMap& t1, const GemvParams& P, int grid,
                        cudaStream_t s) {
  constexpr int W = Shape<NT>::WARPS, S = Shape<NT>::STAGES;
  auto kern = gemv_kernel<NMAT, NT, S, W>;
  const size_t smem = (size_t)W * S * (16 * BLK + 8) + (size_t)(W / NMAT) * 2 * 32 * NT * 2 * 4;
  static uint64_t attr_set = 0;  // one bit per device: the attribute is set per function and device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !(attr_set >> dev & 1)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (dev < 64) attr_set |= 1ull << dev;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(W * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, t0, t1, P);
}

// Weight matrix [rows][nsb blocks] as a 2-D tensor of 8-byte elements (18 per
// block), loaded 16 rows x 1 superblock at a time.
bool weight_map(CUtensorMap* m, const void* w, int rows, int nsb) {
  return tmap_2d(m, CU_TENSOR_MAP_DATA_TYPE_UINT64, w, (uint64_t)rows, (uint64_t)nsb * (BLK / 8),
                 (uint64_t)nsb * BLK, BLK / 8, 16, CU_TENSOR_MAP_SWIZZLE_NONE);
}

// Choose the number of K-splits. A CTA walks its contiguous range of units with
// `streams` independent unit streams (warps, or warp pairs for gate/up); the
// cost is the longest stream's superblock steps plus about one step of
// split-K fixup per unit when K is split.
void choose_split(int nsb, int nrt, int grid, int streams, int* nks_out, int* kc_out) {
  double best = 1e30;
  int best_nks = 1, best_kc = nsb;
  for (int t = 1; t <= nsb; ++t) {
    const int kc = (nsb + t - 1) / t;
    const int nks = (nsb + kc - 1) / kc;
    if (nks != t) continue;
    const int64_t units = (int64_t)nks * nrt;
    const int64_t per_cta = (units + grid - 1) / grid;
    const int64_t per_stream = (per_cta + streams - 1) / streams;
    const double cost = (double)per_stream * kc + (nks > 1 ? (double)per_stream : 0.0);
    if (cost < best - 1e-9) {
      best = cost;
      best_nks = nks;
      best_kc = kc;
    }
  }
  *nks_out = best_nks;
  *kc_out = best_kc;
}

inline size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

}  // namespace

bool decode_plan(int64_t m, int64_t hidden, int64_t inter, int num_sms, DecodePlan* p) {
  if (m < 1 || m > 8) return false;
  p->m = (int)m;
  p->hidden = (int)hidden;
  p->inter = (int)inter;
  p->nt = (int)((m + 3) / 4);
  const int nsb1 = (int)(hidden / QK), nsb2 = (int)(inter / QK);
  const int nrt1 = (int)(inter / 16), nrt2 = (int)(hidden / 16);
  const int w = p->nt == 1 ? Shape<1>::WARPS : Shape<2>::WARPS;
  choose_split(nsb1, nrt1, num_sms, w / 2, &p->nks1, &p->kc1);
  choose_split(nsb2, nrt2, num_sms, w, &p->nks2, &p->kc2);
  p->grid1 = (int)std::min<int64_t>(num_sms, (int64_t)p->nks1 * nrt1);
  p->grid2 = (int)std::min<int64_t>(num_sms, (int64_t)p->nks2 * nrt2);
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align256(o + bytes);
    return at;
  };
  p->off_fx1 = take((size_t)nsb1 * 16 * p->nt * 32 * 8);
  p->off_fm1 = take((size_t)nsb1 * p->nt * 32 * 4);
  p->off_sc1 = take((size_t)nsb1 * 8 * 4);
  p->off_fx2 = take((size_t)nsb2 * 16 * p->nt * 32 * 8);
  p->off_fm2 = take((size_t)nsb2 * p->nt * 32 * 4);
  p->off_sc2 = take((size_t)nsb2 * 8 * 4);
  p->off_h = take((size_t)m * inter * 4);
  p->off_p1 = take(p->nks1 > 1 ? (size_t)p->nks1 * 2 * m * inter * 4 : 0);
  p->off_p2 = take(p->nks2 > 1 ? (size_t)p->nks2 * m * hidden * 4 : 0);
  p->off_sem1 = take((size_t)nrt1 * 4);
  p->off_cnt2 = take((size_t)nsb2 * 4);
  p->off_sem2 = take((size_t)nrt2 * 4);
  p->ws_bytes = o;
  return true;
}

cudaError_t launch_decode(const DecodePlan& p, const void* x, int bf16, const void* wg, const void* wu, const void* wd,
                          float* y, void* ws, uint32_t* err, cudaStream_t s, const ProfileEvents& prof) {
  uint8_t* W = (uint8_t*)ws;
  FragPtrs f1{(uint2*)(W + p.off_fx1), (uint32_t*)(W + p.off_fm1), (float*)(W + p.off_sc1)};
  FragPtrs f2{(uint2*)(W + p.off_fx2), (uint32_t*)(W + p.off_fm2), (float*)(W + p.off_sc2)};
  const int nsb1 = p.hidden / QK;
  // K0: not a dependent launch, so it also orders this call after the previous one on the stream
  uint32_t* counters = (uint32_t*)(W + p.off_sem1);
  const int ncounters = (int)((p.ws_bytes - p.off_sem1) / 4);
  prof.before(0, s);
  if (bf16)
    prep_x_kernel<__nv_bfloat16>
        <<<nsb1, 128 * p.nt, 0, s>>>((const __nv_bfloat16*)x, p.hidden, p.m, p.nt, f1, counters, ncounters);
  else
    prep_x_kernel<float><<<nsb1, 128 * p.nt, 0, s>>>((const float*)x, p.hidden, p.m, p.nt, f1, counters, ncounters);
  prof.after(0, s);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  GemvParams g1{};
  g1.w0 = (const uint8_t*)wg;
  g1.w1 = (const uint8_t*)wu;
  g1.rows = p.inter;
  g1.nsb = nsb1;
  g1.m = p.m;
  g1.kc = p.kc1;
  g1.nks = p.nks1;
  g1.in = f1;
  g1.part = (float*)(W + p.off_p1);
  g1.sem = (uint32_t*)(W + p.off_sem1);
  g1.out = (float*)(W + p.off_h);
  g1.next = f2;
  g1.cnt_next = (uint32_t*)(W + p.off_cnt2);
  g1.err = err;
  CUtensorMap mg, mu, md;
  if (!weight_map(&mg, wg, p.inter, nsb1) || !weight_map(&mu, wu, p.inter, nsb1) ||
      !weight_map(&md, wd, p.hidden, p.inter / QK))
    return cudaErrorInvalidValue;
  prof.before(1, s);
  e = (p.nt == 1) ? launch_gemv<2, 1>(mg, mu, g1, p.grid1, s) : launch_gemv<2, 2>(mg, mu, g1, p.grid1, s);
  prof.after(1, s);
  if (e != cudaSuccess) return e;

  GemvParams g2{};
  g2.w0 = (const uint8_t*)wd;
  g2.w1 = nullptr;
  g2.rows = p.hidden;
  g2.nsb = p.inter / QK;
  g2.m = p.m;
  g2.kc = p.kc2;
  g2.nks = p.nks2;
  g2.in = f2;
  g2.part = (float*)(W + p.off_p2);
  g2.sem = (uint32_t*)(W + p.off_sem2);
  g2.out = y;
  g2.err = err;
  prof.before(2, s);
  e = (p.nt == 1) ? launch_gemv<1, 1>(md, md, g2, p.grid2, s) : launch_gemv<1, 2>(md, md, g2, p.grid2, s);
  prof.after(2, s);
  return e;
}

}  // namespace q4k
