// Decode regime (m = 1..16 tokens per pass) of the Q4_K SwiGLU FFN on sm_103a.
//
//   K0  prep_x:         x [m][hidden] -> B fragments (below); per token and superblock
//                       (one token: not launched, K1 builds them from x)
//   K1  gemv<gate/up>:  partial g = Wg.x and u = Wu.x per K-chunk, one pass over both
//   K1b finish_gateup:  g, u = sum of the chunks; h = silu(g) * u -> B fragments
//   K2  gemv<down>:     partial y = Wd.h per K-chunk
//   K3  finish_down:    y = sum of the chunks (only when K is split)
// All but the call's first kernel (K0, or K1 for one token) are launched with
// programmatic dependent launch: each starts (and streams its first weight tiles)
// while the previous kernel drains.
// Source: realizar src/cuda/executor/layers/ffn.rs, fused_ffn_swiglu_gpu
// (gate and up GEMVs of the same input, SwiGLU, down GEMV, chained on one
// stream without synchronisation); realizar q4k_gemv_cached_uses.rs,
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
// Streaming. A CTA walks a contiguous range of units; a unit is a set of
// 16-row tiles (gate and up of one tile in K1, COMBOS consecutive tiles of
// W_down in K2) over one K-chunk. Each step loads, with one 3-D TMA box per
// matrix, the next group of SLICES consecutive superblocks of those rows
// (SLICES x 144 contiguous bytes per row) into a stage of a ring shared by the
// CTA; in shared memory the box is laid out
// superblock-major, 144 bytes per row, so the fragment loads are free of bank
// conflicts. Each warp takes TPW of the unit's tiles at one superblock of the
// group; with one token tile it keeps that superblock's B fragments in
// registers while it stays the same. At the end of a unit an owner warp
// (rotating) sums the SLICES partial dot products through shared memory and
// stores them; the chunks are summed by K1b / K3 in a fixed order, so results
// are deterministic.
#include <algorithm>
#include <cmath>

#include "common.cuh"
#include "gemv_stream.cuh"
#include "kernels.h"
#include "q8_1.cuh"

namespace q4k {

namespace {

// 2^e entries per superblock: 8 up to two token tiles, 4 per tile beyond
__host__ __device__ constexpr int sc_stride(int nt) { return nt <= 2 ? 8 : 4 * nt; }

struct FragPtrs {
  uint2* fx;     // [nsb][16 k-steps][nt][32 lanes] main B fragments
  uint32_t* fm;  // [nsb][nt][32 lanes] min-term B fragments (b0b1; b2b3 are zero)
  float* sc;     // [nsb][sc_stride(nt)] 2^e per token
};

// One warp turns the 256 inputs of token t of superblock `sb` (this lane holds
// inputs 8*lane .. 8*lane+7 in v) into B fragments; `zero` writes the zeros of
// a padding token.
__device__ __forceinline__ void frag_token(const float v_in[8], bool zero, int t, int nt, int sb, FragPtrs f) {
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
    if (lane == 0) f.sc[(int64_t)sb * sc_stride(nt) + t] = 1.f;
    return;
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v_in[i]));
  amax = warp_max(amax);
  int e = 0;
  if (amax > 0.f) e = max((int)((__float_as_uint(amax) >> 23) & 0xFF) - 127 - 14, -100);
  const float s = __uint_as_float((uint32_t)(127 - e) << 23);  // 2^-e
  __half hi[8], lo[8];
  float xsum = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float y = v_in[i] * s;
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
  if (lane == 0) f.sc[(int64_t)sb * sc_stride(nt) + t] = __uint_as_float((uint32_t)(127 + e) << 23);
}

// One token (m = 1): block-diagonal B. Quad thread tig of an MMA owns quant
// group tig of every row (sub-blocks 2tig and 2tig+1) and supplies 4 of its
// weights per row and MMA as fp16 subnormals q * 2^-24 (low nibbles) or
// 16q * 2^-24 (high nibbles), straight from the quant word with one AND. The
// B column pair (2tig, 2tig+1) holds the hi and lo parts of x at exactly those
// k rows and is zero elsewhere, so C column pair tig collects sub-block
// 2tig's (or 2tig+1's) partial dot product alone and the 6-bit scale is
// applied once per superblock in float32. MMA index k: 0..7 = low nibbles of
// quant bytes 4k..4k+3 of the group, 8..15 = their high nibbles. Layout per
// superblock, one record of DREC bytes at fx + sb * DREC (a multiple of 16, so a
// group of records is one bulk copy): [16 MMAs][8 lanes with data: lane 4g +
// (g >> 1)] uint2 (b0 = x at bytes 0 and 2 of the word, b1 = x at bytes 1 and 3;
// g = 2tig + part), then 8 floats: the sub-block sums of x * 2^-e, then 2^e.
// Lane L holds x[8L .. 8L+7] of the superblock: quant group L >> 3, nibble half
// (L >> 2) & 1, MMAs 2(L & 3) and 2(L & 3) + 1.
constexpr int DREC = 1088;
constexpr int DREC_X = 1024, DREC_SC = 1056;  // byte offsets of the sums and of 2^e
__device__ __forceinline__ void frag_token_diag(const float v_in[8], int sb, FragPtrs f) {
  const int lane = threadIdx.x & 31;
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v_in[i]));
  amax = warp_max(amax);
  int e = 0;
  if (amax > 0.f) e = max((int)((__float_as_uint(amax) >> 23) & 0xFF) - 127 - 14, -100);
  const float s = __uint_as_float((uint32_t)(127 - e) << 23);  // 2^-e
  __half hi[8], lo[8];
  float xsum = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float y = v_in[i] * s;
    hi[i] = __float2half_rn(y);
    lo[i] = __float2half_rn(y - __half2float(hi[i]));
    xsum += y;
  }
  xsum += __shfl_xor_sync(0xffffffffu, xsum, 1);  // lanes 4j .. 4j+3 hold sub-block j
  xsum += __shfl_xor_sync(0xffffffffu, xsum, 2);
  uint8_t* rec = reinterpret_cast<uint8_t*>(f.fx) + (int64_t)sb * DREC;
  if ((lane & 3) == 0) reinterpret_cast<float*>(rec + DREC_X)[lane >> 2] = xsum;
  const int tig = lane >> 3, half = (lane >> 2) & 1, s0 = 2 * (lane & 3);
  uint2* fx = reinterpret_cast<uint2*>(rec);
#pragma unroll
  for (int ss = 0; ss < 2; ++ss) {
    const int k = half * 8 + s0 + ss;
#pragma unroll
    for (int part = 0; part < 2; ++part) {
      const __half* h8 = part ? lo : hi;
      uint2 fr;
      fr.x = h2_as_u32(__halves2half2(h8[4 * ss + 0], h8[4 * ss + 2]));
      fr.y = h2_as_u32(__halves2half2(h8[4 * ss + 1], h8[4 * ss + 3]));
      fx[k * 8 + 2 * tig + part] = fr;
    }
  }
  if (lane == 0) reinterpret_cast<float*>(rec + DREC_SC)[0] = __uint_as_float((uint32_t)(127 + e) << 23);
}

// One warp, one token: the block-diagonal B operand of superblock sb of x, straight into this
// lane's registers (the record frag_token_diag would write, as the gate/up GEMV reads it):
// bc[k] for MMA k, and the sub-block sums and scale of this lane's quant group. Lane L
// computes x[8L .. 8L+7] as frag_token_diag does; entry (k, 2p + part) of the record comes
// from lane 8p + 4(k >> 3) + ((k & 7) >> 1), half k & 1, and lane (g, tig) takes entry
// (k, g) when g >> 1 == tig (zeros otherwise).
__device__ __forceinline__ void diag_frags_from_x(const void* x, int xbf16, int sb, uint2 bc[16], float& xlo,
                                                  float& xhi, float& xsc) {
  const int lane = threadIdx.x & 31, g = lane >> 2, tig = lane & 3;
  float v[8];
  if (xbf16)
    load8(reinterpret_cast<const __nv_bfloat16*>(x) + (int64_t)sb * QK + lane * 8, v);
  else
    load8(reinterpret_cast<const float*>(x) + (int64_t)sb * QK + lane * 8, v);
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
  xsum += __shfl_xor_sync(0xffffffffu, xsum, 1);  // lanes 4j .. 4j+3 hold sub-block j
  xsum += __shfl_xor_sync(0xffffffffu, xsum, 2);
  uint2 E[2][2];  // this lane's entries: [half ss][part (hi, lo)]
#pragma unroll
  for (int ss = 0; ss < 2; ++ss)
#pragma unroll
    for (int part = 0; part < 2; ++part) {
      const __half* h8 = part ? lo : hi;
      E[ss][part] = make_uint2(h2_as_u32(__halves2half2(h8[4 * ss + 0], h8[4 * ss + 2])),
                               h2_as_u32(__halves2half2(h8[4 * ss + 1], h8[4 * ss + 3])));
    }
  const bool act = (g >> 1) == tig;
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const int src = 8 * tig + 4 * (k >> 3) + ((k & 7) >> 1), ss = k & 1;
    uint2 a0, a1;
    a0.x = __shfl_sync(0xffffffffu, E[ss][0].x, src);
    a0.y = __shfl_sync(0xffffffffu, E[ss][0].y, src);
    a1.x = __shfl_sync(0xffffffffu, E[ss][1].x, src);
    a1.y = __shfl_sync(0xffffffffu, E[ss][1].y, src);
    bc[k] = act ? ((g & 1) ? a1 : a0) : make_uint2(0u, 0u);
  }
  xlo = __shfl_sync(0xffffffffu, xsum, 8 * tig);
  xhi = __shfl_sync(0xffffffffu, xsum, 8 * tig + 4);
  xsc = __uint_as_float((uint32_t)(127 + e) << 23) * 1048576.f;  // 2^e * 2^20
}

// Q8: x (or h) is first rounded to Q8_1 (blocks of 32 = 4 lanes) and its
// dequantized values q * d become the B operand, the activations of the Q8_1
// entry point; the token slot's warp is whole, so the shuffles are safe.
__device__ __forceinline__ void round_q8_1(float v[8], int8_t q[8], float& d, float& s) {
  q8_1_block8(v, q, d, s);
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = (float)q[i] * d;
}

// K0: one CTA per superblock of x, one warp per token slot. DIAG: one token, x in host
// memory (with x in device memory the gate/up GEMV builds the block-diagonal fragments
// itself, diag_frags_from_x, and K0 is not launched).
template <typename T, bool Q8, bool DIAG = false>
__global__ void prep_x_kernel(const T* __restrict__ x, int hidden, int m, int nt, FragPtrs f) {
  pdl_launch_dependents();
  const int t = threadIdx.x >> 5, sb = blockIdx.x, lane = threadIdx.x & 31;
  float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (t < m) {
    load8(x + (int64_t)t * hidden + (int64_t)sb * QK + lane * 8, v);
    if (Q8) {
      int8_t q[8];
      float d, s;
      round_q8_1(v, q, d, s);
    }
  }
  if constexpr (DIAG)
    frag_token_diag(v, sb, f);
  else
    frag_token(v, t >= m, t, nt, sb, f);
}

// silu(z) = z * sigmoid(z), with t = e^-|z| in (0, 1]: sigmoid is 1 / (1 + t) for z >= 0
// and t / (1 + t) below. Nothing overflows, the divisor is in [1, 2] (where __fdividef
// is within 2 ulp), and there is no branch: the IEEE division's slow path had serialised
// the 8 values of a lane and made this the longest step of the SwiGLU kernel.
__device__ __forceinline__ float silu_f(float z) {
  const float t = expf(-fabsf(z));  // in (0, 1]
  return z * __fdividef(z >= 0.f ? 1.0f : t, 1.0f + t);
}

// K1b: one CTA per 256-row block of h, one warp per token slot. Sums the
// gate/up chunks in order, applies SwiGLU and writes the fragments of h (Q8: of
// Q8_1(h), whose quants and (d, s) also go to hq [m][inter] and hds [m][inter/32]).
template <bool Q8, bool DIAG = false>
__global__ void finish_gateup_kernel(const float* __restrict__ part, int nks, int m, int inter, int nt, FragPtrs f,
                                     uint8_t* __restrict__ hq, float2* __restrict__ hds) {
  pdl_launch_dependents();
  pdl_wait();
  const int t = threadIdx.x >> 5, sb = blockIdx.x, lane = threadIdx.x & 31;
  float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (t < m) {
    const int64_t i0 = (int64_t)sb * QK + lane * 8;
    float g[8], u[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) g[i] = u[i] = 0.f;
    // Batches of 4 chunks: all of a batch's loads are issued before the first add (a
    // loop over a run-time count would wait for each load in turn); sums in chunk order.
    for (int k0 = 0; k0 < nks; k0 += 4) {
      float a[4][8], b[4][8];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (k0 + j < nks) {
          load8(part + (((int64_t)(k0 + j) * 2 + 0) * m + t) * inter + i0, a[j]);
          load8(part + (((int64_t)(k0 + j) * 2 + 1) * m + t) * inter + i0, b[j]);
        }
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (k0 + j < nks)
#pragma unroll
          for (int i = 0; i < 8; ++i) g[i] += a[j][i], u[i] += b[j][i];
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = silu_f(g[i]) * u[i];
    if (Q8) {
      int8_t q[8];
      float d, s;
      round_q8_1(v, q, d, s);
      uint2 pk;
      pk.x = (uint32_t)(uint8_t)q[0] | (uint32_t)(uint8_t)q[1] << 8 | (uint32_t)(uint8_t)q[2] << 16 |
             (uint32_t)(uint8_t)q[3] << 24;
      pk.y = (uint32_t)(uint8_t)q[4] | (uint32_t)(uint8_t)q[5] << 8 | (uint32_t)(uint8_t)q[6] << 16 |
             (uint32_t)(uint8_t)q[7] << 24;
      *reinterpret_cast<uint2*>(hq + (int64_t)t * inter + i0) = pk;
      if ((lane & 3) == 0) hds[((int64_t)t * inter + i0) / Q8B] = make_float2(d, s);
    }
  }
  if constexpr (DIAG)
    frag_token_diag(v, sb, f);
  else
    frag_token(v, t >= m, t, nt, sb, f);
}

// Bytes of one stage: the weight boxes, then (one token, down projection) the input
// records, rounded up so that every stage's first box starts on a 128-byte boundary
// (the destination alignment of a tensor copy into shared memory).
__host__ __device__ constexpr int stage_total(int box_bytes, int rec_bytes) {
  return (box_bytes + rec_bytes + 127) / 128 * 128;
}

struct GemvParams {
  int rows;           // output rows of each matrix
  int nsb;            // superblocks along K
  int m;              // tokens
  int gpc;            // superblock groups per K-chunk
  int nks;            // K-chunks
  FragPtrs in;        // B fragments of the input
  float* out;         // chunk sums: [nks][2][m][rows] (gate/up) or [nks][m][rows] (down)
  uint32_t* err;
  int diag;           // one token with block-diagonal B fragments (frag_token_diag)
  const void* x;      // one-token gate/up: x itself, the fragments built in the kernel (or null: read
                      // the records K0 wrote)
  int xbf16;          // ... as bf16 (else float32)
};

__device__ __forceinline__ void mma16816(float c[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// COMBOS 16-row tiles per superblock and step (gate and up of the same rows, or
// COMBOS consecutive tiles of W_down); each warp takes TPW of them (sharing the
// B operand) at one of the SLICES superblocks.
template <bool GATEUP, int NT, int COMBOS, int TPW, int SLICES, int STAGES, int CPS, bool DIAG>
__global__ void __launch_bounds__(COMBOS / TPW * SLICES * 32, CPS)
    gemv_kernel(const __grid_constant__ CUtensorMap tm0, const __grid_constant__ CUtensorMap tm1,
                const GemvParams P) {
  static_assert(!DIAG || NT == 1, "the block-diagonal operand carries one token");
  constexpr int TG = COMBOS / TPW;  // tile groups
  constexpr int WARPS = TG * SLICES;
  static_assert(COMBOS % TPW == 0, "tiles split evenly over warps");
  constexpr int ROWS = 16;
  constexpr int RU = GATEUP ? ROWS : ROWS * COMBOS;    // output rows of a unit (per matrix)
  constexpr int MATS = GATEUP ? 2 : 1;
  constexpr int BOX_BYTES = SLICES * RU * BLK;        // one box: [SLICES][RU rows][144 B]
  constexpr int STAGE_BYTES = MATS * BOX_BYTES;
  // One token, down projection: each step's superblocks change, so their B records
  // travel with the weights, one bulk copy per stage behind the boxes.
  constexpr bool BSMEM = DIAG && !GATEUP;
  constexpr int STAGE_TOTAL = stage_total(STAGE_BYTES, BSMEM ? SLICES * DREC : 0);
  static_assert(BOX_BYTES % 128 == 0 && STAGE_TOTAL % 128 == 0, "TMA boxes land on 128-byte boundaries");
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_TOTAL);
  uint64_t* empty = full + STAGES;
  float* red = reinterpret_cast<float*>(empty + STAGES);  // [2][WARPS][32 lanes][TPW][NT][2]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(red + 2 * WARPS * 32 * TPW * NT * 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, tig = lane & 3;
  const int tgrp = warp % TG, slice = warp / TG;
  const int nru = P.rows / RU;
  const int ngroups = (P.nsb + SLICES - 1) / SLICES;
  const int U = P.nks * nru;  // at most 16 chunks x 2^16 row units
  const int u0 = (int)((int64_t)U * blockIdx.x / gridDim.x), u1 = (int)((int64_t)U * (blockIdx.x + 1) / gridDim.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], WARPS);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  // ---------------------------------------------------------------- producer (warp 0, lane 0)
  const bool producer = (warp == 0 && lane == 0);
  // Unit u = ks * nru + ru: K-chunk ks, row unit ru, superblock groups [g, ge).
  // One division places a walk at its first unit; later units follow by counting.
  struct Walk {
    int u, ks, ru, g, ge;
  };
  auto walk_start = [&](Walk& w, int u) {
    w.u = u;
    w.ks = u / nru;
    w.ru = u - w.ks * nru;
    w.g = w.ks * P.gpc;
    w.ge = min(ngroups, w.g + P.gpc);
  };
  auto walk_next = [&](Walk& w) {
    ++w.u;
    if (++w.ru == nru) {
      w.ru = 0;
      ++w.ks;
    }
    w.g = w.ks * P.gpc;
    w.ge = min(ngroups, w.g + P.gpc);
  };
  Walk pw;
  walk_start(pw, u0);
  int pstep = 0;
  const uint64_t pol = policy_evict_first();
  // B records of superblock group grp into the stage of step `step` (after the input is ready)
  auto issue_b = [&](int step, int grp) {
    const int n = min(SLICES, P.nsb - grp * SLICES);
    bulk_g2s(smem + (step % STAGES) * STAGE_TOTAL + STAGE_BYTES,
             reinterpret_cast<const uint8_t*>(P.in.fx) + (int64_t)grp * SLICES * DREC, (uint32_t)(n * DREC),
             &full[step % STAGES]);
  };
  int pre_grp[STAGES];  // groups of the steps issued before the input was ready
  auto produce = [&](bool input_ready) -> bool {  // issue the next step's loads; false on a timed-out wait
    const int s = pstep % STAGES;
    if (pstep >= STAGES && !mbar_wait(&empty[s], (uint32_t)((pstep / STAGES) - 1) & 1u, P.err)) return false;
    uint8_t* st = smem + s * STAGE_TOTAL;
    const int bbytes = BSMEM ? min(SLICES, P.nsb - pw.g * SLICES) * DREC : 0;
    mbar_arrive_expect_tx(&full[s], STAGE_BYTES + bbytes);
    tma_box3(st, &tm0, pw.ru * RU, pw.g * SLICES, &full[s], pol);
    if (GATEUP) tma_box3(st + BOX_BYTES, &tm1, pw.ru * RU, pw.g * SLICES, &full[s], pol);
    if (BSMEM) {
      if (input_ready)
        issue_b(pstep, pw.g);
      else
        pre_grp[pstep] = pw.g;
    }
    ++pstep;
    if (++pw.g == pw.ge) walk_next(pw);
    return true;
  };
  bool failed = false;  // warp-uniform once the loop starts
  if (producer) {
    for (int i = 0; i < STAGES - 1 && pw.u < u1; ++i)
      if (!produce(false)) {
        failed = true;
        *abort_flag = 1;
        break;
      }
  }
  failed = __any_sync(0xffffffffu, failed);
  pdl_launch_dependents();
  pdl_wait();  // input fragments come from the previous kernel
  if (BSMEM && producer)
    for (int i = 0; i < pstep; ++i) issue_b(i, pre_grp[i]);

  // B fragment lane to read for token tile n: this lane when its token is real,
  // else the same position of token 4n (always real); the columns of padding
  // tokens then hold copies that are never stored.
  int flane[NT];
#pragma unroll
  for (int n = 0; n < NT; ++n) flane[n] = ((lane >> 3) < P.m - 4 * n) ? lane : (lane & 7);
  // Sub-blocks 2*tig and 2*tig+1 of a row are this thread's. Their 6-bit scales
  // and mins are gathered from the 12-byte field with byte permutes whose
  // selectors and masks depend only on tig: for sub-blocks 0-3 a scale (min) is
  // the low 6 bits of byte j (j+4); for 4-7 it is the low (high) nibble of
  // byte j+4 with the top two bits of byte j-4 (j) above it.
  const uint32_t bb = 2u * (uint32_t)(tig & 1);
  const bool shigh = tig >= 2;
  const uint32_t selS0 = shigh ? ((4u + bb) | bb << 4 | (4u + bb) << 8 | bb << 12) : bb * 0x1111u;
  const uint32_t selS1 = selS0 + 0x1111u;
  const uint32_t selM = shigh ? ((4u + bb) | bb << 4 | (5u + bb) << 8 | (bb + 1u) << 12)
                              : (bb | bb << 4 | (bb + 1u) << 8 | (bb + 1u) << 12);
  const uint32_t mL = shigh ? 0x000F000Fu : 0x003F003Fu, mH = shigh ? 0x00300030u : 0u, sM = shigh ? 4u : 0u;

  // ---------------------------------------------------------------- consumer (all warps)
  Walk cw;
  walk_start(cw, u0);
  int nunit = 0, cstep = 0;
  float acc[TPW][NT][2];
#pragma unroll
  for (int t = 0; t < TPW; ++t)
#pragma unroll
    for (int n = 0; n < NT; ++n) acc[t][n][0] = acc[t][n][1] = 0.f;
  // A warp keeps the B fragments of its superblock in registers for as long as
  // that superblock stays the same (with one group per K-chunk: until its chunk
  // changes). With two token tiles they take 64 registers, which leave no room
  // for two CTAs per SM; there they are read through L1 at each use.
  constexpr bool CACHEB = NT == 1 || CPS == 1;
  uint2 bc[CACHEB ? 16 : 1][NT];
  uint32_t bmc[NT];
  float xsc[NT];
  float xlo = 0.f, xhi = 0.f;  // DIAG: sums of x * 2^-e over sub-blocks 2tig and 2tig+1
  int csb = -1;
  if constexpr (DIAG && GATEUP) {  // x's fragments of the first superblock, while the first weights arrive
    const int sb0 = cw.g * SLICES + slice;
    if (P.x && cw.u < u1 && sb0 < min(P.nsb, (cw.ks + 1) * P.gpc * SLICES)) {
      uint2 bt[16];
      diag_frags_from_x(P.x, P.xbf16, sb0, bt, xlo, xhi, xsc[0]);
#pragma unroll
      for (int k = 0; k < 16; ++k) bc[k][0] = bt[k];
      csb = sb0;
    }
  }

  // A warp whose wait timed out raises the CTA's abort flag and stops waiting,
  // copying and computing, but still walks its units so that every warp reaches
  // every unit-end barrier.
#pragma unroll 1
  while (cw.u < u1) {
    bool pf = false;
    if (producer && !failed && pw.u < u1) pf = !produce(true);
    if (__any_sync(0xffffffffu, pf)) {
      failed = true;
      *abort_flag = 1;
    }
    const int s = cstep % STAGES;
    if (!failed) {
      if (*abort_flag) {
        failed = true;
      } else {
        const bool ok = mbar_wait(&full[s], (uint32_t)(cstep / STAGES) & 1u, P.err);
        if (__any_sync(0xffffffffu, !ok)) failed = true;
      }
      if (failed) *abort_flag = 1;
    }
    const int sb = cw.g * SLICES + slice;
    const int chunk_end = min(P.nsb, (cw.ks + 1) * P.gpc * SLICES);
    if (DIAG && !failed && sb < chunk_end) {
      // ------------------------------------------ TPW 16-row tiles of one superblock, one token
      const bool act = (g >> 1) == tig;  // this lane's B column pair belongs to its own quant group
      if (BSMEM || sb != csb) {
        if constexpr (BSMEM) {  // h's record, copied into the stage with the weights
          const uint8_t* rec = smem + s * STAGE_TOTAL + STAGE_BYTES + slice * DREC;
          const uint2* fxd = reinterpret_cast<const uint2*>(rec);
#pragma unroll
          for (int k = 0; k < 16; ++k) bc[k][0] = act ? fxd[k * 8 + g] : make_uint2(0u, 0u);
          xlo = reinterpret_cast<const float*>(rec + DREC_X)[2 * tig];
          xhi = reinterpret_cast<const float*>(rec + DREC_X)[2 * tig + 1];
          xsc[0] = reinterpret_cast<const float*>(rec + DREC_SC)[0] * 1048576.f;  // 2^e * 2^20
        } else if (P.x) {  // x's fragments, built here from x (no separate kernel)
          uint2 bt[16];
          diag_frags_from_x(P.x, P.xbf16, sb, bt, xlo, xhi, xsc[0]);
#pragma unroll
          for (int k = 0; k < 16; ++k) bc[k][0] = bt[k];
        } else {  // x's record, written by K0
          const uint8_t* rec = reinterpret_cast<const uint8_t*>(P.in.fx) + (int64_t)sb * DREC;
          const uint2* fxd = reinterpret_cast<const uint2*>(rec);
#pragma unroll
          for (int k = 0; k < 16; ++k) bc[k][0] = act ? fxd[k * 8 + g] : make_uint2(0u, 0u);
          xlo = reinterpret_cast<const float*>(rec + DREC_X)[2 * tig];
          xhi = reinterpret_cast<const float*>(rec + DREC_X)[2 * tig + 1];
          xsc[0] = reinterpret_cast<const float*>(rec + DREC_SC)[0] * 1048576.f;  // 2^e * 2^20
        }
        csb = sb;
      }
#pragma unroll
      for (int t = 0; t < TPW; ++t) {
        const int cb = tgrp * TPW + t;
        const uint8_t* base = smem + s * STAGE_TOTAL + (GATEUP ? cb * BOX_BYTES + slice * RU * BLK
                                                                  : (slice * RU + cb * ROWS) * BLK);
        uint4 hd[2], q0[2], q1[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const uint8_t* rb = base + (g + 8 * r) * BLK;
          hd[r] = *reinterpret_cast<const uint4*>(rb);
          q0[r] = *reinterpret_cast<const uint4*>(rb + 16 + 32 * tig);
          q1[r] = *reinterpret_cast<const uint4*>(rb + 32 + 32 * tig);
        }
        // clo: sub-block 2tig (low nibbles, q * 2^-24); chi: sub-block 2tig+1 (high nibbles, q * 2^-20).
        // Columns 2tig and 2tig+1 hold the hi and lo parts of x.
        float clo[4] = {0.f, 0.f, 0.f, 0.f}, chi[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int w = 0; w < 8; ++w) {
          const uint4& qa = (w < 4) ? q0[0] : q1[0];
          const uint4& qb = (w < 4) ? q0[1] : q1[1];
          const uint32_t w0 = (w & 3) == 0 ? qa.x : (w & 3) == 1 ? qa.y : (w & 3) == 2 ? qa.z : qa.w;
          const uint32_t w1 = (w & 3) == 0 ? qb.x : (w & 3) == 1 ? qb.y : (w & 3) == 2 ? qb.z : qb.w;
          const uint32_t t0 = w0 >> 8, t1 = w1 >> 8;
          mma16816(clo, w0 & 0x000F000Fu, w1 & 0x000F000Fu, t0 & 0x000F000Fu, t1 & 0x000F000Fu, bc[w][0].x,
                   bc[w][0].y);
          mma16816(chi, w0 & 0x00F000F0u, w1 & 0x00F000F0u, t0 & 0x00F000F0u, t1 & 0x00F000F0u, bc[8 + w][0].x,
                   bc[8 + w][0].y);
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          // (scale, scale) and (min, min) of sub-blocks 2tig and 2tig+1 as fp16 1024 + value
          const uint32_t ps = prmt(hd[r].y, hd[r].w, selM), pm = prmt(hd[r].z, hd[r].w, selM);
          const uint32_t scb = lop3_and_or(ps, mL, lop3_and_or(ps >> 10, mH, 0x64006400u));
          const uint32_t mnb = lop3_and_or(pm >> sM, mL, lop3_and_or(pm >> 10, mH, 0x64006400u));
          // (16 * scale_2tig, scale_2tig+1) and (min_2tig, min_2tig+1), exact
          const float2 sf = __half22float2(__hfma2(u32_as_h2(scb), u32_as_h2(0x3C004C00u), u32_as_h2(0xE400F400u)));
          const float2 mf = __half22float2(__hsub2(u32_as_h2(mnb), u32_as_h2(0x64006400u)));
          const float2 dd = __half22float2(u32_as_h2(hd[r].x));
          const float tq = fmaf(sf.y, chi[2 * r] + chi[2 * r + 1], sf.x * (clo[2 * r] + clo[2 * r + 1]));
          const float tm = fmaf(mf.y, xhi, mf.x * xlo);
          const float S = fmaf(dd.x, tq, -(dd.y * 9.5367431640625e-07f) * tm);  // dmin * 2^-20
          acc[t][0][r] = fmaf(S, xsc[0], acc[t][0][r]);
        }
      }
    } else if (!DIAG && !failed && sb < chunk_end) {
      // ------------------------------------------ TPW 16-row tiles of one superblock
      uint4 q0[TPW][2], q1[TPW][2];
      uint32_t A_min[TPW][2];
      __half2 mlo[TPW][2], alo[TPW][2], mhi[TPW][2], ahi[TPW][2];
      float dd[TPW][2], dm[TPW][2];
#pragma unroll
      for (int t = 0; t < TPW; ++t) {
        const int cb = tgrp * TPW + t;
        const uint8_t* base = smem + s * STAGE_TOTAL + (GATEUP ? cb * BOX_BYTES + slice * RU * BLK
                                                                  : (slice * RU + cb * ROWS) * BLK);
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const uint8_t* rb = base + (g + 8 * r) * BLK;
          const uint4 hd = *reinterpret_cast<const uint4*>(rb);
          q0[t][r] = *reinterpret_cast<const uint4*>(rb + 16 + 32 * tig);
          q1[t][r] = *reinterpret_cast<const uint4*>(rb + 32 + 32 * tig);
          const float2 dpair = __half22float2(u32_as_h2(hd.x));
          dd[t][r] = dpair.x;
          dm[t][r] = dpair.y;
          // 0x6400 | value in each half: fp16 1024 + value
          const uint32_t p0 = prmt(hd.y, hd.w, selS0), p1 = prmt(hd.y, hd.w, selS1), pm = prmt(hd.z, hd.w, selM);
          const uint32_t s0b = lop3_and_or(p0, mL, lop3_and_or(p0 >> 10, mH, 0x64006400u));
          const uint32_t s1b = lop3_and_or(p1, mL, lop3_and_or(p1 >> 10, mH, 0x64006400u));
          const uint32_t mnb = lop3_and_or(pm >> sM, mL, lop3_and_or(pm >> 10, mH, 0x64006400u));
          mlo[t][r] = __hsub2(u32_as_h2(s0b), u32_as_h2(0x64006400u));                        // scale, scale
          alo[t][r] = __hmul2(mlo[t][r], u32_as_h2(0xE400E400u));                             // * -1024
          mhi[t][r] = __hfma2(u32_as_h2(s1b), u32_as_h2(0x2C002C00u), u32_as_h2(0xD400D400u));  // scale / 16
          ahi[t][r] = __hmul2(mhi[t][r], u32_as_h2(0xE400E400u));                             // -64 * scale
          A_min[t][r] = h2_as_u32(__hsub2(u32_as_h2(mnb), u32_as_h2(0x64006400u)));
        }
      }
      // Low-nibble (sub-block 2tig) and high-nibble (2tig+1) weights both enter as
      // exact q * scale, so one accumulator per tile and token tile takes both.
      float c[TPW][NT][4], cm[TPW][NT][4];
#pragma unroll
      for (int t = 0; t < TPW; ++t)
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
          for (int i = 0; i < 4; ++i) c[t][n][i] = cm[t][n][i] = 0.f;
      const uint2* fx = P.in.fx + (int64_t)sb * 16 * NT * 32;
      if (sb != csb) {
        if constexpr (CACHEB) {
#pragma unroll
          for (int k = 0; k < 16; ++k)
#pragma unroll
            for (int n = 0; n < NT; ++n) bc[k][n] = fx[(k * NT + n) * 32 + flane[n]];
        }
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          bmc[n] = P.in.fm[((int64_t)sb * NT + n) * 32 + flane[n]];
          xsc[n] = P.in.sc[(int64_t)sb * sc_stride(NT) + n * 4 + tig];
        }
        csb = sb;
      }
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        uint2 b0[NT], b1[NT];
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          if constexpr (CACHEB) {
            b0[n] = bc[2 * w][n];
            b1[n] = bc[2 * w + 1][n];
          } else {
            b0[n] = __ldg(fx + (2 * w * NT + n) * 32 + flane[n]);
            b1[n] = __ldg(fx + ((2 * w + 1) * NT + n) * 32 + flane[n]);
          }
        }
#pragma unroll
        for (int t = 0; t < TPW; ++t) {
          uint32_t L0[2], L1[2], H0[2], H1[2];
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const uint4& qq = (w < 4) ? q0[t][r] : q1[t][r];
            const uint32_t wd = (w & 3) == 0 ? qq.x : (w & 3) == 1 ? qq.y : (w & 3) == 2 ? qq.z : qq.w;
            const uint32_t t8 = wd >> 8;
            L0[r] = h2_as_u32(__hfma2(u32_as_h2(lop3_and_or(wd, 0x000F000Fu, 0x64006400u)), mlo[t][r], alo[t][r]));
            L1[r] = h2_as_u32(__hfma2(u32_as_h2(lop3_and_or(t8, 0x000F000Fu, 0x64006400u)), mlo[t][r], alo[t][r]));
            H0[r] = h2_as_u32(__hfma2(u32_as_h2(lop3_and_or(wd, 0x00F000F0u, 0x64006400u)), mhi[t][r], ahi[t][r]));
            H1[r] = h2_as_u32(__hfma2(u32_as_h2(lop3_and_or(t8, 0x00F000F0u, 0x64006400u)), mhi[t][r], ahi[t][r]));
          }
#pragma unroll
          for (int n = 0; n < NT; ++n) {
            mma16816(c[t][n], L0[0], L0[1], L1[0], L1[1], b0[n].x, b0[n].y);
            mma16816(c[t][n], H0[0], H0[1], H1[0], H1[1], b1[n].x, b1[n].y);
          }
        }
      }
      {
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          const uint32_t bm = bmc[n];
#pragma unroll
          for (int t = 0; t < TPW; ++t) mma16816(cm[t][n], A_min[t][0], A_min[t][1], 0u, 0u, bm, 0u);
        }
      }
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        const float xs = xsc[n];
#pragma unroll
        for (int t = 0; t < TPW; ++t)
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const float main = c[t][n][2 * r] + c[t][n][2 * r + 1];
            const float mins = cm[t][n][2 * r] + cm[t][n][2 * r + 1];
            acc[t][n][r] = fmaf(main, dd[t][r] * xs, acc[t][n][r]);
            acc[t][n][r] = fmaf(-mins, dm[t][r] * (64.f * xs), acc[t][n][r]);
          }
      }
    }
    __syncwarp();
    if (lane == 0 && !failed) mbar_arrive(&empty[s]);
    ++cstep;
    // ------------------------------------------------ end of a unit
    if (++cw.g == cw.ge) {
      if constexpr (DIAG) {  // quad thread tig summed its own sub-blocks only
#pragma unroll
        for (int t = 0; t < TPW; ++t)
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            acc[t][0][r] += __shfl_xor_sync(0xffffffffu, acc[t][0][r], 1);
            acc[t][0][r] += __shfl_xor_sync(0xffffffffu, acc[t][0][r], 2);
          }
      }
      constexpr int PER_LANE = TPW * NT * 2;
      float* slot = red + (size_t)((nunit & 1) * WARPS + warp) * 32 * PER_LANE + lane * PER_LANE;
#pragma unroll
      for (int t = 0; t < TPW; ++t)
#pragma unroll
        for (int n = 0; n < NT; ++n) slot[(t * NT + n) * 2] = acc[t][n][0], slot[(t * NT + n) * 2 + 1] = acc[t][n][1];
      __syncwarp();
      asm volatile("bar.sync 1, %0;" ::"r"(WARPS * 32) : "memory");
      if (warp == 1 + (nunit % (WARPS - 1)) && !*abort_flag) {
        // owner: sum the SLICES partial dot products of every tile and store this chunk's sums
        const float* rs = red + (size_t)(nunit & 1) * WARPS * 32 * PER_LANE + lane * PER_LANE;
        const int row0 = cw.ru * RU;
#pragma unroll
        for (int cb = 0; cb < COMBOS; ++cb)
#pragma unroll
          for (int n = 0; n < NT; ++n) {
            float s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int sl = 0; sl < SLICES; ++sl) {
              const float* q = rs + (size_t)(sl * TG + cb / TPW) * 32 * PER_LANE + ((cb % TPW) * NT + n) * 2;
              s0 += q[0];
              s1 += q[1];
            }
            const int tok = n * 4 + tig;
            if (tok < P.m) {
              float* o = GATEUP ? P.out + (((int64_t)cw.ks * 2 + cb) * P.m + tok) * P.rows + row0
                                : P.out + ((int64_t)cw.ks * P.m + tok) * P.rows + row0 + ROWS * cb;
              o[g] = s0;
              o[g + 8] = s1;
            }
          }
      }
#pragma unroll
      for (int t = 0; t < TPW; ++t)
#pragma unroll
        for (int n = 0; n < NT; ++n) acc[t][n][0] = acc[t][n][1] = 0.f;
      ++nunit;
      walk_next(cw);
    }
  }
  if (producer && *abort_flag) {
    // let copies already in flight land before the CTA's shared memory goes away
    for (int t = max(0, pstep - STAGES); t < pstep; ++t)
      (void)mbar_wait(&full[t % STAGES], (uint32_t)(t / STAGES) & 1u, nullptr);
  }
}

// CTA shapes. Up to 4 tokens, 8 warps and two CTAs per SM (they drift apart, so
// one's loads and waits overlap the other's arithmetic): K1 two tiles per warp
// (gate and up of the same rows) sharing the B operand, gate and up boxes of 16
// rows x 8 superblocks, two stages; K2 one 16-row tile per unit and warp (boxes
// of 16 rows x 8 superblocks, three stages), which gives enough units to leave K
// unsplit on large layers, so no chunk sum follows. 5-16 tokens (two to four token tiles;
// B read through L1, so that a thread fits in 128 registers): small CTAs, many
// per SM, which keeps 16 warps per SM without tying them to one CTA barrier per
// step; K1 4 warps (gate or up tile at 2 superblocks), boxes of 16 rows x 2
// superblocks, two stages, four CTAs per SM; K2 2 warps, boxes of 16 rows x 2
// superblocks, three stages, eight CTAs per SM.
template <bool GATEUP, int NT> struct Shape;
template <> struct Shape<true, 1> { static constexpr int COMBOS = 2, TPW = 2, SLICES = 8, STAGES = 2, CPS = 2; };
template <> struct Shape<false, 1> { static constexpr int COMBOS = 1, TPW = 1, SLICES = 8, STAGES = 3, CPS = 2; };
template <> struct Shape<true, 2> { static constexpr int COMBOS = 2, TPW = 1, SLICES = 2, STAGES = 2, CPS = 4; };
template <> struct Shape<false, 2> { static constexpr int COMBOS = 1, TPW = 1, SLICES = 2, STAGES = 3, CPS = 8; };
template <> struct Shape<true, 3> : Shape<true, 2> {};
template <> struct Shape<false, 3> : Shape<false, 2> {};
template <> struct Shape<true, 4> : Shape<true, 2> {};
template <> struct Shape<false, 4> : Shape<false, 2> {};

struct ShapeVals {
  int slices, combos, cps;
};
template <bool GATEUP, int NT>
constexpr ShapeVals shape_vals() {
  return {Shape<GATEUP, NT>::SLICES, Shape<GATEUP, NT>::COMBOS, Shape<GATEUP, NT>::CPS};
}
template <bool GATEUP>
ShapeVals shape_of(int nt) {
  return nt == 1   ? shape_vals<GATEUP, 1>()
         : nt == 2 ? shape_vals<GATEUP, 2>()
         : nt == 3 ? shape_vals<GATEUP, 3>()
                   : shape_vals<GATEUP, 4>();
}
template <bool GATEUP>
cudaError_t launch_gemv_nt(int nt, const CUtensorMap& t0, const CUtensorMap& t1, const GemvParams& P, int grid,
                           cudaStream_t s);

template <bool GATEUP, int NT, bool DIAG>
constexpr size_t gemv_smem() {
  using S = Shape<GATEUP, NT>;
  constexpr size_t stage = stage_total(S::COMBOS * 16 * S::SLICES * BLK, DIAG && !GATEUP ? S::SLICES * DREC : 0);
  return S::STAGES * stage + 2 * S::STAGES * 8 + (size_t)2 * S::COMBOS * S::SLICES * 32 * NT * 2 * 4 + 16;
}

template <bool GATEUP, int NT, bool DIAG = false>
cudaError_t launch_gemv(const CUtensorMap& t0, const CUtensorMap& t1, const GemvParams& P, int grid,
                        cudaStream_t s) {
  using S = Shape<GATEUP, NT>;
  auto kern = gemv_kernel<GATEUP, NT, S::COMBOS, S::TPW, S::SLICES, S::STAGES, S::CPS, DIAG>;
  constexpr size_t smem = gemv_smem<GATEUP, NT, DIAG>();
  static uint64_t attr_set = 0;  // one bit per device
  const cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), smem, &attr_set);
  if (e != cudaSuccess) return e;
  void* args[] = {const_cast<CUtensorMap*>(&t0), const_cast<CUtensorMap*>(&t1), const_cast<GemvParams*>(&P)};
  // the one-token gate/up GEMV that builds x's fragments itself is the call's first kernel
  return launch_pdl(reinterpret_cast<const void*>(kern), dim3(grid), dim3(S::COMBOS / S::TPW * S::SLICES * 32), smem, s,
                    args, !(GATEUP && DIAG && P.x));
}

template <bool GATEUP>
cudaError_t launch_gemv_nt(int nt, const CUtensorMap& t0, const CUtensorMap& t1, const GemvParams& P, int grid,
                           cudaStream_t s) {
  return P.diag ? launch_gemv<GATEUP, 1, true>(t0, t1, P, grid, s)
         : nt == 1 ? launch_gemv<GATEUP, 1>(t0, t1, P, grid, s)
         : nt == 2 ? launch_gemv<GATEUP, 2>(t0, t1, P, grid, s)
         : nt == 3 ? launch_gemv<GATEUP, 3>(t0, t1, P, grid, s)
                   : launch_gemv<GATEUP, 4>(t0, t1, P, grid, s);
}

}  // namespace

bool decode_plan(int64_t m, int64_t hidden, int64_t inter, int num_sms, DecodePlan* p) {
  if (m < 1 || m > DECODE_PASS_MAX) return false;
  p->m = (int)m;
  p->hidden = (int)hidden;
  p->inter = (int)inter;
  p->nt = (int)((m + 3) / 4);
  const int nsb1 = (int)(hidden / QK), nsb2 = (int)(inter / QK);
  const bool one = p->nt == 1;
  const ShapeVals s1 = shape_of<true>(p->nt), s2 = shape_of<false>(p->nt);
  const int sl1 = s1.slices, sl2 = s2.slices, cb2 = s2.combos;
  const int nru1 = (int)(inter / 16), nru2 = (int)(hidden / (16 * cb2));
  // at most 16 chunks x 4 tokens of partial sums: with hidden, inter <= 16384 the
  // whole workspace stays under 13.1 MiB
  const int max_nks = 16 / p->nt;
  const int ctas1 = num_sms * s1.cps, ctas2 = num_sms * s2.cps;
  choose_split((nsb1 + sl1 - 1) / sl1, nru1, ctas1, max_nks, &p->nks1, &p->kc1);
  // K2 leaves K unsplit when its row units alone fill half the CTA slots (no chunk sum to follow)
  choose_split((nsb2 + sl2 - 1) / sl2, nru2, ctas2, (one && 2 * nru2 >= ctas2) ? 1 : max_nks, &p->nks2, &p->kc2);
  p->grid1 = (int)std::min<int64_t>(ctas1, (int64_t)p->nks1 * nru1);
  p->grid2 = (int)std::min<int64_t>(ctas2, (int64_t)p->nks2 * nru2);
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align256(o + bytes);
    return at;
  };
  p->off_fx1 = take((size_t)nsb1 * 16 * p->nt * 32 * 8);
  p->off_fm1 = take((size_t)nsb1 * p->nt * 32 * 4);
  p->off_sc1 = take((size_t)nsb1 * sc_stride(p->nt) * 4);
  p->off_fx2 = take((size_t)nsb2 * 16 * p->nt * 32 * 8);
  p->off_fm2 = take((size_t)nsb2 * p->nt * 32 * 4);
  p->off_sc2 = take((size_t)nsb2 * sc_stride(p->nt) * 4);
  p->off_p1 = take((size_t)p->nks1 * 2 * m * inter * 4);
  p->off_p2 = take((size_t)p->nks2 * m * hidden * 4);  // also the float32 y of a bf16-output call
  p->ws_bytes = o;
  return true;
}

bool device_resident(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

int decode_kernels(const DecodePlan& p, bool q8, int ybf16, const void* x) {
  const bool no_k0 = p.m == 1 && !q8 && device_resident(x);  // K1 builds x's fragments
  return (no_k0 ? 3 : 4) + (p.nks2 > 1 || ybf16);
}

cudaError_t launch_decode(const DecodePlan& p, const void* x, int bf16, const void* wg, const void* wu, const void* wd,
                          void* y, void* ws, uint32_t* err, cudaStream_t s, const ProfileEvents& prof, int ybf16,
                          uint8_t* q8h) {
  const bool q8 = q8h != nullptr;  // activations rounded to Q8_1 (x, and h stored at q8h)
  uint8_t* W = (uint8_t*)ws;
  FragPtrs f1{(uint2*)(W + p.off_fx1), (uint32_t*)(W + p.off_fm1), (float*)(W + p.off_sc1)};
  FragPtrs f2{(uint2*)(W + p.off_fx2), (uint32_t*)(W + p.off_fm2), (float*)(W + p.off_sc2)};
  float* p1 = (float*)(W + p.off_p1);
  const bool k3 = p.nks2 > 1 || ybf16;  // K3 sums the chunks and/or stores bf16
  float* p2 = k3 ? (float*)(W + p.off_p2) : (float*)y;
  const int nsb1 = p.hidden / QK, nsb2 = p.inter / QK;
  const ShapeVals s1 = shape_of<true>(p.nt), s2 = shape_of<false>(p.nt);
  const int sl1 = s1.slices, sl2 = s2.slices, cb2 = s2.combos;
  CUtensorMap mg, mu, md;
  if (!weight_map(&mg, wg, p.inter, nsb1, 16, sl1) || !weight_map(&mu, wu, p.inter, nsb1, 16, sl1) ||
      !weight_map(&md, wd, p.hidden, nsb2, 16 * cb2, sl2))
    return cudaErrorInvalidValue;

  // One token on the float32 path: block-diagonal operands (see frag_token_diag). With x in
  // device memory K1 builds x's fragments itself and is the call's first kernel (no K0).
  // With x in host memory K0 reads it once (every K1 warp reading it across the host link
  // cost several microseconds) and writes the records K1 reads.
  const bool diag = p.m == 1 && !q8;
  const bool k0 = !diag || !device_resident(x);
  // K0: not a dependent launch, so it also orders this call after the previous one on the stream
  prof.before(0, s);
  if (diag && k0 && bf16)
    prep_x_kernel<__nv_bfloat16, false, true><<<nsb1, 32, 0, s>>>((const __nv_bfloat16*)x, p.hidden, 1, 1, f1);
  else if (diag && k0)
    prep_x_kernel<float, false, true><<<nsb1, 32, 0, s>>>((const float*)x, p.hidden, 1, 1, f1);
  else if (!diag) {
    const int nw = 128 * p.nt;  // one warp per token slot
    if (bf16 && q8)
      prep_x_kernel<__nv_bfloat16, true><<<nsb1, nw, 0, s>>>((const __nv_bfloat16*)x, p.hidden, p.m, p.nt, f1);
    else if (bf16)
      prep_x_kernel<__nv_bfloat16, false><<<nsb1, nw, 0, s>>>((const __nv_bfloat16*)x, p.hidden, p.m, p.nt, f1);
    else if (q8)
      prep_x_kernel<float, true><<<nsb1, nw, 0, s>>>((const float*)x, p.hidden, p.m, p.nt, f1);
    else
      prep_x_kernel<float, false><<<nsb1, nw, 0, s>>>((const float*)x, p.hidden, p.m, p.nt, f1);
  }
  prof.after(0, s);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  GemvParams g1{p.inter, nsb1, p.m, p.kc1, p.nks1, f1, p1, err, diag, k0 ? nullptr : x, bf16};
  prof.before(1, s);
  e = launch_gemv_nt<true>(p.nt, mg, mu, g1, p.grid1, s);
  prof.after(1, s);
  if (e != cudaSuccess) return e;

  {
    const float* pp = p1;
    int nks = p.nks1, m = p.m, inter = p.inter, nt = p.nt;
    FragPtrs f = f2;
    uint8_t* hq = q8h;
    float2* hds = q8 ? (float2*)(q8h + (size_t)p.m * p.inter) : nullptr;
    void* args[] = {&pp, &nks, &m, &inter, &nt, &f, &hq, &hds};
    const void* fn = q8     ? reinterpret_cast<const void*>(finish_gateup_kernel<true>)
                     : diag ? reinterpret_cast<const void*>(finish_gateup_kernel<false, true>)
                            : reinterpret_cast<const void*>(finish_gateup_kernel<false>);
    prof.before(2, s);
    e = launch_pdl(fn, dim3(nsb2), dim3(diag ? 32 : 128 * p.nt), 0, s, args);
    prof.after(2, s);
    if (e != cudaSuccess) return e;
  }

  GemvParams g2{p.hidden, nsb2, p.m, p.kc2, p.nks2, f2, p2, err, diag, nullptr, 0};
  prof.before(3, s);
  e = launch_gemv_nt<false>(p.nt, md, md, g2, p.grid2, s);
  prof.after(3, s);
  if (e != cudaSuccess) return e;

  prof.before(4, s);  // the down-chunk sum (absent when K is not split)
  if (k3) e = launch_finish_down(p2, p.nks2, (int64_t)p.m * p.hidden, y, ybf16, s);
  prof.after(4, s);
  return e;
}

}  // namespace q4k
