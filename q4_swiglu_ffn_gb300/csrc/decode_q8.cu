// Decode regime (m = 1..16 tokens per pass) with Q8_1 activations, on sm_103a. One or two
// tokens run the integer kernels of this file; three to sixteen run the float32
// decode path's kernels (decode.cu) on Q8_1-rounded x and h, whose fp16 tensor
// cores take 4 to 16 token columns at once where the integer epilogue per
// 32-weight sub-block would dominate.
//
//   K0  q8_1(x):           x [m][hidden] -> planar Q8_1 (the stand-alone quantizer's kernel)
//   K1  gemv_q8<gate/up>:  partial g = Wg.xq and u = Wu.xq per K-chunk, one pass over both
//   K1b finish_gateup_q8:  g, u = sum of the chunks; h = silu(g) * u -> planar Q8_1
//   K2  gemv_q8<down>:     partial y = Wd.hq per K-chunk
//   K3  finish_down:       y = sum of the chunks (only when K is split)
// K1, K1b, K2 and K3 are launched with programmatic dependent launch.
// Source: realizar src/cuda/executor/layers/ffn.rs, fused_ffn_swiglu_gpu_true_dp4a
// (x quantized to Q8_1 once and shared by the gate and up GEMVs, integer dot
// products of the 4-bit quants with the int8 activations, h re-quantized to
// Q8_1 before the down GEMV); the per-block correction is that of
// spark_model/layers/ops/q4k_mmq.rs, q4k_mmq_gemm (d, dmin, 6-bit scales and
// mins applied to the integer sums).
//
// Arithmetic. For one weight row, sub-block j (32 weights: 4-bit q, 6-bit scale
// sc_j and min m_j, block factors d and dmin) against the Q8_1 block with int8
// quants q8, scale d8_j and s8_j = d8_j * sum(q8):
//     dot = d * sum_j sc_j * d8_j * I_j  -  dmin * sum_j m_j * s8_j,
//     I_j = sum_i q_i * q8_i   (an exact int32).
// I_j comes from dp4a (four u8 x s8 products and a 32-bit add per instruction).
// A 32-bit word of quants holds, in its low nibbles, 4 consecutive weights of
// sub-block 2G and, in its high nibbles, the 4 weights of sub-block 2G+1 at the
// same positions: the low nibbles are masked out, the high nibbles are masked
// in place (16 q) and the factor 16 is shifted out of the integer sum exactly.
// |I_j * sc_j| <= 32 * 15 * 127 * 63 < 2^24, so its conversion to float32 is exact;
// the remaining arithmetic is float32.
//
// Streaming is that of the float32 decode GEMV: a CTA walks a contiguous range
// of units (K-chunk x row unit), loading per step one 3-D TMA box per matrix
// (SLICES superblocks x the unit's rows, superblock-major, 144 bytes per row)
// into a ring of stages; each warp takes TPW 16-row tiles at one superblock of
// the step. Lane (g, tig) owns rows g and g+8 of each tile and quant group tig
// (sub-blocks 2 tig and 2 tig + 1), so its quant bytes per row (32) and its
// activation bytes per token (64, plus two {d8, s8} pairs) are contiguous. At
// the end of a unit the four lanes of a row are summed by shuffles and an owner
// warp sums the SLICES partial dot products through shared memory; the chunks
// are summed by K1b / K3 in chunk order, so results are deterministic.
#include <algorithm>
#include <cmath>

#include "common.cuh"
#include "gemv_stream.cuh"
#include "kernels.h"
#include "q8_1.cuh"

namespace q4k {

namespace {

struct GemvQ8Params {
  int rows;            // output rows of each matrix
  int nsb;             // superblocks along K
  int m;               // tokens
  int gpc;             // superblock groups per K-chunk
  int nks;             // K-chunks
  const uint8_t* xq;   // Q8_1 quants of the input [m][nsb * 256]
  const float4* xds;   // {d8, s8} of blocks 2i and 2i+1 of the input: [m][nsb * 4]
  float* out;          // chunk sums: [nks][2][m][rows] (gate/up) or [nks][m][rows] (down)
  uint32_t* err;
  const void* x;       // gate/up: x itself, quantized in the kernel (or null: xq, xds from K0)
  int xbf16;           // ... as bf16 (else float32)
};

// One warp: Q8_1 of token tt's superblock sb of x, as lane (g, tig) of the GEMV reads it from
// K0's planar output: the 64 quants of blocks 2 tig and 2 tig + 1 (w) and their {d8, s8}
// (d). Lane L quantizes x[8L .. 8L+7] (q8_1_block8, the stand-alone quantizer's rule, so the
// bytes are K0's); the lanes of quant group tig then gather lanes 8 tig .. 8 tig + 7.
__device__ __forceinline__ void q8_frags_from_x(const void* x, int xbf16, int64_t kq, int tt, int sb, uint4 w[4],
                                                float4& d) {
  const int lane = threadIdx.x & 31, tig = lane & 3;
  const int64_t off = (int64_t)tt * kq + (int64_t)sb * QK + lane * 8;
  float v[8];
  if (xbf16) {
    const uint4 a = *reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(x) + off);
    const uint32_t u[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(u[i] << 16);
      v[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
    }
  } else {
    const float4* p = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(x) + off);
    const float4 a = p[0], b = p[1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
  int8_t q[8];
  float dd, ss;
  q8_1_block8(v, q, dd, ss);
  const uint32_t w0 = (uint32_t)(uint8_t)q[0] | (uint32_t)(uint8_t)q[1] << 8 | (uint32_t)(uint8_t)q[2] << 16 |
                      (uint32_t)(uint8_t)q[3] << 24;
  const uint32_t w1 = (uint32_t)(uint8_t)q[4] | (uint32_t)(uint8_t)q[5] << 8 | (uint32_t)(uint8_t)q[6] << 16 |
                      (uint32_t)(uint8_t)q[7] << 24;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int la = 8 * tig + 2 * i;
    w[i].x = __shfl_sync(0xffffffffu, w0, la);
    w[i].y = __shfl_sync(0xffffffffu, w1, la);
    w[i].z = __shfl_sync(0xffffffffu, w0, la + 1);
    w[i].w = __shfl_sync(0xffffffffu, w1, la + 1);
  }
  d.x = __shfl_sync(0xffffffffu, dd, 8 * tig);
  d.y = __shfl_sync(0xffffffffu, ss, 8 * tig);
  d.z = __shfl_sync(0xffffffffu, dd, 8 * tig + 4);
  d.w = __shfl_sync(0xffffffffu, ss, 8 * tig + 4);
}

// dp4a with an unsigned first and a signed second operand.
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Shared memory of a CTA: the stage ring, the stage barriers, the unit-end
// reduction slots and the abort flag.
template <bool GATEUP, int MT, int COMBOS, int TPW, int SLICES, int STAGES>
struct Q8Smem {
  static constexpr int WARPS = COMBOS / TPW * SLICES;
  static constexpr int RU = GATEUP ? 16 : 16 * COMBOS;
  static constexpr int BOX_BYTES = SLICES * RU * BLK;
  static constexpr int STAGE_BYTES = (GATEUP ? 2 : 1) * BOX_BYTES;
  static constexpr int PER_WARP = 8 * TPW * MT * 2;
  static constexpr size_t OFF_BAR = (size_t)STAGES * STAGE_BYTES;
  static constexpr size_t OFF_RED = OFF_BAR + 2 * STAGES * 8;
  static constexpr size_t OFF_FLAG = OFF_RED + (size_t)2 * WARPS * PER_WARP * 4;
  static constexpr size_t BYTES = OFF_FLAG + 16;
};

// COMBOS 16-row tiles per superblock and step (gate and up of the same rows, or
// COMBOS consecutive tiles of W_down); each warp takes TPW of them at one of the
// SLICES superblocks. MT (1 or 2) >= m tokens, whose activations for the warp's
// superblock stay in registers; dp4a forms the integer sums.
template <bool GATEUP, int MT, int COMBOS, int TPW, int SLICES, int STAGES, int CPS>
__global__ void __launch_bounds__(COMBOS / TPW * SLICES * 32, CPS)
    gemv_q8_kernel(const __grid_constant__ CUtensorMap tm0, const __grid_constant__ CUtensorMap tm1,
                   const GemvQ8Params P) {
  constexpr int TG = COMBOS / TPW;  // tile groups
  constexpr int WARPS = TG * SLICES;
  static_assert(COMBOS % TPW == 0, "tiles split evenly over warps");
  constexpr int ROWS = 16;
  constexpr int RU = GATEUP ? ROWS : ROWS * COMBOS;  // output rows of a unit (per matrix)
  constexpr int MATS = GATEUP ? 2 : 1;
  constexpr int BOX_BYTES = SLICES * RU * BLK;      // one box: [SLICES][RU rows][144 B]
  constexpr int STAGE_BYTES = MATS * BOX_BYTES;
  constexpr int PER_WARP = 8 * TPW * MT * 2;         // reduction slot: [8 g][TPW][MT][2 rows]
  using L = Q8Smem<GATEUP, MT, COMBOS, TPW, SLICES, STAGES>;
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* empty = full + STAGES;
  float* red = reinterpret_cast<float*>(smem + L::OFF_RED);  // [2][WARPS][PER_WARP]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_FLAG);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, tig = lane & 3;
  const int tgrp = warp % TG, slice = warp / TG;
  const int nru = P.rows / RU;
  const int ngroups = (P.nsb + SLICES - 1) / SLICES;
  const int U = P.nks * nru;
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
  auto produce = [&]() -> bool {  // issue the next step's loads; false on a timed-out wait
    const int s = pstep % STAGES;
    if (pstep >= STAGES && !mbar_wait(&empty[s], (uint32_t)((pstep / STAGES) - 1) & 1u, P.err)) return false;
    uint8_t* st = smem + s * STAGE_BYTES;
    mbar_arrive_expect_tx(&full[s], STAGE_BYTES);
    tma_box3(st, &tm0, pw.ru * RU, pw.g * SLICES, &full[s], pol);
    if (GATEUP) tma_box3(st + BOX_BYTES, &tm1, pw.ru * RU, pw.g * SLICES, &full[s], pol);
    ++pstep;
    if (++pw.g == pw.ge) walk_next(pw);
    return true;
  };
  bool failed = false;  // warp-uniform once the loop starts
  if (producer) {
    for (int i = 0; i < STAGES - 1 && pw.u < u1; ++i)
      if (!produce()) {
        failed = true;
        *abort_flag = 1;
        break;
      }
  }
  failed = __any_sync(0xffffffffu, failed);
  pdl_launch_dependents();
  pdl_wait();  // the Q8_1 input comes from the previous kernel

  // Sub-blocks 2*tig and 2*tig+1 of a row are this lane's. One byte permute
  // gathers, for both, the bytes their 6-bit scales (mins) are made of into the
  // two 16-bit halves of a word; masks and shifts that depend only on tig then
  // finish them: for sub-blocks 0-3 a scale (min) is the low 6 bits of byte j
  // (j+4); for 4-7 it is the low (high) nibble of byte j+4 with the top two bits
  // of byte j-4 (j) above it.
  const uint32_t bb = 2u * (uint32_t)(tig & 1);
  const bool shigh = tig >= 2;
  const uint32_t sel = shigh ? ((4u + bb) | bb << 4 | (5u + bb) << 8 | (bb + 1u) << 12)
                             : (bb | bb << 4 | (bb + 1u) << 8 | (bb + 1u) << 12);
  const uint32_t mL = shigh ? 0x000F000Fu : 0x003F003Fu, mH = shigh ? 0x00300030u : 0u, sM = shigh ? 4u : 0u;
  const int64_t kq = (int64_t)P.nsb * QK;  // activation bytes per token

  // ---------------------------------------------------------------- consumer (all warps)
  Walk cw;
  walk_start(cw, u0);
  int nunit = 0, cstep = 0;
  float acc[TPW][MT][2];
#pragma unroll
  for (int t = 0; t < TPW; ++t)
#pragma unroll
    for (int k = 0; k < MT; ++k) acc[t][k][0] = acc[t][k][1] = 0.f;
  static_assert(MT <= 2, "one or two tokens");
  uint4 xa[MT][4];  // activation words of sub-block 2 tig (xa[.][0..1]) and 2 tig + 1 (xa[.][2..3])
  float4 xd[MT];    // {d8, s8} of those two blocks
  int csb = -1;
  auto load_x = [&](int tok, int sb, uint4 w[4], float4& d) {
    const int tt = min(tok, P.m - 1);  // padding tokens read a real token; their sums are never stored
    if (GATEUP && P.x) {  // warp-uniform: quantize x here (no K0)
      q8_frags_from_x(P.x, P.xbf16, kq, tt, sb, w, d);
      return;
    }
    const uint4* xp = reinterpret_cast<const uint4*>(P.xq + (int64_t)tt * kq + (int64_t)sb * QK + 64 * tig);
#pragma unroll
    for (int i = 0; i < 4; ++i) w[i] = xp[i];
    d = P.xds[((int64_t)tt * P.nsb + sb) * 4 + tig];
  };
  if (GATEUP && P.x) {  // the first superblock's activations, while the first weights arrive
    const int sb0 = cw.g * SLICES + slice;
    if (cw.u < u1 && sb0 < min(P.nsb, (cw.ks + 1) * P.gpc * SLICES)) {
#pragma unroll
      for (int k = 0; k < MT; ++k) load_x(k, sb0, xa[k], xd[k]);
      csb = sb0;
    }
  }

#pragma unroll 1
  while (cw.u < u1) {
    bool pf = false;
    if (producer && !failed && pw.u < u1) pf = !produce();
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
    if (!failed && sb < chunk_end) {
      // ------------------------------------------ TPW 16-row tiles of one superblock
      uint4 q0[TPW][2], q1[TPW][2];
      int scl[TPW][2], sch[TPW][2];
      float mnl[TPW][2], mnh[TPW][2], dd[TPW][2], dm[TPW][2];
#pragma unroll
      for (int t = 0; t < TPW; ++t) {
        const int cb = tgrp * TPW + t;
        const uint8_t* base = smem + s * STAGE_BYTES + (GATEUP ? cb * BOX_BYTES + slice * RU * BLK
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
          const uint32_t vs = prmt(hd.y, hd.w, sel), vm = prmt(hd.z, hd.w, sel);
          const uint32_t scp = (vs & mL) | ((vs >> 10) & mH);
          const uint32_t mnp = ((vm >> sM) & mL) | ((vm >> 10) & mH);
          scl[t][r] = (int)(scp & 0xFFFFu);
          sch[t][r] = (int)(scp >> 16);
          // small non-negative integers to float: 2^23 + v has v in its mantissa
          mnl[t][r] = __uint_as_float(prmt(mnp, 0x4B000000u, 0x7440u)) - 8388608.f;
          mnh[t][r] = __uint_as_float(prmt(mnp, 0x4B000000u, 0x7442u)) - 8388608.f;
        }
      }
      if (sb != csb) {
#pragma unroll
        for (int k = 0; k < MT; ++k) load_x(k, sb, xa[k], xd[k]);
        csb = sb;
      }
#pragma unroll
      for (int k = 0; k < MT; ++k) {
        uint4 xw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) xw[i] = xa[k][i];
        const float4 dsv = xd[k];
        const uint32_t xl[8] = {xw[0].x, xw[0].y, xw[0].z, xw[0].w, xw[1].x, xw[1].y, xw[1].z, xw[1].w};
        const uint32_t xh[8] = {xw[2].x, xw[2].y, xw[2].z, xw[2].w, xw[3].x, xw[3].y, xw[3].z, xw[3].w};
#pragma unroll
        for (int t = 0; t < TPW; ++t)
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const uint32_t w[8] = {q0[t][r].x, q0[t][r].y, q0[t][r].z, q0[t][r].w,
                                   q1[t][r].x, q1[t][r].y, q1[t][r].z, q1[t][r].w};
            int il = 0, ih = 0;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              il = dp4a_us(w[c] & 0x0F0F0F0Fu, xl[c], il);
              ih = dp4a_us(w[c] & 0xF0F0F0F0u, xh[c], ih);
            }
            // |I * scale| < 2^22: 1.5 * 2^23 + v holds v exactly in its mantissa
            const float fl = __int_as_float(il * scl[t][r] + 0x4B400000) - 12582912.f;
            const float fh = __int_as_float((ih >> 4) * sch[t][r] + 0x4B400000) - 12582912.f;
            const float sm = fmaf(fl, dsv.x, fh * dsv.z);
            const float mn = fmaf(mnl[t][r], dsv.y, mnh[t][r] * dsv.w);
            acc[t][k][r] = fmaf(dd[t][r], sm, fmaf(-dm[t][r], mn, acc[t][k][r]));
          }
      }
    }
    __syncwarp();
    if (lane == 0 && !failed) mbar_arrive(&empty[s]);
    ++cstep;
    // ------------------------------------------------ end of a unit
    if (++cw.g == cw.ge) {
      // the four lanes of a row hold different sub-blocks: sum them; lane tig
      // then writes the tokens congruent to tig mod 4
      float* slot = red + (size_t)((nunit & 1) * WARPS + warp) * PER_WARP + g * TPW * MT * 2;
#pragma unroll
      for (int t = 0; t < TPW; ++t)
#pragma unroll
        for (int k = 0; k < MT; ++k)
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            float v = acc[t][k][r];
            v += __shfl_xor_sync(0xffffffffu, v, 1);
            v += __shfl_xor_sync(0xffffffffu, v, 2);
            if ((k & 3) == tig) slot[(t * MT + k) * 2 + r] = v;
          }
      __syncwarp();
      asm volatile("bar.sync 1, %0;" ::"r"(WARPS * 32) : "memory");
      if (warp == 1 + (nunit % (WARPS - 1)) && !*abort_flag) {
        // owner: sum the SLICES partial dot products of every tile and store this chunk's sums
        const float* rs = red + (size_t)(nunit & 1) * WARPS * PER_WARP + g * TPW * MT * 2;
        const int row0 = cw.ru * RU;
#pragma unroll
        for (int cb = 0; cb < COMBOS; ++cb)
#pragma unroll
          for (int k = 0; k < MT; ++k) {
            if ((k & 3) != tig || k >= P.m) continue;
            float s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int sl = 0; sl < SLICES; ++sl) {
              const float* q = rs + (size_t)(sl * TG + cb / TPW) * PER_WARP + ((cb % TPW) * MT + k) * 2;
              s0 += q[0];
              s1 += q[1];
            }
            float* o = GATEUP ? P.out + (((int64_t)cw.ks * 2 + cb) * P.m + k) * P.rows + row0
                              : P.out + ((int64_t)cw.ks * P.m + k) * P.rows + row0 + ROWS * cb;
            o[g] = s0;
            o[g + 8] = s1;
          }
      }
#pragma unroll
      for (int t = 0; t < TPW; ++t)
#pragma unroll
        for (int k = 0; k < MT; ++k) acc[t][k][0] = acc[t][k][1] = 0.f;
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

// CTA shapes: 8 warps, two CTAs per SM. K1: gate and up boxes of 16 rows x 8
// superblocks, two tiles per warp (gate and up), two stages. K2: one tile per warp,
// boxes of 16 rows x 8 superblocks, three stages, and K left unsplit when the row
// units fill half the CTA slots (no chunk sum follows).
template <bool GATEUP, int MT> struct ShapeQ8;
template <int MT> struct ShapeQ8<true, MT> {
  static constexpr int COMBOS = 2, TPW = 2, SLICES = 8, STAGES = 2, CPS = 2;
};
template <int MT> struct ShapeQ8<false, MT> {
  static constexpr int COMBOS = 1, TPW = 1, SLICES = 8, STAGES = 3, CPS = 2;
};

template <bool GATEUP, int MT>
constexpr size_t gemv_q8_smem() {
  using S = ShapeQ8<GATEUP, MT>;
  return Q8Smem<GATEUP, MT, S::COMBOS, S::TPW, S::SLICES, S::STAGES>::BYTES;
}

template <bool GATEUP, int MT>
cudaError_t launch_gemv_q8(const CUtensorMap& t0, const CUtensorMap& t1, const GemvQ8Params& P, int grid,
                           cudaStream_t s) {
  using S = ShapeQ8<GATEUP, MT>;
  auto kern = gemv_q8_kernel<GATEUP, MT, S::COMBOS, S::TPW, S::SLICES, S::STAGES, S::CPS>;
  constexpr size_t smem = gemv_q8_smem<GATEUP, MT>();
  static uint64_t attr_set = 0;  // one bit per device
  const cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), smem, &attr_set);
  if (e != cudaSuccess) return e;
  void* args[] = {const_cast<CUtensorMap*>(&t0), const_cast<CUtensorMap*>(&t1), const_cast<GemvQ8Params*>(&P)};
  // the gate/up GEMV that quantizes x itself is the call's first kernel
  return launch_pdl(reinterpret_cast<const void*>(kern), dim3(grid), dim3(S::COMBOS / S::TPW * S::SLICES * 32), smem,
                    s, args, !(GATEUP && P.x));
}

template <bool GATEUP>
cudaError_t launch_gemv_q8_mt(int mt, const CUtensorMap& t0, const CUtensorMap& t1, const GemvQ8Params& P, int grid,
                              cudaStream_t s) {
  return mt == 1 ? launch_gemv_q8<GATEUP, 1>(t0, t1, P, grid, s) : launch_gemv_q8<GATEUP, 2>(t0, t1, P, grid, s);
}

template <bool GATEUP>
void shape_q8(int mt, int* combos, int* slices, int* cps) {
  auto get = [&](auto tag) {
    using S = decltype(tag);
    *combos = S::COMBOS;
    *slices = S::SLICES;
    *cps = S::CPS;
  };
  if (mt == 1)
    get(ShapeQ8<GATEUP, 1>{});
  else
    get(ShapeQ8<GATEUP, 2>{});
}

// silu(z) = z * sigmoid(z), with t = e^-|z| in (0, 1]: sigmoid is 1 / (1 + t) for z >= 0
// and t / (1 + t) below. Nothing overflows, the divisor is in [1, 2] (where __fdividef
// is within 2 ulp), and there is no branch: the IEEE division's slow path had serialised
// the 8 values of a lane and made this the longest step of the SwiGLU kernel.
__device__ __forceinline__ float silu_f(float z) {
  const float t = expf(-fabsf(z));  // in (0, 1]
  return z * __fdividef(z >= 0.f ? 1.0f : t, 1.0f + t);
}

__device__ __forceinline__ void load8f(const float* p, float v[8]) {
  const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// K1b: one warp per 256 values of h (8 Q8_1 blocks), 8 values per lane. Sums
// the gate/up chunks in order, applies SwiGLU and quantizes h to planar Q8_1.
__global__ void finish_gateup_q8_kernel(const float* __restrict__ part, int nks, int m, int inter,
                                        uint8_t* __restrict__ hq, float2* __restrict__ hds) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 8;  // m * inter is a multiple of 256
  const int t = (int)(i / inter);
  const int64_t c = i - (int64_t)t * inter;
  float g[8], u[8], v[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) g[j] = u[j] = 0.f;
  // Batches of 4 chunks: all of a batch's loads are issued before the first add (a loop
  // over a run-time count would wait for each load in turn); sums in chunk order.
  for (int k0 = 0; k0 < nks; k0 += 4) {
    float a[4][8], b[4][8];
#pragma unroll
    for (int jj = 0; jj < 4; ++jj)
      if (k0 + jj < nks) {
        load8f(part + (((int64_t)(k0 + jj) * 2 + 0) * m + t) * inter + c, a[jj]);
        load8f(part + (((int64_t)(k0 + jj) * 2 + 1) * m + t) * inter + c, b[jj]);
      }
#pragma unroll
    for (int jj = 0; jj < 4; ++jj)
      if (k0 + jj < nks)
#pragma unroll
        for (int j = 0; j < 8; ++j) g[j] += a[jj][j], u[j] += b[jj][j];
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) v[j] = silu_f(g[j]) * u[j];
  int8_t q[8];
  float d, s;
  q8_1_block8(v, q, d, s);
  uint2 packed;
  packed.x = (uint32_t)(uint8_t)q[0] | ((uint32_t)(uint8_t)q[1] << 8) | ((uint32_t)(uint8_t)q[2] << 16) |
             ((uint32_t)(uint8_t)q[3] << 24);
  packed.y = (uint32_t)(uint8_t)q[4] | ((uint32_t)(uint8_t)q[5] << 8) | ((uint32_t)(uint8_t)q[6] << 16) |
             ((uint32_t)(uint8_t)q[7] << 24);
  *reinterpret_cast<uint2*>(hq + i) = packed;
  if ((threadIdx.x & 3) == 0) hds[i / Q8B] = make_float2(d, s);
}

}  // namespace

int decode_q8_tokens(int64_t m) { return m <= 1 ? 1 : m == 2 ? 2 : m <= 4 ? 4 : 8; }

bool decode_q8_plan(int64_t m, int64_t hidden, int64_t inter, int num_sms, DecodeQ8Plan* p) {
  if (m < 1 || m > DECODE_PASS_MAX) return false;
  p->m = (int)m;
  p->hidden = (int)hidden;
  p->inter = (int)inter;
  p->mt = decode_q8_tokens(m);
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align256(o + bytes);
    return at;
  };
  p->fpath = p->mt > 2;
  if (p->fpath) {
    // 3-16 tokens: the float32 path's GEMVs (fp16 tensor cores, 4 to 16 token columns) on
    // Q8_1-rounded x and h beat the integer kernels here, whose every 32-weight
    // sub-block needs its own scale and min epilogue
    if (!decode_plan(m, hidden, inter, num_sms, &p->fp)) return false;
    p->nks1 = p->fp.nks1, p->nks2 = p->fp.nks2;
    p->off_xq = 0;
    p->off_hq = take((size_t)m * inter + (size_t)m * (inter / Q8B) * 8);
    p->off_fp = take(p->fp.ws_bytes);
    p->off_p1 = p->off_p2 = 0;
    p->ws_bytes = o;
    return true;
  }
  const int nsb1 = (int)(hidden / QK), nsb2 = (int)(inter / QK);
  int cb1, sl1, cps1, cb2, sl2, cps2;
  shape_q8<true>(p->mt, &cb1, &sl1, &cps1);
  shape_q8<false>(p->mt, &cb2, &sl2, &cps2);
  const int nru1 = (int)(inter / 16), nru2 = (int)(hidden / (16 * cb2));
  const int max_nks = 16;
  choose_split((nsb1 + sl1 - 1) / sl1, nru1, num_sms * cps1, max_nks, &p->nks1, &p->kc1);
  choose_split((nsb2 + sl2 - 1) / sl2, nru2, num_sms * cps2, 2 * nru2 >= num_sms * cps2 ? 1 : max_nks,
               &p->nks2, &p->kc2);
  p->grid1 = (int)std::min<int64_t>((int64_t)num_sms * cps1, (int64_t)p->nks1 * nru1);
  p->grid2 = (int)std::min<int64_t>((int64_t)num_sms * cps2, (int64_t)p->nks2 * nru2);
  p->off_fp = 0;
  p->off_xq = take((size_t)m * hidden + (size_t)m * (hidden / Q8B) * 8);
  p->off_hq = take((size_t)m * inter + (size_t)m * (inter / Q8B) * 8);
  p->off_p1 = take((size_t)p->nks1 * 2 * m * inter * 4);
  p->off_p2 = take((size_t)p->nks2 * m * hidden * 4);  // also the float32 y of a bf16-output call
  p->ws_bytes = o;
  return true;
}

int decode_q8_kernels(const DecodeQ8Plan& p, const void* x) {
  if (p.fpath) return decode_kernels(p.fp, true, 0, x);
  return (device_resident(x) ? 3 : 4) + (p.nks2 > 1);  // K0 only for x in host memory
}

cudaError_t launch_decode_q8(const DecodeQ8Plan& p, const void* x, int bf16, const void* wg, const void* wu,
                             const void* wd, void* y, void* ws, uint32_t* err, cudaStream_t s,
                             const ProfileEvents& prof, int ybf16) {
  uint8_t* W = (uint8_t*)ws;
  if (p.fpath) return launch_decode(p.fp, x, bf16, wg, wu, wd, y, W + p.off_fp, err, s, prof, ybf16, W + p.off_hq);
  uint8_t* xq = W + p.off_xq;
  uint8_t* hq = W + p.off_hq;
  const float4* xds = (const float4*)(xq + (size_t)p.m * p.hidden);
  float2* hds = (float2*)(hq + (size_t)p.m * p.inter);
  float* p1 = (float*)(W + p.off_p1);
  const bool k3 = p.nks2 > 1 || ybf16;  // K3 sums the chunks and/or stores bf16
  float* p2 = k3 ? (float*)(W + p.off_p2) : (float*)y;
  const int nsb1 = p.hidden / QK, nsb2 = p.inter / QK;
  int cb1, sl1, cps1, cb2, sl2, cps2;
  shape_q8<true>(p.mt, &cb1, &sl1, &cps1);
  shape_q8<false>(p.mt, &cb2, &sl2, &cps2);
  CUtensorMap mg, mu, md;
  if (!weight_map(&mg, wg, p.inter, nsb1, 16, sl1) || !weight_map(&mu, wu, p.inter, nsb1, 16, sl1) ||
      !weight_map(&md, wd, p.hidden, nsb2, 16 * cb2, sl2))
    return cudaErrorInvalidValue;

  // K0: not a dependent launch, so it also orders this call after the previous one on the stream.
  // With x in device memory K1 quantizes it itself and is the call's first kernel instead.
  const bool k0 = !device_resident(x);
  prof.before(0, s);
  cudaError_t e = k0 ? launch_q8_1(x, bf16, p.m, p.hidden, xq, s) : cudaSuccess;
  prof.after(0, s);
  if (e != cudaSuccess) return e;

  GemvQ8Params g1{p.inter, nsb1, p.m, p.kc1, p.nks1, xq, xds, p1, err, k0 ? nullptr : x, bf16};
  prof.before(1, s);
  e = launch_gemv_q8_mt<true>(p.mt, mg, mu, g1, p.grid1, s);
  prof.after(1, s);
  if (e != cudaSuccess) return e;

  {
    const float* pp = p1;
    int nks = p.nks1, m = p.m, inter = p.inter;
    uint8_t* hqq = hq;
    float2* hd = hds;
    void* args[] = {&pp, &nks, &m, &inter, &hqq, &hd};
    const unsigned warps = (unsigned)((int64_t)p.m * p.inter / QK);
    prof.before(2, s);
    e = launch_pdl(reinterpret_cast<const void*>(finish_gateup_q8_kernel), dim3(warps), dim3(32), 0, s, args);
    prof.after(2, s);
    if (e != cudaSuccess) return e;
  }

  GemvQ8Params g2{p.hidden, nsb2, p.m, p.kc2, p.nks2, hq, (const float4*)hds, p2, err, nullptr, 0};
  prof.before(3, s);
  e = launch_gemv_q8_mt<false>(p.mt, md, md, g2, p.grid2, s);
  prof.after(3, s);
  if (e != cudaSuccess) return e;

  prof.before(4, s);  // the down-chunk sum (absent when K is not split)
  if (k3) e = launch_finish_down(p2, p.nks2, (int64_t)p.m * p.hidden, y, ybf16, s);
  prof.after(4, s);
  return e;
}

}  // namespace q4k
