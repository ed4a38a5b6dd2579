// Prefill regime (m >= 25 tokens) of the Q4_K SwiGLU FFN on sm_103a.
//
//   P0 quant_expand(x)     x -> Q8_1 (the ABI's q8_1_quantize_act rule) -> tensor-core B
//                          operand planes (below), in one pass per token row
//   P2 mmq<gate/up>        G = deq(Wg) . deq(xq), U = deq(Wu) . deq(xq) on tcgen05,
//                          h = silu(G) * U, h -> planar Q8_1 (hq)
//   P3 expand(hq)
//   P4 mmq<down>           y = deq(Wd) . deq(hq), float32 (at small m split into K slices
//                          that fill one wave, each writing partial sums; at large m
//                          only the last, partial round of tiles is split)
//   P4b finish_tail        the split tail tiles' sum, in slice order (only then)
//   P5 finish_down         the slices' sum in slice order, and/or y stored as bf16 (only then)
// Both MMQ kernels are persistent: one CTA per SM walks the (row tile, token tile)
// items with its pipelines running on across items.
// Source: spark_model/layers/ops/q4k_mmq.rs (per-prefill activations to Q8_1,
// then the Q4_K MMQ GEMM C[m, n] = A_q8[m, k] x W_q4k[n, k]); realizar
// layers/ffn.rs, fused_ffn_swiglu_gpu_true_dp4a (x quantized to Q8_1 once for
// gate and up; the activated vector quantized again before down).
//
// Arithmetic. GB300's int8 tensor path (mma.sync s8) is slow and tcgen05 has no
// integer kind on sm_103a, so the Q4_K x Q8_1 products run on tcgen05.mma
// kind::f16 with operands that carry the integers exactly:
//   A (weights, M = 128 rows):  q * scale_j as fp16 (<= 945, exact), unpacked from
//                               the 4-bit quants by transform warps and stored
//                               straight into tensor memory (row i in TMEM lane i),
//                               so the weights never pass through shared memory.
//   B (activations, 128 tokens): v = q8 * d8 * 2^-e_t split into fp16 hi and lo
//                               (about 22 bits of v; e_t per token keeps |v| < 2^15).
//                               The stage's hi tile and lo tile lie back to back, so
//                               one N = 256 MMA takes both: D_main columns 0-127 get
//                               A . hi, 128-255 A . lo: half the MMA instructions, and
//                               half the predicate and descriptor work between them,
//                               on the one issuing thread.
// Each superblock (256 k) accumulates into D_main afresh; the epilogue warps add
// d * (D_hi + D_lo) - 64*dmin * D_min into registers, where D_min is one
// K = 16 MMA of the 6-bit mins against s8_j * 2^-(e_t+6) (hi and lo), s8_j =
// d8_j * sum(q8) of sub-block j. The closed form per output is
//   sum_b [ d_b * sum_j scale_j * sum_i q_i * v_i  -  dmin_b * sum_j min_j * s8_j ],
// i.e. the dot product of the dequantized Q4_K row with the dequantized Q8_1
// activations. The k order inside every aligned group of 8 is (0,2,1,3,4,6,5,7)
// on both operands, which is the order the nibble unpacking produces.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "gemv_stream.cuh"
#include "kernels.h"
#include "q8_1.cuh"
#include "tc05.cuh"
#include "tmap.h"

namespace q4k {

namespace {

// ------------------------------------------------------------------------- expand
// One CTA (EXP_NT threads) per token row. Writes
//   hi[t][k], lo[t][k]  fp16 planes of q8*d8*2^-e_t at permuted positions,
//   mn[t][sb*64 + 0..15] fp16 of s8_j*2^-(e_t+6): hi of the 8 sub-blocks, then lo,
//   scale[t] = 2^e_t.
// e_t = exponent(127 * max_j d8_j) - 14.

constexpr int EXP_NT = 256;  // threads of an expand CTA

// The row exponent e_t from each thread's running maximum of d8 (all EXP_NT threads call it).
__device__ __forceinline__ int row_exponent(float mx) {
  __shared__ float red[EXP_NT / 32];
  const int tid = threadIdx.x;
  mx = warp_max(mx);
  if ((tid & 31) == 0) red[tid >> 5] = mx;
  __syncthreads();
  mx = red[0];
#pragma unroll
  for (int i = 1; i < EXP_NT / 32; ++i) mx = fmaxf(mx, red[i]);
  const float top = mx * 127.f;
  return top > 0.f ? max((int)((__float_as_uint(top) >> 23) & 0xFF) - 127 - 14, -100) : 0;
}

// The planes of one row from its int8 quants qr[k] and block scales d8 (block j at
// d8[j * dstride]), given e_t.
__device__ __forceinline__ void expand_row(const int8_t* qr, const float* d8p, int dstride, int k, int e,
                                           __half* __restrict__ hr, __half* __restrict__ lr,
                                           __half* __restrict__ mr) {
  const int tid = threadIdx.x, lane = tid & 31;
  const float s = __uint_as_float((uint32_t)(127 - e) << 23);  // 2^-e
  for (int base = 0; base < k; base += EXP_NT * 8) {
    const int c = base + tid * 8;  // 8 values; one warp covers one superblock
    if (c >= k) break;             // k % 256 == 0, so whole warps leave together
    const float d8 = d8p[(c / Q8B) * dstride];
    const float d8s = d8 * s;  // exact power-of-two scaling
    const uint2 raw = *reinterpret_cast<const uint2*>(qr + c);
    int q[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      q[i] = (int)(int8_t)((raw.x >> (8 * i)) & 0xFF);
      q[4 + i] = (int)(int8_t)((raw.y >> (8 * i)) & 0xFF);
    }
    __align__(16) __half vh[8], vl[8];
    int qsum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int src = perm8(i);
      const float v = (float)q[src] * d8s;
      const __half h = __float2half_rn(v);
      vh[i] = h;
      vl[i] = __float2half_rn(fmaf((float)q[src], d8s, -__half2float(h)));
      qsum += q[i];
    }
    *reinterpret_cast<uint4*>(hr + c) = *reinterpret_cast<uint4*>(vh);
    if (lr) *reinterpret_cast<uint4*>(lr + c) = *reinterpret_cast<uint4*>(vl);
    // sub-block sums: 4 lanes per Q8_1 block
    qsum += __shfl_xor_sync(0xffffffffu, qsum, 1);
    qsum += __shfl_xor_sync(0xffffffffu, qsum, 2);
    const float d8m = d8s * 0.015625f;  // 2^-(e+6)
    const float sv = (float)qsum * d8m;
    const __half sh = __float2half_rn(sv);
    const __half sl = __float2half_rn(fmaf((float)qsum, d8m, -__half2float(sh)));
    // lane 4j holds sub-block j of this superblock
    __half* ms = mr + (int64_t)(c / QK) * 64;
    if ((lane & 3) == 0) {
      ms[lane >> 2] = sh;
      ms[8 + (lane >> 2)] = sl;
    }
    if (lane >= 16) ms[lane] = __float2half_rn(0.f);
    if (lane < 16) ms[32 + lane] = __float2half_rn(0.f), ms[48 + lane] = __float2half_rn(0.f);
  }
}

// The planes of a row already quantized to Q8_1 (h, written by the gate/up MMQ's epilogue).
__global__ void __launch_bounds__(EXP_NT) expand_kernel(const int8_t* __restrict__ qs, const float2* __restrict__ ds,
                                                     int k, __half* __restrict__ hi, __half* __restrict__ lo,
                                                     __half* __restrict__ mn, float* __restrict__ scale) {
  const int t = blockIdx.x;
  const int nblk = k / Q8B;
  const float2* dsr = ds + (int64_t)t * nblk;
  float mx = 0.f;
  for (int j = threadIdx.x; j < nblk; j += EXP_NT) mx = fmaxf(mx, fabsf(dsr[j].x));
  const int e = row_exponent(mx);
  if (threadIdx.x == 0) scale[t] = __uint_as_float((uint32_t)(127 + e) << 23);
  expand_row(qs + (int64_t)t * k, reinterpret_cast<const float*>(dsr), 2, k, e, hi + (int64_t)t * k,
             lo ? lo + (int64_t)t * k : nullptr, mn + (int64_t)t * (k / QK) * 64);
}

// x's row quantized to Q8_1 (the stand-alone quantizer's rule, q8_1_block8) and expanded in
// one pass: the quants and block scales wait in shared memory (k + k/8 bytes) while the
// CTA finds e_t. The planes are bit-identical to quantizing x and then expanding it.
template <typename T>
__global__ void __launch_bounds__(EXP_NT) quant_expand_kernel(const T* __restrict__ x, int k, __half* __restrict__ hi,
                                                           __half* __restrict__ lo, __half* __restrict__ mn,
                                                           float* __restrict__ scale) {
  extern __shared__ __align__(16) uint8_t qe_smem[];
  int8_t* sq = reinterpret_cast<int8_t*>(qe_smem);      // k quants
  float* sd = reinterpret_cast<float*>(qe_smem + k);    // k/32 block scales (k % 256 == 0: aligned)
  const int t = blockIdx.x, tid = threadIdx.x;
  const T* xr = x + (int64_t)t * k;
  float mx = 0.f;
  for (int base = 0; base < k; base += EXP_NT * 8) {
    const int c = base + tid * 8;
    if (c >= k) break;  // whole warps leave together: the quad shuffles see only live lanes
    float v[8];
    load8(xr + c, v);
    int8_t q[8];
    float d, ss;
    q8_1_block8(v, q, d, ss);
    uint2 packed;
    packed.x = (uint32_t)(uint8_t)q[0] | ((uint32_t)(uint8_t)q[1] << 8) | ((uint32_t)(uint8_t)q[2] << 16) |
               ((uint32_t)(uint8_t)q[3] << 24);
    packed.y = (uint32_t)(uint8_t)q[4] | ((uint32_t)(uint8_t)q[5] << 8) | ((uint32_t)(uint8_t)q[6] << 16) |
               ((uint32_t)(uint8_t)q[7] << 24);
    *reinterpret_cast<uint2*>(sq + c) = packed;
    if ((tid & 3) == 0) sd[c / Q8B] = d;
    mx = fmaxf(mx, d);
  }
  const int e = row_exponent(mx);  // its barrier also publishes sq and sd
  if (tid == 0) scale[t] = __uint_as_float((uint32_t)(127 + e) << 23);
  expand_row(sq, sd, 1, k, e, hi + (int64_t)t * k, lo ? lo + (int64_t)t * k : nullptr,
             mn + (int64_t)t * (k / QK) * 64);
}

// The largest k the fused x kernel takes (its shared memory stays under the 48 KB default);
// beyond it x is quantized and expanded by two kernels.
constexpr int QE_MAX_K = 43520;
inline size_t quant_expand_smem(int64_t k) { return (size_t)k + (size_t)(k / Q8B) * 4; }

// ------------------------------------------------------------------------- tcgen05 MMQ
constexpr int TM = 128;                   // weight rows per tile
constexpr int TN = 128;                   // tokens per tile
constexpr int KCH = 64;                   // k per chunk (one 128-byte swizzle atom of fp16)
constexpr int CH_PER_SB = 5;              // 4 main chunks + 1 min chunk per superblock
constexpr int STAGES = 4;
constexpr int TILE_BYTES = TM * KCH * 2;  // 16 KB
constexpr int STAGE_BYTES = 2 * TILE_BYTES;  // B hi and lo; A of the stage is in TMEM
constexpr int NWARPS = 14;                // 0 TMA, 1 MMA, 2-5 transform, 6-13 epilogue
constexpr int W_TMA = 0, W_MMA = 1, W_EPI = 6, N_EPI = 8;  // warps W_MMA + 1 .. W_EPI - 1 transform
// TMEM columns: D_main at 0 (fp32, hi products in 0-127, lo in 128-255), D_min at 256,
// the A tile of stage s at 384 + 32 s (64 fp16 per lane, two to a column). D_main and
// D_min have one buffer each: the next superblock's MMAs wait until the epilogue has
// read them.
constexpr uint32_t TMEM_COLS = 512, TM_DMIN = 256, TM_A = 384, A_COLS = KCH / 2;
static_assert(TM_A + STAGES * A_COLS <= TMEM_COLS, "A stages fit in TMEM");
// gate/up exchange: [128 rows][TN + 1] raw sums, then the TN token factors 2^e_t
constexpr int XG_BYTES = (TM * (TN + 1) + TN) * 4;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + XG_BYTES + 1024 /*align*/ + 256 /*barriers*/;

struct MmqParams {
  const uint8_t* w0;   // gate (gate/up kernel) or down
  const uint8_t* w1;   // up (gate/up kernel)
  int nsb;             // superblocks along K
  int m;               // tokens
  int ldo;             // output row length (inter for hq, hidden for y)
  int ntn;             // tiles along N (tokens)
  int ksplit;          // slices of K (down only; 1 for gate/up)
  int tiles;           // (row tile, token tile) pairs
  int nwork;           // work items: tiles x ksplit; item w is slice w / tiles of tile w % tiles
  // Without SPLIT: the tiles from `whole` on (the last, partial round of items on the
  // SMs) are split along K into tail_q > 1 slices, items whole + j for
  // j < (tiles - whole) * tail_q (slice j / (tiles - whole) of tile whole + j % (tiles -
  // whole)), which store partial tiles [tail_q][tiles - whole][TN tokens][TM rows] in tail
  // (scaled by the token factors 2^e_t; for gate/up the raw g and u, SwiGLU and Q8_1 come
  // after the slices' sum)
  int whole, tail_q;
  float* tail;
  int mt_fast;         // consecutive CTAs take consecutive row tiles (else consecutive token tiles)
  const float* tscale; // 2^e_t per token
  int8_t* hq_qs;       // gate/up: Q8_1 quants of h [m][inter]
  float2* hq_ds;       // gate/up: Q8_1 (d, s) of h [m][inter/32]
  float* y;            // down: [ksplit][m][hidden] (the slices' partial sums, or y itself when ksplit = 1)
  uint32_t* err;
};

// The transform warps load each superblock of their rows one superblock ahead into
// registers, and PF_SB superblocks ahead into L2.
constexpr int PF_SB = 3;
__device__ __forceinline__ void prefetch_row_l2(const uint8_t* p) {  // the <= 3 lines of a 144-byte block
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p + 128));
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p + BLK - 1));
}

constexpr int EPI_COLS = 8;  // accumulator columns an epilogue thread reads per TMEM load round
static_assert(EPI_COLS == 8 || EPI_COLS == 16, "tmem_ld8 or tmem_ld16");

constexpr uint32_t IDESC_MAIN = idesc_f16(TM, 2 * TN);  // B = the hi tile, then the lo tile
constexpr uint32_t IDESC_MIN = idesc_f16(TM, TN);

// silu(z) = z * sigmoid(z), with t = e^-|z| in (0, 1]: sigmoid is 1 / (1 + t) for z >= 0
// and t / (1 + t) below. Nothing overflows, the divisor is in [1, 2], where CUDA's
// __fdividef is within 2 ulp, and there is no branch (the IEEE division's slow-path
// branch kept the 32 independent values of an item from overlapping).
__device__ __forceinline__ float silu_f(float z) {
  const float t = expf(-fabsf(z));  // in (0, 1]
  return z * __fdividef(z >= 0.f ? 1.0f : t, 1.0f + t);
}

// SwiGLU + Q8_1 of a finished gate/up tile, shared by 8 warps (ew = 0..7), in
// FINAL_PIECES steps so that the epilogue can run them between the next item's
// superblock hand-overs instead of holding the MMAs up. xg holds, per tile row (0-63
// gate, 64-127 up, same 64 inter indices), the 128 token columns; ts (after xg) their
// factors 2^e_t. Each of the 256 threads owns one item (token e % 128, Q8_1 block
// e / 128 of 32 inter rows) whole: its 32 values are independent, so the max and the
// sum need no shuffles, and its 32 quants leave as two 16-byte stores. Steps 0-3 each
// turn 8 of the item's gate values into h = silu(g) * u in place (the item owns those
// rows of its column) and carry the running max; step 4 quantizes and stores. Reading
// column tt of a row, the lanes of a warp hit consecutive banks (the row pitch is 129
// words).
constexpr int FINAL_PIECES = 5;
__device__ __forceinline__ void gateup_final_piece(float* xg, const MmqParams& P, int mt, int nt, int ew, int lane,
                                                   int piece, float& amax, volatile int* abort_flag) {
  if (*abort_flag) return;
  constexpr int LD = TN + 1;
  const float* ts = xg + TM * LD;
  const int e = ew * 32 + lane, tt = e & (TN - 1), qb = e / TN;
  const int t = nt * TN + tt;
  if (t >= P.m) return;
  float* col = xg + (qb * 32) * LD + tt;  // row qb*32 + j of this item at col[j * LD]
  if (piece < 4) {
    const float sc = ts[tt];
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) {
      const int j = piece * 8 + jj;
      const float g = col[j * LD] * sc;
      const float u = col[(64 + j) * LD] * sc;
      const float h = silu_f(g) * u;
      col[j * LD] = h;
      amax = fmaxf(amax, fabsf(h));
    }
    return;
  }
  const bool nz = amax >= 0x1p-120f;  // below: zero block (127/amax would overflow)
  const float dq = nz ? __fdiv_rn(amax, 127.f) : 0.f;
  const float inv = nz ? __fdiv_rn(127.f, amax) : 0.f;
  int sum = 0;
  uint32_t pk[Q8B / 4];
#pragma unroll
  for (int w = 0; w < Q8B / 4; ++w) {
    uint32_t v = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      float rq = roundf(__fmul_rn(col[(4 * w + b) * LD], inv));
      rq = fminf(fmaxf(rq, -127.f), 127.f);
      const int qi = (int)rq;
      sum += qi;
      v |= ((uint32_t)qi & 0xFFu) << (8 * b);
    }
    pk[w] = v;
  }
  const int irow = mt * 64 + qb * 32;
  uint4* dst = reinterpret_cast<uint4*>(P.hq_qs + (int64_t)t * P.ldo + irow);  // 32-byte aligned
  dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
  P.hq_ds[(int64_t)t * (P.ldo / Q8B) + irow / Q8B] = make_float2(dq, __fmul_rn(dq, (float)sum));
}

// Persistent: one CTA per SM walks the work items blockIdx.x, + gridDim.x, ... with
// every pipeline (stages, TMEM buffers, their barrier phases) running on across
// items, so one item's last superblocks and epilogue overlap the next item's first
// loads and MMAs. SPLIT: the down projection at small m, K split into P.ksplit slices.
// TAIL: the last round's tiles may be split along K (P.tail_q); gate/up builds without it
// when there is no such round, so that its epilogue carries no partial-tile path.
template <bool GATEUP, bool SPLIT, bool TAIL>
__global__ void __launch_bounds__(NWARPS * 32, 1)
    mmq_kernel(const __grid_constant__ CUtensorMap tm_hi, const __grid_constant__ CUtensorMap tm_lo,
               const __grid_constant__ CUtensorMap tm_mn, const MmqParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  float* xg = reinterpret_cast<float*>(smem + STAGES * STAGE_BYTES);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES + XG_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* accf = empty + STAGES;  // D_main and D_min hold a finished superblock
  uint64_t* acce = accf + 1;        // ... and the epilogue has read them
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acce + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nmt = P.tiles / P.ntn;
  const int64_t rowbytes = (int64_t)P.nsb * BLK;
  struct Work {
    int nt, mt, ks, sb0, nsbl;  // token tile, row tile, K slice, its superblocks [sb0, sb0 + nsbl)
    int tl;                     // index among the split tail tiles, or -1
  };
  auto work = [&](int w) {
    Work k;
    k.tl = -1;
    k.ks = SPLIT ? w / P.tiles : 0;
    int tile = w - k.ks * P.tiles;
    if (TAIL && !SPLIT && P.tail_q > 1 && w >= P.whole) {
      const int j = w - P.whole, ntail = P.tiles - P.whole;
      k.tl = j % ntail;
      k.ks = j / ntail;
      tile = P.whole + k.tl;
    }
    k.nt = P.mt_fast ? tile / nmt : tile % P.ntn;
    k.mt = P.mt_fast ? tile % nmt : tile / P.ntn;
    const int nsl = SPLIT ? P.ksplit : k.tl >= 0 ? P.tail_q : 1;  // K slices of this item's tile
    k.sb0 = (int)((int64_t)P.nsb * k.ks / nsl);
    k.nsbl = (int)((int64_t)P.nsb * (k.ks + 1) / nsl) - k.sb0;
    return k;
  };
  // the Q4_K row of tile row r (0-63 gate, 64-127 up for gate/up), at the item's first superblock
  auto row_ptr = [&](const Work& k, int r) {
    const uint8_t* p = GATEUP ? (r < 64 ? P.w0 + (int64_t)(k.mt * 64 + r) * rowbytes
                                        : P.w1 + (int64_t)(k.mt * 64 + r - 64) * rowbytes)
                              : P.w0 + (int64_t)(k.mt * TM + r) * rowbytes;
    return p + (int64_t)k.sb0 * BLK;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 5);   // 4 transform warps + the TMA producer
      mbar_init(&empty[s], 1);  // one tcgen05.commit
    }
    mbar_init(accf, 1);      // tcgen05.commit
    mbar_init(acce, N_EPI);  // the epilogue warps
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == W_MMA) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncwarp();  // every CTA or named barrier below is entered by whole warps
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == W_TMA) {
    // ------------------------------------------------------------ TMA producer (B operand)
    if (lane == 0) {
      int q = 0;
      bool ok = true;
      for (int w = blockIdx.x; w < P.nwork && ok; w += gridDim.x) {
        const Work k = work(w);
        for (int sb = 0; sb < k.nsbl && ok; ++sb) {
          for (int c = 0; c < CH_PER_SB; ++c, ++q) {
            const int s = q % STAGES, u = q / STAGES;
            if (u > 0 && !wait_bar(&empty[s], (u - 1) & 1, abort_flag, P.err)) {
              ok = false;
              break;
            }
            uint8_t* st = smem + s * STAGE_BYTES;
            const int sba = k.sb0 + sb;
            if (c < 4) {
              mbar_arrive_expect_tx(&full[s], 2 * TILE_BYTES);
              tma_load_2d(st, &tm_hi, sba * QK + c * KCH, k.nt * TN, &full[s]);
              tma_load_2d(st + TILE_BYTES, &tm_lo, sba * QK + c * KCH, k.nt * TN, &full[s]);
            } else {
              mbar_arrive_expect_tx(&full[s], TILE_BYTES);
              tma_load_2d(st, &tm_mn, sba * KCH, k.nt * TN, &full[s]);
            }
          }
        }
      }
    }
  } else if (warp == W_MMA) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int q = 0, G = 0;  // chunks and superblocks issued so far (all items)
      bool ok = true;
      for (int w = blockIdx.x; w < P.nwork && ok; w += gridDim.x) {
        const int nsbl = work(w).nsbl;
        for (int sb = 0; sb < nsbl && ok; ++sb, ++G) {
          // one buffer: the epilogue must have read the previous superblock's D_main and D_min
          if (G >= 1 && !wait_bar(acce, (G - 1) & 1, abort_flag, P.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_main = tmem, d_min = tmem + TM_DMIN;
          for (int c = 0; c < CH_PER_SB; ++c, ++q) {
            const int s = q % STAGES, u = q / STAGES;
            if (!wait_bar(&full[s], u & 1, abort_flag, P.err)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t st = smem_u32(smem + s * STAGE_BYTES), a = tmem + TM_A + s * A_COLS;
            const uint64_t b0 = sw128_desc(st);  // hi rows 0-127, then lo rows (the next 16 KB)
            if (c < 4) {
#pragma unroll
              for (int ks = 0; ks < KCH / 16; ++ks) {
                const uint64_t off = (uint64_t)((ks * 32) >> 4);  // 16 fp16 = 32 bytes along K
                mma_f16_ts(d_main, a + ks * 8, b0 + off, IDESC_MAIN, (c | ks) != 0);  // 16 fp16 = 8 TMEM columns
              }
            } else {
              mma_f16_ts(d_min, a, b0, IDESC_MIN, 0u);
            }
            mma_commit(&empty[s]);
          }
          if (!ok) break;
          mma_commit(accf);
        }
      }
    }
  } else if (warp < W_EPI) {
    // ------------------------------------------------------------ transform: Q4_K -> fp16 A tiles in TMEM
    // A warp reaches TMEM lanes 32 * (warp % 4) .. +31 only, so that quarter of the rows is its own.
    const int r = (warp & 3) * 32 + lane;  // tile row 0..127 = TMEM lane
    const uint32_t a_lanes = tmem + ((uint32_t)((warp & 3) * 32) << 16) + TM_A;  // + stage columns
    int w = blockIdx.x;
    if (w < P.nwork) {
      Work k = work(w);
      const uint8_t* src = row_ptr(k, r);
      // the next item's row (for the prefetches that run past this item's last superblock)
      auto next_row = [&](int wc, int& nsbl) -> const uint8_t* {
        if (wc + (int)gridDim.x >= P.nwork) {
          nsbl = 0;
          return nullptr;
        }
        const Work kn = work(wc + gridDim.x);
        nsbl = kn.nsbl;
        return row_ptr(kn, r);
      };
      int nsbl_n;
      const uint8_t* src_n = next_row(w, nsbl_n);
      // The current superblock's 144 bytes. Each chunk's 32 quant bytes are replaced by the next
      // superblock's as soon as they are unpacked, and the header at the superblock's end, so
      // every load has a superblock's time to land and no second copy is held.
      uint4 cur[9];
#pragma unroll
      for (int i = 0; i < 9; ++i) cur[i] = __ldg(reinterpret_cast<const uint4*>(src) + i);
#pragma unroll
      for (int a = 1; a < PF_SB; ++a)
        if (a < k.nsbl) prefetch_row_l2(src + (int64_t)a * BLK);
      int q = 0;
      bool ok = true;
      while (ok) {
        for (int sb = 0; sb < k.nsbl && ok; ++sb) {
          // the next superblock: of this item, else the first of the next
          const uint8_t* nxt = nullptr;
          if (sb + 1 < k.nsbl)
            nxt = src + (int64_t)(sb + 1) * BLK;
          else if (w + (int)gridDim.x < P.nwork)
            nxt = row_ptr(work(w + gridDim.x), r);
          const uint4* nx4 = reinterpret_cast<const uint4*>(nxt);
          const uint4 hd_n = nxt ? __ldg(nx4) : make_uint4(0, 0, 0, 0);
          // and the superblock PF_SB ahead into L2, so that the loads of the next one find it there
          const int ahead = sb + PF_SB;
          if (ahead < k.nsbl)
            prefetch_row_l2(src + (int64_t)ahead * BLK);
          else if (ahead - k.nsbl < nsbl_n)
            prefetch_row_l2(src_n + (int64_t)(ahead - k.nsbl) * BLK);
          // The superblock's 6-bit scales and mins, one byte each, four to a word: sub-blocks
          // 0-3 are the low 6 bits of scale bytes 0-3 (4-7 for the mins); sub-blocks 4-7 take
          // the low (high) nibbles of bytes 8-11 and, as bits 4-5, the top two bits of bytes
          // 0-3 (4-7), the rule scale_min applies one value at a time.
          const uint4 hd = cur[0];
          const uint32_t sc03 = hd.y & 0x3F3F3F3Fu, mn03 = hd.z & 0x3F3F3F3Fu;
          const uint32_t sc47 = (hd.w & 0x0F0F0F0Fu) | ((hd.y >> 2) & 0x30303030u);
          const uint32_t mn47 = ((hd.w >> 4) & 0x0F0F0F0Fu) | ((hd.z >> 2) & 0x30303030u);
#pragma unroll
          for (int c = 0; c < CH_PER_SB; ++c) {
            const int s = q % STAGES, u = q / STAGES;
            ++q;
            if (!ok || (u > 0 && !wait_bar(&empty[s], (u - 1) & 1, abort_flag, P.err))) {
              ok = false;
              break;
            }
            tc_fence_after();  // the MMAs that read this stage have completed
            const uint32_t arow = a_lanes + s * A_COLS;
            if (c < 4) {
              const uint32_t sw = (c < 2 ? sc03 : sc47) >> (16 * (c & 1));  // sub-blocks 2c, 2c + 1
              uint32_t a[16];  // the chunk's two sub-blocks in turn, 16 columns each
              unpack_half<false>(cur[1 + 2 * c], cur[2 + 2 * c], sw & 0xFFu, a);
              tmem_st16(arow, a);
              unpack_half<true>(cur[1 + 2 * c], cur[2 + 2 * c], (sw >> 8) & 0xFFu, a);
              if (nxt) {  // this chunk's quants of the next superblock, into the registers just read
                cur[1 + 2 * c] = __ldg(nx4 + 1 + 2 * c);
                cur[2 + 2 * c] = __ldg(nx4 + 2 + 2 * c);
              }
              tmem_st16(arow + 16, a);
            } else {
              uint32_t mns[8], v[8];
#pragma unroll
              for (int j = 0; j < 4; ++j) mns[j] = (mn03 >> (8 * j)) & 0xFFu, mns[4 + j] = (mn47 >> (8 * j)) & 0xFFu;
              min_operand(mns, v);
              tmem_st8(arow, v);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&full[s]);
          }
          cur[0] = hd_n;
        }
        w += gridDim.x;
        if (w >= P.nwork) break;
        k = work(w);
        src = row_ptr(k, r);
        src_n = next_row(w, nsbl_n);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (8 warps)
    // Warp pair (quarter, half): TMEM lanes 32 * quarter .. +31 (tile rows), token
    // columns 64 * half .. +63. Every epilogue warp walks every item and reaches both
    // named barriers of each, also after an abort (then without waiting or reading).
    const int quarter = warp & 3, half = (warp - W_EPI) >> 2;
    const int r = quarter * 32 + lane, c0 = half * (TN / 2);
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    constexpr int LD = TN + 1;
    int G = 0;  // superblocks consumed so far (all items)
    bool ok = true;
    // gate/up: the previous item's SwiGLU + Q8_1 steps still to run (FINAL_PIECES when none)
    int pend_mt = 0, pend_nt = 0, pend_piece = FINAL_PIECES;
    float pend_amax = 0.f;
    auto final_step = [&]() {
      gateup_final_piece(xg, P, pend_mt, pend_nt, warp - W_EPI, lane, pend_piece, pend_amax, abort_flag);
      ++pend_piece;
    };
    for (int w = blockIdx.x; w < P.nwork; w += gridDim.x) {
      const Work k = work(w);
      const uint8_t* hdr = row_ptr(k, r);
      float acc[TN / 2];
#pragma unroll
      for (int i = 0; i < TN / 2; ++i) acc[i] = 0.f;
      for (int sb = 0; sb < k.nsbl; ++sb, ++G) {
        if (!ok) continue;
        const uint32_t dm2 = __ldg(reinterpret_cast<const uint32_t*>(hdr + (int64_t)sb * BLK));
        const float d = fp16_bits_to_f32(dm2), dmn = -64.f * fp16_bits_to_f32(dm2 >> 16);
        ok = __all_sync(0xffffffffu, wait_bar(accf, G & 1, abort_flag, P.err));
        if (!ok) continue;
        tc_fence_after();
        const uint32_t tm_hi = tmem + lane_addr + c0, tm_min = tmem + lane_addr + TM_DMIN + c0;
        // EPI_COLS columns of each of D_hi, D_lo and D_min per round (fewer live registers
        // than a wider round; the hand-over does not bind)
#pragma unroll
        for (int j = 0; j < TN / 2 / EPI_COLS; ++j) {
          float v[EPI_COLS], vl[EPI_COLS], u[EPI_COLS];
          if constexpr (EPI_COLS == 16) {
            tmem_ld16(tm_hi + j * 16, v);
            tmem_ld16(tm_hi + TN + j * 16, vl);
            tmem_ld16(tm_min + j * 16, u);
          } else {
            tmem_ld8(tm_hi + j * 8, v);
            tmem_ld8(tm_hi + TN + j * 8, vl);
            tmem_ld8(tm_min + j * 8, u);
          }
          tmem_wait_ld();
          if (j == TN / 2 / EPI_COLS - 1) {  // every column of this warp is in registers: release the buffers
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acce);
          }
#pragma unroll
          for (int i = 0; i < EPI_COLS; ++i)
            acc[j * EPI_COLS + i] = fmaf(u[i], dmn, fmaf(v[i] + vl[i], d, acc[j * EPI_COLS + i]));
        }
        // one step of the previous item's tail while the MMAs run this item's next superblock
        if (GATEUP && pend_piece < FINAL_PIECES) final_step();
      }
      if (!ok) *abort_flag = 1;
      const int t0 = k.nt * TN;
      if (GATEUP && (!TAIL || k.tl < 0)) {
        // rows 0-63 hold gate, 64-127 up, for the same 64 inter indices. The previous
        // item's tail (steps left over when this item had fewer superblocks than steps)
        // finishes, and every warp is past it, before the exchange is rewritten.
        while (pend_piece < FINAL_PIECES) final_step();
        __syncwarp();
        asm volatile("bar.sync 2, 256;" ::: "memory");
#pragma unroll
        for (int i = 0; i < TN / 2; ++i) xg[r * LD + c0 + i] = acc[i];
        if (half == 0) xg[TM * LD + r] = t0 + r < P.m ? P.tscale[t0 + r] : 0.f;  // thread r: token r's factor
        __syncwarp();
        asm volatile("bar.sync 2, 256;" ::: "memory");
        pend_mt = k.mt, pend_nt = k.nt, pend_piece = 0, pend_amax = 0.f;
      } else if (TAIL && k.tl >= 0) {
        if (!ok) continue;
        // a slice of a split tail tile: its partial tile, token-major, rows contiguous
        float* so = P.tail + ((int64_t)k.ks * (P.tiles - P.whole) + k.tl) * TM * TN;
#pragma unroll
        for (int i = 0; i < TN / 2; ++i) {
          const int t = t0 + c0 + i;
          so[(int64_t)(c0 + i) * TM + r] = t < P.m ? acc[i] * P.tscale[t] : 0.f;
        }
      } else if (!GATEUP && ok) {
        const int row = k.mt * TM + r;
        float* yo = P.y + (int64_t)k.ks * P.m * P.ldo;
#pragma unroll
        for (int i = 0; i < TN / 2; ++i) {
          const int t = t0 + c0 + i;
          if (t < P.m) yo[(int64_t)t * P.ldo + row] = acc[i] * P.tscale[t];
        }
      }
    }
    if (GATEUP)
      while (pend_piece < FINAL_PIECES) final_step();  // the last item's tail
  }
  // ---------------------------------------------------------------- teardown
  // (lane 0 of the TMA and MMA warps arrives after its loop, the other lanes long before)
  tc_fence_before();
  __syncwarp();
  __syncthreads();
  if (*abort_flag) {
    // let copies and MMAs already in flight land before the shared memory and TMEM go away
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 1000000ull) {
    }
  }
  if (warp == W_MMA) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
  }
}

// The split tail tiles of the down projection: y = the sum of the tail_q partial tiles,
// in slice order. One CTA per (tail tile, 8 tokens), a thread per row.
__global__ void __launch_bounds__(TM) finish_tail_kernel(const float* __restrict__ tail, int whole, int tiles,
                                                         int tail_q, int ntn, int mt_fast, int m, int ldo,
                                                         float* __restrict__ y) {
  pdl_wait();
  const int ntail = tiles - whole, tl = blockIdx.x % ntail, t8 = blockIdx.x / ntail;
  const int tile = whole + tl, nmt = tiles / ntn;
  const int nt = mt_fast ? tile / nmt : tile % ntn, mt = mt_fast ? tile % nmt : tile / ntn;
  const int r = threadIdx.x;
  float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int q = 0; q < tail_q; ++q)  // the 8 tokens' loads of a slice are in flight together
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (nt * TN + t8 * 8 + i < m) v[i] += tail[(((int64_t)q * ntail + tl) * TN + t8 * 8 + i) * TM + r];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int t = nt * TN + t8 * 8 + i;
    if (t < m) y[(int64_t)t * ldo + mt * TM + r] = v[i];
  }
}

// The split tail tiles of the gate/up projection: g and u = the sums of the tail_q partial
// tiles in slice order (already scaled by 2^e_t), then h = silu(g) * u and its Q8_1, the rule
// of the unsplit epilogue. One CTA of 256 threads per tail tile; thread e owns token e % 128
// and the Q8_1 block e / 128 of the tile's 64 inter rows.
__global__ void __launch_bounds__(256) finish_gateup_tail_kernel(const float* __restrict__ tail, int whole, int tiles,
                                                                 int tail_q, int ntn, int mt_fast, int m, int ldo,
                                                                 int8_t* __restrict__ hq_qs, float2* __restrict__ hq_ds) {
  pdl_wait();
  const int ntail = tiles - whole, tl = blockIdx.x;
  const int tile = whole + tl, nmt = tiles / ntn;
  const int nt = mt_fast ? tile / nmt : tile % ntn, mt = mt_fast ? tile % nmt : tile / ntn;
  const int e = threadIdx.x, tt = e & (TN - 1), qb = e / TN;
  const int t = nt * TN + tt;
  if (t >= m) return;
  float h[Q8B], amax = 0.f;
#pragma unroll
  for (int j = 0; j < Q8B; j += 4) {
    float4 g = make_float4(0.f, 0.f, 0.f, 0.f), u = g;
    for (int q = 0; q < tail_q; ++q) {
      const float* pt = tail + (((int64_t)q * ntail + tl) * TN + tt) * TM;
      const float4 gq = *reinterpret_cast<const float4*>(pt + qb * 32 + j);
      const float4 uq = *reinterpret_cast<const float4*>(pt + 64 + qb * 32 + j);
      g.x += gq.x, g.y += gq.y, g.z += gq.z, g.w += gq.w;
      u.x += uq.x, u.y += uq.y, u.z += uq.z, u.w += uq.w;
    }
    h[j] = silu_f(g.x) * u.x;
    h[j + 1] = silu_f(g.y) * u.y;
    h[j + 2] = silu_f(g.z) * u.z;
    h[j + 3] = silu_f(g.w) * u.w;
#pragma unroll
    for (int i = 0; i < 4; ++i) amax = fmaxf(amax, fabsf(h[j + i]));
  }
  const bool nz = amax >= 0x1p-120f;  // below: zero block (127/amax would overflow)
  const float dq = nz ? __fdiv_rn(amax, 127.f) : 0.f;
  const float inv = nz ? __fdiv_rn(127.f, amax) : 0.f;
  int sum = 0;
  uint32_t pk[Q8B / 4];
#pragma unroll
  for (int w = 0; w < Q8B / 4; ++w) {
    uint32_t v = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      float rq = roundf(__fmul_rn(h[4 * w + b], inv));
      rq = fminf(fmaxf(rq, -127.f), 127.f);
      const int qi = (int)rq;
      sum += qi;
      v |= ((uint32_t)qi & 0xFFu) << (8 * b);
    }
    pk[w] = v;
  }
  const int irow = mt * 64 + qb * 32;
  uint4* dst = reinterpret_cast<uint4*>(hq_qs + (int64_t)t * ldo + irow);  // 32-byte aligned
  dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
  hq_ds[(int64_t)t * (ldo / Q8B) + irow / Q8B] = make_float2(dq, __fmul_rn(dq, (float)sum));
}

// Split of the down projection's last, partial round of tiles over num_sms persistent
// CTAs: whole tiles before `whole`, the rest in q > 1 K slices each (q = 0 when the tiles
// make whole rounds, fit one round, or leave too many for two slices each).
void tail_split(int tiles, int num_sms, int* whole, int* q) {
  const int rounds = tiles / num_sms, ntail = tiles - rounds * num_sms;
  *whole = rounds * num_sms;
  *q = (rounds > 0 && ntail > 0 && num_sms / ntail >= 2) ? std::min(num_sms / ntail, 8) : 0;
}

// ------------------------------------------------------------------------- host side
// 2-D fp16 tensor [rows][cols] (row-major), box 64 x 128, 128-byte swizzle; rows beyond
// `rows` read as zeros.
bool make_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols) {
  return tmap_2d(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, base, (uint64_t)rows, (uint64_t)cols, (uint64_t)cols * 2, KCH,
                 TN, CU_TENSOR_MAP_SWIZZLE_128B);
}

// One persistent CTA per SM (at most one per work item).
template <bool GATEUP, bool SPLIT, bool TAIL>
cudaError_t launch_mmq(const CUtensorMap& hi, const CUtensorMap& lo, const CUtensorMap& mn, const MmqParams& P,
                       int num_sms, cudaStream_t s) {
  const int grid = std::min(P.nwork, num_sms);
  auto kern = mmq_kernel<GATEUP, SPLIT, TAIL>;
  static uint64_t attr_set = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !(attr_set >> dev & 1)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (dev < 64) attr_set |= 1ull << dev;
  }
  kern<<<grid, NWARPS * 32, SMEM_BYTES, s>>>(hi, lo, mn, P);
  return cudaGetLastError();
}

struct Operand {
  __half *hi, *lo, *mn;
  float* scale;
};

// The CTAs resident at once (one per SM) share operands through L2. Walking token
// tiles fastest keeps few weight row tiles but every token tile's B planes in
// flight; walking row tiles fastest the reverse. Take the order whose resident
// operands are fewer bytes (at large m the down projection's B planes alone
// exceed L2 in the first order).
int row_tiles_fastest(int64_t nmt, int64_t ntn, int64_t k, int num_sms) {
  const int64_t w_tile = (int64_t)TM * (k / QK) * BLK, b_tile = (int64_t)TN * k * 4;
  const int64_t r = num_sms;
  const int64_t tok_fast = std::min<int64_t>(nmt, (r + ntn - 1) / ntn) * w_tile + std::min<int64_t>(ntn, r) * b_tile;
  const int64_t row_fast = std::min<int64_t>(nmt, r) * w_tile + std::min<int64_t>(ntn, (r + nmt - 1) / nmt) * b_tile;
  return row_fast < tok_fast ? 1 : 0;
}

}  // namespace

// K slices of the down projection: its (row tile, token tile) CTAs number only
// hidden/128 per 128 tokens, fewer than the SMs when m is small. Each slice sums
// part of K into its own partial output, reduced in slice order afterwards. The
// grid is split as far as all slices still run in one wave (and each keeps at
// least two superblocks); a grid of a wave or more is not split, since the
// partial outputs cost traffic that a full grid does not repay.
int down_ksplit(int64_t m, int64_t hidden, int64_t inter, int num_sms) {
  const int64_t ctas = (hidden / TM) * ((m + TN - 1) / TN), nsb = inter / QK;
  int k = 1;
  while (k < 8 && ctas * (k + 1) <= num_sms && nsb / (k + 1) >= 2) ++k;
  return k;
}

bool prefill_plan(int64_t m, int64_t hidden, int64_t inter, int num_sms, PrefillPlan* p) {
  if (m < 9 || num_sms < 1) return false;
  p->m = (int)m;
  p->hidden = (int)hidden;
  p->inter = (int)inter;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align256(o + bytes);
    return at;
  };
  auto op_bytes = [&](int64_t k, bool with_lo) {
    return align256((size_t)m * k * 2) * (with_lo ? 2 : 1) + align256((size_t)m * (k / QK) * 64 * 2) +
           align256((size_t)m * 4);
  };
  p->off_xq = take((size_t)m * hidden + (size_t)m * (hidden / Q8B) * 8);
  p->off_hq = take((size_t)m * inter + (size_t)m * (inter / Q8B) * 8);
  p->off_xop = take(op_bytes(hidden, true));
  p->off_hop = take(op_bytes(inter, true));
  p->off_misc = take(256);
  p->ksplit = down_ksplit(m, hidden, inter, num_sms);
  p->num_sms = num_sms;
  const int dtiles = (int)((hidden / TM) * ((m + TN - 1) / TN));
  p->tail_whole = dtiles, p->tail_q = 0;
  if (p->ksplit == 1) tail_split(dtiles, num_sms, &p->tail_whole, &p->tail_q);
  p->off_tail = take(p->tail_q > 1 ? (size_t)(dtiles - p->tail_whole) * p->tail_q * TM * TN * 4 : 0);
  // gate/up: 64 inter rows (of gate and of up) per tile; slices of at least two superblocks
  const int gtiles = (int)((inter / 64) * ((m + TN - 1) / TN));
  tail_split(gtiles, num_sms, &p->gu_whole, &p->gu_q);
  p->gu_q = std::min<int64_t>(p->gu_q, hidden / QK / 2);
  if (p->gu_q < 2) p->gu_whole = gtiles, p->gu_q = 0;
  p->off_gtail = take(p->gu_q > 1 ? (size_t)(gtiles - p->gu_whole) * p->gu_q * TM * TN * 4 : 0);
  p->off_ypart = take((size_t)p->ksplit * m * hidden * 4);  // also the float32 y of a bf16-output call
  p->ws_bytes = o;
  return true;
}

int prefill_kernels(const PrefillPlan& p, int ybf16) {
  return (p.hidden <= QE_MAX_K ? 4 : 5) + (p.gu_q > 1) + (p.tail_q > 1) + (p.ksplit > 1 || ybf16);
}

cudaError_t launch_prefill(const PrefillPlan& p, const void* x, int bf16, const void* wg, const void* wu,
                           const void* wd, void* y, void* ws, uint32_t* err, cudaStream_t s,
                           const ProfileEvents& prof, int ybf16) {
  uint8_t* W = (uint8_t*)ws;
  const int64_t m = p.m, H = p.hidden, I = p.inter;
  auto split = [&](uint8_t* base, int64_t k, bool with_lo) {
    Operand op;
    size_t o = 0;
    op.hi = (__half*)(base + o);
    o += align256((size_t)m * k * 2);
    op.lo = with_lo ? (__half*)(base + o) : nullptr;
    if (with_lo) o += align256((size_t)m * k * 2);
    op.mn = (__half*)(base + o);
    o += align256((size_t)m * (k / QK) * 64 * 2);
    op.scale = (float*)(base + o);
    return op;
  };
  const Operand xo = split(W + p.off_xop, H, true);
  const Operand ho = split(W + p.off_hop, I, true);
  int8_t* xq = (int8_t*)(W + p.off_xq);
  float2* xds = (float2*)(W + p.off_xq + (size_t)m * H);
  int8_t* hq = (int8_t*)(W + p.off_hq);
  float2* hds = (float2*)(W + p.off_hq + (size_t)m * I);

  CUtensorMap mx_hi, mx_lo, mx_mn, mh_hi, mh_lo, mh_mn;
  if (!make_map(&mx_hi, xo.hi, m, H) || !make_map(&mx_lo, xo.lo, m, H) ||
      !make_map(&mx_mn, xo.mn, m, (H / QK) * 64) || !make_map(&mh_hi, ho.hi, m, I) ||
      !make_map(&mh_lo, ho.lo, m, I) || !make_map(&mh_mn, ho.mn, m, (I / QK) * 64))
    return cudaErrorInvalidValue;

  prof.before(0, s);  // x's operand planes
  cudaError_t e = cudaSuccess;
  if (H <= QE_MAX_K) {
    const size_t sm = quant_expand_smem(H);
    if (bf16)
      quant_expand_kernel<__nv_bfloat16><<<(unsigned)m, EXP_NT, sm, s>>>((const __nv_bfloat16*)x, (int)H, xo.hi,
                                                                      xo.lo, xo.mn, xo.scale);
    else
      quant_expand_kernel<float><<<(unsigned)m, EXP_NT, sm, s>>>((const float*)x, (int)H, xo.hi, xo.lo, xo.mn,
                                                              xo.scale);
    e = cudaGetLastError();
  } else if ((e = launch_q8_1(x, bf16, m, H, xq, s)) == cudaSuccess) {
    expand_kernel<<<(unsigned)m, EXP_NT, 0, s>>>(xq, xds, (int)H, xo.hi, xo.lo, xo.mn, xo.scale);
    e = cudaGetLastError();
  }
  prof.after(0, s);
  if (e != cudaSuccess) return e;

  const int ntn = (int)((m + TN - 1) / TN);
  MmqParams g{};
  g.w0 = (const uint8_t*)wg;
  g.w1 = (const uint8_t*)wu;
  g.nsb = (int)(H / QK);
  g.m = (int)m;
  g.ldo = (int)I;
  g.ntn = ntn;
  g.ksplit = 1;
  g.mt_fast = row_tiles_fastest(I / 64, ntn, H, p.num_sms);
  g.tiles = g.nwork = (int)(I / 64) * ntn;
  g.whole = p.gu_whole;
  g.tail_q = p.gu_q;
  g.tail = (float*)(W + p.off_gtail);
  if (p.gu_q > 1) g.nwork = p.gu_whole + (g.tiles - p.gu_whole) * p.gu_q;
  g.tscale = xo.scale;
  g.hq_qs = hq;
  g.hq_ds = hds;
  g.err = err;
  prof.before(1, s);
  e = p.gu_q > 1 ? launch_mmq<true, false, true>(mx_hi, mx_lo, mx_mn, g, p.num_sms, s)
                 : launch_mmq<true, false, false>(mx_hi, mx_lo, mx_mn, g, p.num_sms, s);
  if (e == cudaSuccess && p.gu_q > 1) {  // the split tail tiles' sum, SwiGLU and Q8_1
    finish_gateup_tail_kernel<<<g.tiles - p.gu_whole, 256, 0, s>>>(g.tail, p.gu_whole, g.tiles, p.gu_q, ntn,
                                                                   g.mt_fast, (int)m, (int)I, hq, hds);
    e = cudaGetLastError();
  }
  prof.after(1, s);
  if (e != cudaSuccess) return e;

  prof.before(2, s);
  expand_kernel<<<(unsigned)m, EXP_NT, 0, s>>>(hq, hds, (int)I, ho.hi, ho.lo, ho.mn, ho.scale);
  prof.after(2, s);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  MmqParams dn{};
  dn.w0 = (const uint8_t*)wd;
  dn.nsb = (int)(I / QK);
  dn.m = (int)m;
  dn.ldo = (int)H;
  dn.ntn = ntn;
  dn.ksplit = p.ksplit;
  dn.mt_fast = row_tiles_fastest(H / TM, ntn, I, p.num_sms);
  dn.tiles = (int)(H / TM) * ntn;
  dn.nwork = dn.tiles * p.ksplit;
  dn.whole = p.tail_whole;
  dn.tail_q = p.tail_q;
  dn.tail = (float*)(W + p.off_tail);
  if (p.tail_q > 1) dn.nwork = p.tail_whole + (dn.tiles - p.tail_whole) * p.tail_q;
  dn.tscale = ho.scale;
  float* ypart = (float*)(W + p.off_ypart);
  const bool fin = p.ksplit > 1 || ybf16;  // the slice sum and/or the bf16 store
  dn.y = fin ? ypart : (float*)y;
  dn.err = err;
  prof.before(3, s);  // the down MMQ, and the sum of its K slices when there are several
  e = p.ksplit > 1 ? launch_mmq<false, true, false>(mh_hi, mh_lo, mh_mn, dn, p.num_sms, s)
                   : launch_mmq<false, false, true>(mh_hi, mh_lo, mh_mn, dn, p.num_sms, s);
  if (e == cudaSuccess && p.tail_q > 1) {
    const int ntail = dn.tiles - p.tail_whole;
    finish_tail_kernel<<<ntail * (TN / 8), TM, 0, s>>>(dn.tail, p.tail_whole, dn.tiles, p.tail_q, ntn, dn.mt_fast,
                                                     (int)m, (int)H, dn.y);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess && fin) e = launch_finish_down(ypart, p.ksplit, m * H, y, ybf16, s);
  prof.after(3, s);
  return e;
}

}  // namespace q4k
