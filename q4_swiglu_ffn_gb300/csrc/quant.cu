// Q4_K dequantisation (test hook), Q8_1 activation quantisation, and the
// load-time Q4_K weight quantizer, for sm_103a.
//
// Block format (spark_model/layers/ops/q4k_mmq.rs: QK_K = 256, 144-byte
// block_q4_K): bytes 0-1 fp16 d, 2-3 fp16 dmin, 4-15 packed 6-bit scales and
// mins of 8 sub-blocks of 32, 16-143 the 4-bit quants in four groups of 32
// bytes (group g: low nibble of byte i = weight 64g+i, high nibble = weight
// 64g+32+i).
#include "common.cuh"
#include "kernels.h"
#include "q8_1.cuh"

namespace q4k {

// ------------------------------------------------------------------------- dequantize
// One warp per block; lane t covers group t/8, bytes 4(t%8)..4(t%8)+3 of it, i.e.
// four weights of sub-block 2g (low nibbles) and the same four of 2g+1 (high).
// w = d*scale*q - dmin*min: d*scale and dmin*min are exact in float32 (11+6 bits),
// so one fma rounds the exact value once.
__global__ void dequant_kernel(const uint8_t* __restrict__ w, float* __restrict__ out, int64_t nblocks,
                               int nb_per_row) {
  const int64_t blk = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  if (blk >= nblocks) return;
  const int lane = threadIdx.x & 31;
  const uint8_t* b = w + blk * BLK;
  const uint4 hdr = *reinterpret_cast<const uint4*>(b);
  const float d = fp16_bits_to_f32(hdr.x), dmin = fp16_bits_to_f32(hdr.x >> 16);
  const int grp = lane >> 3, pos = (lane & 7) * 4;
  uint32_t sl, ml, sh, mh;
  scale_min(hdr.y, hdr.z, hdr.w, 2 * grp, sl, ml);
  scale_min(hdr.y, hdr.z, hdr.w, 2 * grp + 1, sh, mh);
  const float dl = __fmul_rn(d, (float)sl), ol = __fmul_rn(dmin, (float)ml);
  const float dh = __fmul_rn(d, (float)sh), oh = __fmul_rn(dmin, (float)mh);
  const uint32_t q = *reinterpret_cast<const uint32_t*>(b + 16 + 32 * grp + pos);
  float4 lo, hi;
  lo.x = fmaf(dl, (float)(q & 15), -ol);
  lo.y = fmaf(dl, (float)((q >> 8) & 15), -ol);
  lo.z = fmaf(dl, (float)((q >> 16) & 15), -ol);
  lo.w = fmaf(dl, (float)((q >> 24) & 15), -ol);
  hi.x = fmaf(dh, (float)((q >> 4) & 15), -oh);
  hi.y = fmaf(dh, (float)((q >> 12) & 15), -oh);
  hi.z = fmaf(dh, (float)((q >> 20) & 15), -oh);
  hi.w = fmaf(dh, (float)((q >> 28) & 15), -oh);
  const int64_t row = blk / nb_per_row, col = (blk % nb_per_row) * QK + 64 * grp + pos;
  float* o = out + row * (int64_t)nb_per_row * QK + col;
  *reinterpret_cast<float4*>(o) = lo;
  *reinterpret_cast<float4*>(o + 32) = hi;
}

cudaError_t launch_dequant(const void* w, float* out, int64_t rows, int64_t cols, cudaStream_t s) {
  const int64_t nb = rows * (cols / QK);
  const int warps = 8;
  const int64_t grid = (nb + warps - 1) / warps;
  dequant_kernel<<<(unsigned)grid, warps * 32, 0, s>>>((const uint8_t*)w, out, nb, (int)(cols / QK));
  return cudaGetLastError();
}

// ------------------------------------------------------------------------- Q8_1 quantize
// Each lane holds 8 consecutive values; 4 lanes make a block of 32. All float32
// operations are written with explicit round-to-nearest intrinsics:
// d = amax/127, inv = 127/amax, q = roundf(x*inv) (ties away from zero), s = d*sum(q).
template <typename T>
__global__ void q8_1_kernel(const T* __restrict__ x, int8_t* __restrict__ qs, float2* __restrict__ ds,
                            int64_t m, int64_t k) {
  // one thread per 8 values; 4 threads per Q8_1 block; rows of k values
  pdl_launch_dependents();  // a dependent GEMV may start streaming its weights (it waits before reading q)
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t per_row = k / 8;
  const bool active = gid < m * per_row;
  const int64_t g = active ? gid : 0;
  const int64_t row = g / per_row, c8 = (g % per_row) * 8;
  float v[8];
  load8(x + row * k + c8, v);
  int8_t q[8];
  float d, s;
  q8_1_block8(v, q, d, s);  // all lanes of the warp take part in the shuffles
  if (!active) return;
  uint2 packed;
  packed.x = (uint32_t)(uint8_t)q[0] | ((uint32_t)(uint8_t)q[1] << 8) | ((uint32_t)(uint8_t)q[2] << 16) |
             ((uint32_t)(uint8_t)q[3] << 24);
  packed.y = (uint32_t)(uint8_t)q[4] | ((uint32_t)(uint8_t)q[5] << 8) | ((uint32_t)(uint8_t)q[6] << 16) |
             ((uint32_t)(uint8_t)q[7] << 24);
  *reinterpret_cast<uint2*>(qs + row * k + c8) = packed;
  if ((threadIdx.x & 3) == 0) ds[row * (k / Q8B) + c8 / Q8B] = make_float2(d, s);
}

cudaError_t launch_q8_1(const void* x, int bf16, int64_t m, int64_t k, void* out, cudaStream_t s) {
  int8_t* qs = (int8_t*)out;
  float2* ds = (float2*)((uint8_t*)out + m * k);
  const int64_t threads = m * (k / 8);
  const int tpb = 256;
  const int64_t grid = (threads + tpb - 1) / tpb;
  if (bf16)
    q8_1_kernel<__nv_bfloat16><<<(unsigned)grid, tpb, 0, s>>>((const __nv_bfloat16*)x, qs, ds, m, k);
  else
    q8_1_kernel<float><<<(unsigned)grid, tpb, 0, s>>>((const float*)x, qs, ds, m, k);
  return cudaGetLastError();
}

// ------------------------------------------------------------------------- weight quantizer
// Deterministic min-max Q4_K quantizer in float64, one warp per block, lane L
// holding 8 consecutive values of sub-block L/4. Every operation is an explicit
// round-to-nearest intrinsic so that no multiply-add is fused.
__device__ __forceinline__ double fp16_up(double v, bool& bad) {
  // smallest fp16 >= v (v >= 0)
  if (!(v <= 65504.0)) { bad = true; return 0.0; }
  __half h = __double2half(v);
  unsigned short bits = __half_as_ushort(h);
  if ((double)__half2float(h) < v) bits = (unsigned short)(bits + 1);
  if (bits > 0x7BFF) { bad = true; return 0.0; }
  return (double)__half2float(__ushort_as_half(bits));
}
__device__ __forceinline__ double smallest_fp16_cover(double total, double mult, bool& bad) {
  double f = fp16_up(__ddiv_rn(total, mult), bad);
  if (__dmul_rn(f, mult) < total) {
    unsigned short bits = (unsigned short)(__half_as_ushort(__double2half(f)) + 1);
    if (bits > 0x7BFF) bad = true;
    f = (double)__half2float(__ushort_as_half(bits));
  }
  return f;
}
__device__ __forceinline__ int smallest_int_cover(double need, double step, int top) {
  if (!(step > 0.0)) return 0;
  double n = ceil(__ddiv_rn(need, step));
  n = fmin(fmax(n, 0.0), (double)top);
  if (__dmul_rn(step, n) < need && n < top) n = __dadd_rn(n, 1.0);
  if (n >= 1.0 && __dmul_rn(step, __dadd_rn(n, -1.0)) >= need) n = __dadd_rn(n, -1.0);
  return (int)n;
}
__device__ __forceinline__ double round_half_away(double v) {
  const double a = fabs(v), f = floor(a);
  const double r = (__dadd_rn(a, -f) >= 0.5) ? __dadd_rn(f, 1.0) : f;
  return copysign(r, v);
}

template <typename T>
__global__ void quantize_weights_kernel(const T* __restrict__ w, uint8_t* __restrict__ out, int64_t nblocks,
                                        int nb_per_row, uint32_t* err) {
  const int64_t blk = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  if (blk >= nblocks) return;  // whole warps exit together
  const int lane = threadIdx.x & 31, j = lane >> 2;
  const int64_t row = blk / nb_per_row, c = (blk % nb_per_row) * QK + lane * 8;
  float vf[8];
  load8(w + row * (int64_t)nb_per_row * QK + c, vf);
  double x[8];
  double mn = 0.0, mx = 0.0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    x[i] = (double)vf[i];
    mn = fmin(mn, x[i]);
    mx = fmax(mx, x[i]);
  }
  mn = fmin(mn, __shfl_xor_sync(0xffffffffu, mn, 1));
  mn = fmin(mn, __shfl_xor_sync(0xffffffffu, mn, 2));
  mx = fmax(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
  mx = fmax(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
  const double lo = __dadd_rn(fmax(0.0, -mn), 0.0), hi = __dadd_rn(fmax(0.0, mx), 0.0);
  double L = lo;
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) L = fmax(L, __shfl_xor_sync(0xffffffffu, L, o));
  bool bad = false;
  const double dmin = smallest_fp16_cover(L, 63.0, bad);
  const int mq = smallest_int_cover(lo, dmin, 63);
  const double r = __dadd_rn(hi, __dmul_rn(dmin, (double)mq));
  double R = r;
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) R = fmax(R, __shfl_xor_sync(0xffffffffu, R, o));
  const double d = smallest_fp16_cover(R, 945.0, bad);
  const int sq = smallest_int_cover(r, __dmul_rn(15.0, d), 63);
  const double step = __dmul_rn(d, (double)sq);
  const double off = __dmul_rn(dmin, (double)mq);
  uint32_t nib[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    double q = 0.0;
    if (step > 0.0) q = fmin(fmax(round_half_away(__ddiv_rn(__dadd_rn(x[i], off), step)), 0.0), 15.0);
    nib[i] = (uint32_t)q;
  }
  const bool any_bad = __any_sync(0xffffffffu, bad);
  uint8_t* o = out + blk * BLK;
  // quant bytes: sub-block 2g in low nibbles, 2g+1 in high nibbles of group g
  uint32_t w0 = nib[0] | (nib[1] << 8) | (nib[2] << 16) | (nib[3] << 24);
  uint32_t w1 = nib[4] | (nib[5] << 8) | (nib[6] << 16) | (nib[7] << 24);
  const uint32_t h0 = __shfl_down_sync(0xffffffffu, w0, 4), h1 = __shfl_down_sync(0xffffffffu, w1, 4);
  if ((j & 1) == 0) {
    const int grp = j >> 1;
    uint2 v = any_bad ? make_uint2(0u, 0u) : make_uint2(w0 | (h0 << 4), w1 | (h1 << 4));
    *reinterpret_cast<uint2*>(o + 16 + 32 * grp + (lane & 3) * 8) = v;
  }
  // gather scales and mins of the 8 sub-blocks into lane 0 and pack them
  uint32_t scs[8], mns[8];
#pragma unroll
  for (int jj = 0; jj < 8; ++jj) {
    scs[jj] = (uint32_t)__shfl_sync(0xffffffffu, sq, 4 * jj);
    mns[jj] = (uint32_t)__shfl_sync(0xffffffffu, mq, 4 * jj);
  }
  if (lane == 0) {
    uint32_t bytes[12];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      bytes[t] = (scs[t] & 63u) | ((scs[t + 4] >> 4) << 6);
      bytes[t + 4] = (mns[t] & 63u) | ((mns[t + 4] >> 4) << 6);
      bytes[t + 8] = (scs[t + 4] & 15u) | ((mns[t + 4] & 15u) << 4);
    }
    uint4 hdr;
    const uint32_t dbits = __half_as_ushort(__double2half(d));
    const uint32_t mbits = __half_as_ushort(__double2half(dmin));
    hdr.x = dbits | (mbits << 16);
    hdr.y = bytes[0] | (bytes[1] << 8) | (bytes[2] << 16) | (bytes[3] << 24);
    hdr.z = bytes[4] | (bytes[5] << 8) | (bytes[6] << 16) | (bytes[7] << 24);
    hdr.w = bytes[8] | (bytes[9] << 8) | (bytes[10] << 16) | (bytes[11] << 24);
    if (any_bad) {
      hdr = make_uint4(0u, 0u, 0u, 0u);
      set_error(err, ERRBIT_RANGE);
    }
    *reinterpret_cast<uint4*>(o) = hdr;
  }
}

cudaError_t launch_quantize_weights(const void* w, int bf16, int64_t rows, int64_t cols, void* out,
                                    uint32_t* err, cudaStream_t s) {
  const int64_t nb = rows * (cols / QK);
  const int warps = 4;
  const int64_t grid = (nb + warps - 1) / warps;
  if (bf16)
    quantize_weights_kernel<__nv_bfloat16>
        <<<(unsigned)grid, warps * 32, 0, s>>>((const __nv_bfloat16*)w, (uint8_t*)out, nb, (int)(cols / QK), err);
  else
    quantize_weights_kernel<float>
        <<<(unsigned)grid, warps * 32, 0, s>>>((const float*)w, (uint8_t*)out, nb, (int)(cols / QK), err);
  return cudaGetLastError();
}

}  // namespace q4k
