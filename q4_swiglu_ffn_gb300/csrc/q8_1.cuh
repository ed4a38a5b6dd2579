// Q8_1 quantisation of one block of 32 activations held by 4 lanes (8 each),
// shared by the stand-alone quantizer and the kernels that re-quantize h.
// Source: realizar src/cuda/executor/layers/ffn.rs, fused_ffn_swiglu_gpu_true_dp4a
// (per-block scale + 32 x int8); spark_model/layers/ops/q4k_mmq.rs,
// quantize_act_q8_1. Every float32 operation is an explicit round-to-nearest
// intrinsic: d = amax/127, inv = 127/amax, q = roundf(x*inv) (ties away from
// zero) clamped to +-127, s = d*sum(q); a block whose amax is below 2^-120 is
// all zero.
#pragma once
#include "common.cuh"

namespace q4k {

// Eight consecutive activations (16-byte aligned), float32 or bf16, widened exactly to float32.
__device__ __forceinline__ void load8(const float* p, float v[8]) {
  const float4 a = *reinterpret_cast<const float4*>(p), b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void load8(const __nv_bfloat16* p, float v[8]) {
  const uint4 a = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// The 4 lanes of a block must be aligned quads of the warp, and every lane of
// the warp must call this (it shuffles).
__device__ __forceinline__ void q8_1_block8(const float v[8], int8_t q[8], float& d, float& s) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  const bool nz = amax >= 0x1p-120f;  // below: zero block (127/amax would overflow)
  d = nz ? __fdiv_rn(amax, 127.f) : 0.f;
  const float inv = nz ? __fdiv_rn(127.f, amax) : 0.f;
  int sum = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float r = roundf(__fmul_rn(v[i], inv));
    r = fminf(fmaxf(r, -127.f), 127.f);
    q[i] = (int8_t)(int)r;
    sum += (int)r;
  }
  sum += __shfl_xor_sync(0xffffffffu, sum, 1);
  sum += __shfl_xor_sync(0xffffffffu, sum, 2);
  s = __fmul_rn(d, (float)sum);
}

}  // namespace q4k
