// Pieces shared by the two decode GEMV families (float32 activations in
// decode.cu, Q8_1 activations in decode_q8.cu): the 3-D TMA box of a weight
// matrix, the choice of the K split, programmatic dependent launch, and the
// down-projection chunk sum.
#pragma once
#include <algorithm>
#include <climits>

#include "common.cuh"
#include "tmap.h"

namespace q4k {
namespace {

// 3-D box {18 x 8-byte elements of a block, rows, superblocks} of a weight matrix.
__device__ __forceinline__ void tma_box3(void* dst, const CUtensorMap* tm, int row, int sb, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(0), "r"(row), "r"(sb), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void store4(float* y, int64_t i, float4 s) { reinterpret_cast<float4*>(y)[i] = s; }
__device__ __forceinline__ void store4(__nv_bfloat16* y, int64_t i, float4 s) {
  // round to nearest even, once
  const __nv_bfloat162 a = __floats2bfloat162_rn(s.x, s.y), b = __floats2bfloat162_rn(s.z, s.w);
  uint2 v;
  v.x = *reinterpret_cast<const uint32_t*>(&a);
  v.y = *reinterpret_cast<const uint32_t*>(&b);
  reinterpret_cast<uint2*>(y)[i] = v;
}

// y = sum over the K-chunks of the down partials, in chunk order (float32, or
// bf16 rounded once from the float32 sum).
template <typename T>
__global__ void finish_down_kernel(const float* __restrict__ part, int nks, int64_t n, T* __restrict__ y) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (4 * i >= n) return;
  float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
  // Batches of 8 chunks: all of a batch's loads are issued before the first add (a
  // loop over a run-time count would wait for each load in turn); sums in chunk order.
  for (int k0 = 0; k0 < nks; k0 += 8) {
    float4 a[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (k0 + j < nks) a[j] = reinterpret_cast<const float4*>(part + (int64_t)(k0 + j) * n)[i];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (k0 + j < nks) s.x += a[j].x, s.y += a[j].y, s.z += a[j].z, s.w += a[j].w;
  }
  store4(y, i, s);
}

// pdl = false: an ordinary launch (the first kernel of a call, ordered after all earlier work).
inline cudaError_t launch_pdl(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t s, void** args,
                              bool pdl = true) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

// Launches K3 (n = m * hidden outputs): the sum of the down projection's K-chunks,
// and the store of y as float32 or (ybf16) bf16.
inline cudaError_t launch_finish_down(const float* part, int nks, int64_t n, void* y, int ybf16, cudaStream_t s) {
  void* args[] = {&part, &nks, &n, &y};
  const void* fn = ybf16 ? reinterpret_cast<const void*>(finish_down_kernel<__nv_bfloat16>)
                         : reinterpret_cast<const void*>(finish_down_kernel<float>);
  // small CTAs spread the sums over more SMs (more loads in flight)
  return launch_pdl(fn, dim3((unsigned)((n / 4 + 63) / 64)), dim3(64), 0, s, args);
}

// Weight matrix [rows][nsb blocks] as a 3-D tensor {18 x 8-byte elements of a
// block, rows, blocks}; a box of box_rows rows x slices superblocks lands in
// shared memory superblock-major, 144 bytes per row.
inline bool weight_map(CUtensorMap* m, const void* w, int rows, int nsb, int box_rows, int slices) {
  const cuuint64_t dims[3] = {(cuuint64_t)(BLK / 8), (cuuint64_t)rows, (cuuint64_t)nsb};
  const cuuint64_t strides[2] = {(cuuint64_t)nsb * BLK, (cuuint64_t)BLK};
  const cuuint32_t box[3] = {(cuuint32_t)(BLK / 8), (cuuint32_t)box_rows, (cuuint32_t)slices};
  return tmap_encode_cached(m, CU_TENSOR_MAP_DATA_TYPE_UINT64, 3, w, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

// Number of K-chunks: the most, up to max_nks, among those that minimise the longest CTA's
// group steps. The cap bounds the partial-sum buffers (nks x m x rows floats).
inline void choose_split(int ngroups, int nru, int grid, int max_nks, int* nks_out, int* gpc_out) {
  int64_t best = INT64_MAX;
  int best_nks = 1, best_gpc = ngroups;
  for (int t = 1; t <= ngroups && t <= max_nks; ++t) {
    const int gpc = (ngroups + t - 1) / t;
    const int nks = (ngroups + gpc - 1) / gpc;
    if (nks != t) continue;
    const int64_t per_cta = ((int64_t)nks * nru + grid - 1) / grid;
    const int64_t cost = per_cta * gpc;
    if (cost <= best) {  // ties go to more chunks: one group per chunk lets warps keep their inputs
      best = cost;
      best_nks = nks;
      best_gpc = gpc;
    }
  }
  *nks_out = best_nks;
  *gpc_out = best_gpc;
}

inline size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

// Sets the dynamic shared memory limit of a kernel once per device (the
// attribute belongs to the function and the device).
inline cudaError_t set_smem_once(const void* kern, size_t smem, uint64_t* done_mask) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !(*done_mask >> dev & 1)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (dev < 64) *done_mask |= 1ull << dev;
  }
  return cudaSuccess;
}

}  // namespace
}  // namespace q4k
