// Host-side encoding of TMA tensor maps (driver entry point fetched through the
// runtime, so the library does not link libcuda directly).
#pragma once
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

namespace q4k {

inline PFN_cuTensorMapEncodeTiled_v12000 tmap_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Encodes a tiled tensor map, reusing the result of an earlier call with the
// same arguments. A map only describes an address range, so a cached one stays
// exact for the same arguments (even when that memory was freed and allocated
// again); the cache saves the host-side encode on every call of a layer whose
// weights stay put.
inline bool tmap_encode_cached(CUtensorMap* m, CUtensorMapDataType elem, cuuint32_t rank, const void* base,
                               const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                               CUtensorMapSwizzle swz) {
  struct Entry {
    bool used;
    CUtensorMapDataType elem;
    cuuint32_t rank;
    const void* base;
    cuuint64_t dims[3], strides[2];
    cuuint32_t box[3];
    CUtensorMapSwizzle swz;
    CUtensorMap map;
  };
  constexpr int N = 64;
  static Entry table[N] = {};
  static int next = 0;
  static std::mutex mu;
  Entry key{};
  key.elem = elem;
  key.rank = rank;
  key.base = base;
  for (cuuint32_t i = 0; i < rank && i < 3; ++i) key.dims[i] = dims[i], key.box[i] = box[i];
  for (cuuint32_t i = 0; i + 1 < rank && i < 2; ++i) key.strides[i] = strides[i];
  key.swz = swz;
  auto same = [&](const Entry& e) {
    if (!e.used || e.elem != key.elem || e.rank != key.rank || e.base != key.base || e.swz != key.swz) return false;
    for (int i = 0; i < 3; ++i)
      if (e.dims[i] != key.dims[i] || e.box[i] != key.box[i]) return false;
    for (int i = 0; i < 2; ++i)
      if (e.strides[i] != key.strides[i]) return false;
    return true;
  };
  {
    std::lock_guard<std::mutex> lk(mu);
    for (const Entry& e : table)
      if (same(e)) {
        *m = e.map;
        return true;
      }
  }
  auto fn = tmap_encode_fn();
  if (!fn) return false;
  const cuuint32_t estr[3] = {1, 1, 1};
  if (fn(m, elem, rank, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  std::lock_guard<std::mutex> lk(mu);
  key.used = true;
  key.map = *m;
  table[next] = key;
  next = (next + 1) % N;
  return true;
}

// 2-D tensor [rows][cols] of `elem`-typed elements, row pitch `pitch_bytes`,
// loaded in boxes of box_cols x box_rows. Out-of-range elements read as zero.
inline bool tmap_2d(CUtensorMap* m, CUtensorMapDataType elem, const void* base, uint64_t rows, uint64_t cols,
                    uint64_t pitch_bytes, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle swz) {
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)pitch_bytes};
  const cuuint32_t box[2] = {box_cols, box_rows};
  return tmap_encode_cached(m, elem, 2, base, dims, strides, box, swz);
}

}  // namespace q4k
