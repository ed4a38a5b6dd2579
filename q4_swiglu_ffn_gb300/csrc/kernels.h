// Host-side launch interface of the sm_103a kernels (internal to the library).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace q4k {

// Optional per-kernel timing: when ev != nullptr, the FFN launchers record
// ev[2i] before and ev[2i+1] after their i-th kernel (i < n / 2) on the call's stream.
struct ProfileEvents {
  cudaEvent_t* ev = nullptr;
  int n = 0;
  void before(int i, cudaStream_t s) const { if (ev && 2 * i + 1 < n) cudaEventRecord(ev[2 * i], s); }
  void after(int i, cudaStream_t s) const { if (ev && 2 * i + 1 < n) cudaEventRecord(ev[2 * i + 1], s); }
};

cudaError_t launch_dequant(const void* w, float* out, int64_t rows, int64_t cols, cudaStream_t s);
cudaError_t launch_q8_1(const void* x, int bf16, int64_t m, int64_t k, void* out, cudaStream_t s);
cudaError_t launch_quantize_weights(const void* w, int bf16, int64_t rows, int64_t cols, void* out,
                                    uint32_t* err, cudaStream_t s);

// ---------------------------------------------------------------- decode (m <= 16 per pass)
constexpr int DECODE_PASS_MAX = 16;  // tokens of one decode pass

// The allocation-free decode entry point: its static scratch array and the
// largest shapes it accepts (every such shape's plan fits in the array).
constexpr size_t NOALLOC_SCRATCH_BYTES = size_t(16) << 20;
constexpr int NOALLOC_MAX_TOKENS = 8;
constexpr int NOALLOC_MAX_DIM = 16384;
struct DecodePlan {
  int m, hidden, inter;
  int nt;              // n-tiles of 4 tokens (1 to 4)
  int nks1, kc1;       // gate/up K-chunks and superblock groups per chunk
  int nks2, kc2;       // down K-chunks and superblock groups per chunk
  int grid1, grid2;    // CTAs
  size_t ws_bytes;     // workspace bytes
  // workspace offsets (bytes): fragments of x and of h, gate/up and down chunk sums
  size_t off_fx1, off_fm1, off_sc1, off_fx2, off_fm2, off_sc2, off_p1, off_p2;
};
bool decode_plan(int64_t m, int64_t hidden, int64_t inter, int num_sms, DecodePlan* p);
// Kernels one launch_decode call enqueues (q8: with q8h; x as passed to launch_decode).
int decode_kernels(const DecodePlan& p, bool q8, int ybf16, const void* x);
// x (or any pointer) is in device or managed memory (not page-locked host memory).
bool device_resident(const void* p);
// y is float32, or bf16 when ybf16 (rounded once by the final chunk-sum kernel).
// With q8h, x and h are rounded to Q8_1 before they become the B operand, and the
// Q8_1 of h (quants [m][inter], then (d, s) [m][inter/32]) is stored at q8h.
cudaError_t launch_decode(const DecodePlan& p, const void* x, int bf16, const void* wg, const void* wu, const void* wd,
                          void* y, void* ws, uint32_t* err, cudaStream_t s, const ProfileEvents& prof, int ybf16 = 0,
                          uint8_t* q8h = nullptr);

// ---------------------------------------------------------------- decode with Q8_1 activations (m <= 16 per pass)
struct DecodeQ8Plan {
  int m, hidden, inter;
  int mt;              // tokens the GEMV kernels are compiled for (1, 2, 4 or 8; >= m)
  int fpath;           // 3-16 tokens: the float32 path's kernels on Q8_1-rounded activations (fp below)
  DecodePlan fp;       // that path's plan; its workspace starts at off_fp
  int nks1, kc1;       // gate/up K-chunks and superblock groups per chunk
  int nks2, kc2;       // down K-chunks and superblock groups per chunk
  int grid1, grid2;    // CTAs
  size_t ws_bytes;     // workspace bytes
  // workspace offsets (bytes): planar Q8_1 of x and of h, gate/up and down chunk sums
  size_t off_xq, off_hq, off_p1, off_p2, off_fp;
};
int decode_q8_tokens(int64_t m);
bool decode_q8_plan(int64_t m, int64_t hidden, int64_t inter, int num_sms, DecodeQ8Plan* p);
cudaError_t launch_decode_q8(const DecodeQ8Plan& p, const void* x, int bf16, const void* wg, const void* wu,
                             const void* wd, void* y, void* ws, uint32_t* err, cudaStream_t s,
                             const ProfileEvents& prof, int ybf16 = 0);
// Kernels one launch_decode_q8 call enqueues (x as passed to it).
int decode_q8_kernels(const DecodeQ8Plan& p, const void* x);

// ---------------------------------------------------------------- Q6_K GEMV (m <= 8)
struct Q6Plan {
  int m, n, k;
  int nt;              // n-tiles of 4 tokens (1 or 2)
  int cps, grid;       // CTAs per SM and CTAs
  size_t smem;         // dynamic shared memory per CTA
  size_t ws_bytes;     // workspace bytes
  size_t off_fx, off_sc;  // workspace offsets: B fragments of x and their 2^e factors
};
bool q6k_plan(int64_t m, int64_t n, int64_t k, int num_sms, Q6Plan* p);
cudaError_t launch_q6k_gemv(const Q6Plan& p, const void* x, int bf16, const void* w, float* y, void* ws,
                            uint32_t* err, cudaStream_t s, const ProfileEvents& prof);
cudaError_t launch_q6k_dequant(const void* w, float* out, int64_t rows, int64_t cols, cudaStream_t s);

// ---------------------------------------------------------------- prefill (m >= 25)
struct PrefillPlan {
  int m, hidden, inter;
  size_t ws_bytes;
  size_t off_xq, off_hq;  // planar Q8_1 of x and of h
  size_t off_xop, off_hop;  // tensor-core operands
  size_t off_misc;
  int ksplit;             // K slices of the down projection
  int num_sms;            // SMs (resident CTAs of the GEMMs, for their tile order)
  int tail_whole, tail_q; // down projection: tiles from tail_whole on split into tail_q K slices
  size_t off_tail;        // their partial tiles
  int gu_whole, gu_q;     // the same for the gate/up projection (its SwiGLU after the slices' sum)
  size_t off_gtail;       // their partial tiles
  size_t off_ypart;       // their partial outputs [ksplit][m][hidden] (ksplit > 1)
};
bool prefill_plan(int64_t m, int64_t hidden, int64_t inter, int num_sms, PrefillPlan* p);
// Kernels one prefill call launches.
int prefill_kernels(const PrefillPlan& p, int ybf16);
cudaError_t launch_prefill(const PrefillPlan& p, const void* x, int bf16, const void* wg, const void* wu,
                           const void* wd, void* y, void* ws, uint32_t* err, cudaStream_t s,
                           const ProfileEvents& prof, int ybf16 = 0);

}  // namespace q4k
