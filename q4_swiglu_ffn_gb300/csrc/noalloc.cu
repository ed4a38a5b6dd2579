// Decode-regime feed-forward entry point that allocates no device memory.
//
// Some callers cannot call cudaMalloc: a serving process that hands all device
// memory to its own pool at start-up and forbids later allocations, or a
// latency-critical loop in which cudaMalloc/cudaFree (which may synchronise
// the whole device) are not acceptable. ffn_q4k_swiglu grows a workspace with
// cudaMalloc and ffn_q4k_swiglu_ex needs the caller to allocate one; this entry
// point instead runs the decode kernels on a fixed scratch array that lives in
// the library image itself (a file-scope __device__ array, present on every
// GPU that loads the library, until the process exits). Its device wait
// timeouts go to the library's error word (itself a static __device__ word),
// so q4k_check_device_error reports them like any other call's.
#include <cstdint>
#include <mutex>

#include "api_internal.h"
#include "common.cuh"
#include "kernels.h"
#include "q4kffn.h"

namespace {

static __device__ __align__(256) uint8_t g_noalloc_scratch[q4k::NOALLOC_SCRATCH_BYTES];

std::mutex g_noalloc_mu;
void* g_noalloc_scratch_addr[64];  // device address of g_noalloc_scratch, per device (null until resolved)

// Once per device, with that device current: turn the host-side name of the
// static array into this device's address of it.
q4k_status noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return Q4K_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) {
      (void)cudaGetLastError();
      return Q4K_ERR_CUDA;
    }
    g_noalloc_scratch_addr[dev] = p;
  }
  *out = g_noalloc_scratch_addr[dev];
  return Q4K_OK;
}

q4k_status noalloc_call(const void* x, int64_t m, int64_t hidden, int64_t inter, const void* W_gate,
                        const void* W_up, const void* W_down, float* y, q4k_stream_t stream) {
  if (!x || !W_gate || !W_up || !W_down || !y) return Q4K_ERR_NULL;
  if (m < 1 || m > q4k::NOALLOC_MAX_TOKENS) return Q4K_ERR_SHAPE;  // decode regime only
  if (hidden <= 0 || inter <= 0 || hidden % q4k::QK || inter % q4k::QK || hidden > q4k::NOALLOC_MAX_DIM ||
      inter > q4k::NOALLOC_MAX_DIM)
    return Q4K_ERR_SHAPE;
  const uintptr_t any = reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(W_gate) |
                        reinterpret_cast<uintptr_t>(W_up) | reinterpret_cast<uintptr_t>(W_down) |
                        reinterpret_cast<uintptr_t>(y);
  if (any & 15u) return Q4K_ERR_ALIGN;
  int sms = 0;
  uint32_t* err = nullptr;
  q4k_status st = q4k::current_device(&sms, &err);
  if (st != Q4K_OK) return st;
  st = q4k::resolve_host_io(&x, &y);  // device memory, or mapped page-locked host memory
  if (st != Q4K_OK) return st;
  void* scratch = nullptr;
  st = noalloc_scratch(&scratch);
  if (st != Q4K_OK) return st;
  q4k::DecodePlan p;
  if (!q4k::decode_plan(m, hidden, inter, sms, &p)) return Q4K_ERR_SHAPE;
  if (p.ws_bytes > q4k::NOALLOC_SCRATCH_BYTES) return Q4K_ERR_NOMEM;  // more scratch than the array holds
  q4k::record_kernels(q4k::decode_kernels(p, false, 0, x));          // K0 (not for one token in device memory), K1, K1b, K2 (+ K3)
  const cudaError_t e = q4k::launch_decode(p, x, 0, W_gate, W_up, W_down, y, scratch, err,
                                           static_cast<cudaStream_t>(stream), q4k::ProfileEvents{});
  return e == cudaSuccess ? Q4K_OK : Q4K_ERR_CUDA;
}

}  // namespace

extern "C" q4k_status ffn_q4k_swiglu_noalloc(const void* x, int64_t m, int64_t hidden, int64_t inter,
                                             const void* W_gate, const void* W_up, const void* W_down, float* y,
                                             q4k_stream_t stream) {
  const q4k_status st = noalloc_call(x, m, hidden, inter, W_gate, W_up, W_down, y, stream);
  return st == Q4K_OK ? st : q4k::record_failure(st);
}
