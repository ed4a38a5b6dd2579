// Decode-regime feed-forward entry point that allocates no device memory.
//
// Some callers cannot call cudaMalloc: a serving process that hands all device
// memory to its own pool at start-up and forbids later allocations, or a
// latency-critical loop in which cudaMalloc/cudaFree (which may synchronise
// the whole device) are not acceptable. ffn_q4k_swiglu grows a workspace with
// cudaMalloc and ffn_q4k_swiglu_ex needs the caller to allocate one; this entry
// point instead runs the decode kernels on a fixed scratch array that lives in
// the library image itself (a file-scope __device__ array, present on every
// GPU that loads the library, until the process exits).
#include <cstdint>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "q4kffn.h"

namespace {

// Large enough for every decode shape with m <= 8 and hidden, inter <= 16384 (the
// largest of them needs about 13 MiB, depending on the SM count).
constexpr size_t NOALLOC_SCRATCH_BYTES = size_t(16) << 20;

static __device__ __align__(256) uint8_t g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];
static __device__ uint32_t g_noalloc_err;  // device error word of this entry point

struct NoallocDevice {
  bool ready = false;
  bool ok = false;
  int sms = 0;
  void* scratch = nullptr;  // device address of g_noalloc_scratch on this device
  uint32_t* err = nullptr;  // device address of g_noalloc_err on this device
};
std::mutex g_noalloc_mu;
NoallocDevice g_noalloc_dev[64];

// Once per device, with that device current: check the architecture and turn the
// host-side names of the static arrays into device addresses.
q4k_status noalloc_setup(NoallocDevice** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return Q4K_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  NoallocDevice& d = g_noalloc_dev[dev];
  if (!d.ready) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return Q4K_ERR_CUDA;
    d.ok = (major == 10 && minor == 3);
    if (d.ok) {
      if (cudaGetSymbolAddress(&d.scratch, g_noalloc_scratch) != cudaSuccess) return Q4K_ERR_CUDA;
      if (cudaGetSymbolAddress(reinterpret_cast<void**>(&d.err), g_noalloc_err) != cudaSuccess)
        return Q4K_ERR_CUDA;
    }
    d.ready = true;
  }
  if (!d.ok) return Q4K_ERR_ARCH;
  *out = &d;
  return Q4K_OK;
}

}  // namespace

extern "C" q4k_status ffn_q4k_swiglu_noalloc(const void* x, int64_t m, int64_t hidden, int64_t inter,
                                             const void* W_gate, const void* W_up, const void* W_down, float* y,
                                             q4k_stream_t stream) {
  if (!x || !W_gate || !W_up || !W_down || !y) return Q4K_ERR_NULL;
  if (m < 1 || m > 8) return Q4K_ERR_SHAPE;  // decode regime only
  if (hidden <= 0 || inter <= 0 || hidden % q4k::QK || inter % q4k::QK || hidden > 16384 || inter > 16384)
    return Q4K_ERR_SHAPE;
  const uintptr_t any = reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(W_gate) |
                        reinterpret_cast<uintptr_t>(W_up) | reinterpret_cast<uintptr_t>(W_down) |
                        reinterpret_cast<uintptr_t>(y);
  if (any & 15u) return Q4K_ERR_ALIGN;
  NoallocDevice* d = nullptr;
  q4k_status st = noalloc_setup(&d);
  if (st != Q4K_OK) return st;
  q4k::DecodePlan p;
  if (!q4k::decode_plan(m, hidden, inter, d->sms, &p)) return Q4K_ERR_SHAPE;
  if (p.ws_bytes > NOALLOC_SCRATCH_BYTES) return Q4K_ERR_NOMEM;  // shape needs more scratch than the array holds
  const cudaError_t e = q4k::launch_decode(p, x, 0, W_gate, W_up, W_down, y, d->scratch, d->err,
                                           static_cast<cudaStream_t>(stream), q4k::ProfileEvents{});
  return e == cudaSuccess ? Q4K_OK : Q4K_ERR_CUDA;
}
