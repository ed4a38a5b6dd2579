// C ABI of the Q4_K SwiGLU FFN library: argument validation, per-device state
// (architecture check, error word, default workspace), dispatch by regime, and
// replay of repeated decode calls from recorded CUDA graphs.
// Conventions (see include/q4kffn.h): device pointers owned by the caller,
// work enqueued on the caller's stream without synchronisation, argument
// errors returned before anything is launched (realizar
// q4k_gemv_cached_uses.rs, q4k_gemv_indexed_async: refuse a null weight
// pointer before launch; libmir micro_moe.rs: checked size arithmetic).
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "api_internal.h"
#include "common.cuh"
#include "kernels.h"
#include "q4kffn.h"

namespace {

// The device error word: a file-scope __device__ word, so that no entry point
// has to allocate device memory for it (every GPU that loads the library holds
// its own copy, zero at load). Host code turns its name into this device's
// address with cudaGetSymbolAddress once per device.
__device__ uint32_t g_error_word;

thread_local q4k_status g_last = Q4K_OK;
thread_local q4k::ProfileEvents g_prof;
thread_local int g_kernels = 0;  // kernels the last FFN or GEMV call launched (or replayed)

q4k_status fail(q4k_status s) {
  g_last = s;
  return s;
}

constexpr int MAX_DEV = 64;
constexpr int64_t MAX_DIM = int64_t(1) << 20;   // rows, columns and tokens
constexpr int64_t MAX_ELEMS = int64_t(1) << 36; // elements of one operand

struct DeviceState {
  bool checked = false;
  bool ok = false;
  int sms = 0;
  uint32_t* err = nullptr;  // device address of g_error_word on this device
  void* ws = nullptr;       // default workspace of ffn_q4k_swiglu
  size_t ws_bytes = 0;
  std::mutex mu;
};
std::mutex g_mu;
DeviceState g_dev[MAX_DEV];

q4k_status device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEV) return Q4K_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& d = g_dev[dev];
  if (!d.checked) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return Q4K_ERR_CUDA;
    d.ok = (major == 10 && minor == 3);
    if (d.ok && cudaGetSymbolAddress(reinterpret_cast<void**>(&d.err), g_error_word) != cudaSuccess) {
      (void)cudaGetLastError();
      return Q4K_ERR_CUDA;
    }
    d.checked = true;
  }
  if (!d.ok) return Q4K_ERR_ARCH;
  *out = &d;
  return Q4K_OK;
}

bool dim_ok(int64_t v) { return v > 0 && v <= MAX_DIM && v % q4k::QK == 0; }
bool tokens_ok(int64_t m) { return m >= 1 && m <= MAX_DIM; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

q4k_status check_ffn_args(const void* x, int dtype, int64_t m, int64_t hidden, int64_t inter, const void* wg,
                          const void* wu, const void* wd, const float* y) {
  if (!x || !wg || !wu || !wd || !y) return Q4K_ERR_NULL;
  if (dtype != Q4K_F32 && dtype != Q4K_BF16) return Q4K_ERR_DTYPE;
  if (!tokens_ok(m) || !dim_ok(hidden) || !dim_ok(inter)) return Q4K_ERR_SHAPE;
  if (m * hidden > MAX_ELEMS || m * inter > MAX_ELEMS || hidden * inter > MAX_ELEMS) return Q4K_ERR_SHAPE;
  if (!aligned16(x) || !aligned16(wg) || !aligned16(wu) || !aligned16(wd) || !aligned16(y)) return Q4K_ERR_ALIGN;
  return Q4K_OK;
}

// Up to DECODE_MAX tokens the call runs the decode kernels, in passes of at most
// DECODE_CHUNK tokens (four token tiles of 4). A pass streams all the weights
// once: on the LLaMA-7B FFN one 16-token pass takes 56 us and the prefill GEMM
// at one token tile 122 us, so 24 tokens take 95 us in two passes. From 25 tokens
// on the prefill GEMM runs (two passes would still win by about 8% up to 32).
constexpr int64_t DECODE_CHUNK = q4k::DECODE_PASS_MAX;
constexpr int64_t DECODE_MAX = 24;
bool is_decode(int64_t m) { return m <= DECODE_MAX; }
int64_t last_chunk(int64_t m) { return m - DECODE_CHUNK * ((m - 1) / DECODE_CHUNK); }

// x and y may be device (or managed) memory, used as is, or page-locked host
// memory mapped into the device's address space: on GB300 the host memory is
// coherent over NVLink-C2C, so the kernels then read x and write y across the
// link with no separate copy. Host memory without a device mapping (pageable,
// or registered without one) is refused, so no kernel touches an address the
// device cannot reach.
q4k_status resolve_io(const void* p, const void** out) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return Q4K_ERR_MEMORY;
  }
  if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) {
    *out = p;
    return Q4K_OK;
  }
  if (a.type == cudaMemoryTypeHost && a.devicePointer) {
    *out = a.devicePointer;
    return Q4K_OK;
  }
  return Q4K_ERR_MEMORY;
}

q4k_status resolve_xy(const void** x, float** y) {
  const void* yy = *y;
  q4k_status st = resolve_io(*x, x);
  if (st == Q4K_OK) st = resolve_io(yy, &yy);
  *y = const_cast<float*>(static_cast<const float*>(yy));
  return st;
}

size_t plan_bytes(int64_t m, int64_t hidden, int64_t inter, int sms) {
  if (is_decode(m)) {
    q4k::DecodePlan a, b;
    if (!q4k::decode_plan(std::min(m, DECODE_CHUNK), hidden, inter, sms, &a) ||
        !q4k::decode_plan(last_chunk(m), hidden, inter, sms, &b))
      return 0;
    return std::max(a.ws_bytes, b.ws_bytes);
  }
  q4k::PrefillPlan p;
  return q4k::prefill_plan(m, hidden, inter, sms, &p) ? p.ws_bytes : 0;
}

size_t plan_bytes_q8(int64_t m, int64_t hidden, int64_t inter, int sms) {
  if (is_decode(m)) {
    q4k::DecodeQ8Plan a, b;
    if (!q4k::decode_q8_plan(std::min(m, DECODE_CHUNK), hidden, inter, sms, &a) ||
        !q4k::decode_q8_plan(last_chunk(m), hidden, inter, sms, &b))
      return 0;
    return std::max(a.ws_bytes, b.ws_bytes);
  }
  return plan_bytes(m, hidden, inter, sms);
}

// Decode calls repeat with the same buffers token after token, so each distinct
// call (path, buffers, shape, dtype) is recorded once as a CUDA graph of its
// kernel launches and replayed afterwards: one graph launch instead of five
// kernel launches. The first call of a kind runs directly (which also prepares
// each kernel) and then records the graph on a private stream. Calls made while
// the caller's stream is being captured, or with the profiling hook on, launch
// directly.
struct DecodeGraph {
  bool used = false;
  int path = 0;  // 0: float32 activations, 1: Q8_1 activations, 2: Q6_K GEMV (wg = W, hidden = k, inter = n)
  const void *x = nullptr, *wg = nullptr, *wu = nullptr, *wd = nullptr, *ws = nullptr;
  float* y = nullptr;
  int dtype = 0;
  int ybf16 = 0;  // y stored as bf16
  int64_t m = 0, hidden = 0, inter = 0;
  uint64_t last = 0;
  cudaGraphExec_t exec = nullptr;
};
struct GraphCache {
  static constexpr int N = 32;
  std::mutex mu;
  DecodeGraph g[N];
  uint64_t tick = 0;
  cudaStream_t cap = nullptr;  // private stream the graphs are recorded on
};
GraphCache g_graphs[MAX_DEV];

// `launch(stream, profile)` enqueues the call's kernels on `stream`.
template <class Launch>
q4k_status run_graphed(const DecodeGraph& key, cudaStream_t s, Launch launch) {
  int dev = 0;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  const bool graphs = !g_prof.ev && cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < MAX_DEV &&
                      cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusNone;
  if (!graphs) return launch(s, g_prof) == cudaSuccess ? Q4K_OK : Q4K_ERR_CUDA;
  GraphCache& gc = g_graphs[dev];
  std::lock_guard<std::mutex> lk(gc.mu);
  ++gc.tick;
  for (DecodeGraph& g : gc.g)
    if (g.used && g.path == key.path && g.x == key.x && g.y == key.y && g.wg == key.wg && g.wu == key.wu &&
        g.wd == key.wd && g.ws == key.ws && g.dtype == key.dtype && g.ybf16 == key.ybf16 && g.m == key.m &&
        g.hidden == key.hidden && g.inter == key.inter) {
      g.last = gc.tick;
      return cudaGraphLaunch(g.exec, s) == cudaSuccess ? Q4K_OK : Q4K_ERR_CUDA;
    }
  // first call of this kind: run it directly, then record it for the next ones
  if (launch(s, q4k::ProfileEvents{}) != cudaSuccess) return Q4K_ERR_CUDA;
  if (!gc.cap && cudaStreamCreateWithFlags(&gc.cap, cudaStreamNonBlocking) != cudaSuccess) {
    gc.cap = nullptr;
    return Q4K_OK;  // no graph this time; the call itself has been issued
  }
  cudaGraph_t graph = nullptr;
  if (cudaStreamBeginCapture(gc.cap, cudaStreamCaptureModeThreadLocal) != cudaSuccess) return Q4K_OK;
  const cudaError_t le = launch(gc.cap, q4k::ProfileEvents{});
  const cudaError_t ce = cudaStreamEndCapture(gc.cap, &graph);
  cudaGraphExec_t exec = nullptr;
  if (le != cudaSuccess || ce != cudaSuccess || !graph || cudaGraphInstantiate(&exec, graph, 0) != cudaSuccess) {
    if (graph) cudaGraphDestroy(graph);
    (void)cudaGetLastError();  // a failed recording leaves the direct path as it was
    return Q4K_OK;
  }
  cudaGraphDestroy(graph);
  DecodeGraph* slot = &gc.g[0];
  for (DecodeGraph& g : gc.g) {
    if (!g.used) {
      slot = &g;
      break;
    }
    if (g.last < slot->last) slot = &g;
  }
  if (slot->used) cudaGraphExecDestroy(slot->exec);  // freed once any launch in flight completes
  *slot = key;
  slot->used = true;
  slot->last = gc.tick;
  slot->exec = exec;
  return Q4K_OK;
}

q4k_status run_decode(const q4k::DecodePlan& p, const void* x, int dtype, const void* wg, const void* wu,
                      const void* wd, void* y, int ybf16, void* ws, DeviceState* d, cudaStream_t s) {
  g_kernels += q4k::decode_kernels(p, false, ybf16, x);  // K0 (not for one token in device memory), K1, K1b, K2 (+ K3)
  DecodeGraph key;
  key.path = 0;
  key.x = x, key.wg = wg, key.wu = wu, key.wd = wd, key.ws = ws, key.y = static_cast<float*>(y);
  key.dtype = dtype, key.ybf16 = ybf16, key.m = p.m, key.hidden = p.hidden, key.inter = p.inter;
  return run_graphed(key, s, [&](cudaStream_t st, const q4k::ProfileEvents& pr) {
    return q4k::launch_decode(p, x, dtype == Q4K_BF16, wg, wu, wd, y, ws, d->err, st, pr, ybf16);
  });
}

q4k_status run_decode_q8(const q4k::DecodeQ8Plan& p, const void* x, int dtype, const void* wg, const void* wu,
                         const void* wd, float* y, void* ws, DeviceState* d, cudaStream_t s) {
  g_kernels += q4k::decode_q8_kernels(p, x);  // K0 (not for 1-2 tokens in device memory), K1, K1b, K2 (+ K3)
  DecodeGraph key;
  key.path = 1;
  key.x = x, key.wg = wg, key.wu = wu, key.wd = wd, key.ws = ws, key.y = y;
  key.dtype = dtype, key.m = p.m, key.hidden = p.hidden, key.inter = p.inter;
  return run_graphed(key, s, [&](cudaStream_t st, const q4k::ProfileEvents& pr) {
    return q4k::launch_decode_q8(p, x, dtype == Q4K_BF16, wg, wu, wd, y, ws, d->err, st, pr);
  });
}

q4k_status run_q6k(const q4k::Q6Plan& p, const void* x, int dtype, const void* w, float* y, void* ws, DeviceState* d,
                   cudaStream_t s) {
  g_kernels = 2;
  DecodeGraph key;
  key.path = 2;
  key.x = x, key.wg = w, key.ws = ws, key.y = y;
  key.dtype = dtype, key.m = p.m, key.hidden = p.k, key.inter = p.n;
  return run_graphed(key, s, [&](cudaStream_t st, const q4k::ProfileEvents& pr) {
    return q4k::launch_q6k_gemv(p, x, dtype == Q4K_BF16, w, y, ws, d->err, st, pr);
  });
}

q4k_status run_ffn(const void* x, int dtype, int64_t m, int64_t hidden, int64_t inter, const void* wg,
                   const void* wu, const void* wd, void* y, void* ws, DeviceState* d, cudaStream_t s,
                   int ybf16 = 0) {
  const int64_t yrow = hidden * (ybf16 ? 2 : 4);  // bytes of one token of y
  cudaError_t e;
  if (is_decode(m)) {
    const int64_t xrow = hidden * (dtype == Q4K_BF16 ? 2 : 4);  // bytes of one token of x
    g_kernels = 0;
    for (int64_t t0 = 0; t0 < m; t0 += DECODE_CHUNK) {
      q4k::DecodePlan p;
      if (!q4k::decode_plan(std::min(DECODE_CHUNK, m - t0), hidden, inter, d->sms, &p)) return Q4K_ERR_SHAPE;
      const q4k_status st = run_decode(p, static_cast<const uint8_t*>(x) + t0 * xrow, dtype, wg, wu, wd,
                                       static_cast<uint8_t*>(y) + t0 * yrow, ybf16, ws, d, s);
      if (st != Q4K_OK) return st;
    }
    return Q4K_OK;
  } else {
    q4k::PrefillPlan p;
    if (!q4k::prefill_plan(m, hidden, inter, d->sms, &p)) return Q4K_ERR_SHAPE;
    // x quantize+expand, MMQ, expand, MMQ (+ the split tail tiles' sum) (+ slice sum / bf16 store)
    g_kernels = q4k::prefill_kernels(p, ybf16);
    e = q4k::launch_prefill(p, x, dtype == Q4K_BF16, wg, wu, wd, y, ws, d->err, s, g_prof, ybf16);
  }
  return e == cudaSuccess ? Q4K_OK : Q4K_ERR_CUDA;
}

}  // namespace

namespace q4k {

q4k_status current_device(int* sms, uint32_t** err) {
  DeviceState* d = nullptr;
  const q4k_status st = device_state(&d);
  if (st != Q4K_OK) return st;
  *sms = d->sms;
  *err = d->err;
  return Q4K_OK;
}

q4k_status resolve_host_io(const void** x, float** y) { return resolve_xy(x, y); }

q4k_status record_failure(q4k_status s) { return fail(s); }

void record_kernels(int n) { g_kernels = n; }

}  // namespace q4k

extern "C" {

size_t q4k_weight_bytes(int64_t rows, int64_t cols) {
  if (rows <= 0 || rows > MAX_DIM || !dim_ok(cols)) return 0;
  return (size_t)rows * (size_t)(cols / q4k::QK) * q4k::BLK;
}

size_t q8_1_bytes(int64_t m, int64_t k) {
  if (!tokens_ok(m) || !dim_ok(k)) return 0;
  return (size_t)m * (size_t)k + (size_t)m * (size_t)(k / q4k::Q8B) * 8;
}

q4k_status q4k_quantize_weights(const void* W, q4k_dtype dtype, int64_t rows, int64_t cols, void* out_q4k,
                                q4k_stream_t stream) {
  if (!W || !out_q4k) return fail(Q4K_ERR_NULL);
  if (dtype != Q4K_F32 && dtype != Q4K_BF16) return fail(Q4K_ERR_DTYPE);
  if (rows <= 0 || rows > MAX_DIM || !dim_ok(cols) || rows * cols > MAX_ELEMS) return fail(Q4K_ERR_SHAPE);
  if (!aligned16(W) || !aligned16(out_q4k)) return fail(Q4K_ERR_ALIGN);
  DeviceState* d = nullptr;
  q4k_status st = device_state(&d);
  if (st != Q4K_OK) return fail(st);
  if (q4k::launch_quantize_weights(W, dtype == Q4K_BF16, rows, cols, out_q4k, d->err, (cudaStream_t)stream) !=
      cudaSuccess)
    return fail(Q4K_ERR_CUDA);
  return Q4K_OK;
}

q4k_status q8_1_quantize_act(const void* x, q4k_dtype dtype, int64_t m, int64_t k, void* out_q8,
                             q4k_stream_t stream) {
  if (!x || !out_q8) return fail(Q4K_ERR_NULL);
  if (dtype != Q4K_F32 && dtype != Q4K_BF16) return fail(Q4K_ERR_DTYPE);
  if (!tokens_ok(m) || !dim_ok(k) || m * k > MAX_ELEMS) return fail(Q4K_ERR_SHAPE);
  if (!aligned16(x) || !aligned16(out_q8)) return fail(Q4K_ERR_ALIGN);
  DeviceState* d = nullptr;
  q4k_status st = device_state(&d);
  if (st != Q4K_OK) return fail(st);
  if (q4k::launch_q8_1(x, dtype == Q4K_BF16, m, k, out_q8, (cudaStream_t)stream) != cudaSuccess)
    return fail(Q4K_ERR_CUDA);
  return Q4K_OK;
}

q4k_status ffn_q4k_swiglu(const void* x, int64_t m, int64_t hidden, int64_t inter, const void* W_gate,
                          const void* W_up, const void* W_down, float* y, q4k_stream_t stream) {
  q4k_status st = check_ffn_args(x, Q4K_F32, m, hidden, inter, W_gate, W_up, W_down, y);
  if (st != Q4K_OK) return fail(st);
  DeviceState* d = nullptr;
  st = device_state(&d);
  if (st != Q4K_OK) return fail(st);
  st = resolve_xy(&x, &y);
  if (st != Q4K_OK) return fail(st);
  std::lock_guard<std::mutex> lk(d->mu);
  const size_t need = plan_bytes(m, hidden, inter, d->sms);
  if (need == 0) return fail(Q4K_ERR_SHAPE);
  if (d->ws_bytes < need) {
    if (d->ws) cudaFree(d->ws);  // synchronises the device, so no call still uses it
    d->ws = nullptr;
    d->ws_bytes = 0;
    if (cudaMalloc(&d->ws, need) != cudaSuccess) return fail(Q4K_ERR_NOMEM);
    if (cudaMemset(d->ws, 0, need) != cudaSuccess) return fail(Q4K_ERR_CUDA);
    d->ws_bytes = need;
  }
  st = run_ffn(x, Q4K_F32, m, hidden, inter, W_gate, W_up, W_down, y, d->ws, d, (cudaStream_t)stream);
  return st == Q4K_OK ? st : fail(st);
}

q4k_status ffn_q4k_swiglu_ex(const void* x, q4k_dtype dtype, int64_t m, int64_t hidden, int64_t inter,
                             const void* W_gate, const void* W_up, const void* W_down, float* y, void* workspace,
                             size_t ws_bytes, q4k_stream_t stream) {
  q4k_status st = check_ffn_args(x, dtype, m, hidden, inter, W_gate, W_up, W_down, y);
  if (st != Q4K_OK) return fail(st);
  if (!workspace) return fail(Q4K_ERR_NULL);
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return fail(Q4K_ERR_ALIGN);
  DeviceState* d = nullptr;
  st = device_state(&d);
  if (st != Q4K_OK) return fail(st);
  st = resolve_xy(&x, &y);
  if (st != Q4K_OK) return fail(st);
  const size_t need = plan_bytes(m, hidden, inter, d->sms);
  if (need == 0) return fail(Q4K_ERR_SHAPE);
  if (ws_bytes < need) return fail(Q4K_ERR_NOMEM);
  st = run_ffn(x, dtype, m, hidden, inter, W_gate, W_up, W_down, y, workspace, d, (cudaStream_t)stream);
  return st == Q4K_OK ? st : fail(st);
}

q4k_status ffn_q4k_swiglu_q8_1(const void* x, q4k_dtype dtype, int64_t m, int64_t hidden, int64_t inter,
                               const void* W_gate, const void* W_up, const void* W_down, float* y, void* workspace,
                               size_t ws_bytes, q4k_stream_t stream) {
  q4k_status st = check_ffn_args(x, dtype, m, hidden, inter, W_gate, W_up, W_down, y);
  if (st != Q4K_OK) return fail(st);
  if (!workspace) return fail(Q4K_ERR_NULL);
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return fail(Q4K_ERR_ALIGN);
  DeviceState* d = nullptr;
  st = device_state(&d);
  if (st != Q4K_OK) return fail(st);
  st = resolve_xy(&x, &y);
  if (st != Q4K_OK) return fail(st);
  const size_t need = plan_bytes_q8(m, hidden, inter, d->sms);
  if (need == 0) return fail(Q4K_ERR_SHAPE);
  if (ws_bytes < need) return fail(Q4K_ERR_NOMEM);
  if (!is_decode(m)) {  // the prefill path already quantizes its activations to Q8_1
    st = run_ffn(x, dtype, m, hidden, inter, W_gate, W_up, W_down, y, workspace, d, (cudaStream_t)stream);
    return st == Q4K_OK ? st : fail(st);
  }
  const int64_t xrow = hidden * (dtype == Q4K_BF16 ? 2 : 4);  // bytes of one token of x
  g_kernels = 0;
  for (int64_t t0 = 0; t0 < m; t0 += DECODE_CHUNK) {
    q4k::DecodeQ8Plan p;
    if (!q4k::decode_q8_plan(std::min(DECODE_CHUNK, m - t0), hidden, inter, d->sms, &p)) return fail(Q4K_ERR_SHAPE);
    st = run_decode_q8(p, static_cast<const uint8_t*>(x) + t0 * xrow, dtype, W_gate, W_up, W_down, y + t0 * hidden,
                       workspace, d, (cudaStream_t)stream);
    if (st != Q4K_OK) return fail(st);
  }
  return Q4K_OK;
}

q4k_status ffn_q4k_swiglu_ex_y(const void* x, q4k_dtype dtype, int64_t m, int64_t hidden, int64_t inter,
                               const void* W_gate, const void* W_up, const void* W_down, void* y, q4k_dtype ydtype,
                               void* workspace, size_t ws_bytes, q4k_stream_t stream) {
  if (ydtype != Q4K_F32 && ydtype != Q4K_BF16) return fail(Q4K_ERR_DTYPE);
  q4k_status st = check_ffn_args(x, dtype, m, hidden, inter, W_gate, W_up, W_down, static_cast<const float*>(y));
  if (st != Q4K_OK) return fail(st);
  if (!workspace) return fail(Q4K_ERR_NULL);
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return fail(Q4K_ERR_ALIGN);
  DeviceState* d = nullptr;
  st = device_state(&d);
  if (st != Q4K_OK) return fail(st);
  const void* yy = y;
  st = resolve_io(x, &x);
  if (st == Q4K_OK) st = resolve_io(y, &yy);
  if (st != Q4K_OK) return fail(st);
  const size_t need = plan_bytes(m, hidden, inter, d->sms);
  if (need == 0) return fail(Q4K_ERR_SHAPE);
  if (ws_bytes < need) return fail(Q4K_ERR_NOMEM);
  st = run_ffn(x, dtype, m, hidden, inter, W_gate, W_up, W_down, const_cast<void*>(yy), workspace, d,
               (cudaStream_t)stream, ydtype == Q4K_BF16);
  return st == Q4K_OK ? st : fail(st);
}

size_t ffn_q4k_q8_1_workspace_bytes(int64_t m, int64_t hidden, int64_t inter) {
  if (!tokens_ok(m) || !dim_ok(hidden) || !dim_ok(inter)) return 0;
  DeviceState* d = nullptr;
  if (device_state(&d) != Q4K_OK) return 0;
  return plan_bytes_q8(m, hidden, inter, d->sms);
}

size_t ffn_q4k_q8_1_workspace_h_offset(int64_t m, int64_t hidden, int64_t inter) {
  if (!tokens_ok(m) || !dim_ok(hidden) || !dim_ok(inter)) return 0;
  DeviceState* d = nullptr;
  if (device_state(&d) != Q4K_OK) return 0;
  if (is_decode(m)) {
    q4k::DecodeQ8Plan p;  // one decode pass holds one h; calls of several passes have none to show
    return m <= DECODE_CHUNK && q4k::decode_q8_plan(m, hidden, inter, d->sms, &p) ? p.off_hq : 0;
  }
  q4k::PrefillPlan p;
  return q4k::prefill_plan(m, hidden, inter, d->sms, &p) ? p.off_hq : 0;
}

size_t q6k_weight_bytes(int64_t rows, int64_t cols) {
  if (rows <= 0 || rows > MAX_DIM || !dim_ok(cols)) return 0;
  return (size_t)rows * (size_t)(cols / q4k::QK) * 210;
}

size_t q6k_gemv_workspace_bytes(int64_t m, int64_t n, int64_t k) {
  DeviceState* d = nullptr;
  if (device_state(&d) != Q4K_OK) return 0;
  q4k::Q6Plan p;
  return q4k::q6k_plan(m, n, k, d->sms, &p) ? p.ws_bytes : 0;
}

q4k_status q6k_gemv(const void* x, q4k_dtype dtype, int64_t m, int64_t n, int64_t k, const void* W, float* y,
                    void* workspace, size_t ws_bytes, q4k_stream_t stream) {
  if (!x || !W || !y || !workspace) return fail(Q4K_ERR_NULL);
  if (dtype != Q4K_F32 && dtype != Q4K_BF16) return fail(Q4K_ERR_DTYPE);
  if (m < 1 || m > 8 || n < 16 || n > MAX_DIM || n % 16 != 0 || !dim_ok(k) || k > 8192) return fail(Q4K_ERR_SHAPE);
  if (!aligned16(x) || !aligned16(W) || !aligned16(y) || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(Q4K_ERR_ALIGN);
  DeviceState* d = nullptr;
  q4k_status st = device_state(&d);
  if (st != Q4K_OK) return fail(st);
  st = resolve_xy(&x, &y);
  if (st != Q4K_OK) return fail(st);
  q4k::Q6Plan p;
  if (!q4k::q6k_plan(m, n, k, d->sms, &p)) return fail(Q4K_ERR_SHAPE);
  if (ws_bytes < p.ws_bytes) return fail(Q4K_ERR_NOMEM);
  st = run_q6k(p, x, dtype, W, y, workspace, d, (cudaStream_t)stream);
  return st == Q4K_OK ? st : fail(st);
}

q4k_status q6k_dequantize(const void* q6k, int64_t rows, int64_t cols, float* out, q4k_stream_t stream) {
  if (!q6k || !out) return fail(Q4K_ERR_NULL);
  if (rows <= 0 || rows > MAX_DIM || !dim_ok(cols) || rows * cols > MAX_ELEMS) return fail(Q4K_ERR_SHAPE);
  if (!aligned16(out)) return fail(Q4K_ERR_ALIGN);
  DeviceState* d = nullptr;
  q4k_status st = device_state(&d);
  if (st != Q4K_OK) return fail(st);
  if (q4k::launch_q6k_dequant(q6k, out, rows, cols, (cudaStream_t)stream) != cudaSuccess) return fail(Q4K_ERR_CUDA);
  return Q4K_OK;
}

size_t ffn_q4k_workspace_bytes(int64_t m, int64_t hidden, int64_t inter) {
  if (!tokens_ok(m) || !dim_ok(hidden) || !dim_ok(inter)) return 0;
  DeviceState* d = nullptr;
  if (device_state(&d) != Q4K_OK) return 0;
  return plan_bytes(m, hidden, inter, d->sms);
}

size_t ffn_q4k_workspace_h_q8_1_offset(int64_t m, int64_t hidden, int64_t inter) {
  if (!tokens_ok(m) || !dim_ok(hidden) || !dim_ok(inter) || is_decode(m)) return 0;
  DeviceState* d = nullptr;
  if (device_state(&d) != Q4K_OK) return 0;
  q4k::PrefillPlan p;
  return q4k::prefill_plan(m, hidden, inter, d->sms, &p) ? p.off_hq : 0;
}

q4k_status q4k_dequantize(const void* q4k_, int64_t rows, int64_t cols, float* out, q4k_stream_t stream) {
  if (!q4k_ || !out) return fail(Q4K_ERR_NULL);
  if (rows <= 0 || rows > MAX_DIM || !dim_ok(cols) || rows * cols > MAX_ELEMS) return fail(Q4K_ERR_SHAPE);
  if (!aligned16(q4k_) || !aligned16(out)) return fail(Q4K_ERR_ALIGN);
  DeviceState* d = nullptr;
  q4k_status st = device_state(&d);
  if (st != Q4K_OK) return fail(st);
  if (q4k::launch_dequant(q4k_, out, rows, cols, (cudaStream_t)stream) != cudaSuccess) return fail(Q4K_ERR_CUDA);
  return Q4K_OK;
}

q4k_status q4k_check_device_error(q4k_stream_t stream) {
  DeviceState* d = nullptr;
  q4k_status st = device_state(&d);
  if (st != Q4K_OK) return fail(st);
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return fail(Q4K_ERR_CUDA);
  uint32_t word = 0;
  if (cudaMemcpy(&word, d->err, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return fail(Q4K_ERR_CUDA);
  if (word && cudaMemset(d->err, 0, sizeof(word)) != cudaSuccess) return fail(Q4K_ERR_CUDA);
  if (word & q4k::ERRBIT_TIMEOUT) return fail(Q4K_ERR_TIMEOUT);
  if (word & q4k::ERRBIT_RANGE) return fail(Q4K_ERR_RANGE);
  return Q4K_OK;
}

namespace {
// One warp waits on an mbarrier that nothing will complete, through the same
// bounded wait as the FFN kernels, then returns: the wait gives up after
// limit_ns and records the timeout in the device error word.
__global__ void bounded_wait_probe_kernel(uint64_t limit_ns, uint32_t* err) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    q4k::mbar_init(&bar, 1);
    q4k::fence_mbar_init();
  }
  __syncwarp();
  (void)q4k::mbar_wait(&bar, 0u, err, limit_ns);
}
}  // namespace

q4k_status q4k_test_bounded_wait(uint64_t limit_ns, q4k_stream_t stream) {
  if (limit_ns < 1000 || limit_ns > q4k::WAIT_LIMIT_NS) return fail(Q4K_ERR_SHAPE);
  DeviceState* d = nullptr;
  q4k_status st = device_state(&d);
  if (st != Q4K_OK) return fail(st);
  bounded_wait_probe_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(limit_ns, d->err);
  return cudaGetLastError() == cudaSuccess ? Q4K_OK : fail(Q4K_ERR_CUDA);
}

q4k_status q4k_set_profile_events(void* const* events, int n) {
  if (n < 0 || (n > 0 && !events)) return fail(Q4K_ERR_NULL);
  g_prof.ev = n > 0 ? reinterpret_cast<cudaEvent_t*>(const_cast<void**>(events)) : nullptr;
  g_prof.n = n;
  return Q4K_OK;
}

q4k_status q4k_get_last_error(void) { return g_last; }

int q4k_last_call_kernels(void) { return g_kernels; }

const char* q4k_status_string(q4k_status s) {
  switch (s) {
    case Q4K_OK: return "ok";
    case Q4K_ERR_NULL: return "null pointer";
    case Q4K_ERR_SHAPE: return "invalid shape";
    case Q4K_ERR_ALIGN: return "pointer not 16-byte aligned";
    case Q4K_ERR_DTYPE: return "unsupported dtype";
    case Q4K_ERR_CUDA: return "CUDA error";
    case Q4K_ERR_ARCH: return "device is not sm_103";
    case Q4K_ERR_TIMEOUT: return "bounded device wait timed out";
    case Q4K_ERR_NOMEM: return "workspace allocation failed or too small";
    case Q4K_ERR_RANGE: return "quantized scale outside the fp16 range";
    case Q4K_ERR_MEMORY: return "pointer is neither device memory nor mapped page-locked host memory";
  }
  return "unknown status";
}

}  // extern "C"
