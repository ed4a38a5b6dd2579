/*
 * q4kffn.h -- C ABI of the GB300 (sm_103a) Q4_K SwiGLU feed-forward library.
 *
 * The library computes the LLaMA-style feed-forward block
 *     y = W_down . ( silu(W_gate . x) * (W_up . x) )
 * with weights stored as rows of GGML Q4_K blocks (256 weights in 144 bytes:
 * fp16 d, fp16 dmin, 12 bytes of packed 6-bit scales and mins for 8
 * sub-blocks of 32, 128 bytes of 4-bit quants).
 *   Source: realizar src/cuda/executor/layers/ffn.rs, fused_ffn_swiglu_gpu
 *   ("down(swiglu(gate(x), up(x)))", gate and up over the same input, all
 *   launches chained on one stream with no synchronisation) and
 *   fused_ffn_swiglu_gpu_true_dp4a (activations quantized to Q8_1 once for
 *   gate and up, the activated vector re-quantized before down);
 *   spark_model/layers/ops/q4k_mmq.rs (QK_K = 256, 144-byte blocks,
 *   q4k_weight_bytes, quantize_act_q8_1, q4k_mmq_gemm, quantize_weight_q4k).
 *
 * Conventions for every entry point
 *   - Pointers are DEVICE pointers owned by the caller unless a comment says
 *     otherwise; the library never frees them. They must be 16-byte aligned.
 *   - For ffn_q4k_swiglu, ffn_q4k_swiglu_ex, ffn_q4k_swiglu_q8_1 and q6k_gemv,
 *     x and y may also be page-locked host memory mapped into the device's
 *     address space (cudaHostAlloc / cudaHostRegister, which map by default
 *     under unified addressing). GB300's host memory is coherent over
 *     NVLink-C2C, so the kernels then read x and write y across the link
 *     directly, with no separate copy. Other host memory (pageable, or without
 *     a device mapping) returns Q4K_ERR_MEMORY before anything is launched.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and the call returns without synchronising.
 *   - Argument errors are detected on the host before anything is launched and
 *     returned synchronously; nothing is written in that case.
 *   - Faults inside kernels (a bounded device wait that ran out, a weight
 *     block whose scale would overflow fp16) are recorded in a per-device
 *     error word and returned by q4k_check_device_error().
 *   - Shapes: hidden and inter (and every quantized dimension) must be
 *     positive multiples of 256; m >= 1.
 *   - Layouts: x and y are row-major [m][hidden]. W_gate and W_up hold `inter`
 *     rows of hidden/256 blocks, W_down holds `hidden` rows of inter/256
 *     blocks (row = output feature, blocks run along the input dimension;
 *     realizar q4k_gemv_cached_uses.rs, q4k_gemv_cached: n = output, k = input).
 *   - Regimes: m <= 24 runs the decode path (float32 activations, no
 *     activation quantization) in passes of at most 16 tokens; m >= 25 runs the
 *     prefill path (activations quantized to Q8_1, Q4_K x Q8_1 GEMM on the
 *     tensor cores). ffn_q4k_swiglu_q8_1 quantizes the activations to Q8_1 at
 *     every m (decode passes up to 24 tokens, the prefill path above).
 */
#ifndef Q4KFFN_H
#define Q4KFFN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  Q4K_OK = 0,
  Q4K_ERR_NULL = 1,      /* a required pointer is NULL                                 */
  Q4K_ERR_SHAPE = 2,     /* dim not a positive multiple of 256, m < 1, or size overflow */
  Q4K_ERR_ALIGN = 3,     /* a pointer is not 16-byte aligned                           */
  Q4K_ERR_DTYPE = 4,     /* unknown activation dtype                                   */
  Q4K_ERR_CUDA = 5,      /* a CUDA runtime call or launch failed                       */
  Q4K_ERR_ARCH = 6,      /* current device is not compute capability 10.3              */
  Q4K_ERR_TIMEOUT = 7,   /* a bounded device wait ran out (reported after the fact)    */
  Q4K_ERR_NOMEM = 8,     /* workspace allocation failed or caller workspace too small  */
  Q4K_ERR_RANGE = 9,     /* weight quantizer: a block scale does not fit in fp16       */
  Q4K_ERR_MEMORY = 10    /* x or y is neither device memory nor mapped pinned host memory */
} q4k_status;

typedef enum { Q4K_F32 = 0, Q4K_BF16 = 1 } q4k_dtype;

/* A cudaStream_t passed as an opaque handle. */
typedef void* q4k_stream_t;

/* Bytes of a Q4_K matrix of `rows` rows of `cols` inputs: rows*(cols/256)*144.
 * Source: spark_model/layers/ops/q4k_mmq.rs, q4k_weight_bytes. Returns 0 for an
 * invalid shape. */
size_t q4k_weight_bytes(int64_t rows, int64_t cols);

/* Bytes of a planar Q8_1 buffer for [m][k] activations: m*k int8 quants followed
 * by m*(k/32) {float d, float s} pairs (d = block scale, s = d * sum of the 32
 * quants). Returns 0 for an invalid shape. */
size_t q8_1_bytes(int64_t m, int64_t k);

/* Quantize float32 or bf16 weights [rows][cols] (row-major) to Q4_K blocks.
 * Source: spark_model/layers/ops/q4k_mmq.rs, quantize_weight_q4k (load-time
 * bf16 -> block_q4_K); the pages give no algorithm, so this is a deterministic
 * min-max quantizer: per block, dmin is the smallest fp16 with 63*dmin covering
 * the largest sub-block negative range, each 6-bit min the smallest integer
 * covering its sub-block, d the smallest fp16 with 945*d covering the largest
 * (max + dmin*min), each 6-bit scale the smallest integer covering its
 * sub-block, and q = round((x + dmin*min)/(d*scale)) clamped to 0..15, all in
 * float64 with one rounding per operation. Every value ends within half a
 * quant step of its input. out_q4k: q4k_weight_bytes(rows, cols) bytes.
 * A block whose scale would exceed 65504 sets Q4K_ERR_RANGE in the device
 * error word (that block is written with zeros). */
q4k_status q4k_quantize_weights(const void* W, q4k_dtype dtype, int64_t rows, int64_t cols,
                                void* out_q4k, q4k_stream_t stream);

/* Quantize float32 or bf16 activations [m][k] to planar Q8_1 (see q8_1_bytes).
 * Source: realizar ffn.rs, fused_ffn_swiglu_gpu_true_dp4a ("per-block scale +
 * 32 x int8"); spark_model q4k_mmq.rs, quantize_act_q8_1. Per block of 32, in
 * float32 with one rounding per operation: d = amax/127, inv = 127/amax,
 * q = round(x*inv) ties away from zero, s = d*sum(q); an all-zero block gives
 * zeros. bf16 input is widened exactly. Output is bit-exact with that rule. */
q4k_status q8_1_quantize_act(const void* x, q4k_dtype dtype, int64_t m, int64_t k,
                             void* out_q8, q4k_stream_t stream);

/* The feed-forward block with float32 activations x [m][hidden] and float32
 * output y [m][hidden]. Uses a per-device workspace that the library grows on
 * demand (cudaMalloc, guarded by a mutex, kept until process exit). The first
 * call on a device also checks that it is an sm_103 part. Concurrent calls on
 * different streams of one device must use ffn_q4k_swiglu_ex with separate
 * workspaces. y must not alias x or the weights. */
q4k_status ffn_q4k_swiglu(const void* x, int64_t m, int64_t hidden, int64_t inter,
                          const void* W_gate, const void* W_up, const void* W_down,
                          float* y, q4k_stream_t stream);

/* As ffn_q4k_swiglu, with an explicit activation dtype (Q4K_F32 or Q4K_BF16)
 * and a caller-owned device workspace of at least
 * ffn_q4k_workspace_bytes(m, hidden, inter) bytes, 256-byte aligned. Its
 * contents need no initialisation (every call sets up what it reads). Calls
 * sharing one workspace must not overlap on the GPU. */
q4k_status ffn_q4k_swiglu_ex(const void* x, q4k_dtype dtype, int64_t m, int64_t hidden,
                             int64_t inter, const void* W_gate, const void* W_up,
                             const void* W_down, float* y, void* workspace, size_t ws_bytes,
                             q4k_stream_t stream);

/* As ffn_q4k_swiglu_ex, with the dtype of y: Q4K_F32, or Q4K_BF16 (each output
 * is the float32 result rounded once to bf16, round to nearest even, by the
 * final kernel that sums the down projection's K-chunks). Source: spark_model/
 * layers/ops/q4k_mmq.rs, q4k_mmq_gemm (the MMQ's fused bf16 store). y is
 * [m][hidden] of that dtype; the workspace is sized by ffn_q4k_workspace_bytes. */
q4k_status ffn_q4k_swiglu_ex_y(const void* x, q4k_dtype dtype, int64_t m, int64_t hidden,
                               int64_t inter, const void* W_gate, const void* W_up,
                               const void* W_down, void* y, q4k_dtype ydtype, void* workspace,
                               size_t ws_bytes, q4k_stream_t stream);
/* The feed-forward block with Q8_1 activations at every m: x is quantized to
 * Q8_1 once and shared by the gate and up projections, h = silu(g) * u is
 * re-quantized to Q8_1 before the down projection, and every dot product is
 * the Q4_K x Q8_1 block product
 *     d * sum_j scale_j * d8_j * sum_i(q_i * q8_i) - dmin * sum_j min_j * s8_j
 * with exact integer inner sums. Source: realizar src/cuda/executor/layers/
 * ffn.rs, fused_ffn_swiglu_gpu_true_dp4a (the decode pipeline with quantized
 * activations and integer dot products); spark_model/layers/ops/q4k_mmq.rs,
 * q4k_mmq_gemm (the block correction). For m = 1..24 it runs decode passes of at
 * most 16 tokens (x Q8_1, gate+up GEMV, chunk sum + SwiGLU + Q8_1 of h, down GEMV,
 * down chunk sum); a pass of 1-2 tokens forms integer dot products, one of 3-16
 * tokens multiplies the dequantized Q8_1 values (q * d) on the fp16 tensor cores
 * with float32 accumulation; for m >= 25 it is the same computation as
 * ffn_q4k_swiglu_ex's prefill path (and gives the same bytes). x is float32 or bf16 [m][hidden] (bf16 is
 * widened exactly before quantization), y float32 [m][hidden]. The workspace is
 * caller-owned, 256-byte aligned, of at least ffn_q4k_q8_1_workspace_bytes(m,
 * hidden, inter) bytes, needs no initialisation, and must not be shared by
 * calls that overlap on the GPU. Repeated decode calls with the same buffers
 * are replayed from a recorded CUDA graph, as for ffn_q4k_swiglu. */
q4k_status ffn_q4k_swiglu_q8_1(const void* x, q4k_dtype dtype, int64_t m, int64_t hidden,
                               int64_t inter, const void* W_gate, const void* W_up,
                               const void* W_down, float* y, void* workspace, size_t ws_bytes,
                               q4k_stream_t stream);
/* Workspace bytes ffn_q4k_swiglu_q8_1 needs for this shape (0 for an invalid shape). */
size_t ffn_q4k_q8_1_workspace_bytes(int64_t m, int64_t hidden, int64_t inter);
/* Test hook: byte offset, inside an ffn_q4k_swiglu_q8_1 workspace, of the
 * planar Q8_1 copy of h = silu(gate)*up (q8_1_bytes(m, inter) bytes) that the
 * call feeds to the down projection; 0 for an invalid shape and for 9..24
 * tokens (several decode passes, each with its own h). */
size_t ffn_q4k_q8_1_workspace_h_offset(int64_t m, int64_t hidden, int64_t inter);
/* Decode-regime variant of ffn_q4k_swiglu (float32 x, m = 1..8, hidden and
 * inter multiples of 256 up to 16384) that allocates no device memory, for
 * callers that cannot call cudaMalloc: a serving process whose memory pool owns
 * all device memory after start-up, or a latency-critical loop that cannot
 * afford cudaMalloc's possible device-wide synchronisation. It has no
 * counterpart on the source pages. Its scratch is a 16 MiB array inside the
 * library image (a file-scope __device__ array that every GPU loading the
 * library holds until the process exits), enough for every accepted shape; m
 * outside 1..8 or a dimension above 16384 returns Q4K_ERR_SHAPE, and a shape
 * whose scratch would still exceed 16 MiB returns Q4K_ERR_NOMEM, both without
 * launching. x and y follow the other FFN entry points: device memory, or
 * mapped page-locked host memory (anything else returns Q4K_ERR_MEMORY before
 * launch). The first call on a device checks the architecture and resolves
 * the array's device address (cudaGetSymbolAddress), so make that first call
 * before any stream capture. Every call on a device shares the one array and
 * each call re-initialises what it reads; calls that overlap on the GPU
 * (different streams, no ordering) race on it and must not be issued. Device
 * wait timeouts are recorded in the library's error word (q4k_check_device_error);
 * failed calls set q4k_get_last_error and successful ones q4k_last_call_kernels,
 * as for the other entry points. */
q4k_status ffn_q4k_swiglu_noalloc(const void* x, int64_t m, int64_t hidden, int64_t inter,
                                  const void* W_gate, const void* W_up, const void* W_down,
                                  float* y, q4k_stream_t stream);

/* ---- Q6_K GEMV (the LM head) ----
 * Q6_K block (GGML block_q6_K, 256 weights in 210 bytes): ql[128] low 4 bits
 * of the quants, qh[64] high 2 bits, 16 signed 8-bit sub-block scales, fp16 d.
 * Weight i is d * scale[i / 16] * (q_i - 32); in half h (weights 128h..128h+127),
 * weight 128h + 32s + l (s = 0..3, l = 0..31) takes its low 4 bits from the
 * low (s < 2) or high (s >= 2) nibble of ql[64h + l + 32*(s % 2)] and its high 2
 * bits from bits 2s..2s+1 of qh[32h + l]. */
/* Bytes of a Q6_K matrix of `rows` rows of `cols` inputs: rows*(cols/256)*210
 * (0 for an invalid shape). */
size_t q6k_weight_bytes(int64_t rows, int64_t cols);
/* Workspace bytes q6k_gemv needs (0 for a shape q6k_gemv rejects). */
size_t q6k_gemv_workspace_bytes(int64_t m, int64_t n, int64_t k);
/* y[t][r] = sum_c W[r][c] * x[t][c] for t < m, r < n: the GEMV of a Q6_K weight
 * matrix W (n rows of k/256 blocks, row = output) with float32 or bf16
 * activations x [m][k] (bf16 widened exactly), float32 output y [m][n].
 * Source: realizar src/cuda/executor/q4k_gemv_cached_uses.rs,
 * q6k_gemv_cached_async (the Q4_K GEMV's contract for Q6_K weights, used for the
 * LM head). Shapes: 1 <= m <= 8, n a positive multiple of 16, k a multiple of
 * 256 up to 8192 (else Q4K_ERR_SHAPE). x, W, y 16-byte aligned; the workspace
 * caller-owned, 256-byte aligned, at least q6k_gemv_workspace_bytes(m, n, k)
 * bytes, no initialisation needed, not shared by calls that overlap on the GPU.
 * Repeated calls with the same buffers are replayed from a recorded CUDA graph. */
q4k_status q6k_gemv(const void* x, q4k_dtype dtype, int64_t m, int64_t n, int64_t k,
                    const void* W, float* y, void* workspace, size_t ws_bytes,
                    q4k_stream_t stream);
/* Test hook: dequantize a Q6_K matrix to float32 [rows][cols]; every value
 * d*scale*(q-32) is exact in float32. */
q4k_status q6k_dequantize(const void* q6k, int64_t rows, int64_t cols, float* out,
                          q4k_stream_t stream);
/* Workspace bytes ffn_q4k_swiglu_ex needs for this shape (0 for an invalid shape). */
size_t ffn_q4k_workspace_bytes(int64_t m, int64_t hidden, int64_t inter);

/* Byte offset and size, inside an ffn_q4k_swiglu_ex workspace, of the planar
 * Q8_1 copy of the activated vector h = silu(gate)*up that the prefill path
 * feeds to the down projection (m >= 25 only; test hook, offset 0 / size 0 for
 * decode shapes). */
size_t ffn_q4k_workspace_h_q8_1_offset(int64_t m, int64_t hidden, int64_t inter);

/* Test hook: dequantize a Q4_K matrix to float32 [rows][cols]. Every value is
 * d*scale*q - dmin*min rounded once to float32 (bit-exact). */
q4k_status q4k_dequantize(const void* q4k, int64_t rows, int64_t cols, float* out,
                          q4k_stream_t stream);

/* Synchronise `stream`, then read and clear the device error word of the
 * current device. Returns Q4K_OK, Q4K_ERR_TIMEOUT, Q4K_ERR_RANGE or
 * Q4K_ERR_CUDA (a sticky runtime error). */
q4k_status q4k_check_device_error(q4k_stream_t stream);

/* Test hook for the bounded device waits (no counterpart on the source pages).
 * Enqueues on `stream` one warp that waits, through the same bounded wait as
 * the FFN kernels, on a barrier that nothing completes. The wait gives up after
 * limit_ns nanoseconds (1e3..2e9; otherwise Q4K_ERR_SHAPE, nothing launched)
 * and records a timeout in the device error word, so that the next
 * q4k_check_device_error() returns Q4K_ERR_TIMEOUT and the context stays
 * usable. No memory of the caller is touched. */
q4k_status q4k_test_bounded_wait(uint64_t limit_ns, q4k_stream_t stream);

/* Per-kernel timing hook (for benchmarks). After this call, every FFN call made
 * on this thread records events[2i] (cudaEvent_t) before and events[2i+1] after
 * its i-th kernel, for i < n/2, on the call's stream. Decode calls launch up to
 * 5 (activation fragments, gate+up GEMV, chunk sum + SwiGLU + h fragments, down
 * GEMV, down chunk sum when K is split or y is bf16; a slot whose kernel does not
 * run records two adjacent events), prefill calls 4 (Q8_1 of x and its operand
 * expansion, gate+up MMQ + SwiGLU + Q8_1 of h, operand expansion of h, down MMQ;
 * the second and fourth slots also cover the sums of their split tiles or K
 * slices when there are some). Decode calls of
 * 9..24 tokens record each pass's kernels into the same slots. Q6_K GEMV calls
 * record 2 (x fragments, GEMV). The events stay owned by the caller; n = 0 (events NULL) turns the
 * hook off. Recording between kernels serialises them, so timed runs of the
 * whole call leave the hook off. */
q4k_status q4k_set_profile_events(void* const* events, int n);

/* Q4_K x Q8_1 GEMM with FP8 tensor-core operands (tcgen05 kind::f8f6f4, E4M3 x
 * E4M3, exact integer products): out[t][r] = sum_k deq(W)[r][k] * deq(xq)[t][k]
 * for t < m tokens and r < n rows. Source: spark_model/layers/ops/q4k_mmq.rs,
 * q4k_mmq_gemm (C[m, n] = A_q8[m, k] x W_q4k[n, k]^T, activations quantized to
 * Q8_1 before the GEMM). The 4-bit quants enter the MMA unscaled as E4M3 codes
 * (exact), each Q8_1 quant as 16*h + l with both parts exact in E4M3, and one
 * MMA of K = 32 forms one sub-block's integer dot product exactly; the 6-bit
 * scales, the Q8_1 scales and the min terms are applied in float32 per
 * sub-block. xq8: planar Q8_1 of the activations [m][k] (q8_1_bytes(m, k)
 * bytes, as written by q8_1_quantize_act); W: n rows of k/256 Q4_K blocks
 * (row = output); out float32 [m][n]. k a multiple of 256, n a multiple of
 * 128, m >= 1 (else Q4K_ERR_SHAPE). Workspace: caller-owned, 256-byte aligned,
 * q4k_mmq_fp8_workspace_bytes(m, k) bytes (the two E4M3 planes of the
 * activations), no initialisation needed. Launches two kernels on `stream`. */
q4k_status q4k_mmq_fp8(const void* xq8, int64_t m, int64_t k, const void* W, int64_t n, float* out,
                       void* workspace, size_t ws_bytes, q4k_stream_t stream);
/* Workspace bytes q4k_mmq_fp8 needs (0 for an invalid shape). */
size_t q4k_mmq_fp8_workspace_bytes(int64_t m, int64_t k);

/* Benchmark hook (no counterpart on the source pages): the int8 tensor-core
 * rate. Enqueues on `stream` one kernel in which every warp issues `iters`
 * rounds of 8 independent mma.sync.m16n8k32 s8 x s8 -> s32 operations (the
 * int8 tensor instruction of sm_103a; tcgen05.mma has no integer kind here) and
 * nothing else, 4 CTAs of 8 warps per SM. *ops_per_launch receives the integer
 * operations the launch performs (2*16*8*32 per MMA); the caller times the
 * launch (CUDA events on `stream`) and divides. iters in 1..2^24, else
 * Q4K_ERR_SHAPE; ops_per_launch NULL gives Q4K_ERR_NULL. Touches no memory of
 * the caller. */
q4k_status q4k_bench_int8_mma(int64_t iters, double* ops_per_launch, q4k_stream_t stream);

/* Benchmark hook (no counterpart on the source pages): the issue rate of
 * tcgen05.mma kind::f16 (M = 128, K = 16, N = n; A in tensor memory, fp32
 * accumulators) when `issuers` threads per CTA issue back to back into their own
 * accumulators, one CTA per SM, `iters` rounds of 4 MMAs per thread, one commit
 * per round. Runs on `stream` and waits for it; *cycles_per_mma receives the SM
 * cycles per MMA of one issuing thread (averaged over the CTAs): the tensor pipe's
 * own rate is 4096 multiply-adds per cycle, 128 * n * 16 per MMA. n in {64, 128,
 * 256}, issuers in {1, 2, 4}, n * issuers <= 256 and iters in 1..2^20, else
 * Q4K_ERR_SHAPE; cycles_per_mma NULL gives Q4K_ERR_NULL. Its waits are bounded
 * (q4k_check_device_error reports a timeout). Touches no memory of the caller. */
q4k_status q4k_bench_tcgen05_issue(int n, int issuers, int64_t iters, double* cycles_per_mma, q4k_stream_t stream);

/* Benchmark hook: how many kernels the most recent FFN or Q6_K GEMV call on
 * this thread launched (directly, or as nodes of the replayed graph). */
int q4k_last_call_kernels(void);
/* Status of the most recent failed host-side call on this thread (Q4K_OK if none). */
q4k_status q4k_get_last_error(void);

/* Static, human-readable name of a status. */
const char* q4k_status_string(q4k_status status);

#ifdef __cplusplus
}
#endif

#endif /* Q4KFFN_H */
