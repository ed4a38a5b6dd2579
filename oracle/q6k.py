"""Plain CPU restatement of the Q6_K GEMV (test infrastructure only).

Source restated here: realizar src/cuda/executor/q4k_gemv_cached_uses.rs,
``q6k_gemv_cached_async`` -- the same GEMV as the Q4_K one (y[n] over the k
inputs of row n, float32 input, float32 output, k a multiple of 256) for
weights stored as Q6_K blocks, used for the LM head.

The pages name the Q6_K format but do not print its bytes. The reading used
here is the GGML ``block_q6_K`` layout, 256 weights in 210 bytes:

* bytes   0-127  ``ql``: low 4 bits of the quants,
* bytes 128-191  ``qh``: high 2 bits of the quants,
* bytes 192-207  ``scales``: 16 signed 8-bit sub-block scales,
* bytes 208-209  ``d``: fp16 super-block scale.

The block holds two halves of 128 weights. In half h (``ql`` bytes
64h..64h+63, ``qh`` bytes 32h..32h+31), for l in 0..31 and part s in 0..3,
weight 128h + 32s + l has the 6-bit quant

    q = (nibble of ql[64h + l + 32*(s % 2)], low for s < 2, high for s >= 2)
        | ((qh[32h + l] >> 2s) & 3) << 4

so weight i belongs to sub-block i // 16 and its value is

    w_i = d * scales[i // 16] * (q_i - 32).

Every factor is an integer times a power of two with at most 11 + 8 + 6
significant bits, so the float64 result is exact (and so is float32).
"""
from __future__ import annotations

import numpy as np

from .q4k import QK_K, fp16_bits_to_f64

Q6K_BLOCK_BYTES = 210


def q6k_fields(blocks: np.ndarray):
    """Decode Q6_K blocks [..., 210] -> d (float64, exact), scales[..., 16] (int),
    q[..., 256] (int 0..63, in weight order)."""
    b = np.asarray(blocks, dtype=np.uint8)
    ql = b[..., 0:128].astype(np.int64)
    qh = b[..., 128:192].astype(np.int64)
    scales = b[..., 192:208].view(np.int8).astype(np.int64)
    d = fp16_bits_to_f64(b[..., 208:210].copy().view(np.uint16)[..., 0])
    q = np.empty(b.shape[:-1] + (QK_K,), dtype=np.int64)
    for h in range(2):
        for s in range(4):
            nib_bytes = ql[..., 64 * h + 32 * (s % 2): 64 * h + 32 * (s % 2) + 32]
            nib = (nib_bytes & 0x0F) if s < 2 else (nib_bytes >> 4)
            hi2 = (qh[..., 32 * h: 32 * h + 32] >> (2 * s)) & 3
            q[..., 128 * h + 32 * s: 128 * h + 32 * s + 32] = nib | (hi2 << 4)
    return d, scales, q


def dequantize_q6k(blocks: np.ndarray) -> np.ndarray:
    """Exact float64 weights of a Q6_K matrix [rows, nblk, 210] -> [rows, nblk*256]."""
    d, scales, q = q6k_fields(blocks)
    sub = np.arange(QK_K) // 16
    w = (d[..., None] * scales[..., sub]) * (q - 32)
    return w.reshape(w.shape[:-2] + (w.shape[-2] * QK_K,))


def gemv_q6k(x: np.ndarray, blocks: np.ndarray) -> np.ndarray:
    """y[t, n] = sum_k W[n, k] x[t, k] in float64 over the exact weights.

    x: [m, k] (float32 values, or bf16 values widened exactly); blocks: [n, k/256, 210].
    """
    w = dequantize_q6k(blocks)
    return np.asarray(x, dtype=np.float64) @ w.T
