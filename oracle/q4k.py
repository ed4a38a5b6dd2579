"""Plain CPU restatement of the Q4_K SwiGLU FFN (test infrastructure only).

Sources restated here (page title, then the item on it):

* spark_model/layers/ops/q4k_mmq.rs -- constants ``QK_K`` (256 weights per
  block) and ``Q4K_BLOCK_BYTES`` (144), ``q4k_weight_bytes`` (rows x blocks x
  144), ``quantize_act_q8_1`` (bf16 activations to Q8_1 before the GEMM),
  ``q4k_mmq_gemm`` (C[m, n] = A_q8[m, k] x W_q4k[n, k]) and the header's
  pipeline (per-prefill activations to Q8_1, then the Q4_K MMQ).
* realizar src/cuda/executor/layers/ffn.rs -- ``fused_ffn_swiglu_gpu``:
  LLaMA-style ``down(swiglu(gate(x), up(x)))`` with gate and up as GEMVs of
  the same input; ``fused_ffn_swiglu_gpu_true_dp4a``: activations quantized
  to Q8_1 once ("per-block scale + 32 x int8") and shared by gate and up,
  then the activated vector quantized again before the down GEMV.
* realizar src/cuda/executor/q4k_gemv_cached_uses.rs -- ``q4k_gemv_cached``:
  y[n] over the k inputs of row n, weights stored as rows of Q4_K blocks
  (``n`` = output dimension, ``k`` = input dimension, k divisible by 256).

The GGML Q4_K byte layout (fp16 d, fp16 dmin, 12 bytes of packed 6-bit
scales and mins for 8 sub-blocks of 32, 128 bytes of 4-bit quants) is the
format those pages store; its bit packing is restated in ``unpack_scales_mins``
and ``q4k_fields``. Readings taken where the pages are silent are listed in
the module docstrings of the functions concerned.
"""
from __future__ import annotations

import numpy as np

QK_K = 256
BLOCK_BYTES = 144
Q8_BLOCK = 32


# ----------------------------------------------------------------------------------------
# Q4_K block decoding
# ----------------------------------------------------------------------------------------

def fp16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    """IEEE binary16 bit patterns (uint16) to their exact float64 values."""
    return np.ascontiguousarray(b, dtype=np.uint16).view(np.float16).astype(np.float64)


def unpack_scales_mins(s12: np.ndarray):
    """The 12 packed bytes of a Q4_K block -> (scale[8], min[8]), each 6 bits.

    Sub-blocks 0-3: scale = low 6 bits of byte j, min = low 6 bits of byte j+4.
    Sub-blocks 4-7: scale = low nibble of byte j+4 with the top two bits of
    byte j-4 as bits 4-5; min = high nibble of byte j+4 with the top two bits
    of byte j as bits 4-5.
    """
    s = np.asarray(s12, dtype=np.uint8).astype(np.int64)
    sc = np.empty(s.shape[:-1] + (8,), dtype=np.int64)
    mn = np.empty_like(sc)
    for j in range(4):
        sc[..., j] = s[..., j] & 63
        mn[..., j] = s[..., j + 4] & 63
    for j in range(4, 8):
        sc[..., j] = (s[..., j + 4] & 0x0F) | ((s[..., j - 4] >> 6) << 4)
        mn[..., j] = (s[..., j + 4] >> 4) | ((s[..., j] >> 6) << 4)
    return sc, mn


def pack_scales_mins(sc: np.ndarray, mn: np.ndarray) -> np.ndarray:
    """Inverse of ``unpack_scales_mins``: (scale[8], min[8]) in 0..63 -> 12 bytes."""
    sc = np.asarray(sc, dtype=np.int64)
    mn = np.asarray(mn, dtype=np.int64)
    out = np.zeros(sc.shape[:-1] + (12,), dtype=np.int64)
    for j in range(4):
        out[..., j] = (sc[..., j] & 63) | ((sc[..., j + 4] >> 4) << 6)
        out[..., j + 4] = (mn[..., j] & 63) | ((mn[..., j + 4] >> 4) << 6)
        out[..., j + 8] = (sc[..., j + 4] & 0x0F) | ((mn[..., j + 4] & 0x0F) << 4)
    return out.astype(np.uint8)


def q4k_fields(blocks: np.ndarray):
    """Decode the fields of Q4_K blocks [..., 144].

    Returns d, dmin (float64, exact), scale[..., 8], min[..., 8] (int) and
    q[..., 256] (int 0..15, in weight order). The 128 quant bytes form four
    groups of 32; in group g, the low nibble of byte i is weight 64g+i
    (sub-block 2g) and the high nibble is weight 64g+32+i (sub-block 2g+1).
    """
    b = np.asarray(blocks, dtype=np.uint8)
    d = fp16_bits_to_f64(b[..., 0:2].copy().view(np.uint16)[..., 0])
    dmin = fp16_bits_to_f64(b[..., 2:4].copy().view(np.uint16)[..., 0])
    sc, mn = unpack_scales_mins(b[..., 4:16])
    qs = b[..., 16:144].astype(np.int64).reshape(b.shape[:-1] + (4, 32))
    lo = qs & 0x0F
    hi = qs >> 4
    q = np.stack([lo, hi], axis=-2).reshape(b.shape[:-1] + (256,))
    return d, dmin, sc, mn, q


def dequantize_q4k(blocks: np.ndarray) -> np.ndarray:
    """Exact float64 weights of a Q4_K matrix [rows, nblk, 144] -> [rows, nblk*256].

    Weight i of sub-block j is d*scale_j*q_i - dmin*min_j. Every term is an
    integer multiple of 2**-24 below 2**27 in magnitude, so the float64 result
    is the exact real value.
    """
    d, dmin, sc, mn, q = q4k_fields(blocks)
    sub = np.arange(256) // 32
    w = (d[..., None] * sc[..., sub]) * q - (dmin[..., None] * mn[..., sub])
    return w.reshape(w.shape[:-2] + (w.shape[-2] * 256,))


def dequantize_q4k_f32(blocks: np.ndarray) -> np.ndarray:
    """Exact weights rounded once to float32 (round to nearest even)."""
    return dequantize_q4k(blocks).astype(np.float32)


# ----------------------------------------------------------------------------------------
# Q8_1 activation quantization
# ----------------------------------------------------------------------------------------

def _round_half_away(v: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest integer, ties away from zero (exact)."""
    a = np.abs(v)
    f = np.floor(a)
    r = f + ((a - f) >= 0.5)
    return np.copysign(r, v)


def quantize_q8_1(x: np.ndarray):
    """Q8_1 quantization of float32 activations [m, k] (k % 32 == 0).

    Per block of 32 consecutive values, in float32 with one rounding per
    operation (the reading of "round-to-nearest of x*127/absmax"):
      amax = max|x|; d = amax/127; inv = 127/amax; q = round(x*inv) with ties
      away from zero, clamped to [-127, 127]; s = d * sum(q).
    A block whose amax is below 2**-120 (zero, or so small that 127/amax would
    overflow float32) gives d = s = 0 and q = 0.
    Returns (q int8 [m, k], d float32 [m, k/32], s float32 [m, k/32]).
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    m, k = x.shape
    assert k % Q8_BLOCK == 0
    xb = x.reshape(m, k // Q8_BLOCK, Q8_BLOCK)
    amax = np.max(np.abs(xb), axis=-1)
    nz = amax >= np.float32(2.0 ** -120)
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        d = np.where(nz, amax / np.float32(127.0), np.float32(0.0)).astype(np.float32)
        inv = np.where(nz, np.float32(127.0) / amax, np.float32(0.0)).astype(np.float32)
    v = (xb * inv[..., None]).astype(np.float32)
    q = np.clip(_round_half_away(v.astype(np.float64)), -127, 127).astype(np.int64)
    sq = q.sum(axis=-1).astype(np.float32)
    s = (d * sq).astype(np.float32)
    return q.reshape(m, k).astype(np.int8), d, s


def dequantize_q8_1(q: np.ndarray, d: np.ndarray) -> np.ndarray:
    """float64 value q*d of every Q8_1 element (exact)."""
    m, k = q.shape
    return (q.reshape(m, k // Q8_BLOCK, Q8_BLOCK).astype(np.float64)
            * d.astype(np.float64)[..., None]).reshape(m, k)


def q8_1_to_bytes(q: np.ndarray, d: np.ndarray, s: np.ndarray) -> np.ndarray:
    """Planar Q8_1 buffer: int8 quants [m][k], then {float d, float s} pairs [m][k/32].

    This planar byte layout is a reading: the pages name Q8_1 as "per-block
    scale + 32 x int8" and a "DS4 layout" without defining its bytes.
    """
    m, k = q.shape
    ds = np.stack([d.astype(np.float32), s.astype(np.float32)], axis=-1)
    return np.concatenate([q.astype(np.int8).view(np.uint8).reshape(-1),
                           ds.view(np.uint8).reshape(-1)])


def q8_1_from_bytes(buf: np.ndarray, m: int, k: int):
    buf = np.asarray(buf, dtype=np.uint8)
    q = buf[: m * k].view(np.int8).reshape(m, k)
    ds = buf[m * k: m * k + m * (k // Q8_BLOCK) * 8].view(np.float32).reshape(m, k // Q8_BLOCK, 2)
    return q, ds[..., 0].copy(), ds[..., 1].copy()


# ----------------------------------------------------------------------------------------
# The feed-forward block
# ----------------------------------------------------------------------------------------

def silu(z: np.ndarray) -> np.ndarray:
    """silu(z) = z / (1 + exp(-z)) in float64 (gives -0 for very negative z)."""
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def _matvec_rows(blocks: np.ndarray, a: np.ndarray, chunk: int = 2048) -> np.ndarray:
    """a [m, k] float64 times the transpose of the dequantized rows of ``blocks``.

    Rows of the weight matrix are dequantized ``chunk`` at a time to bound
    memory; each output element is still one dot product over all k inputs.
    """
    rows = blocks.shape[0]
    out = np.empty((a.shape[0], rows), dtype=np.float64)
    for r0 in range(0, rows, chunk):
        w = dequantize_q4k(blocks[r0:r0 + chunk])
        out[:, r0:r0 + chunk] = a @ w.T
    return out


def ffn_decode(x: np.ndarray, wg: np.ndarray, wu: np.ndarray, wd: np.ndarray):
    """Decode regime: y = W_down (silu(W_gate x) * (W_up x)), all in float64.

    x is float32 [m, hidden] used as given (no activation quantization on this
    path, the reading of the fp32-activation GEMV pipeline). Weight matrices
    are Q4_K rows: wg, wu [inter, hidden/256, 144]; wd [hidden, inter/256, 144].
    Returns (y float64 [m, hidden], h float64 [m, inter]).
    """
    a = np.asarray(x, dtype=np.float32).astype(np.float64)
    g = _matvec_rows(wg, a)
    u = _matvec_rows(wu, a)
    h = silu(g) * u
    y = _matvec_rows(wd, h)
    return y, h


def gate_up_h(xq: np.ndarray, xd: np.ndarray, wg: np.ndarray, wu: np.ndarray) -> np.ndarray:
    """Prefill gate/up stage on Q8_1 activations: h = silu(g) * u in float64."""
    a = dequantize_q8_1(xq, xd)
    g = _matvec_rows(wg, a)
    u = _matvec_rows(wu, a)
    return silu(g) * u


def ffn_down_from_q8_1(hq: np.ndarray, hd: np.ndarray, wd: np.ndarray) -> np.ndarray:
    """Prefill down stage: y = W_down deq(hq) in float64."""
    return _matvec_rows(wd, dequantize_q8_1(hq, hd))


def ffn_prefill(x: np.ndarray, wg: np.ndarray, wu: np.ndarray, wd: np.ndarray):
    """Prefill regime with Q8_1 activations.

    1. xq = Q8_1(x)                          (x float32, bf16 inputs widened exactly)
    2. g, u = deq(W) . deq(xq) in float64
    3. h = silu(g) * u, rounded to float32 (the reading: h is a float32 tensor)
    4. hq = Q8_1(h)
    5. y = deq(W_down) . deq(hq) in float64
    Returns a dict with y, h (float32), and both Q8_1 tensors as (q, d, s).
    """
    xq, xd, xs = quantize_q8_1(x)
    h = gate_up_h(xq, xd, wg, wu).astype(np.float32)
    hq, hd, hs = quantize_q8_1(h)
    y = ffn_down_from_q8_1(hq, hd, wd)
    return {"y": y, "h": h, "xq": (xq, xd, xs), "hq": (hq, hd, hs)}


# ----------------------------------------------------------------------------------------
# Closed form of one Q4_K x Q8_1 block dot product
# ----------------------------------------------------------------------------------------

def q4k_q8_1_dot(block: np.ndarray, q8: np.ndarray, d8: np.ndarray, s8: np.ndarray) -> float:
    """sum_j [ d*scale_j*d8_j*sum_{i in j} q4_i*q8_i - dmin*min_j*s8_j ] over the 8 sub-blocks.

    block: one Q4_K block (144 bytes); q8: 256 int8 quants; d8, s8: the 8
    Q8_1 scales and sums of the same 256 positions. With s8_j = d8_j*sum(q8)
    this equals the dot product of the dequantized vectors exactly.
    """
    d, dmin, sc, mn, q = q4k_fields(np.asarray(block, dtype=np.uint8)[None])
    q = q[0].reshape(8, 32)
    q8 = np.asarray(q8, dtype=np.int64).reshape(8, 32)
    isum = (q * q8).sum(axis=1)                       # exact integers
    tot = 0.0
    for j in range(8):
        tot += float(d[0]) * int(sc[0, j]) * float(d8[j]) * int(isum[j])
        tot -= float(dmin[0]) * int(mn[0, j]) * float(s8[j])
    return tot


# ----------------------------------------------------------------------------------------
# Q4_K weight quantizer (load-time)
# ----------------------------------------------------------------------------------------

FP16_MAX = 65504.0


def _fp16_up(v: np.ndarray) -> np.ndarray:
    """Smallest float16 >= v for float64 v >= 0 (raises if v exceeds the fp16 range)."""
    if np.any(v > FP16_MAX):
        raise ValueError("Q4_K scale exceeds the fp16 range")
    f = v.astype(np.float16)
    bits = f.view(np.uint16).astype(np.uint32)
    bits = bits + (f.astype(np.float64) < v)
    if np.any(bits > 0x7BFF):
        raise ValueError("Q4_K scale exceeds the fp16 range")
    return bits.astype(np.uint16).view(np.float16)


def _smallest_fp16_cover(total: np.ndarray, mult: float) -> np.ndarray:
    """Smallest float16 f with mult*f >= total (total >= 0), as float16."""
    f = _fp16_up(total / mult)
    short = f.astype(np.float64) * mult < total
    if np.any(short):
        bits = f.view(np.uint16).astype(np.uint32) + short
        if np.any(bits > 0x7BFF):
            raise ValueError("Q4_K scale exceeds the fp16 range")
        f = bits.astype(np.uint16).view(np.float16)
    return f


def _smallest_int_cover(need: np.ndarray, step: np.ndarray, top: int) -> np.ndarray:
    """Smallest integer n in [0, top] with step*n >= need (0 where step == 0)."""
    with np.errstate(divide="ignore", invalid="ignore"):
        n = np.where(step > 0, np.ceil(need / np.where(step > 0, step, 1.0)), 0.0)
    n = np.clip(n, 0, top)
    n = np.where((step > 0) & (step * n < need) & (n < top), n + 1, n)
    n = np.where((step > 0) & (n >= 1) & (step * (n - 1) >= need), n - 1, n)
    return n.astype(np.int64)


def quantize_q4k(w: np.ndarray) -> np.ndarray:
    """Deterministic min-max Q4_K quantizer: float32 [rows, cols] -> uint8 [rows, cols/256, 144].

    The pages give only the launch of their load-time quantizer, so the
    algorithm is this reading (float64, every operation rounded once):
      per sub-block j: lo_j = max(0, -min x), hi_j = max(0, max x)
      dmin = smallest fp16 with 63*dmin >= max_j lo_j
      min_j = smallest integer with dmin*min_j >= lo_j           (<= 63)
      r_j = hi_j + dmin*min_j
      d = smallest fp16 with 945*d >= max_j r_j
      scale_j = smallest integer with 15*d*scale_j >= r_j        (<= 63)
      q_i = clamp(round_half_away((x_i + dmin*min_j) / (d*scale_j)), 0, 15), 0 if d*scale_j == 0
    so every x of the block lies within half a quant step d*scale_j of its
    dequantized value.
    """
    w = np.ascontiguousarray(w, dtype=np.float32)
    rows, cols = w.shape
    assert cols % QK_K == 0
    nb = cols // QK_K
    x = w.astype(np.float64).reshape(rows, nb, 8, 32)
    lo = np.maximum(0.0, -x.min(axis=-1)) + 0.0      # + 0.0 turns -0.0 into +0.0
    hi = np.maximum(0.0, x.max(axis=-1)) + 0.0
    dmin = _smallest_fp16_cover(lo.max(axis=-1), 63.0)
    dmin64 = dmin.astype(np.float64)
    mn = _smallest_int_cover(lo, dmin64[..., None], 63)
    r = hi + dmin64[..., None] * mn
    d = _smallest_fp16_cover(r.max(axis=-1), 945.0)
    d64 = d.astype(np.float64)
    sc = _smallest_int_cover(r, 15.0 * d64[..., None], 63)
    step = d64[..., None] * sc                                  # [rows, nb, 8]
    with np.errstate(divide="ignore", invalid="ignore"):
        v = (x + (dmin64[..., None] * mn)[..., None]) / np.where(step > 0, step, 1.0)[..., None]
    q = np.clip(_round_half_away(v), 0, 15)
    q = np.where(step[..., None] > 0, q, 0).astype(np.int64)    # [rows, nb, 8, 32]

    out = np.zeros((rows, nb, BLOCK_BYTES), dtype=np.uint8)
    out[..., 0:2] = d.reshape(rows, nb, 1).view(np.uint8)
    out[..., 2:4] = dmin.reshape(rows, nb, 1).view(np.uint8)
    out[..., 4:16] = pack_scales_mins(sc, mn)
    qq = q.reshape(rows, nb, 4, 2, 32)                          # group g: sub-blocks 2g, 2g+1
    out[..., 16:144] = (qq[..., 0, :] | (qq[..., 1, :] << 4)).reshape(rows, nb, 128).astype(np.uint8)
    return out
