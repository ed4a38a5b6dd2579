"""Seeded synthetic workloads for the Q4_K SwiGLU FFN (inputs only).

This module is the one piece shared by the CPU oracle side (tests) and the
GPU side (bench, smoke). It draws random numbers and lays them out as input
buffers; it performs none of the method's arithmetic (no dequantisation, no
quantisation, no dot products).

Random source: SplitMix64 (Steele, Lea & Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014), used counter-style: element i
of stream s under seed S is mix64(key(S, s) + (i + 1) * GAMMA) with
key(S, s) = mix64(S + s * GAMMA). Normals come from Box-Muller in float64.

Workload shapes follow the five configurations of the Q4_K SwiGLU FFN
benchmark (tiny decode, LLaMA-7B-shaped decode, 13B-shaped batched decode,
8B-shaped prefill, 27B-shaped long prefill). Q4_K weight blocks are
generated directly as bytes of the 144-byte GGML block: fp16 ``d`` and
``dmin`` drawn from U[0.001, 0.05] and rounded to fp16, and uniformly random
bytes for the 12 packed scale/min bytes and the 128 quant bytes. Uniform
bytes make every 6-bit scale and min uniform on 0..63 and every 4-bit quant
uniform on 0..15 without this module knowing how the bits are packed.
"""
from __future__ import annotations

import dataclasses
import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
QK_K = 256          # weights per Q4_K block
BLOCK_BYTES = 144   # bytes per Q4_K block

# stream ids within one seed
S_WG, S_WU, S_WD, S_X, S_OUTLIER_POS, S_OUTLIER_VAL = 1, 2, 3, 4, 5, 6


def _mix64(z: np.ndarray) -> np.ndarray:
    z = z.astype(np.uint64, copy=True)
    with np.errstate(over="ignore"):
        z ^= z >> np.uint64(30)
        z *= np.uint64(0xBF58476D1CE4E5B9)
        z ^= z >> np.uint64(27)
        z *= np.uint64(0x94D049BB133111EB)
        z ^= z >> np.uint64(31)
    return z


def u64_stream(seed: int, stream: int, n: int, offset: int = 0) -> np.ndarray:
    """n consecutive 64-bit outputs (starting at counter ``offset``) of one stream."""
    with np.errstate(over="ignore"):
        key = _mix64(np.array([np.uint64(seed) + np.uint64(stream) * GAMMA], dtype=np.uint64))[0]
        ctr = np.arange(offset + 1, offset + n + 1, dtype=np.uint64)
        return _mix64(key + ctr * GAMMA)


def uniform(seed: int, stream: int, n: int, offset: int = 0) -> np.ndarray:
    """float64 uniforms on [0, 1) with 53 random bits."""
    return (u64_stream(seed, stream, n, offset) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def random_bytes(seed: int, stream: int, n: int) -> np.ndarray:
    words = u64_stream(seed, stream, (n + 7) // 8)
    return words.view(np.uint8)[:n].copy()


def normal(seed: int, stream: int, n: int) -> np.ndarray:
    """float64 N(0,1) by Box-Muller (one normal per pair of uniforms)."""
    u = uniform(seed, stream, 2 * n)
    u1 = 1.0 - u[0::2]          # (0, 1]
    u2 = u[1::2]
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (round-to-nearest-even); returns uint16 bit patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def q4k_blocks(seed: int, stream: int, rows: int, cols: int,
               d_lo: float = 0.001, d_hi: float = 0.05) -> np.ndarray:
    """Random Q4_K weight matrix: uint8 array [rows, cols/256, 144].

    Bytes 0-1 hold fp16 d, bytes 2-3 fp16 dmin (both U[d_lo, d_hi] rounded to
    fp16), bytes 4-143 are uniformly random.
    """
    assert cols % QK_K == 0
    nb = rows * (cols // QK_K)
    raw = random_bytes(seed, stream, nb * BLOCK_BYTES).reshape(nb, BLOCK_BYTES)
    u = uniform(seed, stream + 100, 2 * nb).reshape(nb, 2)
    dd = (d_lo + (d_hi - d_lo) * u).astype(np.float16)
    raw[:, 0:4] = dd.view(np.uint8).reshape(nb, 4)
    return raw.reshape(rows, cols // QK_K, BLOCK_BYTES)


Q6K_BLOCK_BYTES = 210  # bytes per Q6_K block


def q6k_blocks(seed: int, stream: int, rows: int, cols: int,
               d_lo: float = 0.0005, d_hi: float = 0.002) -> np.ndarray:
    """Random Q6_K weight matrix: uint8 array [rows, cols/256, 210].

    Bytes 208-209 hold fp16 d (U[d_lo, d_hi] rounded to fp16); bytes 0-207
    (the quant bits and the 16 signed 8-bit scales) are uniformly random, so
    every 6-bit quant is uniform on 0..63 and every scale on -128..127.
    """
    assert cols % QK_K == 0
    nb = rows * (cols // QK_K)
    raw = random_bytes(seed, stream, nb * Q6K_BLOCK_BYTES).reshape(nb, Q6K_BLOCK_BYTES)
    u = uniform(seed, stream + 100, nb)
    dd = (d_lo + (d_hi - d_lo) * u).astype(np.float16)
    raw[:, 208:210] = dd.view(np.uint8).reshape(nb, 2)
    return raw.reshape(rows, cols // QK_K, Q6K_BLOCK_BYTES)


@dataclasses.dataclass(frozen=True)
class LMHeadConfig:
    """A Q6_K GEMV workload: y [m, n] = x [m, k] . W[n, k]^T (an LM head)."""
    index: int
    name: str
    n: int      # output rows (vocabulary)
    k: int      # inputs (hidden)
    m: int      # tokens

    @property
    def seed(self) -> int:
        return 0x5EED0600 + self.index

    def weight_bytes(self) -> int:
        return self.n * self.k // QK_K * Q6K_BLOCK_BYTES


# LLaMA-7B's output projection (vocabulary 32000, hidden 4096) at decode, and a small case
LMHEADS = [
    LMHeadConfig(0, "tiny-lmhead-q6k-n512-k256-m1", 512, 256, 1),
    LMHeadConfig(1, "llama7b-lmhead-q6k-n32000-k4096-m1", 32000, 4096, 1),
]


def lmhead_weights(cfg: LMHeadConfig) -> np.ndarray:
    return q6k_blocks(cfg.seed, S_WG, cfg.n, cfg.k)


def lmhead_x(cfg: LMHeadConfig, m: int | None = None) -> np.ndarray:
    m = cfg.m if m is None else m
    return normal(cfg.seed, S_X, m * cfg.k).reshape(m, cfg.k).astype(np.float32)


@dataclasses.dataclass(frozen=True)
class Config:
    index: int
    name: str
    hidden: int
    inter: int
    m: int
    x_dtype: str            # "f32" or "bf16"
    outliers: tuple | None  # ("channels", frac, scale) or ("entries", frac, absval)

    @property
    def seed(self) -> int:
        return 0x5EED0000 + self.index

    @property
    def regime(self) -> str:
        return "decode" if self.m <= 8 else "prefill"

    def weight_bytes(self) -> int:
        return 3 * self.hidden * self.inter // QK_K * BLOCK_BYTES

    def int8_ops(self) -> int:
        return 2 * self.m * self.hidden * self.inter * 3


CONFIGS = [
    Config(0, "tiny-decode-h256-i768-m1", 256, 768, 1, "f32", None),
    Config(1, "llama7b-decode-h4096-i11008-m1", 4096, 11008, 1, "f32", None),
    Config(2, "13b-batched-decode-h5120-i13824-m8", 5120, 13824, 8, "f32", ("channels", 0.005, 50.0)),
    Config(3, "8b-prefill-h4096-i14336-m512", 4096, 14336, 512, "bf16", ("channels", 0.001, 100.0)),
    Config(4, "27b-long-prefill-h5120-i17408-m2048", 5120, 17408, 2048, "bf16", ("entries", 0.0005, 900.0)),
]
TINY_DECODE, LLAMA7B_DECODE, BATCHED_13B_DECODE, PREFILL_8B, LONG_PREFILL_27B = CONFIGS


def _choose(seed: int, stream: int, n: int, k: int) -> np.ndarray:
    """k distinct indices of range(n), chosen by sorting seeded uniform keys."""
    keys = uniform(seed, stream, n)
    return np.sort(np.argsort(keys, kind="stable")[:k])


def activations(cfg: Config, m: int | None = None, seed: int | None = None):
    """Activations x [m, hidden].

    Returns (x_f32, x_bits): x_f32 is the float32 value of every element (for
    bf16 workloads the exactly widened bf16 value), x_bits is the buffer a
    caller hands to the library (float32 array, or uint16 bf16 bit patterns).
    """
    m = cfg.m if m is None else m
    seed = cfg.seed if seed is None else seed
    H = cfg.hidden
    x = normal(seed, S_X, m * H).reshape(m, H)
    if cfg.outliers is not None:
        kind, frac, val = cfg.outliers
        if kind == "channels":
            nch = max(1, int(round(frac * H)))
            ch = _choose(seed, S_OUTLIER_POS, H, nch)
            x[:, ch] *= val
        elif kind == "entries":
            nent = max(1, int(round(frac * m * H)))
            pos = _choose(seed, S_OUTLIER_POS, m * H, nent)
            u = uniform(seed, S_OUTLIER_VAL, 2 * nent).reshape(nent, 2)
            mag = val * (0.5 + 0.5 * u[:, 0])
            mag[0] = val                     # at least one entry exactly +-val
            sign = np.where(u[:, 1] < 0.5, -1.0, 1.0)
            flat = x.reshape(-1)
            flat[pos] = sign * mag
        else:
            raise ValueError(kind)
    xf = x.astype(np.float32)
    if cfg.x_dtype == "bf16":
        bits = f32_to_bf16_bits(xf)
        return bf16_bits_to_f32(bits).reshape(m, H), bits.reshape(m, H)
    return xf, xf


def weights(cfg: Config, seed: int | None = None):
    """(Wg, Wu, Wd) as uint8 Q4_K block arrays.

    Wg, Wu: [inter, hidden/256, 144] (one row per output feature);
    Wd:     [hidden, inter/256, 144].
    """
    seed = cfg.seed if seed is None else seed
    wg = q4k_blocks(seed, S_WG, cfg.inter, cfg.hidden)
    wu = q4k_blocks(seed, S_WU, cfg.inter, cfg.hidden)
    wd = q4k_blocks(seed, S_WD, cfg.hidden, cfg.inter)
    return wg, wu, wd


def small_config(hidden: int, inter: int, m: int, x_dtype: str = "f32",
                 outliers=None, index: int = 100) -> Config:
    """A shape for parity sweeps that is not one of the five named workloads."""
    return Config(index, f"sweep-h{hidden}-i{inter}-m{m}", hidden, inter, m, x_dtype, outliers)
