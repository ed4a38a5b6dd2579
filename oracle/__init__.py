"""CPU oracle for the Q4_K SwiGLU feed-forward block -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The GPU library never calls it, links
it or falls back to it, and the two share no code: the only thing both sides
use is the seeded input generator in ``workloads/``.

What it computes (plain numpy, float64 unless the definition fixes float32):

* ``dequantize_q4k``   -- exact value of every weight of a GGML Q4_K block.
* ``quantize_q8_1``    -- Q8_1 activation blocks (int8 quants, fp32 scale, fp32 sum),
                          bit-exact float32 rules.
* ``ffn_decode``       -- y = W_down (silu(W_gate x) * (W_up x)) over exact weights.
* ``ffn_prefill``      -- the same block with activations quantized to Q8_1 before
                          gate/up and the activated vector re-quantized before down.
* ``quantize_q4k``     -- deterministic min-max Q4_K weight quantizer.
* ``q4k_q8_1_dot``     -- the closed form of one Q4_K x Q8_1 block dot product.
* ``dequantize_q6k``   -- exact value of every weight of a GGML Q6_K block.
* ``gemv_q6k``         -- y = W x over exact Q6_K weights (the LM-head GEMV).

Pins (tests/test_oracle_*.py) tie every function to something other than
itself: hand-built blocks whose values follow from the block definition,
bit-level bijection of the scale packing, closed forms, a pure-Python scalar
brute force on tiny inputs, one-hot weight matrices that turn the FFN into a
gather, round-trip bounds and tie cases of the rounding rule.
"""
from .q4k import (  # noqa: F401
    QK_K, BLOCK_BYTES, Q8_BLOCK,
    fp16_bits_to_f64, unpack_scales_mins, pack_scales_mins, q4k_fields,
    dequantize_q4k, dequantize_q4k_f32,
    quantize_q8_1, dequantize_q8_1, q8_1_to_bytes, q8_1_from_bytes,
    silu, ffn_decode, ffn_prefill, ffn_down_from_q8_1, gate_up_h,
    quantize_q4k, q4k_q8_1_dot,
)
from .q6k import Q6K_BLOCK_BYTES, q6k_fields, dequantize_q6k, gemv_q6k  # noqa: F401
