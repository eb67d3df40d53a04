"""CPU oracle of the TACO fused compress / decompress-reduce operator.

Test infrastructure: only the tests, the smoke check and the benchmark's CPU
baseline leg use it. The product path never imports it.
"""
from .taco_oracle import *  # noqa: F401,F403
from .taco_oracle import (  # noqa: F401
    BLOCK_SIZES, DEFAULT_TARGET_ENERGY, FORMAT_E4M3, FORMAT_INT8, Q_MAX, Q_MAX_INT8, VARIANT_ABSMAX, VARIANT_DUAL, VARIANT_STATIC, VARIANTS,
    bf16_bits_to_f64, compress, compress_stages, compress_values_stages, decompress_one_f64,
    decompress_reduce, decompress_reduce_f64, e4m3_decode, e4m3_decode_table,
    e4m3_encode, f64_to_bf16_bits, int8_decode, int8_encode, q_max, reduce_recompress, round_to_bf16, static_scale, sylvester_hadamard,
    wire_bytes_per_element,
)
