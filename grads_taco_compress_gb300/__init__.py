"""GB300-native TACO fused compress / decompress-reduce operator.

The operator lives in libtaco (CUDA, sm_103a) behind the C ABI of
include/taco.h; ``binding`` wraps it for torch tensors.
"""

from .binding import (  # noqa: F401
    DEFAULT_TARGET_ENERGY, HEADER_BYTES, HEADER_DTYPE, MAX_SHARDS,
    VARIANT_ABSMAX, VARIANT_DUAL, VARIANT_STATIC,
    TacoError, library, new_workspace, parse_headers, shard_bytes, shard_scales_offset, shard_views,
    taco_compress, taco_compress_shards, taco_compress_shards_fwht, taco_compress_shards_int8,
    taco_compress_shards_mma,
    taco_compress_shards_noalloc, taco_decompress_reduce, taco_decompress_reduce_int8,
    taco_decompress_reduce_mma, taco_decompress_reduce_mma_ptrs, taco_decompress_reduce_ptrs,
    taco_decompress_shards, taco_decompress_shards_ptrs, taco_e4m3_decode_f32, taco_e4m3_encode_f32,
    taco_reduce_recompress, taco_reduce_recompress_ptrs, taco_reduce_recompress_int8_ptrs,
    taco_decompress_shards_int8_ptrs, taco_reduce_recompress_batched_ptrs, FORMAT_E4M3, FORMAT_INT8,
    workspace_bytes,
)
