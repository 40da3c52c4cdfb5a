"""GB300-native (sm_103a) KV-cache codec for multi-agent KV sharing.

SharedKVPool ("PolyKV": int8 keys with a per-tensor scale; values rotated by
a Walsh-Hadamard transform and coded at 3 bits with the Lloyd-Max N(0,1)
codebook; fan-out decode into N agent caches) and CacheCard ("QKVShare":
per-token {2,4,8,16}-bit asymmetric group quantization with metadata), as a
C-ABI CUDA library (include/kvpool.h) with this thin ctypes binding.
"""
from .binding import (  # noqa: F401
    KVP_ERR_ALIGN, KVP_ERR_ARG, KVP_ERR_BITS, KVP_ERR_CUDA, KVP_ERR_HEADER, KVP_ERR_NONFINITE,
    KVP_ERR_RANGE, KVP_ERR_SIZE, KVP_ERR_TIMEOUT, KVP_ERR_UNSUPPORTED_D, KVP_MAX_LAYERS, KVP_OK, CardHeader, KVPError,
    Shape, cachecard_bytes, cachecard_pack, cachecard_read_header, cachecard_status, cachecard_unpack,
    cachecard_unpack_at,
    check, declared_functions, kvp_bandwidth_probe, KVP_PROBE_STORE, KVP_PROBE_BULK_STORE, KVP_PROBE_COPY,
    kvp_launch_count, kvp_test_fail_next_encode, kvp_test_limit_next_attend, kvp_test_limit_next_unpack, kvp_strerror, kvpool_attend, kvpool_attend_workspace_bytes, kvpool_attend_lora,
    kvpool_attend_lora_workspace_bytes, kvpool_decode_into, kvpool_encode, kvpool_encode_ex, kvpool_encode_noalloc, KVP_NOALLOC_SCRATCH_BYTES,
    kvpool_pool_bytes, kvpool_pool_bytes_ex, kvpool_status, KVP_K_PER_TENSOR, KVP_K_Q8_0, kvpool_workspace_bytes, load,
)
