"""Sub-byte quantized KV cache with fused-dequantization decode attention for GB300 (sm_103a).

The compute path is the CUDA library built from ``csrc/`` (C ABI in
``include/kvq.h``); :mod:`.kvq` is its thin Python binding.
"""
from .kvq import (KVQError, QuantizedKVCache, kvq_block_bytes, kvq_decode_attention, kvq_decode_num_splits,  # noqa: F401
                  kvq_decode_split, kvq_decode_combine, kvq_decode_workspace_bytes,
                  kvq_decode_attention_noalloc, kvq_dequantize, kvq_project_append, kvq_quantize_append, kvq_status_string,
                  kvq_version)
