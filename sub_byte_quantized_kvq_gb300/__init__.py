"""Sub-byte quantized KV cache with fused-dequantization decode attention for GB300 (sm_103a)."""
