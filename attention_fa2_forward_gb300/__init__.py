"""GB300-native fused multi-head attention forward (no KV cache)."""
