"""GB300-native per-token-group fp8 e4m3 quantization (placeholder)."""
