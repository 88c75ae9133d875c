"""GB300-native fused multi-query FlashAttention forward (DeepSeek V4 Flash shape)."""
