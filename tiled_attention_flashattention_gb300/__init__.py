"""GB300-native fused attention forward: tiled FlashAttention prefill and MLA decode."""
