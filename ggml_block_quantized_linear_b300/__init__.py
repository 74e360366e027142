"""B300-native GGML block-quantized linear layers (Q8_0, Q4_K)."""
