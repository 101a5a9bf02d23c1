"""GB300-native split-K BF16 decode GEMM (placeholder until the binding lands)."""
