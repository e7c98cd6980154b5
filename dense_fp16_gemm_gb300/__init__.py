"""GB300-native dense fp16 NT GEMM (placeholder; binding follows)."""
