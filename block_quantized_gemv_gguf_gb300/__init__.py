"""Block-quantized (GGUF Q8_0 / Q4_0 / Q4_K / Q6_K) GEMV and GEMM for GB300."""
