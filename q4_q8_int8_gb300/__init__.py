"""q4_K x q8_1 quantized GEMM for GB300 (sm_103a)."""
