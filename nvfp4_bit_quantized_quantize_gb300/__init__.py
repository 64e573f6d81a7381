"""NVFP4 quantize + block-scaled GEMM for GB300 (sm_103a)."""
