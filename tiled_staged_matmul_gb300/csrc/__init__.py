"""CUDA sources of the GEMM library and their build step."""
