"""Bit-exact block-scaled int8 GEMM for GB300 (sm_103a)."""
