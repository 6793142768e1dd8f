"""Fused Hadamard rotation + NVFP4 quantization for GB300 (sm_103a)."""
