"""GB300-native GGUF block-quantized mul_mat (Q8_0 / Q4_K / Q6_K weights, fp32 activations).

The compute path is the C-ABI library ``libsyn.so`` built from ``csrc/`` for sm_103a;
``syn`` is its thin ctypes binding.  Importing this package does not load the library;
``from gguf_block_quantized_gb300 import syn`` does, and fails loudly if it is missing.
"""
__all__ = ["syn", "synth", "workloads"]
