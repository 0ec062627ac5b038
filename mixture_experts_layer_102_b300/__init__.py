"""B300-native forward pass of a top-k routed Mixture-of-Experts FFN layer.

The compute runs in hand-written sm_103a CUDA kernels behind a C-ABI shared library
(``libmoe_b300.so``, built in this directory). ``mixture_experts_layer_102_b300.moe``
is the thin Python binding over that library; ``configs`` and ``inputs`` hold the named
workloads and the seeded synthetic input generator.
"""
__all__ = ["configs", "inputs", "moe"]
