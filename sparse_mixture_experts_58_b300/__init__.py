"""B300-native (sm_103a) Mixtral sparse mixture-of-experts feed-forward layer.

``sparse_mixture_experts_58_b300.moe`` is the Python binding over the C-ABI
library ``libmoe.so`` (every step runs in hand-written CUDA kernels; importing
it without the built library raises).  ``sparse_mixture_experts_58_b300.inputs``
draws the seeded synthetic workloads and needs no GPU.
"""
__all__ = ["inputs", "moe"]
