"""GB300-native batched routed-MoE FFN (sm_103a CUDA kernels behind a C ABI).

``workloads`` (seeded synthetic inputs) imports nothing else from the package.
The CUDA library is loaded on first use by ``mixture_experts_ffn_top_gb300.ops``;
a missing library is an error, never a fallback.
"""
__all__ = ["workloads"]
