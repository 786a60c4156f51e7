"""GB300 (sm_103a) fused causal attention with grouped KV heads: libxattn and its binding.

Importing the package loads nothing. ``bwd_xattn_fwd_gb300.xattn`` loads the CUDA
library (and fails loudly if it has not been built); ``workloads`` holds the seeded
input recipes.
"""
__all__ = ["xattn", "workloads"]
