"""B300-native latent mixture-of-experts layer (Edge0-145B form).

The layer -- router, top-k with softmax renormalisation, the token
permutation by group then expert, shared int4 projections around a
per-expert latent SwiGLU, the optional Recover-LoRA branch and the weighted
combine -- runs in hand-written CUDA kernels for sm_103a behind the C ABI of
include/lmoe.h (liblmoe.so, built in-tree). This package is the thin Python
binding: `capi` has the C functions by name, `LatentMoE` wraps a handle with
torch-allocated device memory.
"""
from . import capi  # noqa: F401  (loads liblmoe.so; raises ImportError if it is not built)
from .capi import LmoeError, PATH_AUTO, PATH_DECODE, PATH_PREFILL  # noqa: F401
from .layer import LatentMoE  # noqa: F401

__all__ = ["capi", "LatentMoE", "LmoeError", "PATH_AUTO", "PATH_DECODE", "PATH_PREFILL"]
