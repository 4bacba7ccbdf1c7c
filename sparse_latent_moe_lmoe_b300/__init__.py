"""B300-native latent mixture-of-experts layer (Edge0-145B form).

The layer -- router, top-k with softmax renormalisation, the token
permutation by group then expert, shared int4 projections around a
per-expert latent SwiGLU, the optional Recover-LoRA branch and the weighted
combine -- runs in hand-written CUDA kernels for sm_103a behind the C ABI of
include/lmoe.h (liblmoe.so, built in-tree by `python -m
sparse_latent_moe_lmoe_b300.build`). This package is the thin Python binding:
`capi` has the C functions by name, `LatentMoE` wraps a handle with
torch-allocated device memory, `LatentMoEStack` runs a stack of them. Touching either loads the library and raises
ImportError if it has not been built -- there is no fallback.
"""
import importlib

__all__ = ["capi", "LatentMoE", "LatentMoEStack", "LmoeError", "PATH_AUTO", "PATH_DECODE", "PATH_PREFILL"]


def __getattr__(name):
    if name == "capi":
        return importlib.import_module(".capi", __name__)
    if name in ("LatentMoE", "LatentMoEStack"):
        return getattr(importlib.import_module(".layer", __name__), name)
    if name in ("LmoeError", "PATH_AUTO", "PATH_DECODE", "PATH_PREFILL"):
        return getattr(importlib.import_module(".capi", __name__), name)
    raise AttributeError(name)
