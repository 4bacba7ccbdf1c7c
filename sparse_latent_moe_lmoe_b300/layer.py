"""A torch-facing handle around the C ABI: device weight upload, workspace
allocation and stream plumbing. Argument marshalling only -- every step of
the layer runs in liblmoe.so's CUDA kernels."""
from __future__ import annotations

import ctypes

import numpy as np
import torch

from . import capi
from .capi import LmoeConfig, LmoePerm, LmoeWeights

_DT = {np.dtype(np.float32): torch.float32, np.dtype(np.uint8): torch.uint8, np.dtype(np.uint16): torch.int16,
       np.dtype(np.int32): torch.int32}


def to_device(a, device) -> torch.Tensor:
    """numpy (uint16 = bf16 bits) or torch tensor -> contiguous device tensor."""
    if a is None:
        return None
    if isinstance(a, torch.Tensor):
        return a.to(device).contiguous()
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to(device).contiguous()


def to_pinned(a):
    """A numpy array (or tensor) as page-locked host memory the device can address."""
    if a is None:
        return None
    t = a if isinstance(a, torch.Tensor) else torch.from_numpy(
        np.ascontiguousarray(a).view(np.int16) if a.dtype == np.uint16 else np.ascontiguousarray(a))
    return t.cpu().contiguous().pin_memory()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


class LatentMoE:
    """One latent MoE layer on one GPU.

    shape: any object with d, E, G, k, L, f, lora_rank, has_bias attributes
    (and optionally wfmt: "int4" or "nvfp4").
    weights: dict with the keys of capi.WEIGHT_FIELDS (numpy arrays or torch
    tensors in the layouts of include/lmoe.h; bf16 as uint16 bits).
    """

    def __init__(self, shape, weights: dict, device: int = 0, force_path: int = capi.PATH_AUTO,
                 decode_max_T: int = 0, timeout_cycles: int = 0, flags: int = 0, expert_slots: int = 0,
                 expert_weights_on_host: bool = False):
        self.shape = shape
        self.device = torch.device("cuda", device)
        # staged experts may keep gate / up / Down in page-locked host memory
        host = ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s") if expert_weights_on_host else ()
        self.dev_weights = {n: (to_pinned(weights.get(n)) if n in host else to_device(weights.get(n), self.device))
                            for n in capi.WEIGHT_FIELDS}
        nvfp4 = getattr(shape, "wfmt", "int4") == "nvfp4"
        self.cfg = LmoeConfig(shape.d, shape.E, shape.G, shape.k, shape.L, shape.f, 16 if nvfp4 else 32,
                              shape.lora_rank, 1 if shape.has_bias else 0, flags, timeout_cycles, decode_max_T,
                              force_path, capi.WEIGHTS_NVFP4 if nvfp4 else capi.WEIGHTS_INT4, expert_slots)
        self.wts = LmoeWeights(*[None if t is None else t.data_ptr() for t in
                                 (self.dev_weights[n] for n in capi.WEIGHT_FIELDS)])
        self.h = capi.lmoe_create(self.cfg, self.wts, device)
        self._ws = None
        self._ws_bytes = {}  # (T, host_staging) -> bytes (fixed per handle)

    # ----------------------------------------------------------- plumbing
    def workspace(self, T: int, host_staging: bool = False) -> torch.Tensor:
        n = self._ws_bytes.get((T, host_staging))
        if n is None:
            n = capi.lmoe_workspace_size(self.h, T)
            if host_staging:
                n = ((n + 255) // 256) * 256 + capi.lmoe_host_staging_size(self.h, T)
            self._ws_bytes[(T, host_staging)] = n
        if self._ws is None or self._ws.numel() < n:
            self._ws = torch.empty(max(n, 256), dtype=torch.uint8, device=self.device)
        return self._ws

    def close(self):
        if getattr(self, "h", None):
            capi.lmoe_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def check(self, stream=None):
        capi.lmoe_check(self.h, _stream(stream))

    # ------------------------------------------------------------ steps
    def route(self, x: torch.Tensor, want_logits: bool = False, stream=None):
        T = x.shape[0]
        sh = self.shape
        idx = torch.empty((T, sh.k), dtype=torch.int32, device=self.device)
        w = torch.empty((T, sh.k), dtype=torch.float32, device=self.device)
        logits = torch.empty((T, sh.E), dtype=torch.float32, device=self.device) if want_logits else None
        capi.lmoe_route(self.h, _ptr(x), T, _ptr(idx), _ptr(w), _ptr(logits), _ptr(self.workspace(T)),
                        _stream(stream))
        return idx, w, logits

    def alloc_perm(self, T: int) -> dict:
        sh = self.shape
        n = max(1, T * sh.k)
        z = lambda m: torch.empty(max(1, m), dtype=torch.int32, device=self.device)  # noqa: E731
        return dict(expert_offsets=z(sh.E + 1), sorted_assign=z(n), inv=z(n), group_offsets=z(sh.G + 1),
                    group_tok_offsets=z(sh.G + 1), group_tokens=z(T * min(sh.G, sh.k)), assign_row=z(n))

    @staticmethod
    def perm_struct(perm: dict) -> LmoePerm:
        return LmoePerm(*[perm[n].data_ptr() for n in capi.PERM_FIELDS])

    def permute(self, idx: torch.Tensor, stream=None) -> dict:
        T = idx.shape[0]
        perm = self.alloc_perm(T)
        capi.lmoe_permute(self.h, _ptr(idx), T, self.perm_struct(perm), _ptr(self.workspace(T)), _stream(stream))
        return perm

    def expert_forward(self, x, idx, w, perm: dict, stream=None) -> torch.Tensor:
        T = x.shape[0]
        sh = self.shape
        Y = torch.empty((max(1, T * min(sh.G, sh.k)), sh.d), dtype=torch.float32, device=self.device)
        capi.lmoe_expert_forward(self.h, _ptr(x), T, _ptr(idx), _ptr(w), self.perm_struct(perm), _ptr(Y),
                                 _ptr(self.workspace(T)), _stream(stream))
        return Y

    def combine(self, Y, idx, perm: dict, T: int, residual=None, stream=None) -> torch.Tensor:
        y = torch.empty((T, self.shape.d), dtype=torch.bfloat16, device=self.device)
        capi.lmoe_combine(self.h, _ptr(Y), _ptr(idx), self.perm_struct(perm), T, _ptr(residual), _ptr(y),
                          _stream(stream))
        return y

    def forward(self, x: torch.Tensor, residual=None, out=None, stream=None) -> torch.Tensor:
        T = x.shape[0]
        y = out if out is not None else torch.empty((T, self.shape.d), dtype=torch.bfloat16, device=self.device)
        capi.lmoe_layer_forward(self.h, _ptr(x), T, _ptr(residual), _ptr(y), _ptr(self.workspace(T)),
                                _stream(stream))
        return y

    def prefetch_experts(self, x: torch.Tensor, stream=None):
        """Staged experts: the prerouter stages this layer's predicted experts
        for the tokens x (lmoe_prefetch_experts)."""
        capi.lmoe_prefetch_experts(self.h, _ptr(x), x.shape[0], _stream(stream))

    def stage_stats(self) -> dict:
        return capi.lmoe_get_stage_stats(self.h)

    def last_decode_routing(self, T: int, stream=None):
        """(idx, w, logits) that the last decode-path forward of T <= 16 tokens
        on this layer's workspace selected (lmoe_decode_routing)."""
        sh = self.shape
        idx = torch.empty((T, sh.k), dtype=torch.int32, device=self.device)
        w = torch.empty((T, sh.k), dtype=torch.float32, device=self.device)
        logits = torch.empty((T, sh.E), dtype=torch.float32, device=self.device)
        capi.lmoe_decode_routing(self.h, _ptr(self.workspace(T)), T, _ptr(idx), _ptr(w), _ptr(logits),
                                 _stream(stream))
        return idx, w, logits

    def forward_noalloc(self, x: torch.Tensor, residual=None, out=None, stream=None) -> torch.Tensor:
        """The layer for T <= 16 tokens with the library's fixed per-device
        scratch instead of a workspace (lmoe_layer_forward_noalloc): the C call
        allocates nothing. `out` must be given by a caller that cannot allocate."""
        T = x.shape[0]
        y = out if out is not None else torch.empty((T, self.shape.d), dtype=torch.bfloat16, device=self.device)
        capi.lmoe_layer_forward_noalloc(self.h, _ptr(x), T, _ptr(residual), _ptr(y), _stream(stream))
        return y

    def forward_host(self, x_host: torch.Tensor, y_host: torch.Tensor, residual_host=None, stream=None):
        """Host (ideally pinned) bf16 tensors in and out; waits for the result."""
        T = x_host.shape[0]
        ws = self.workspace(T, host_staging=True)
        capi.lmoe_layer_forward_host(self.h, _ptr(x_host), T, _ptr(residual_host), _ptr(y_host), _ptr(ws),
                                     _stream(stream))
        return y_host


class LatentMoEStack:
    """A stack of LatentMoE layers of one shape (lmoe_stack_forward):
    x_{l+1} = bf16(x_l + bf16(layer_l(x_l)))."""

    def __init__(self, layers):
        self.layers = list(layers)
        if not self.layers:
            raise ValueError("empty stack")
        self.device = self.layers[0].device
        self._ws = None

    def workspace(self, T: int) -> torch.Tensor:
        n = capi.lmoe_stack_workspace_size(self.layers[0].h, T)
        if self._ws is None or self._ws.numel() < n:
            self._ws = torch.empty(max(n, 256), dtype=torch.uint8, device=self.device)
        return self._ws

    def forward(self, x: torch.Tensor, out=None, stream=None) -> torch.Tensor:
        T = x.shape[0]
        y = out if out is not None else torch.empty_like(x)
        capi.lmoe_stack_forward([m.h for m in self.layers], _ptr(x), T, _ptr(y), _ptr(self.workspace(T)),
                                _stream(stream))
        return y
