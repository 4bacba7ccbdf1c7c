"""Seeded synthetic inputs for the latent MoE layer.

Shapes and distributions follow the workloads the Edge0-145B pages describe
(512 experts in groups of 64 sharing two large matrices, top-10 routing, int4
frozen base, optional Recover-LoRA branch) at the concrete sizes this library
is measured on. The module draws inputs only: it holds none of the layer's
arithmetic, and both the CPU oracle and the CUDA library consume the arrays it
returns as plain bytes.

Layouts (all C-contiguous numpy arrays; bf16 values are uint16 bit patterns):

  W_r    f32  [E][d]            router weights
  b_r    f32  [E]               router bias (Zipf popularity), or None
  W_in_q u8   [G][L][d/2]       shared down-projection, int4 packed
  W_in_s u16  [G][L][d/32]      its bf16 scales
  W_out_q u8  [G][d][L/2]       shared up-projection
  W_out_s u16 [G][d][L/32]
  gate_q, up_q  u8 [E][f][L/2]  per-expert SwiGLU gate / up (scales [E][f][L/32])
  down_q        u8 [E][L][f/2]  per-expert down (scales [E][L][f/32])
  A_in  bf16 [G][d][r], B_in bf16 [G][r][L], A_out bf16 [G][L][r], B_out bf16 [G][r][d]
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, replace

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "_synth.so")
_lib = None

# stream ids: one independent random stream per logical tensor
S_WR, S_BIAS, S_WIN, S_WOUT, S_GATE, S_UP, S_DOWN = 1, 2, 3, 4, 5, 6, 7
S_AIN, S_BIN, S_AOUT, S_BOUT, S_X = 8, 9, 10, 11, 12


def build(force: bool = False) -> str:
    """Compile synth.c into _synth.so (gcc, -O2)."""
    src = os.path.join(_HERE, "synth.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        tmp = _SO + ".tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-D_DEFAULT_SOURCE", "-fPIC", "-shared", src,
                               "-o", tmp, "-lm", "-lpthread"])
        os.replace(tmp, _SO)
    return _SO


def _L():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_SO)
        u64, i64, d, p = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
        lib.synth_normal_f32.argtypes = [u64, u64, i64, d, p]
        lib.synth_normal_bf16.argtypes = [u64, u64, i64, d, p]
        lib.synth_int4_matrix.argtypes = [u64, u64, i64, ctypes.c_int, d, p, p]
        lib.synth_int4_matrix.restype = ctypes.c_int
        lib.synth_int4_source.argtypes = [u64, u64, i64, ctypes.c_int, d, p]
        lib.synth_nvfp4_matrix.argtypes = [u64, u64, i64, ctypes.c_int, d, i64, p, p, p]
        lib.synth_e4m3_rne.argtypes = [ctypes.c_float]
        lib.synth_e4m3_rne.restype = ctypes.c_uint8
        lib.synth_zipf_bias.argtypes = [u64, ctypes.c_int, d, p]
        lib.synth_routing.argtypes = [u64, ctypes.c_int, ctypes.c_int, ctypes.c_int, d, p, p]
        lib.synth_set_threads.argtypes = [ctypes.c_int]
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags.c_contiguous
    return a.ctypes.data_as(ctypes.c_void_p)


def set_threads(n: int) -> None:
    """Host threads used by the generators (0 = all online cores)."""
    _L().synth_set_threads(int(n))


def normal_f32(seed: int, stream: int, shape, sigma: float) -> np.ndarray:
    out = np.empty(shape, np.float32)
    _L().synth_normal_f32(seed, stream, out.size, sigma, _ptr(out))
    return out


def normal_bf16(seed: int, stream: int, shape, sigma: float) -> np.ndarray:
    out = np.empty(shape, np.uint16)
    _L().synth_normal_bf16(seed, stream, out.size, sigma, _ptr(out))
    return out


def int4_matrix(seed: int, stream: int, rows: int, K: int, sigma: float):
    """(q packed u8 [rows][K/2], scales bf16 bits u16 [rows][K/32])"""
    q = np.empty((rows, K // 2), np.uint8)
    s = np.empty((rows, K // 32), np.uint16)
    rc = _L().synth_int4_matrix(seed, stream, rows, K, sigma, _ptr(q), _ptr(s))
    if rc != 0:
        raise ValueError("K must be a multiple of 32")
    return q, s


def nvfp4_matrix(seed: int, stream: int, rows: int, K: int, sigma: float, rows_per_tensor: int):
    """The same draws as int4_matrix in NVFP4: (E2M1 codes u8 [rows][K/2],
    E4M3 block scales u8 [rows][K/16], fp32 tensor scales [rows/rows_per_tensor])."""
    q = np.empty((rows, K // 2), np.uint8)
    s = np.empty((rows, K // 16), np.uint8)
    gs = np.empty(rows // rows_per_tensor, np.float32)
    rc = _L().synth_nvfp4_matrix(seed, stream, rows, K, sigma, rows_per_tensor, _ptr(q), _ptr(s), _ptr(gs))
    if rc != 0:
        raise ValueError("K must be a multiple of 16 and rows a multiple of rows_per_tensor")
    return q, s, gs


def e4m3_rne(x: float) -> int:
    """The quantiser's fp32 -> E4M3 rounding (x >= 0, saturating at 448)."""
    return int(_L().synth_e4m3_rne(float(x)))


def int4_source(seed: int, stream: int, rows: int, K: int, sigma: float) -> np.ndarray:
    """The fp32 draws that int4_matrix quantises."""
    out = np.empty((rows, K), np.float32)
    _L().synth_int4_source(seed, stream, rows, K, sigma, _ptr(out))
    return out


def zipf_bias(seed: int, E: int, s: float = 1.1) -> np.ndarray:
    out = np.empty(E, np.float32)
    _L().synth_zipf_bias(seed, E, s, _ptr(out))
    return out


def routing(seed: int, T: int, E: int, k: int, skew: float = 0.0):
    """Synthetic (idx i32 [T][k], w f32 [T][k]): distinct experts per token,
    weights positive, descending and summing to 1."""
    if k > 64 or k > E:
        raise ValueError("k must be <= min(64, E)")
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float32)
    _L().synth_routing(seed, T, E, k, skew, _ptr(idx), _ptr(w))
    return idx, w


@dataclass(frozen=True)
class LayerShape:
    d: int
    E: int
    G: int
    k: int
    L: int
    f: int
    lora_rank: int = 0
    has_bias: bool = False
    wfmt: str = "int4"  # or "nvfp4"

    @property
    def epg(self) -> int:
        return self.E // self.G


# the workloads: a tiny layer the oracle finishes in seconds, and the
# Edge0-shaped layer (512 experts / 8 groups / top-10, latent 1024, expert 256)
TINY = LayerShape(d=256, E=16, G=2, k=2, L=64, f=32)
EDGE0 = LayerShape(d=4096, E=512, G=8, k=10, L=1024, f=256)

WORKLOADS = {
    # name: (shape, T, weight seed, x seed, bias seed or None, lora seed or None)
    "tiny_t64": (TINY, 64, 0, 0, None, None),
    "decode_t8": (EDGE0, 8, 0, 1, None, None),
    "prefill_t16384_zipf": (replace(EDGE0, has_bias=True), 16384, 0, 1, 2, None),
    "lora_t16": (replace(EDGE0, lora_rank=64), 16, 0, 1, None, 3),
    # a small layer within the single-kernel decode pass's shapes (d 1024, L 256), for quick path tests
    "small_t16_nvfp4": (LayerShape(d=1024, E=64, G=4, k=10, L=256, f=256, wfmt="nvfp4"), 16, 0, 1, None, None),
    "small_t256_nvfp4": (LayerShape(d=1024, E=64, G=4, k=10, L=256, f=256, wfmt="nvfp4"), 256, 0, 1, None, None),
    # the same layers with NVFP4 weights (the same fp32 draws, quantised to NVIDIA's FP4 format)
    "tiny_t64_nvfp4": (replace(TINY, wfmt="nvfp4"), 64, 0, 0, None, None),
    "decode_t8_nvfp4": (replace(EDGE0, wfmt="nvfp4"), 8, 0, 1, None, None),
    "prefill_t16384_zipf_nvfp4": (replace(EDGE0, has_bias=True, wfmt="nvfp4"), 16384, 0, 1, 2, None),
    # the 16K prefill layer with its rank-64 Recover-LoRA branch
    "prefill_t16384_zipf_lora": (replace(EDGE0, has_bias=True, lora_rank=64), 16384, 0, 1, 2, 3),
}

W_SIGMA = 0.02       # int4 weights and router before quantisation
LORA_A_SIGMA = 0.02
LORA_B_SIGMA = 0.002


def make_layer(shape: LayerShape, seed: int, bias_seed: int | None = None, lora_seed: int | None = None,
               zipf_s: float = 1.1) -> dict:
    d, E, G, L, f, r = shape.d, shape.E, shape.G, shape.L, shape.f, shape.lora_rank
    W = {}
    W["W_r"] = normal_f32(seed, S_WR, (E, d), W_SIGMA)
    W["b_r"] = zipf_bias(bias_seed, E, zipf_s) if shape.has_bias else None
    # (name, stream, tensors, rows per tensor, K)
    mats = [("W_in", S_WIN, G, L, d), ("W_out", S_WOUT, G, d, L), ("gate", S_GATE, E, f, L), ("up", S_UP, E, f, L),
            ("down", S_DOWN, E, L, f)]
    for name, stream, nt, rows, K in mats:
        if shape.wfmt == "nvfp4":
            q, s, gs = nvfp4_matrix(seed, stream, nt * rows, K, W_SIGMA, rows)
            W[name + "_q"], W[name + "_s"], W[name + "_gs"] = q.reshape(nt, rows, K // 2), s.reshape(nt, rows, K // 16), gs
        else:
            q, s = int4_matrix(seed, stream, nt * rows, K, W_SIGMA)
            W[name + "_q"], W[name + "_s"], W[name + "_gs"] = q.reshape(nt, rows, K // 2), s.reshape(nt, rows, K // 32), None
    if r > 0:
        ls = seed if lora_seed is None else lora_seed
        W["A_in"] = normal_bf16(ls, S_AIN, (G, d, r), LORA_A_SIGMA)
        W["B_in"] = normal_bf16(ls, S_BIN, (G, r, L), LORA_B_SIGMA)
        W["A_out"] = normal_bf16(ls, S_AOUT, (G, L, r), LORA_A_SIGMA)
        W["B_out"] = normal_bf16(ls, S_BOUT, (G, r, d), LORA_B_SIGMA)
    else:
        W["A_in"] = W["B_in"] = W["A_out"] = W["B_out"] = None
    return W


def make_x(T: int, d: int, seed: int) -> np.ndarray:
    """Activations: bf16 bits [T][d], N(0, 1)."""
    return normal_bf16(seed, S_X, (T, d), 1.0)


def make_workload(name: str):
    """(shape, T, weights dict, x)"""
    shape, T, ws, xs, bs, lsd = WORKLOADS[name]
    return shape, T, make_layer(shape, ws, bs, lsd), make_x(T, shape.d, xs)


def stack_layer_seed(layer: int) -> int:
    """Per-layer seed of the 48-layer stack (router and all weights)."""
    return 1000 + layer


def make_stack_layer(shape: LayerShape, layer: int) -> dict:
    """Weights of layer `layer` of a stack of `shape` layers."""
    return make_layer(shape, stack_layer_seed(layer))


STACK_WORKLOADS = {
    # name: (layer shape, layers, tokens per step, x seed)
    "stack48_t1": (EDGE0, 48, 1, 1),
    "stack48_t8": (EDGE0, 48, 8, 1),
    "stack48_prefill_t4096": (EDGE0, 48, 4096, 1),
}

# stacks whose expert weights stay in page-locked host memory with a fixed
# number of GPU slots per layer (the staged expert cache):
# name: (layer shape, layers, tokens per step, x seed, GPU slots per layer)
STAGED_STACK_WORKLOADS = {
    "stack8_t1_staged": (EDGE0, 8, 1, 1, 160),
    "stack8_t8_staged": (EDGE0, 8, 8, 1, 160),
}


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32)
