"""TEST INFRASTRUCTURE: the CPU oracle for the latent MoE layer.

A plain single-threaded fp64 C implementation (oracle.c) of what the layer
computes, wrapped with ctypes. Only the test suite, the smoke check and the
benchmark's CPU-baseline leg may import this package; the CUDA library never
uses it. See oracle.c for the definitions and the passages they follow.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c (gcc -O2, strict IEEE double: no fast-math, no FMA contraction)."""
    src = os.path.join(_HERE, "oracle.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        tmp = _SO + ".tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", src, "-o", tmp,
                               "-lm"])
        os.replace(tmp, _SO)
    return _SO


_GS = ("W_in_gs", "W_out_gs", "gate_gs", "up_gs", "down_gs")


class _Layer(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("d", "E", "G", "k", "L", "f", "r")] + [
        (n, ctypes.c_void_p) for n in ("W_r", "b_r", "W_in_q", "W_in_s", "W_out_q", "W_out_s", "gate_q", "gate_s",
                                       "up_q", "up_s", "down_q", "down_s", "A_in", "B_in", "A_out", "B_out")] + [
        ("wfmt", ctypes.c_int)] + [(n, ctypes.c_void_p) for n in _GS]


def _p(a):
    if a is None:
        return None
    assert a.flags.c_contiguous
    return a.ctypes.data_as(ctypes.c_void_p).value


def _lib_():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_SO)
        P, I, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
        lib.oracle_bf16_round.argtypes = [ctypes.c_double]
        lib.oracle_bf16_round.restype = ctypes.c_uint16
        lib.oracle_bf16_round_array.argtypes = [I64, P, P]
        lib.oracle_int4_at.argtypes = [P, I]
        lib.oracle_int4_at.restype = I
        lib.oracle_dequant_rows.argtypes = [P, P, I, I64, I, P]
        lib.oracle_e2m1_value.argtypes = [I]
        lib.oracle_e2m1_value.restype = ctypes.c_double
        lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_value.restype = ctypes.c_double
        lib.oracle_nvfp4_dequant_rows.argtypes = [P, P, ctypes.c_double, I, I64, I, P]
        lib.oracle_router_logits.argtypes = [P, I, P, P]
        lib.oracle_topk.argtypes = [I, I, I, P, P, P]
        lib.oracle_permute.argtypes = [I, I, I, I, P, P, P, P, P, P, P, P]
        lib.oracle_permute.restype = I
        lib.oracle_shared_in.argtypes = [P, I, P, P]
        lib.oracle_shared_out.argtypes = [P, I, P, P]
        lib.oracle_expert_latent.argtypes = [P, I, P, P]
        lib.oracle_forward_routed.argtypes = [P, I, P, P, P, P]
        lib.oracle_forward_routed_factored.argtypes = [P, I, P, P, P, P]
        lib.oracle_layer_forward.argtypes = [P, I, P, P, P, P, P]
        lib.oracle_group_row.argtypes = [P, I, P, P, P, P]
        lib.oracle_residual.argtypes = [I64, P, P, P]
        lib.oracle_combine.argtypes = [I, I, I, I, I, P, P, P, P, P]
        _lib = lib
    return _lib


class Layer:
    """Binds a weights dict (lmoe_synth layout) for the C oracle. Keeps the
    arrays alive while the struct points at them."""

    def __init__(self, shape, W: dict):
        self.shape = shape
        self._keep = {k: (None if v is None else np.ascontiguousarray(v)) for k, v in W.items()}
        k = self._keep
        self.s = _Layer(shape.d, shape.E, shape.G, shape.k, shape.L, shape.f, shape.lora_rank,
                        *[_p(k.get(n)) for n in ("W_r", "b_r", "W_in_q", "W_in_s", "W_out_q", "W_out_s", "gate_q",
                                                 "gate_s", "up_q", "up_s", "down_q", "down_s", "A_in", "B_in",
                                                 "A_out", "B_out")])
        if shape.lora_rank == 0:
            self.s.A_in = self.s.B_in = self.s.A_out = self.s.B_out = None
        self.s.wfmt = 1 if getattr(shape, "wfmt", "int4") == "nvfp4" else 0
        for n in _GS:
            setattr(self.s, n, _p(k.get(n)))
        if self.s.wfmt == 1 and any(k.get(n) is None for n in _GS):
            raise ValueError("NVFP4 weights need every per-tensor scale array")

    @property
    def ref(self):
        return ctypes.byref(self.s)


# ------------------------------------------------------------------ formats

def bf16_round(v) -> np.ndarray:
    """bf16 RNE (single rounding from fp64) -> uint16 bit patterns."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, np.uint16)
    _lib_().oracle_bf16_round_array(v.size, _p(v), _p(out))
    return out


def bf16_value(b) -> np.ndarray:
    b = np.asarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def int4_at(row: np.ndarray, k: int) -> int:
    row = np.ascontiguousarray(row, dtype=np.uint8)
    return _lib_().oracle_int4_at(_p(row), k)


def dequant(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """All rows of a packed int4 matrix q [rows][K/2] with scales [rows][K/32]."""
    q = np.ascontiguousarray(q.reshape(-1, q.shape[-1]))
    s = np.ascontiguousarray(s.reshape(-1, s.shape[-1]))
    rows, K = q.shape[0], q.shape[1] * 2
    out = np.empty((rows, K), np.float64)
    _lib_().oracle_dequant_rows(_p(q), _p(s), K, 0, rows, _p(out))
    return out


def e2m1_value(code: int) -> float:
    """Value of an FP4 E2M1 code (0..15)."""
    return _lib_().oracle_e2m1_value(int(code))


def e4m3_value(b: int) -> float:
    """Value of an FP8 E4M3 byte (finite-only format; NaN for S.1111.111)."""
    return _lib_().oracle_e4m3_value(int(b))


def nvfp4_dequant(q: np.ndarray, s: np.ndarray, gs: float) -> np.ndarray:
    """All rows of one NVFP4 tensor: codes q [rows][K/2], E4M3 block scales
    s [rows][K/16] (bytes), fp32 tensor scale gs."""
    q = np.ascontiguousarray(q.reshape(-1, q.shape[-1]))
    s = np.ascontiguousarray(s.reshape(-1, s.shape[-1]), dtype=np.uint8)
    rows, K = q.shape[0], q.shape[1] * 2
    out = np.empty((rows, K), np.float64)
    _lib_().oracle_nvfp4_dequant_rows(_p(q), _p(s), float(gs), K, 0, rows, _p(out))
    return out


# ------------------------------------------------------------------- steps

def router_logits(layer: Layer, x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, np.uint16)
    n = x.shape[0]
    out = np.empty((n, layer.shape.E), np.float64)
    _lib_().oracle_router_logits(layer.ref, n, _p(x), _p(out))
    return out


def topk(logits: np.ndarray, k: int):
    logits = np.ascontiguousarray(logits, np.float64)
    n, E = logits.shape
    idx = np.empty((n, k), np.int32)
    w = np.empty((n, k), np.float64)
    _lib_().oracle_topk(n, E, k, _p(logits), _p(idx), _p(w))
    return idx, w


def permute(idx: np.ndarray, E: int, G: int) -> dict:
    idx = np.ascontiguousarray(idx, np.int32)
    T, k = idx.shape
    n = T * k
    out = dict(expert_offsets=np.empty(E + 1, np.int32), sorted_assign=np.empty(n, np.int32),
               inv=np.empty(n, np.int32), group_offsets=np.empty(G + 1, np.int32),
               group_tok_offsets=np.empty(G + 1, np.int32), group_tokens=np.empty(max(1, T * min(G, k)), np.int32),
               assign_row=np.empty(n, np.int32))
    rows = _lib_().oracle_permute(T, E, G, k, _p(idx), *[_p(out[n_]) for n_ in (
        "expert_offsets", "sorted_assign", "inv", "group_offsets", "group_tok_offsets", "group_tokens",
        "assign_row")])
    out["group_tokens"] = out["group_tokens"][:rows].copy()
    out["rows"] = rows
    return out


def shared_in(layer: Layer, g: int, x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, np.float64)
    h = np.empty(layer.shape.L, np.float64)
    _lib_().oracle_shared_in(layer.ref, g, _p(x), _p(h))
    return h


def shared_out(layer: Layer, g: int, u: np.ndarray) -> np.ndarray:
    u = np.ascontiguousarray(u, np.float64)
    o = np.empty(layer.shape.d, np.float64)
    _lib_().oracle_shared_out(layer.ref, g, _p(u), _p(o))
    return o


def expert_latent(layer: Layer, e: int, h: np.ndarray) -> np.ndarray:
    h = np.ascontiguousarray(h, np.float64)
    u = np.empty(layer.shape.L, np.float64)
    _lib_().oracle_expert_latent(layer.ref, e, _p(h), _p(u))
    return u


def forward_routed(layer: Layer, x: np.ndarray, idx: np.ndarray, w: np.ndarray, factored: bool = False):
    x = np.ascontiguousarray(x, np.uint16)
    idx = np.ascontiguousarray(idx, np.int32)
    w = np.ascontiguousarray(w, np.float64)
    n = x.shape[0]
    sh = layer.shape
    if x.shape != (n, sh.d) or idx.shape != (n, sh.k) or w.shape != (n, sh.k):
        raise ValueError("x must be [n][d], idx and w [n][k]")
    if idx.size and (idx.min() < 0 or idx.max() >= sh.E):
        raise ValueError("expert index out of range")
    y = np.empty((n, layer.shape.d), np.float64)
    fn = _lib_().oracle_forward_routed_factored if factored else _lib_().oracle_forward_routed
    fn(layer.ref, n, _p(x), _p(idx), _p(w), _p(y))
    return y


def layer_forward(layer: Layer, x: np.ndarray):
    """(y fp64 [n][d], idx [n][k], w fp64 [n][k], logits fp64 [n][E])"""
    x = np.ascontiguousarray(x, np.uint16)
    n = x.shape[0]
    sh = layer.shape
    if x.shape != (n, sh.d):
        raise ValueError("x must be [n][d]")
    y = np.empty((n, sh.d), np.float64)
    idx = np.empty((n, sh.k), np.int32)
    w = np.empty((n, sh.k), np.float64)
    logits = np.empty((n, sh.E), np.float64)
    _lib_().oracle_layer_forward(layer.ref, n, _p(x), _p(y), _p(idx), _p(w), _p(logits))
    return y, idx, w, logits


def group_row(layer: Layer, g: int, x_t: np.ndarray, idx_t: np.ndarray, w_t: np.ndarray) -> np.ndarray:
    x_t = np.ascontiguousarray(x_t, np.uint16)
    idx_t = np.ascontiguousarray(idx_t, np.int32)
    w_t = np.ascontiguousarray(w_t, np.float64)
    sh = layer.shape
    if x_t.shape != (sh.d,) or idx_t.shape != (sh.k,) or w_t.shape != (sh.k,) or not 0 <= g < sh.G:
        raise ValueError("x_t must be [d], idx_t and w_t [k], 0 <= g < G")
    y = np.empty(layer.shape.d, np.float64)
    _lib_().oracle_group_row(layer.ref, g, _p(x_t), _p(idx_t), _p(w_t), _p(y))
    return y


def residual(x: np.ndarray, y: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, np.uint16)
    y = np.ascontiguousarray(y, np.float64)
    out = np.empty(x.shape, np.uint16)
    _lib_().oracle_residual(x.size, _p(x), _p(y), _p(out))
    return out


def combine(Y: np.ndarray, idx: np.ndarray, assign_row: np.ndarray, E: int, G: int, residual=None) -> np.ndarray:
    """fp64 combine of per-(group, token) rows Y [rows][d] (fp32)."""
    Y = np.ascontiguousarray(Y, np.float32)
    idx = np.ascontiguousarray(idx, np.int32)
    assign_row = np.ascontiguousarray(assign_row, np.int32)
    T, k = idx.shape
    d = Y.shape[1]
    if residual is not None:
        residual = np.ascontiguousarray(residual, np.uint16)
    y = np.empty((T, d), np.float64)
    _lib_().oracle_combine(T, d, k, G, E // G, _p(Y), _p(idx), _p(assign_row), _p(residual), _p(y))
    return y
