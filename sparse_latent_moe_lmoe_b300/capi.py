"""ctypes binding of liblmoe.so, with the C ABI's names (include/lmoe.h).

Argument marshalling only: every step of the layer runs in the library's
CUDA kernels. Functions raise LmoeError on a non-OK status. Importing this
module loads the library and fails loudly if it has not been built.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liblmoe.so")

LMOE_OK = 0
STATUS = {0: "LMOE_OK", 1: "LMOE_ERR_INVALID_ARG", 2: "LMOE_ERR_UNSUPPORTED", 3: "LMOE_ERR_ALIGNMENT",
          4: "LMOE_ERR_CUDA", 5: "LMOE_ERR_TIMEOUT", 6: "LMOE_ERR_DEVICE_CHECK", 7: "LMOE_ERR_NO_MEMORY"}
PATH_AUTO, PATH_DECODE, PATH_PREFILL = 0, 1, 2
FLAG_MULTI_KERNEL_DECODE = 1
FLAG_STAGED_EXPERTS = 2

EXPORTS = ("lmoe_status_string", "lmoe_version", "lmoe_create", "lmoe_destroy", "lmoe_workspace_size", "lmoe_route",
           "lmoe_permute", "lmoe_expert_forward", "lmoe_combine", "lmoe_layer_forward", "lmoe_layer_forward_noalloc",
           "lmoe_layer_forward_host", "lmoe_stack_forward", "lmoe_stack_workspace_size",
           "lmoe_host_staging_size", "lmoe_check", "lmoe_set_timeout", "lmoe_set_stage_events", "lmoe_stage_name",
           "lmoe_launch_count", "lmoe_decode_routing", "lmoe_prefetch_experts", "lmoe_get_stage_stats")


class LmoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} ({_status_string(status)})")


class LmoeConfig(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int), ("E", ctypes.c_int), ("G", ctypes.c_int), ("k", ctypes.c_int),
                ("L", ctypes.c_int), ("f", ctypes.c_int), ("qgroup", ctypes.c_int), ("lora_rank", ctypes.c_int),
                ("has_bias", ctypes.c_int), ("flags", ctypes.c_uint), ("timeout_cycles", ctypes.c_longlong),
                ("decode_max_T", ctypes.c_int), ("force_path", ctypes.c_int), ("weight_format", ctypes.c_int),
                ("expert_slots", ctypes.c_int)]


WEIGHTS_INT4, WEIGHTS_NVFP4 = 0, 1

WEIGHT_FIELDS = ("W_r", "b_r", "W_in_q", "W_in_s", "W_out_q", "W_out_s", "gate_q", "gate_s", "up_q", "up_s", "down_q",
                 "down_s", "A_in", "B_in", "A_out", "B_out", "W_in_gs", "W_out_gs", "gate_gs", "up_gs", "down_gs")


class LmoeWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in WEIGHT_FIELDS]


PERM_FIELDS = ("expert_offsets", "sorted_assign", "inv", "group_offsets", "group_tok_offsets", "group_tokens",
               "assign_row")


class LmoeStageStats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_ulonglong) for n in ("passes", "routed", "hits", "staged_on_demand", "prefetched",
                                                   "bytes_copied")]


class LmoePerm(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in PERM_FIELDS]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with `python -m sparse_latent_moe_lmoe_b300.build` "
                          "(there is no fallback implementation)")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_int
    sz = ctypes.c_size_t
    sig = {
        "lmoe_status_string": ([I], ctypes.c_char_p),
        "lmoe_version": ([], I),
        "lmoe_create": ([ctypes.POINTER(P), ctypes.POINTER(LmoeConfig), ctypes.POINTER(LmoeWeights), I], S),
        "lmoe_destroy": ([P], S),
        "lmoe_workspace_size": ([P, I], sz),
        "lmoe_host_staging_size": ([P, I], sz),
        "lmoe_route": ([P, P, I, P, P, P, P, P], S),
        "lmoe_permute": ([P, P, I, ctypes.POINTER(LmoePerm), P, P], S),
        "lmoe_expert_forward": ([P, P, I, P, P, ctypes.POINTER(LmoePerm), P, P, P], S),
        "lmoe_combine": ([P, P, P, ctypes.POINTER(LmoePerm), I, P, P, P], S),
        "lmoe_layer_forward": ([P, P, I, P, P, P, P], S),
        "lmoe_layer_forward_noalloc": ([P, P, I, P, P, P], S),
        "lmoe_layer_forward_host": ([P, P, I, P, P, P, P], S),
        "lmoe_stack_forward": ([P, I, P, I, P, P, P], S),
        "lmoe_stack_workspace_size": ([P, I], sz),
        "lmoe_check": ([P, P], S),
        "lmoe_set_timeout": ([P, ctypes.c_longlong], S),
        "lmoe_set_stage_events": ([P, P, I], S),
        "lmoe_stage_name": ([P, I, I, ctypes.POINTER(I)], ctypes.c_char_p),
        "lmoe_launch_count": ([P, I], I),
        "lmoe_decode_routing": ([P, P, I, P, P, P, P], S),
        "lmoe_prefetch_experts": ([P, P, I, P], S),
        "lmoe_get_stage_stats": ([P, ctypes.POINTER(LmoeStageStats)], S),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


_lib = _load()


def _status_string(s: int) -> str:
    return _lib.lmoe_status_string(int(s)).decode()


def _ok(status: int, where: str):
    if status != LMOE_OK:
        raise LmoeError(status, where)


def library():
    return _lib


# ----------------------------------------------------------- C ABI, by name

def lmoe_status_string(status: int) -> str:
    return _status_string(status)


def lmoe_version() -> int:
    return _lib.lmoe_version()


def lmoe_create(cfg: LmoeConfig, weights: LmoeWeights, device: int) -> int:
    h = ctypes.c_void_p()
    _ok(_lib.lmoe_create(ctypes.byref(h), ctypes.byref(cfg), ctypes.byref(weights), int(device)), "lmoe_create")
    return h.value


def lmoe_destroy(h: int) -> None:
    _ok(_lib.lmoe_destroy(h), "lmoe_destroy")


def lmoe_workspace_size(h: int, T: int) -> int:
    return _lib.lmoe_workspace_size(h, int(T))


def lmoe_host_staging_size(h: int, T: int) -> int:
    return _lib.lmoe_host_staging_size(h, int(T))


def lmoe_route(h, x, T, idx, w, logits, ws, stream) -> None:
    _ok(_lib.lmoe_route(h, x, int(T), idx, w, logits, ws, stream), "lmoe_route")


def lmoe_permute(h, idx, T, perm: LmoePerm, ws, stream) -> None:
    _ok(_lib.lmoe_permute(h, idx, int(T), ctypes.byref(perm), ws, stream), "lmoe_permute")


def lmoe_expert_forward(h, x, T, idx, w, perm: LmoePerm, Y, ws, stream) -> None:
    _ok(_lib.lmoe_expert_forward(h, x, int(T), idx, w, ctypes.byref(perm), Y, ws, stream), "lmoe_expert_forward")


def lmoe_combine(h, Y, idx, perm: LmoePerm, T, residual, y, stream) -> None:
    _ok(_lib.lmoe_combine(h, Y, idx, ctypes.byref(perm), int(T), residual, y, stream), "lmoe_combine")


def lmoe_layer_forward(h, x, T, residual, y, ws, stream) -> None:
    _ok(_lib.lmoe_layer_forward(h, x, int(T), residual, y, ws, stream), "lmoe_layer_forward")


def lmoe_layer_forward_noalloc(h, x, T, residual, y, stream) -> None:
    _ok(_lib.lmoe_layer_forward_noalloc(h, x, int(T), residual, y, stream), "lmoe_layer_forward_noalloc")


NOALLOC_MAX_T = 16
NOALLOC_SCRATCH_BYTES = 32 << 20


def lmoe_stack_forward(handles, x, T, y, ws, stream) -> None:
    arr = (ctypes.c_void_p * len(handles))(*handles)
    _ok(_lib.lmoe_stack_forward(arr, len(handles), x, int(T), y, ws, stream), "lmoe_stack_forward")


def lmoe_stack_workspace_size(h, T: int) -> int:
    return _lib.lmoe_stack_workspace_size(h, int(T))


def lmoe_layer_forward_host(h, x_host, T, residual_host, y_host, ws, stream) -> None:
    _ok(_lib.lmoe_layer_forward_host(h, x_host, int(T), residual_host, y_host, ws, stream), "lmoe_layer_forward_host")


def lmoe_check(h, stream) -> None:
    _ok(_lib.lmoe_check(h, stream), "lmoe_check")


def lmoe_check_status(h, stream) -> int:
    """lmoe_check's raw status (no exception)."""
    return _lib.lmoe_check(h, stream)


def lmoe_decode_routing(h, ws, T, idx, w, logits, stream) -> None:
    _ok(_lib.lmoe_decode_routing(h, ws, int(T), idx, w, logits, stream), "lmoe_decode_routing")


def lmoe_set_timeout(h, cycles: int) -> None:
    _ok(_lib.lmoe_set_timeout(h, int(cycles)), "lmoe_set_timeout")


def lmoe_set_stage_events(h, events_ptr, n: int) -> None:
    _ok(_lib.lmoe_set_stage_events(h, events_ptr, int(n)), "lmoe_set_stage_events")


def lmoe_launch_count(h, T: int) -> int:
    return int(_lib.lmoe_launch_count(h, int(T)))


def lmoe_stage_name(h, T: int, i: int):
    cnt = ctypes.c_int(0)
    name = _lib.lmoe_stage_name(h, int(T), int(i), ctypes.byref(cnt))
    return name.decode(), cnt.value


def lmoe_prefetch_experts(h, x, T, stream) -> None:
    _ok(_lib.lmoe_prefetch_experts(h, x, T, stream), "lmoe_prefetch_experts")


def lmoe_get_stage_stats(h) -> dict:
    st = LmoeStageStats()
    _ok(_lib.lmoe_get_stage_stats(h, ctypes.byref(st)), "lmoe_get_stage_stats")
    return {n: int(getattr(st, n)) for n, _ in LmoeStageStats._fields_}
