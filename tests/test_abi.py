"""The C ABI library without a GPU: it loads, exports every entry point the
header declares, and rejects bad arguments on the host before touching CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    src = open(os.path.join(ROOT, "include", "lmoe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(lmoe_[a-z_]+)\s*\(", src)))


def test_library_exports_every_declared_function():
    from sparse_latent_moe_lmoe_b300 import capi
    lib = ctypes.CDLL(capi.LIB_PATH)
    names = header_functions()
    assert len(names) >= 16
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(capi.EXPORTS)


def test_host_side_validation_without_gpu():
    from sparse_latent_moe_lmoe_b300 import capi
    lib = capi.library()
    assert capi.lmoe_version() == 101
    assert lib.lmoe_workspace_size(None, 8) == 0
    assert lib.lmoe_route(None, None, 8, None, None, None, None, None) == 1
    assert lib.lmoe_layer_forward(None, None, 8, None, None, None, None) == 1
    assert lib.lmoe_layer_forward_noalloc(None, None, 8, None, None, None) == 1
    assert lib.lmoe_set_timeout(None, 5) == 1
    assert lib.lmoe_decode_routing(None, None, 8, None, None, None, None) == 1
    assert lib.lmoe_check(None, None) == 1
    assert lib.lmoe_destroy(None) == 0
    h = ctypes.c_void_p()
    cfg = capi.LmoeConfig(256, 16, 2, 2, 64, 32, 16, 0, 0, 0, 0, 0, 0)  # qgroup 16: unsupported
    w = capi.LmoeWeights()
    assert lib.lmoe_create(ctypes.byref(h), ctypes.byref(cfg), ctypes.byref(w), 0) == 2
    cfg.qgroup = 32
    cfg.G = 3  # E % G != 0
    assert lib.lmoe_create(ctypes.byref(h), ctypes.byref(cfg), ctypes.byref(w), 0) == 1
    cfg.G = 2
    assert lib.lmoe_create(ctypes.byref(h), ctypes.byref(cfg), ctypes.byref(w), 0) == 1  # null weights
    cfg.weight_format = 2  # no such format
    assert lib.lmoe_create(ctypes.byref(h), ctypes.byref(cfg), ctypes.byref(w), 0) == 1
    cfg.weight_format = capi.WEIGHTS_NVFP4  # NVFP4 scales come per 16 elements
    assert lib.lmoe_create(ctypes.byref(h), ctypes.byref(cfg), ctypes.byref(w), 0) == 2
    cfg.qgroup = 16
    assert lib.lmoe_create(ctypes.byref(h), ctypes.byref(cfg), ctypes.byref(w), 0) == 1  # null weights
    assert h.value is None
    # staged experts: the slot count must hold a 16-token pass's experts and fit the layer
    cfg.flags = capi.FLAG_STAGED_EXPERTS
    cfg.expert_slots = 0
    assert lib.lmoe_create(ctypes.byref(h), ctypes.byref(cfg), ctypes.byref(w), 0) == 1
    cfg.expert_slots = cfg.E + 1
    assert lib.lmoe_create(ctypes.byref(h), ctypes.byref(cfg), ctypes.byref(w), 0) == 1
    cfg.flags = 8  # no such flag
    cfg.expert_slots = 0
    assert lib.lmoe_create(ctypes.byref(h), ctypes.byref(cfg), ctypes.byref(w), 0) == 2
    assert h.value is None
    assert lib.lmoe_prefetch_experts(None, None, 8, None) == 1
    st = capi.LmoeStageStats()
    assert lib.lmoe_get_stage_stats(None, ctypes.byref(st)) == 1
    for s in range(8):
        assert capi.lmoe_status_string(s)
    name, count = capi.lmoe_stage_name(None, 8, 0)
    assert name == "" and count == 0
    assert capi.lmoe_launch_count(None, 8) == 0


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    """The package has no fallback: a missing library is an ImportError."""
    import importlib
    import sparse_latent_moe_lmoe_b300.capi as capi
    monkeypatch.setattr(capi, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        capi._load()


def test_kblock_reciprocal_is_exact():
    """The W_out GEMM splits K blocks into (group, block) with a multiply-high
    reciprocal, kb / D = (kb * ceil(2^32 / D)) >> 32; exact for kb < 2^32 / D.
    Checked here for every divisor the prefill path can meet (L + rp over 64,
    4..66) and every K block a tile can have (<= 32 groups x D)."""
    for D in range(4, 67):
        m = ((1 << 32) + D - 1) // D
        assert m < (1 << 32)
        for kb in range(0, 32 * D + 64):
            assert (kb * m) >> 32 == kb // D, (D, kb)
