"""lmoe_layer_forward_noalloc (the fixed-scratch decode entry point) against
lmoe_layer_forward (the workspace entry point), through the C ABI, on two
calls in a row. Collected last on purpose: it must pass both in a fresh
process, where its first call looks up the scratch array, and after every
other test has used the library."""
import ctypes

import numpy as np
import pytest
import torch

import lmoe_synth as S
from gpu_util import MAX_ABS, MEAN_REL, bf16_bits, bf16_tensor

pytestmark = pytest.mark.gpu


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _close(a_bits, b_bits):
    a, b = S.bf16_bits_to_f32(a_bits).astype(np.float64), S.bf16_bits_to_f32(b_bits).astype(np.float64)
    mean_rel = np.abs(a - b).sum() / max(np.abs(b).sum(), 1e-300)
    assert mean_rel <= MEAN_REL, mean_rel
    assert np.abs(a - b).max() <= MAX_ABS


@pytest.mark.parametrize("workload,with_residual", [("decode_t8", False), ("decode_t8", True), ("tiny_t64", False),
                                                    ("lora_t16", False)])
def test_noalloc_matches_workspace_entry_point(cuda_device, workload, with_residual):
    """Both entry points run the same decode kernels on the same inputs, and
    those kernels are deterministic: the outputs must agree bit for bit (the
    tolerance check is kept as a second, weaker statement). lora_t16 takes the
    multi-kernel sequence, whose LoRA projections use their own regions of the
    scratch. The second call must not change the device's free memory."""
    from sparse_latent_moe_lmoe_b300 import LatentMoE, capi
    sh, T, W, x = S.make_workload(workload)
    T = min(T, capi.NOALLOC_MAX_T)
    x = x[:T]
    m = LatentMoE(sh, W, device=0)
    xt = bf16_tensor(x, cuda_device)
    res = bf16_tensor(S.make_x(T, sh.d, 77), cuda_device) if with_residual else None
    y_ref = bf16_bits(m.forward(xt, residual=res))
    m.check()
    ys = [torch.empty((T, sh.d), dtype=torch.bfloat16, device=cuda_device) for _ in range(2)]
    outs = []
    for i in range(2):
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        capi.lmoe_layer_forward_noalloc(m.h, _p(xt), T, _p(res), _p(ys[i]), _stream())
        m.check()
        free1 = torch.cuda.mem_get_info()[0]
        if i == 1:
            assert free1 == free0, f"free device memory changed by {free0 - free1} bytes"
        outs.append(bf16_bits(ys[i]))
    for o in outs:
        assert np.array_equal(o, y_ref), "no-alloc result differs from the workspace entry point"
        _close(o, y_ref)
    assert np.array_equal(outs[1], outs[0])
    m.close()


def test_noalloc_rejects_batches_beyond_its_maximum(cuda_device):
    from sparse_latent_moe_lmoe_b300 import LatentMoE, capi
    sh, _, W, x = S.make_workload("tiny_t64")
    m = LatentMoE(sh, W, device=0)
    T = capi.NOALLOC_MAX_T + 1
    xt = bf16_tensor(x[:T], cuda_device)
    y = torch.empty((T, sh.d), dtype=torch.bfloat16, device=cuda_device)
    lib = capi.library()
    st = lib.lmoe_layer_forward_noalloc(m.h, _p(xt), T, None, _p(y), _stream())
    assert st == 1  # LMOE_ERR_INVALID_ARG
    assert lib.lmoe_layer_forward_noalloc(m.h, _p(xt), 0, None, _p(y), _stream()) == 0
    m.check()
    m.close()
