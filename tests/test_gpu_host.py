"""The host-buffer entry point (lmoe_layer_forward_host) against the device
entry point on the same inputs: bit-identical outputs. The handle keeps a
repeated call as a CUDA graph, so the checks cover the first (captured) call,
replays with new contents in the same pinned buffers, a change of buffers (a
new capture), a residual, a timeout change (which drops the graph), and the
prefill path; every result is also checked against the oracle once."""
from dataclasses import replace

import numpy as np
import pytest
import torch

import lmoe_synth as S
import oracle as O
from gpu_util import bf16_bits, bf16_tensor, check_outputs

pytestmark = pytest.mark.gpu


def pinned(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).pin_memory()


def host_bits(t):
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def test_host_call_replays_bit_identical(cuda_device):
    from sparse_latent_moe_lmoe_b300 import LatentMoE, capi
    sh, T, W, x = S.make_workload("decode_t8")
    m = LatentMoE(sh, W, device=0)
    xs = [x, S.make_x(T, sh.d, 71), S.make_x(T, sh.d, 72)]
    xh = pinned(xs[0])
    yh = torch.empty_like(xh).pin_memory()
    for i, xi in enumerate(xs):  # the same pinned buffers, new contents each call
        xh.copy_(pinned(xi))
        m.forward_host(xh, yh)
        y_dev = bf16_bits(m.forward(bf16_tensor(xi, cuda_device)))
        torch.cuda.synchronize()
        m.check()
        assert np.array_equal(host_bits(yh), y_dev), f"call {i}"
        if i == 0:  # the oracle once, on the workload's own input
            check_outputs(host_bits(yh), O.layer_forward(O.Layer(sh, W), xi)[0], "host call")
    # other buffers (captured anew) with a residual, then a timeout change
    res = S.make_x(T, sh.d, 73)
    xh2, rh2, yh2 = pinned(xs[1]), pinned(res), torch.empty_like(xh).pin_memory()
    m.forward_host(xh2, yh2, residual_host=rh2)
    y_dev = bf16_bits(m.forward(bf16_tensor(xs[1], cuda_device), residual=bf16_tensor(res, cuda_device)))
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(yh2), y_dev)
    capi.lmoe_set_timeout(m.h, 1 << 30)
    m.forward_host(xh2, yh2, residual_host=rh2)
    m.check()
    assert np.array_equal(host_bits(yh2), y_dev)


def test_host_call_prefill_path(cuda_device):
    from sparse_latent_moe_lmoe_b300 import LatentMoE, capi
    sh = S.LayerShape(d=256, E=64, G=4, k=4, L=256, f=128)
    W = S.make_layer(sh, 81)
    T = 300
    x = S.make_x(T, sh.d, 82)
    m = LatentMoE(sh, W, device=0, force_path=capi.PATH_PREFILL)
    xh = pinned(x)
    yh = torch.empty_like(xh).pin_memory()
    for _ in range(2):
        m.forward_host(xh, yh)
    y_dev = bf16_bits(m.forward(bf16_tensor(x, cuda_device)))
    torch.cuda.synchronize()
    m.check()
    assert np.array_equal(host_bits(yh), y_dev)


@pytest.mark.parametrize("name,T", [("small", 9000), ("prefill_t16384_zipf", 16384)])
def test_host_call_chunked_prefill(name, T, cuda_device):
    """Prefill-sized host calls run as a pipeline of 4096-token chunks (one
    dequantisation, copies overlapping the compute of neighbouring chunks):
    bit-identical to one device call on all T tokens (every step of the layer
    is per token), with a ragged last chunk and a residual."""
    from sparse_latent_moe_lmoe_b300 import LatentMoE, capi
    if name == "small":
        sh = S.LayerShape(d=256, E=64, G=4, k=4, L=256, f=128)
        W = S.make_layer(sh, 91)
        x = S.make_x(T, sh.d, 92)
    else:
        sh, T, W, x = S.make_workload(name)
    res = S.make_x(T, sh.d, 93)
    m = LatentMoE(sh, W, device=0)
    xh, rh = pinned(x), pinned(res)
    yh = torch.empty_like(xh).pin_memory()
    for _ in range(2):  # captured, then replayed
        m.forward_host(xh, yh, residual_host=rh)
    y_dev = bf16_bits(m.forward(bf16_tensor(x, cuda_device), residual=bf16_tensor(res, cuda_device)))
    torch.cuda.synchronize()
    m.check()
    assert np.array_equal(host_bits(yh), y_dev)


def test_host_call_lora_decode(cuda_device):
    """The LoRA decode sequence (its kernels chained by programmatic dependent
    launch) inside the host call's graph: bit-identical to the device call"""
    from sparse_latent_moe_lmoe_b300 import LatentMoE
    sh, T, W, x = S.make_workload("lora_t16")
    m = LatentMoE(sh, W, device=0)
    xh = pinned(x)
    yh = torch.empty_like(xh).pin_memory()
    for _ in range(3):
        m.forward_host(xh, yh)
    y_dev = bf16_bits(m.forward(bf16_tensor(x, cuda_device)))
    torch.cuda.synchronize()
    m.check()
    assert np.array_equal(host_bits(yh), y_dev)
