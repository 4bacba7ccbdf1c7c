"""GPU parity of the layer with NVFP4 weights (E2M1 codes, E4M3 scales per
16 elements, an fp32 scale per tensor) against the oracle, through the C ABI:
the single-kernel decode pass (one and two token tiles, the Edge0 shape at
8 tokens) and the prefill path (grouped GEMMs on fp16 copies of the weights)."""
import numpy as np
import pytest
import torch

import lmoe_synth as S
import oracle as O
from gpu_util import ambiguous_rows, bf16_bits, bf16_tensor, check_outputs, check_routing

pytestmark = pytest.mark.gpu

_cache = {}


def workload(name):
    if name not in _cache:
        sh, T, W, x = S.make_workload(name)
        y, idx, w, lg = O.layer_forward(O.Layer(sh, W), x)
        _cache[name] = (sh, T, W, x, y, idx, w, lg)
    return _cache[name]


def layer(sh, W, dev, path):
    from sparse_latent_moe_lmoe_b300 import LatentMoE
    return LatentMoE(sh, W, device=dev.index or 0, force_path=path)


def compare(name, sh, got, y_ref, lg_ref):
    tol = 1e-5 * np.abs(lg_ref).max(axis=1)
    keep = ~ambiguous_rows(lg_ref, sh.k, tol)
    mr, ma, _ = check_outputs(got[keep], y_ref[keep], name)
    print(f"{name}: mean rel {mr:.2e}, max abs {ma:.2e}, excluded {int((~keep).sum())} near-tie tokens")


@pytest.mark.parametrize("T", [1, 5, 8, 9, 16])
def test_nvfp4_decode_pass(T, cuda_device):
    from sparse_latent_moe_lmoe_b300 import capi
    sh, _, W, x, y_ref, idx_ref, w_ref, lg_ref = workload("small_t16_nvfp4")
    m = layer(sh, W, cuda_device, capi.PATH_DECODE)
    assert capi.lmoe_stage_name(m.h, T, 0)[0] == "decode_fused"
    got = bf16_bits(m.forward(bf16_tensor(x[:T], cuda_device)))
    torch.cuda.synchronize()
    m.check()
    compare(f"small nvfp4 decode T={T}", sh, got, y_ref[:T], lg_ref[:T])
    idx, w, lg = m.last_decode_routing(T)
    torch.cuda.synchronize()
    check_routing(lg.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy(), lg_ref[:T], idx_ref[:T], w_ref[:T], sh.k)


def test_nvfp4_decode_edge0_t8(cuda_device):
    from sparse_latent_moe_lmoe_b300 import capi
    sh, T, W, x, y_ref, idx_ref, w_ref, lg_ref = workload("decode_t8_nvfp4")
    m = layer(sh, W, cuda_device, capi.PATH_AUTO)
    got = bf16_bits(m.forward(bf16_tensor(x, cuda_device)))
    torch.cuda.synchronize()
    m.check()
    compare("decode_t8_nvfp4", sh, got, y_ref, lg_ref)


def test_nvfp4_prefill_path(cuda_device):
    from sparse_latent_moe_lmoe_b300 import capi
    sh, T, W, x, y_ref, idx_ref, w_ref, lg_ref = workload("small_t256_nvfp4")
    m = layer(sh, W, cuda_device, capi.PATH_PREFILL)
    got = bf16_bits(m.forward(bf16_tensor(x, cuda_device)))
    torch.cuda.synchronize()
    m.check()
    compare("small nvfp4 prefill T=256", sh, got, y_ref, lg_ref)


def test_nvfp4_decode_and_prefill_agree_with_int4_quantisation_gap(cuda_device):
    """The same draws in both formats: the two layers' GPU outputs differ by
    the quantisation gap only (a wrong nibble order or a missing tensor scale
    would make them unrelated)."""
    from sparse_latent_moe_lmoe_b300 import capi
    from dataclasses import replace
    sh, T, W, x, y_ref, idx_ref, w_ref, lg_ref = workload("small_t16_nvfp4")
    sh4 = replace(sh, wfmt="int4")
    W4 = S.make_layer(sh4, 0)
    m4 = layer(sh4, W4, cuda_device, capi.PATH_DECODE)
    mn = layer(sh, W, cuda_device, capi.PATH_DECODE)
    xt = bf16_tensor(x[:8], cuda_device)
    y4 = O.bf16_value(bf16_bits(m4.forward(xt)))
    yn = O.bf16_value(bf16_bits(mn.forward(xt)))
    torch.cuda.synchronize()
    corr = np.corrcoef(y4.ravel(), yn.ravel())[0, 1]
    assert corr > 0.9, corr


def test_nvfp4_per_step_decode_kernels_refuse(cuda_device):
    """The multi-kernel decode sequence reads int4 only: an NVFP4 handle that
    asks for it gets LMOE_ERR_UNSUPPORTED, not a wrong answer."""
    from sparse_latent_moe_lmoe_b300 import LatentMoE, LmoeError, capi
    sh, T, W, x, *_ = workload("small_t16_nvfp4")
    m = LatentMoE(sh, W, device=cuda_device.index or 0, force_path=capi.PATH_DECODE,
                  flags=capi.FLAG_MULTI_KERNEL_DECODE)
    with pytest.raises(LmoeError):
        m.forward(bf16_tensor(x[:4], cuda_device))


@pytest.mark.parametrize("T", [16, 256])
def test_nvfp4_with_lora(T, cuda_device):
    """NVFP4 weights together with a rank-64 Recover-LoRA branch (drawn large
    enough to matter at this shape): the single-kernel pass with the branch's
    kernels around it (T = 16) and the grouped GEMMs with the rank K blocks
    (T = 256), against the oracle"""
    from dataclasses import replace
    from sparse_latent_moe_lmoe_b300 import capi
    sh0, _, _, _ = S.make_workload("small_t16_nvfp4")
    sh = replace(sh0, lora_rank=64)
    W = S.make_layer(sh, 0)
    W["A_in"] = S.normal_bf16(7, S.S_AIN, (sh.G, sh.d, 64), 0.05)
    W["B_in"] = S.normal_bf16(7, S.S_BIN, (sh.G, 64, sh.L), 0.03)
    W["A_out"] = S.normal_bf16(7, S.S_AOUT, (sh.G, sh.L, 64), 0.05)
    W["B_out"] = S.normal_bf16(7, S.S_BOUT, (sh.G, 64, sh.d), 0.03)
    x = S.make_x(T, sh.d, 8)
    y_ref, idx_ref, w_ref, lg_ref = O.layer_forward(O.Layer(sh, W), x)
    W0 = dict(W)
    W0["B_in"] = np.zeros_like(W["B_in"])
    W0["B_out"] = np.zeros_like(W["B_out"])
    y0 = O.layer_forward(O.Layer(sh, W0), x)[0]
    assert np.abs(y0 - y_ref).sum() / np.abs(y_ref).sum() > 30e-3  # the branch moves the output
    m = layer(sh, W, cuda_device, capi.PATH_AUTO)
    expect = "lora_p" if T > 16 else None
    names = [capi.lmoe_stage_name(m.h, T, i)[0] for i in range(capi.lmoe_stage_name(m.h, T, 0)[1])]
    assert (expect in names) if expect else ("decode_fused" in names)
    got = bf16_bits(m.forward(bf16_tensor(x, cuda_device)))
    torch.cuda.synchronize()
    m.check()
    compare(f"NVFP4 + LoRA, T={T}", sh, got, y_ref, lg_ref)
