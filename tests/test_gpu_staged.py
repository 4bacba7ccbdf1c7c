"""Staged experts (LMOE_FLAG_STAGED_EXPERTS): the per-expert weights live in
page-locked host memory and a fixed number of GPU slots; a decode pass
stages its routed experts, the prerouter stages a predicted set ahead. The
output must be bit for bit that of an unstaged handle of the same weights,
whatever the slots held before, and the counters must add up."""
import numpy as np
import pytest
import torch

import lmoe_synth as S
from gpu_util import bf16_bits, bf16_tensor

pytestmark = pytest.mark.gpu

# 256 experts in 4 groups, top-4: 64 slots hold at most a quarter of them
SHAPE = S.LayerShape(d=1024, E=256, G=4, k=4, L=256, f=256)
SLOTS = 64


def handles(cuda_device, seed=5, slots=SLOTS, shape=SHAPE):
    from sparse_latent_moe_lmoe_b300 import LatentMoE, capi
    W = S.make_layer(shape, seed)
    plain = LatentMoE(shape, W, device=cuda_device.index or 0)
    staged = LatentMoE(shape, W, device=cuda_device.index or 0, flags=capi.FLAG_STAGED_EXPERTS, expert_slots=slots,
                       expert_weights_on_host=True)
    return plain, staged


def test_staged_pass_equals_unstaged_through_evictions(cuda_device):
    from sparse_latent_moe_lmoe_b300 import capi
    plain, staged = handles(cuda_device)
    assert [capi.lmoe_stage_name(staged.h, 8, i)[0] for i in range(4)] == ["route", "stage_plan", "stage_copy",
                                                                          "decode_fused"]
    routed = 0
    for step, T in enumerate([8, 16, 1, 8, 16, 3, 16, 8]):  # distinct inputs: the slots keep turning over
        x = bf16_tensor(S.make_x(T, SHAPE.d, 300 + step), cuda_device)
        a = bf16_bits(plain.forward(x))
        b = bf16_bits(staged.forward(x))
        torch.cuda.synchronize()
        assert np.array_equal(a, b), f"step {step}"
        idx, _, _ = staged.last_decode_routing(T)
        routed += len(np.unique(idx.cpu().numpy()))
    staged.check()
    st = staged.stage_stats()
    assert st["passes"] == 8 and st["routed"] == routed
    assert st["hits"] + st["staged_on_demand"] == st["routed"]
    assert st["staged_on_demand"] > SLOTS  # more experts than slots went through them
    assert st["bytes_copied"] == st["staged_on_demand"] * (SHAPE.f // 32) * 3 * 18 * SHAPE.L


def test_repeat_hits_and_prefetch(cuda_device):
    plain, staged = handles(cuda_device, seed=6)
    x = bf16_tensor(S.make_x(16, SHAPE.d, 400), cuda_device)
    staged.forward(x)
    s1 = staged.stage_stats()
    staged.forward(x)  # the same tokens: every routed expert already holds a slot
    s2 = staged.stage_stats()
    assert s2["staged_on_demand"] == s1["staged_on_demand"] and s2["hits"] - s1["hits"] == s2["routed"] - s1["routed"]
    # the prerouter on new tokens, then the pass on the same tokens: no copies left for the pass
    x2 = bf16_tensor(S.make_x(16, SHAPE.d, 401), cuda_device)
    staged.prefetch_experts(x2)
    s3 = staged.stage_stats()
    assert s3["prefetched"] > s2["prefetched"]
    y = bf16_bits(staged.forward(x2))
    s4 = staged.stage_stats()
    assert s4["staged_on_demand"] == s3["staged_on_demand"]
    assert np.array_equal(y, bf16_bits(plain.forward(x2)))
    staged.check()


@pytest.mark.parametrize("T", [1, 8])
def test_staged_stack_with_prerouter_equals_unstaged_stack(T, cuda_device):
    from sparse_latent_moe_lmoe_b300 import LatentMoE, LatentMoEStack, capi
    n = 3
    plain, staged = [], []
    for l in range(n):
        W = S.make_layer(SHAPE, 700 + l)
        plain.append(LatentMoE(SHAPE, W, device=cuda_device.index or 0))
        staged.append(LatentMoE(SHAPE, W, device=cuda_device.index or 0, flags=capi.FLAG_STAGED_EXPERTS,
                                expert_slots=SLOTS, expert_weights_on_host=True))
    sp, ss = LatentMoEStack(plain), LatentMoEStack(staged)
    for step in range(3):
        x = bf16_tensor(S.make_x(T, SHAPE.d, 900 + step), cuda_device)
        a = bf16_bits(sp.forward(x))
        b = bf16_bits(ss.forward(x))
        torch.cuda.synchronize()
        assert np.array_equal(a, b), f"step {step}"
    for m in staged:
        m.check()
    # layers after the first were prefetched by the prerouter (its prediction:
    # the layer's own router on the previous layer's input)
    st = [m.stage_stats() for m in staged]
    assert st[0]["prefetched"] == 0 and all(s["prefetched"] > 0 for s in st[1:])
    assert all(s["hits"] + s["staged_on_demand"] == s["routed"] for s in st)
