"""Top-k selection on exact ties, through the prefill path's router and its
threshold selection (topk.cuh): router rows that are equal give exactly
equal logits on both sides, and the picks must follow the definition --
descending logit, ties to the lower expert index -- also when more than 32
logits tie at the top, where the selection falls back to its round-based
form."""
import numpy as np
import pytest

import lmoe_synth as S
import oracle as O
from gpu_util import bf16_tensor

pytestmark = pytest.mark.gpu

SHAPE = S.LayerShape(d=256, E=64, G=4, k=10, L=256, f=128)


def tied_router(scale_of_expert: np.ndarray) -> dict:
    """A layer whose router row e is scale_of_expert[e] times one shared row
    (small integer scales, so the rows are exact in fp32)."""
    W = S.make_layer(SHAPE, 21)
    base = S.normal_f32(22, 0, (SHAPE.d,), 0.02)
    W["W_r"] = np.ascontiguousarray((scale_of_expert[:, None] * base[None, :]).astype(np.float32))
    return W


def run(W, device, T=64):
    from sparse_latent_moe_lmoe_b300 import LatentMoE, capi
    x = S.make_x(T, SHAPE.d, 23)
    m = LatentMoE(SHAPE, W, device=0, force_path=capi.PATH_PREFILL)
    idx, w, _ = m.route(bf16_tensor(x, device), want_logits=True)
    m.check()
    idx_ref, w_ref = O.topk(O.router_logits(O.Layer(SHAPE, W), x), SHAPE.k)
    return idx.cpu().numpy(), w.cpu().numpy(), idx_ref, w_ref


def test_ties_across_the_kth_place(cuda_device):
    # eight groups of eight equal experts, interleaved over the index range:
    # the top 10 is one whole group and the two lowest indices of the next
    scale = 1.0 + (np.arange(SHAPE.E) % 8).astype(np.float32)
    idx, w, idx_ref, w_ref = run(tied_router(scale), cuda_device)
    assert (idx == idx_ref).all(), np.nonzero((idx != idx_ref).any(1))[0][:5]
    assert np.allclose(w, w_ref, rtol=1e-5, atol=1e-7)


def test_more_than_32_tied_at_the_top(cuda_device):
    # 40 experts share the larger scale: for tokens whose shared dot product
    # is positive all 40 tie at the top (more than the 32 candidates the
    # threshold selection gathers); for the others the 24 remaining ones do
    scale = np.ones(SHAPE.E, np.float32)
    top = np.sort(np.random.default_rng(24).permutation(SHAPE.E)[:40])
    scale[top] = 2.0
    idx, w, idx_ref, w_ref = run(tied_router(scale), cuda_device)
    assert (idx == idx_ref).all(), np.nonzero((idx != idx_ref).any(1))[0][:5]
    assert np.allclose(w, w_ref, rtol=1e-5, atol=1e-7)


# ---------------------------------------------------------------- decode path
# The same two tie patterns through the decode path's two selectors: the
# router kernel of the multi-kernel sequence (lmoe_route at T <= 16), and the
# routing warps inside the single persistent decode kernel, read back from its
# workspace after lmoe_layer_forward. The latter needs a shape the single
# kernel takes (d a multiple of 1024, L and f multiples of 256).
FUSED = S.LayerShape(d=1024, E=64, G=4, k=10, L=256, f=256)


def tied_router_for(shape, scale_of_expert: np.ndarray) -> dict:
    W = S.make_layer(shape, 31)
    base = S.normal_f32(32, 0, (shape.d,), 0.02)
    W["W_r"] = np.ascontiguousarray((scale_of_expert[:, None] * base[None, :]).astype(np.float32))
    return W


def run_decode(shape, W, device, fused: bool, T=16):
    from sparse_latent_moe_lmoe_b300 import LatentMoE, capi
    x = S.make_x(T, shape.d, 33)
    flags = 0 if fused else capi.FLAG_MULTI_KERNEL_DECODE
    m = LatentMoE(shape, W, device=0, force_path=capi.PATH_DECODE, flags=flags)
    xt = bf16_tensor(x, device)
    if fused:
        assert capi.lmoe_stage_name(m.h, T, 0)[0] == "decode_fused"
        m.forward(xt)
        idx, w, _ = m.last_decode_routing(T)
    else:
        idx, w, _ = m.route(xt, want_logits=True)
    m.check()
    idx_ref, w_ref = O.topk(O.router_logits(O.Layer(shape, W), x), shape.k)
    return idx.cpu().numpy(), w.cpu().numpy(), idx_ref, w_ref


def kth_place_scale(E):
    return 1.0 + (np.arange(E) % 8).astype(np.float32)


def many_tied_scale(E, seed=24):
    scale = np.ones(E, np.float32)
    top = np.sort(np.random.default_rng(seed).permutation(E)[:40])
    scale[top] = 2.0
    return scale


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("pattern", ["kth_place", "more_than_32"])
def test_decode_ties(pattern, fused, cuda_device):
    shape = FUSED if fused else SHAPE
    scale = kth_place_scale(shape.E) if pattern == "kth_place" else many_tied_scale(shape.E)
    idx, w, idx_ref, w_ref = run_decode(shape, tied_router_for(shape, scale), cuda_device, fused)
    assert (idx == idx_ref).all(), np.nonzero((idx != idx_ref).any(1))[0][:5]
    assert np.allclose(w, w_ref, rtol=1e-5, atol=1e-7)
