"""GPU parity of the decode path (<= 16 tokens per pass) against the oracle,
through the C ABI. Workloads: the tiny layer (64 tokens, run as four
passes), the Edge0-shaped layer at 8 tokens, and the same layer with the
Recover-LoRA branch at 16 tokens."""
import numpy as np
import pytest
import torch

import lmoe_synth as S
import oracle as O
from gpu_util import (W_RTOL, ambiguous_rows, bf16_bits, bf16_tensor, check_outputs, check_routing, check_rows)

pytestmark = pytest.mark.gpu

_cache = {}


def workload(name):
    if name not in _cache:
        sh, T, W, x = S.make_workload(name)
        Ly = O.Layer(sh, W)
        y, idx, w, lg = O.layer_forward(Ly, x)
        _cache[name] = (sh, T, W, x, Ly, y, idx, w, lg)
    return _cache[name]


def make_layer(sh, W, dev, path=1):
    from sparse_latent_moe_lmoe_b300 import LatentMoE
    return LatentMoE(sh, W, device=dev.index or 0, force_path=path)


@pytest.mark.parametrize("name", ["tiny_t64", "decode_t8", "lora_t16"])
def test_route_parity(name, cuda_device):
    sh, T, W, x, Ly, y, idx_ref, w_ref, lg_ref = workload(name)
    m = make_layer(sh, W, cuda_device)
    xt = bf16_tensor(x, cuda_device)
    idx, w, lg = m.route(xt, want_logits=True)
    torch.cuda.synchronize()
    keep = check_routing(lg.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy(), lg_ref, idx_ref, w_ref, sh.k)
    assert keep.mean() > 0.95
    m.check()


@pytest.mark.parametrize("name", ["tiny_t64", "decode_t8", "lora_t16"])
def test_layer_forward_parity(name, cuda_device):
    sh, T, W, x, Ly, y_ref, idx_ref, w_ref, lg_ref = workload(name)
    m = make_layer(sh, W, cuda_device)
    xt = bf16_tensor(x, cuda_device)
    yt = m.forward(xt)
    torch.cuda.synchronize()
    m.check()
    tol = 1e-5 * np.abs(lg_ref).max(axis=1)
    from gpu_util import ambiguous_rows
    keep = ~ambiguous_rows(lg_ref, sh.k, tol)
    got = bf16_bits(yt)
    mr, ma, _ = check_outputs(got[keep], y_ref[keep], name)
    print(f"{name}: mean rel {mr:.2e}, max abs {ma:.2e}, excluded {int((~keep).sum())} near-tie tokens")


def test_layer_forward_residual_and_repeat(cuda_device):
    """residual add, and two calls in a row give bit-identical results"""
    sh, T, W, x, Ly, y_ref, idx_ref, w_ref, lg_ref = workload("decode_t8")
    m = make_layer(sh, W, cuda_device)
    xt = bf16_tensor(x, cuda_device)
    res_bits = S.make_x(T, sh.d, 7)
    res = bf16_tensor(res_bits, cuda_device)
    y1 = bf16_bits(m.forward(xt, residual=res))
    y2 = bf16_bits(m.forward(xt, residual=res))
    m.check()
    assert np.array_equal(y1, y2)
    ref = O.bf16_value(res_bits) + O.bf16_value(O.bf16_round(y_ref))
    check_outputs(y1, ref, "residual")


@pytest.mark.parametrize("T", [1, 3, 9, 16])
def test_layer_forward_ragged_T(T, cuda_device):
    sh, _, W, x, Ly, y_ref, idx_ref, w_ref, lg_ref = workload("lora_t16")
    m = make_layer(sh, W, cuda_device)
    xt = bf16_tensor(x[:T], cuda_device)
    got = bf16_bits(m.forward(xt))
    m.check()
    check_outputs(got, y_ref[:T], f"T={T}")


@pytest.mark.parametrize("T,E,G,k,skew", [(1, 16, 2, 2, 0.0), (16, 512, 8, 10, 0.0), (64, 16, 2, 2, 0.0),
                                          (1000, 512, 8, 10, 1.1), (16384, 512, 8, 10, 1.1)])
def test_permute_bit_exact(T, E, G, k, skew, cuda_device):
    sh = S.LayerShape(d=256, E=E, G=G, k=k, L=64, f=32)
    W = S.make_layer(sh, 0)
    m = make_layer(sh, W, cuda_device)
    idx, _ = S.routing(100 + T, T, E, k, skew)
    ref = O.permute(idx, E, G)
    perm = m.permute(torch.from_numpy(idx).to(cuda_device))
    torch.cuda.synchronize()
    m.check()
    for n in ("expert_offsets", "sorted_assign", "inv", "group_offsets", "group_tok_offsets", "assign_row"):
        got = perm[n].cpu().numpy()[:ref[n].size]
        assert np.array_equal(got, ref[n]), n
    rows = ref["rows"]
    assert np.array_equal(perm["group_tokens"].cpu().numpy()[:rows], ref["group_tokens"])


@pytest.mark.parametrize("name,T", [("tiny_t64", 64), ("decode_t8", 8), ("lora_t16", 16)])
def test_expert_forward_and_combine(name, T, cuda_device):
    """lmoe_expert_forward and lmoe_combine with a synthetic routing table:
    every Y row against the oracle's (group, token) row, then the combine
    against the oracle's combine of the GPU's own Y rows."""
    sh, _, W, x, Ly, *_ = workload(name)
    m = make_layer(sh, W, cuda_device)
    idx, w = S.routing(5, T, sh.E, sh.k)
    ref_perm = O.permute(idx, sh.E, sh.G)
    dev = cuda_device
    idx_t, w_t = torch.from_numpy(idx).to(dev), torch.from_numpy(w).to(dev)
    perm = m.permute(idx_t)
    xt = bf16_tensor(x[:T], dev)
    Y = m.expert_forward(xt, idx_t, w_t, perm)
    torch.cuda.synchronize()
    m.check()
    Yn = Y.cpu().numpy()
    rows = ref_perm["rows"]
    gto = ref_perm["group_tok_offsets"]
    ref_rows = np.zeros((rows, sh.d))
    for g in range(sh.G):
        for r in range(gto[g], gto[g + 1]):
            t = ref_perm["group_tokens"][r]
            ref_rows[r] = O.group_row(Ly, g, x[t], idx[t], w[t].astype(np.float64))
    err = np.abs(Yn[:rows] - ref_rows).sum() / np.abs(ref_rows).sum()
    assert err < 1e-3, err
    worst = check_rows(Yn[:rows], ref_rows, f"{name} Y rows")
    print(f"{name}: Y rows mean rel {err:.2e}, worst row max-abs / row scale {worst:.2e}")
    y = m.combine(Y, idx_t, perm, T)
    torch.cuda.synchronize()
    y_ref = O.combine(Yn[:max(rows, 1)], idx, ref_perm["assign_row"], sh.E, sh.G)
    check_outputs(bf16_bits(y), y_ref, "combine")


def test_t_zero_is_noop(cuda_device):
    sh, T, W, x, *_ = workload("tiny_t64")
    m = make_layer(sh, W, cuda_device)
    xt = bf16_tensor(x[:1], cuda_device)
    from sparse_latent_moe_lmoe_b300 import capi
    import ctypes
    y = torch.empty_like(xt)
    capi.lmoe_layer_forward(m.h, ctypes.c_void_p(xt.data_ptr()), 0, None, ctypes.c_void_p(y.data_ptr()),
                            ctypes.c_void_p(m.workspace(1).data_ptr()), None)
    m.check()


def test_misaligned_and_bad_args_rejected(cuda_device):
    from sparse_latent_moe_lmoe_b300 import capi
    import ctypes
    sh, T, W, x, *_ = workload("tiny_t64")
    m = make_layer(sh, W, cuda_device)
    xt = bf16_tensor(x, cuda_device)
    ws = m.workspace(T)
    y = torch.empty_like(xt)
    P = ctypes.c_void_p
    with pytest.raises(capi.LmoeError) as e:
        capi.lmoe_layer_forward(m.h, P(xt.data_ptr() + 2), T, None, P(y.data_ptr()), P(ws.data_ptr()), None)
    assert e.value.status == 3
    with pytest.raises(capi.LmoeError) as e:
        capi.lmoe_layer_forward(m.h, P(xt.data_ptr()), -1, None, P(y.data_ptr()), P(ws.data_ptr()), None)
    assert e.value.status == 1
    with pytest.raises(capi.LmoeError) as e:
        capi.lmoe_layer_forward(m.h, P(xt.data_ptr()), T, None, P(xt.data_ptr()), P(ws.data_ptr()), None)
    assert e.value.status == 1
    # out-of-range expert indices are caught on the device
    idx = torch.full((4, sh.k), sh.E + 3, dtype=torch.int32, device=cuda_device)
    m.permute(idx)
    with pytest.raises(capi.LmoeError) as e:
        m.check()
    assert e.value.status == 6


@pytest.mark.parametrize("name", ["tiny_t64", "decode_t8"])
def test_multi_kernel_decode_matches_oracle(name, cuda_device):
    """The per-step kernel sequence (flag) against the oracle, and against
    the single persistent kernel: both deterministic, both within the bar."""
    from sparse_latent_moe_lmoe_b300 import LatentMoE, capi
    sh, T, W, x, Ly, y_ref, idx_ref, w_ref, lg_ref = workload(name)
    xt = bf16_tensor(x, cuda_device)
    multi = LatentMoE(sh, W, device=0, flags=capi.FLAG_MULTI_KERNEL_DECODE)
    fused = LatentMoE(sh, W, device=0)
    if name == "decode_t8":  # the tiny shapes take the per-step kernels either way
        assert capi.lmoe_stage_name(fused.h, T, 0)[0] == "decode_fused"
    assert capi.lmoe_stage_name(multi.h, T, 0)[0] == "route"
    y_m = bf16_bits(multi.forward(xt))
    y_f = bf16_bits(fused.forward(xt))
    y_f2 = bf16_bits(fused.forward(xt))
    multi.check()
    fused.check()
    assert np.array_equal(y_f, y_f2)
    from gpu_util import ambiguous_rows
    keep = ~ambiguous_rows(lg_ref, sh.k, 1e-5 * np.abs(lg_ref).max(axis=1))
    check_outputs(y_m[keep], y_ref[keep], name + " multi-kernel")
    check_outputs(y_f[keep], y_ref[keep], name + " fused")


def test_fused_timeout_path_reports_and_recovers(cuda_device):
    """A one-cycle wait budget makes every grid-barrier wait run out: the
    call finishes, lmoe_check reports LMOE_ERR_TIMEOUT, and with the budget
    restored the next call is correct again (no GPU fault, no hang)."""
    from sparse_latent_moe_lmoe_b300 import LatentMoE, capi
    sh, T, W, x, Ly, y_ref, idx_ref, w_ref, lg_ref = workload("decode_t8")
    m = LatentMoE(sh, W, device=0)
    xt = bf16_tensor(x, cuda_device)
    capi.lmoe_set_timeout(m.h, 1)
    m.forward(xt)
    torch.cuda.synchronize()
    status = capi.lmoe_check_status(m.h, None)
    assert status == 5
    capi.lmoe_set_timeout(m.h, 0)
    y = bf16_bits(m.forward(xt))
    m.check()
    check_outputs(y, y_ref, "after timeout")


@pytest.mark.parametrize("T", [1, 3, 9, 16])
def test_fused_decode_ragged_T(T, cuda_device):
    """The single persistent kernel at token counts that leave ragged token
    tiles (one and two 8-token tiles), against the oracle."""
    from sparse_latent_moe_lmoe_b300 import LatentMoE, capi
    sh, _, W, _x, Ly, _y, _i, _w, _l = workload("decode_t8")
    x = S.make_x(T, sh.d, 40 + T)
    y_ref, idx_ref, w_ref, lg_ref = O.layer_forward(Ly, x)
    m = LatentMoE(sh, W, device=0)
    assert capi.lmoe_stage_name(m.h, T, 0)[0] == "decode_fused"
    xt = bf16_tensor(x, cuda_device)
    idx, w, lg = m.route(xt, want_logits=True)
    got = bf16_bits(m.forward(xt))
    m.check()
    from gpu_util import ambiguous_rows
    keep = ~ambiguous_rows(lg_ref, sh.k, 1e-5 * np.abs(lg_ref).max(axis=1))
    mr, ma, _ = check_outputs(got[keep], y_ref[keep], f"fused T={T}")
    print(f"fused T={T}: mean rel {mr:.2e} max abs {ma:.2e}")


def check_routing_exact(idx_g, w_g, lg_g, lg_ref, k):
    """The routing a pass used against the oracle: logits within the logit bar
    of the oracle's, and the selection equal to the oracle's top-k run on the
    GPU's own fp32 logits -- indices bit for bit (ties included, since both
    sides order the same fp32 values), weights within the weight bar."""
    tol = 1e-5 * np.abs(lg_ref).max(axis=1)
    err = np.abs(lg_g.astype(np.float64) - lg_ref).max(axis=1)
    assert np.all(err <= tol), f"logit error {err.max():.3e}"
    idx_own, w_own = O.topk(lg_g.astype(np.float64), k)
    assert np.array_equal(idx_g, idx_own), np.nonzero((idx_g != idx_own).any(1))[0][:8]
    assert np.allclose(w_g, w_own, rtol=W_RTOL, atol=1e-7), np.abs(w_g - w_own).max()


@pytest.mark.parametrize("T", [1, 3, 8, 9, 16])
@pytest.mark.parametrize("multi", [False, True])
def test_decode_pass_routing_index_for_index(T, multi, cuda_device):
    """The routing computed inside a decode pass (the single persistent
    kernel's routing warps, or route_kernel in the multi-kernel sequence),
    read back from the workspace after lmoe_layer_forward."""
    from sparse_latent_moe_lmoe_b300 import LatentMoE, capi
    sh, _, W, _x, Ly, _y, _i, _w, _l = workload("decode_t8")
    x = S.make_x(T, sh.d, 60 + T)
    lg_ref = O.router_logits(Ly, x)
    m = LatentMoE(sh, W, device=0, flags=capi.FLAG_MULTI_KERNEL_DECODE if multi else 0)
    assert (capi.lmoe_stage_name(m.h, T, 0)[0] == "decode_fused") == (not multi)
    m.forward(bf16_tensor(x, cuda_device))
    idx, w, lg = m.last_decode_routing(T)
    torch.cuda.synchronize()
    m.check()
    check_routing_exact(idx.cpu().numpy(), w.cpu().numpy(), lg.cpu().numpy(), lg_ref, sh.k)
