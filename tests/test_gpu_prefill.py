"""GPU parity of the prefill path (tcgen05 grouped GEMMs) against the oracle,
through the C ABI: a small layer the oracle runs in full (ragged tails in
every grouped GEMM), and the Edge0-shaped layer at 16384 tokens with the Zipf
router bias, checked on a sample of tokens the oracle computes one by one
(tokens are independent in this layer)."""
import numpy as np
import pytest
import torch

import lmoe_synth as S
import oracle as O
from gpu_util import ambiguous_rows, bf16_bits, bf16_tensor, check_outputs, check_routing, check_rows

pytestmark = pytest.mark.gpu

# smallest shape the prefill kernels take: d, L multiples of 256, f of 128
SMALL = S.LayerShape(d=256, E=64, G=4, k=4, L=256, f=128)


def make(sh, W, path):
    from sparse_latent_moe_lmoe_b300 import LatentMoE
    return LatentMoE(sh, W, device=0, force_path=path)


def test_small_layer_prefill_full_oracle(cuda_device):
    from sparse_latent_moe_lmoe_b300 import capi
    sh = SMALL
    W = S.make_layer(sh, 11)
    T = 300
    x = S.make_x(T, sh.d, 12)
    y_ref, idx_ref, w_ref, lg_ref = O.layer_forward(O.Layer(sh, W), x)
    m = make(sh, W, capi.PATH_PREFILL)
    assert capi.lmoe_stage_name(m.h, T, 1)[0] == "permute"
    xt = bf16_tensor(x, cuda_device)
    idx, w, lg = m.route(xt, want_logits=True)
    torch.cuda.synchronize()
    keep = check_routing(lg.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy(), lg_ref, idx_ref, w_ref, sh.k)
    y = bf16_bits(m.forward(xt))
    m.check()
    mr, ma, _ = check_outputs(y[keep], y_ref[keep], "small prefill")
    print(f"small prefill: mean rel {mr:.2e} max abs {ma:.2e}, {int((~keep).sum())} near-tie tokens excluded")
    # residual add and determinism
    res = S.make_x(T, sh.d, 13)
    y1 = bf16_bits(m.forward(xt, residual=bf16_tensor(res, cuda_device)))
    y2 = bf16_bits(m.forward(xt, residual=bf16_tensor(res, cuda_device)))
    m.check()
    assert np.array_equal(y1, y2)
    check_outputs(y1[keep], (O.bf16_value(res) + O.bf16_value(O.bf16_round(y_ref)))[keep], "small prefill residual")


def test_small_expert_forward_prefill(cuda_device):
    from sparse_latent_moe_lmoe_b300 import capi
    sh = SMALL
    W = S.make_layer(sh, 21)
    T = 257
    x = S.make_x(T, sh.d, 22)
    idx, w = S.routing(23, T, sh.E, sh.k, skew=1.1)
    m = make(sh, W, capi.PATH_PREFILL)
    dev = cuda_device
    idx_t, w_t = torch.from_numpy(idx).to(dev), torch.from_numpy(w).to(dev)
    perm = m.permute(idx_t)
    Y = m.expert_forward(bf16_tensor(x, dev), idx_t, w_t, perm)
    torch.cuda.synchronize()
    m.check()
    ref_perm = O.permute(idx, sh.E, sh.G)
    gto, gtok = ref_perm["group_tok_offsets"], ref_perm["group_tokens"]
    Ly = O.Layer(sh, W)
    Yn = Y.cpu().numpy()
    rows = ref_perm["rows"]
    ref = np.zeros((rows, sh.d))
    for g in range(sh.G):
        for r in range(gto[g], gto[g + 1]):
            t = gtok[r]
            ref[r] = O.group_row(Ly, g, x[t], idx[t], w[t].astype(np.float64))
    err = np.abs(Yn[:rows] - ref).sum() / np.abs(ref).sum()
    assert err < 1e-3, err
    worst = check_rows(Yn[:rows], ref, "small prefill Y rows")
    print(f"small prefill Y rows: mean rel {err:.2e}, worst row max-abs / row scale {worst:.2e}")


_big = {}


def big_workload():
    if not _big:
        sh, T, W, x = S.make_workload("prefill_t16384_zipf")
        _big.update(sh=sh, T=T, W=W, x=x)
    return _big


def sample_tokens(idx_gpu, T, n=48, seed=5):
    """A seeded sample that includes tokens routed to the most and the least
    popular experts of the realised routing."""
    rng = np.random.default_rng(seed)
    pick = set(rng.choice(T, n, replace=False).tolist())
    flat = idx_gpu.reshape(-1)
    cnt = np.bincount(flat, minlength=idx_gpu.max() + 1)
    used = np.nonzero(cnt)[0]
    for e in (used[np.argmax(cnt[used])], used[np.argmin(cnt[used])]):
        toks = np.nonzero((idx_gpu == e).any(axis=1))[0]
        pick.update(toks[:4].tolist())
    pick.update([0, T - 1])
    return np.array(sorted(pick))


def test_prefill_16k_sampled_parity(cuda_device):
    from sparse_latent_moe_lmoe_b300 import capi
    b = big_workload()
    sh, T, W, x = b["sh"], b["T"], b["W"], b["x"]
    m = make(sh, W, capi.PATH_AUTO)
    assert capi.lmoe_stage_name(m.h, T, 0)[0] == "route"
    xt = bf16_tensor(x, cuda_device)
    idx, w, lg = m.route(xt, want_logits=True)
    y = bf16_bits(m.forward(xt))
    torch.cuda.synchronize()
    m.check()
    idx_n, w_n, lg_n = idx.cpu().numpy(), w.cpu().numpy(), lg.cpu().numpy()
    # every token: k distinct experts in range, weights positive and summing to 1,
    # ordered by the GPU's own logits (descending, ties to the lower index)
    assert idx_n.min() >= 0 and idx_n.max() < sh.E
    assert all(len(set(r)) == sh.k for r in idx_n)
    assert np.allclose(w_n.sum(1), 1.0, atol=1e-5) and (w_n > 0).all()
    sel = np.take_along_axis(lg_n, idx_n.astype(np.int64), 1)
    assert (np.diff(sel, axis=1) <= 0).all()
    # sampled tokens against the oracle, one by one
    toks = sample_tokens(idx_n, T)
    Ly = O.Layer(sh, W)
    y_ref, idx_ref, w_ref, lg_ref = O.layer_forward(Ly, x[toks])
    keep = check_routing(lg_n[toks], idx_n[toks], w_n[toks], lg_ref, idx_ref, w_ref, sh.k)
    mr, ma, _ = check_outputs(y[toks][keep], y_ref[keep], "prefill 16k sample")
    print(f"prefill 16k: {len(toks)} sampled tokens, mean rel {mr:.2e}, max abs {ma:.2e}")


def test_prefill_router_logits_unbiased(cuda_device):
    """Every logit of 512 tokens through the prefill router GEMM (Edge0 router,
    no bias, so max |l| per token is only a few units) within 1e-5 of the
    token's max |l|, and the top-k of unambiguous tokens bit-exact."""
    from sparse_latent_moe_lmoe_b300 import capi
    sh = S.EDGE0
    W = S.make_layer(sh, 0)
    T = 512
    x = S.make_x(T, sh.d, 61)
    m = make(sh, W, capi.PATH_PREFILL)
    xt = bf16_tensor(x, cuda_device)
    idx, w, lg = m.route(xt, want_logits=True)
    torch.cuda.synchronize()
    m.check()
    Ly = O.Layer(sh, W)
    lg_ref = O.router_logits(Ly, x)
    idx_ref, w_ref = O.topk(lg_ref, sh.k)
    lg_n = lg.cpu().numpy()
    err = np.abs(lg_n.astype(np.float64) - lg_ref).max(axis=1) / np.abs(lg_ref).max(axis=1)
    print(f"prefill router, unbiased: worst |dl| / max|l| = {err.max():.2e}, median {np.median(err):.2e}")
    check_routing(lg_n, idx.cpu().numpy(), w.cpu().numpy(), lg_ref, idx_ref, w_ref, sh.k)


def test_prefill_repeat_is_deterministic(cuda_device):
    b = big_workload()
    sh, T, W, x = b["sh"], b["T"], b["W"], b["x"]
    from sparse_latent_moe_lmoe_b300 import capi
    m = make(sh, W, capi.PATH_AUTO)
    xt = bf16_tensor(x[:4096], cuda_device)
    y1 = bf16_bits(m.forward(xt))
    y2 = bf16_bits(m.forward(xt))
    m.check()
    assert np.array_equal(y1, y2)


# ------------------------------------------------------------ Recover-LoRA
# The branch rides the grouped GEMMs as extra K blocks ([x | P_g] against
# [Win[g] ; B_in[g]], [Z | Q] against [Wout[g] ; B_out[g]]). The LoRA
# matrices here are drawn larger than the workloads' so that either branch
# alone moves the output far beyond the tolerance (checked on the oracle).

def lora_layer(sh, seed, a_sigma=0.08, b_sigma=0.05):
    from dataclasses import replace
    W = S.make_layer(sh, seed)
    r = sh.lora_rank
    W["A_in"] = S.normal_bf16(seed + 1, S.S_AIN, (sh.G, sh.d, r), a_sigma)
    W["B_in"] = S.normal_bf16(seed + 1, S.S_BIN, (sh.G, r, sh.L), b_sigma)
    W["A_out"] = S.normal_bf16(seed + 1, S.S_AOUT, (sh.G, sh.L, r), a_sigma)
    W["B_out"] = S.normal_bf16(seed + 1, S.S_BOUT, (sh.G, r, sh.d), b_sigma)
    return W


def assert_branches_matter(sh, W, x, y_ref):
    """the oracle's output moves by far more than the tolerance when either
    branch is switched off (B_in or B_out zeroed)"""
    for name in ("B_in", "B_out"):
        W0 = dict(W)
        W0[name] = np.zeros_like(W[name])
        y0 = O.layer_forward(O.Layer(sh, W0), x)[0]
        rel = np.abs(y0 - y_ref).sum() / np.abs(y_ref).sum()
        assert rel > 30 * 1e-3, (name, rel)


@pytest.mark.parametrize("G,r,T", [(4, 48, 300), (4, 128, 300), (16, 32, 200)])
def test_small_layer_prefill_lora_full_oracle(G, r, T, cuda_device):
    """rank padding (48 -> 64), two rank K blocks (128), and G = 16 (no token
    order: every (token tile, group) pair)"""
    from dataclasses import replace
    from sparse_latent_moe_lmoe_b300 import capi
    sh = replace(SMALL, G=G, lora_rank=r)
    W = lora_layer(sh, 31 + r)
    x = S.make_x(T, sh.d, 32)
    y_ref, idx_ref, w_ref, lg_ref = O.layer_forward(O.Layer(sh, W), x)
    assert_branches_matter(sh, W, x, y_ref)
    m = make(sh, W, capi.PATH_PREFILL)
    names = [capi.lmoe_stage_name(m.h, T, i)[0] for i in range(capi.lmoe_stage_name(m.h, T, 0)[1])]
    assert "lora_p" in names and "lora_q" in names
    assert names.index("lora_p") < names.index("win") and names.index("lora_q") < names.index("wout")
    assert ("tsort" in names) == (G <= 8)
    xt = bf16_tensor(x, cuda_device)
    idx, w, lg = m.route(xt, want_logits=True)
    torch.cuda.synchronize()
    keep = check_routing(lg.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy(), lg_ref, idx_ref, w_ref, sh.k)
    res = S.make_x(T, sh.d, 33)
    y = bf16_bits(m.forward(xt, residual=bf16_tensor(res, cuda_device)))
    y2 = bf16_bits(m.forward(xt, residual=bf16_tensor(res, cuda_device)))
    m.check()
    assert np.array_equal(y, y2)
    ref = O.bf16_value(res) + O.bf16_value(O.bf16_round(y_ref))
    mr, ma, _ = check_outputs(y[keep], ref[keep], f"prefill LoRA G={G} r={r}")
    print(f"prefill LoRA G={G} r={r}: mean rel {mr:.2e}, max abs {ma:.2e}")


def test_small_expert_forward_prefill_lora(cuda_device):
    """lmoe_expert_forward (group rows, the second mode of the W_out GEMM) with LoRA"""
    from dataclasses import replace
    from sparse_latent_moe_lmoe_b300 import capi
    sh = replace(SMALL, lora_rank=64)
    W = lora_layer(sh, 41)
    T = 257
    x = S.make_x(T, sh.d, 42)
    idx, w = S.routing(43, T, sh.E, sh.k, skew=1.1)
    m = make(sh, W, capi.PATH_PREFILL)
    dev = cuda_device
    idx_t, w_t = torch.from_numpy(idx).to(dev), torch.from_numpy(w).to(dev)
    perm = m.permute(idx_t)
    Y = m.expert_forward(bf16_tensor(x, dev), idx_t, w_t, perm)
    torch.cuda.synchronize()
    m.check()
    ref_perm = O.permute(idx, sh.E, sh.G)
    gto, gtok = ref_perm["group_tok_offsets"], ref_perm["group_tokens"]
    Ly = O.Layer(sh, W)
    rows = ref_perm["rows"]
    ref = np.zeros((rows, sh.d))
    for g in range(sh.G):
        for r in range(gto[g], gto[g + 1]):
            t = gtok[r]
            ref[r] = O.group_row(Ly, g, x[t], idx[t], w[t].astype(np.float64))
    Yn = Y.cpu().numpy()[:rows]
    err = np.abs(Yn - ref).sum() / np.abs(ref).sum()
    assert err < 1e-3, err
    worst = check_rows(Yn, ref, "prefill LoRA Y rows")
    print(f"prefill LoRA Y rows: mean rel {err:.2e}, worst {worst:.2e}")


def test_edge0_lora_prefill_sampled(cuda_device):
    """the Edge0 layer with its r = 64 branch at 2048 tokens through the
    grouped GEMMs, sampled tokens against the oracle"""
    from sparse_latent_moe_lmoe_b300 import capi
    sh, _, W, _ = S.make_workload("lora_t16")
    T = 2048
    x = S.make_x(T, sh.d, 51)
    m = make(sh, W, capi.PATH_AUTO)
    assert capi.lmoe_stage_name(m.h, T, 4)[0] == "lora_p"
    xt = bf16_tensor(x, cuda_device)
    idx, w, lg = m.route(xt, want_logits=True)
    y = bf16_bits(m.forward(xt))
    torch.cuda.synchronize()
    m.check()
    idx_n, w_n, lg_n = idx.cpu().numpy(), w.cpu().numpy(), lg.cpu().numpy()
    toks = sample_tokens(idx_n, T, n=24)
    y_ref, idx_ref, w_ref, lg_ref = O.layer_forward(O.Layer(sh, W), x[toks])
    keep = check_routing(lg_n[toks], idx_n[toks], w_n[toks], lg_ref, idx_ref, w_ref, sh.k)
    mr, ma, _ = check_outputs(y[toks][keep], y_ref[keep], "Edge0 LoRA prefill sample")
    print(f"Edge0 LoRA prefill: {len(toks)} tokens, mean rel {mr:.2e}, max abs {ma:.2e}")
