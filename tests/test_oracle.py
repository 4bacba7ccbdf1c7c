"""Pins for the CPU oracle: each check compares the oracle with something other
than itself -- brute force, closed forms, invariants, special cases that reduce
to a library routine -- so that a dropped term, a wrong sign, a wrong index or
a transposed operand anywhere in it fails at least one test."""
import itertools
from dataclasses import replace

import numpy as np
import pytest

import lmoe_synth as S
import oracle as O

ONE, HALF, TWO, QUARTER = 0x3F80, 0x3F00, 0x4000, 0x3E80  # bf16 bit patterns


# ---------------------------------------------------------------- test helpers

def pack_int4(q: np.ndarray) -> np.ndarray:
    """Independent packer: element 2j -> low nibble of byte j, 2j+1 -> high."""
    q = np.asarray(q, np.int64)
    lo = q[..., 0::2] & 15
    hi = q[..., 1::2] & 15
    return (lo | (hi << 4)).astype(np.uint8)


def unpack_int4(b: np.ndarray) -> np.ndarray:
    b = np.asarray(b, np.int64)
    lo, hi = b & 15, b >> 4
    out = np.stack([lo, hi], axis=-1).reshape(*b.shape[:-1], b.shape[-1] * 2)
    return np.where(out >= 8, out - 16, out)


def bf16_f(bits):
    return (np.asarray(bits, np.uint32) << 16).view(np.float32).astype(np.float64)


def dense(q, s):
    """numpy dequantisation of a packed matrix (independent of the oracle)."""
    v = unpack_int4(q).astype(np.float64)
    sc = np.repeat(bf16_f(s), 32, axis=-1)
    return v * sc


def silu(a):
    return a / (1.0 + np.exp(-a))


def blank_layer(sh: S.LayerShape) -> dict:
    """All-zero weights with unit scales, in the generator's layout."""
    d, E, G, L, f, r = sh.d, sh.E, sh.G, sh.L, sh.f, sh.lora_rank
    W = {
        "W_r": np.zeros((E, d), np.float32),
        "b_r": np.zeros(E, np.float32) if sh.has_bias else None,
        "W_in_q": np.zeros((G, L, d // 2), np.uint8), "W_in_s": np.full((G, L, d // 32), ONE, np.uint16),
        "W_out_q": np.zeros((G, d, L // 2), np.uint8), "W_out_s": np.full((G, d, L // 32), ONE, np.uint16),
        "gate_q": np.zeros((E, f, L // 2), np.uint8), "gate_s": np.full((E, f, L // 32), ONE, np.uint16),
        "up_q": np.zeros((E, f, L // 2), np.uint8), "up_s": np.full((E, f, L // 32), ONE, np.uint16),
        "down_q": np.zeros((E, L, f // 2), np.uint8), "down_s": np.full((E, L, f // 32), ONE, np.uint16),
    }
    for n in ("A_in", "B_in", "A_out", "B_out"):
        W[n] = None
    if r:
        W["A_in"] = np.zeros((G, d, r), np.uint16)
        W["B_in"] = np.zeros((G, r, L), np.uint16)
        W["A_out"] = np.zeros((G, L, r), np.uint16)
        W["B_out"] = np.zeros((G, r, d), np.uint16)
    return W


def bf16_bits(v):
    v = np.asarray(v, np.float32)
    assert np.all(O.bf16_value(O.bf16_round(v)) == v), "value must be exact in bf16"
    return O.bf16_round(v)


# ----------------------------------------------------------------- bf16 format

def test_bf16_round_closed_forms():
    # 8 significant bits (ulp 2^-7 at 1.0); halfway cases round to even
    cases = {1.0: 1.0, 1 + 2 ** -9: 1.0, 1 + 3 * 2 ** -9: 1 + 2 ** -7, 1 + 2 ** -8: 1.0, 1 + 3 * 2 ** -8: 1 + 2 ** -6,
             -(1 + 2 ** -8): -1.0, 255.5: 256.0, 3.0e-3: None, 0.0: 0.0}
    for v, want in cases.items():
        got = O.bf16_value(O.bf16_round(np.array([v])))[0]
        if want is None:
            # nearest of the two neighbouring bf16 values
            e = np.floor(np.log2(abs(v)))
            q = 2.0 ** (e - 7)
            lo, hi = np.floor(v / q) * q, np.ceil(v / q) * q
            want = lo if (v - lo) < (hi - v) else hi
        assert got == want, (v, got, want)
    # a single rounding from fp64: 1 + 2^-8 + 2^-40 is just above the midpoint
    assert O.bf16_value(O.bf16_round(np.array([1 + 2 ** -8 + 2 ** -40])))[0] == 1 + 2 ** -7
    # agrees with round-to-nearest-even of fp32 inputs done by integer arithmetic
    rng = np.random.default_rng(0)
    f = (rng.standard_normal(10000) * 10.0 ** rng.integers(-30, 30, 10000)).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    ref = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    assert np.array_equal(O.bf16_round(f.astype(np.float64)), ref)


# ----------------------------------------------------------------- int4 format

def test_int4_golden_bytes():
    """Byte-level fixture of the packed format (tests/golden/int4_bytes.txt)."""
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "int4_bytes.txt")
    n = 0
    for line in open(path):
        line = line.split("#")[0].strip()
        if not line:
            continue
        byte, lo, hi = (int(v, 0) for v in line.split())
        row = np.array([byte], np.uint8)
        assert O.int4_at(row, 0) == lo and O.int4_at(row, 1) == hi, line
        n += 1
    assert n >= 8


def test_int4_roundtrip_all_values_all_positions():
    vals = np.arange(-7, 8)
    for pos in range(32):
        for v in vals:
            q = np.zeros((1, 32), np.int64)
            q[0, pos] = v
            q[0, (pos + 5) % 32] = -v  # a neighbour with the opposite sign
            packed = pack_int4(q)
            got = [O.int4_at(packed[0], c) for c in range(32)]
            assert got == list(q[0]), (pos, v)
            assert np.array_equal(pack_int4(np.array([got])), packed)


def test_dequant_exact_and_matches_independent_unpack():
    q, s = S.int4_matrix(7, 99, 48, 96, 0.02)
    got = O.dequant(q, s)
    assert np.array_equal(got, dense(q, s))
    # q * s is exact in fp32: a 3-bit integer times an 8-bit significand
    assert np.array_equal(got.astype(np.float32).astype(np.float64), got)


def test_generator_quantiser_is_nearest_level():
    """The generator's symmetric per-32 quantiser against a brute-force search
    over the 15 levels (ties to the even level)."""
    rows, K = 16, 64
    w = S.int4_source(3, 17, rows, K, 0.02)
    q, s = S.int4_matrix(3, 17, rows, K, 0.02)
    qi = unpack_int4(q)
    sv = bf16_f(s)
    for r in range(rows):
        for g in range(K // 32):
            blk = w[r, g * 32:(g + 1) * 32].astype(np.float32)
            amax = np.float32(np.abs(blk).max())
            want_s = O.bf16_value(O.bf16_round(np.array([np.float32(amax / np.float32(7.0))], np.float64)))[0]
            assert sv[r, g] == want_s
            for c in range(32):
                x = np.float32(blk[c] / np.float32(want_s))
                dist = [(abs(float(x) - lv), lv % 2, lv) for lv in range(-7, 8)]
                best = min(dist)[2]
                assert qi[r, g * 32 + c] == best


# ---------------------------------------------------------------------- router

def test_router_one_hot_columns_and_bias():
    sh = replace(S.TINY, has_bias=True)
    W = S.make_layer(sh, 0, bias_seed=2)
    Ly = O.Layer(sh, W)
    # x = one-hot at i  ->  logits = W_r[:, i] + b  (catches a transposed W_r)
    for i in (0, 5, 200, 255):
        x = np.zeros((1, sh.d), np.uint16)
        x[0, i] = ONE
        lg = O.router_logits(Ly, x)
        want = W["W_r"][:, i].astype(np.float64) + W["b_r"].astype(np.float64)
        assert np.array_equal(lg[0], want)
    # zero router weights -> logits are the bias exactly
    W2 = dict(W, W_r=np.zeros_like(W["W_r"]))
    lg = O.router_logits(O.Layer(sh, W2), S.make_x(3, sh.d, 4))
    assert np.array_equal(lg, np.tile(W["b_r"].astype(np.float64), (3, 1)))


def test_router_matches_library_matmul():
    sh = S.TINY
    W = S.make_layer(sh, 0)
    x = S.make_x(9, sh.d, 1)
    lg = O.router_logits(O.Layer(sh, W), x)
    ref = bf16_f(x) @ W["W_r"].astype(np.float64).T
    assert np.allclose(lg, ref, rtol=1e-13, atol=1e-13)


# ----------------------------------------------------------------------- top-k

def brute_topk(l, k):
    key = [(-float(np.float32(v)), e) for e, v in enumerate(l)]
    return [e for _, e in sorted(key)[:k]]


def test_topk_brute_force_random_and_adversarial():
    rng = np.random.default_rng(1)
    cases = [rng.standard_normal((50, 16)),
             np.round(rng.standard_normal((50, 16)) * 2) / 2,          # many exact ties
             np.zeros((3, 16)),                                         # all equal
             np.array([[0.0, -0.0] * 8, [-0.0, 0.0] * 8]),               # signed zeros compare equal
             -1e30 + rng.standard_normal((4, 16)) * 1e14,               # large negatives
             np.tile(np.arange(16)[::-1] * 1e-9, (2, 1)) + 1.0]         # ties only after fp32 rounding
    for lg in cases:
        for k in (1, 2, 5, 16):
            idx, w = O.topk(lg, k)
            for t in range(lg.shape[0]):
                assert list(idx[t]) == brute_topk(lg[t], k), (lg[t], k)


def test_topk_renorm_closed_forms():
    rng = np.random.default_rng(2)
    lg = rng.standard_normal((200, 512)) * 1.3
    idx, w = O.topk(lg, 10)
    assert np.all(np.abs(w.sum(1) - 1) <= 8 * 10 * np.finfo(np.float64).eps)
    assert np.all(np.diff(w, axis=1) <= 0)
    # softmax over the selected logits (library exp on the selected values)
    sel = np.take_along_axis(lg, idx.astype(np.int64), 1)
    ref = np.exp(sel - sel.max(1, keepdims=True))
    assert np.allclose(w, ref / ref.sum(1, keepdims=True), rtol=1e-14)
    # ... equals the full softmax renormalised over the selected experts
    full = np.exp(lg - lg.max(1, keepdims=True))
    full /= full.sum(1, keepdims=True)
    p = np.take_along_axis(full, idx.astype(np.int64), 1)
    assert np.allclose(w, p / p.sum(1, keepdims=True), rtol=1e-12)
    # k = 1 -> weight 1; equal logits -> 1/k
    _, w1 = O.topk(lg, 1)
    assert np.all(w1 == 1.0)
    _, we = O.topk(np.zeros((2, 512)), 10)
    assert np.allclose(we, 0.1, rtol=0, atol=1e-16)


# ----------------------------------------------------------------- permutation

def check_perm(idx, E, G, P):
    T, k = idx.shape
    epg = E // G
    flat = idx.reshape(-1)
    # offsets = exclusive scan of the histogram
    hist = np.bincount(flat, minlength=E)
    assert np.array_equal(P["expert_offsets"], np.concatenate([[0], np.cumsum(hist)]))
    # brute-force stable sort by expert
    want = sorted(range(T * k), key=lambda a: (flat[a], a))
    assert list(P["sorted_assign"]) == want
    # every token exactly k times; inverse round-trips
    assert np.array_equal(np.bincount(P["sorted_assign"] // k, minlength=T), np.full(T, k))
    assert np.array_equal(P["inv"][P["sorted_assign"]], np.arange(T * k))
    assert np.array_equal(P["group_offsets"], P["expert_offsets"][::epg])
    rows = 0
    for g in range(G):
        toks = sorted({t for t in range(T) for j in range(k) if idx[t, j] // epg == g})
        assert P["group_tok_offsets"][g] == rows
        assert list(P["group_tokens"][rows:rows + len(toks)]) == toks
        for t in range(T):
            for j in range(k):
                if idx[t, j] // epg == g:
                    assert P["group_tokens"][P["assign_row"][t * k + j]] == t
                    assert rows <= P["assign_row"][t * k + j] < rows + len(toks)
        rows += len(toks)
    assert P["group_tok_offsets"][G] == rows == P["rows"]


@pytest.mark.parametrize("T,E,G,k,skew", [(1, 16, 2, 2, 0), (7, 16, 2, 2, 0), (37, 64, 8, 10, 0),
                                          (64, 512, 8, 10, 1.1), (300, 32, 4, 3, 2.0)])
def test_permute_brute_force(T, E, G, k, skew):
    idx, _ = S.routing(11 + T, T, E, k, skew)
    check_perm(idx, E, G, O.permute(idx, E, G))


def test_permute_degenerate():
    # every token on the same experts; one group empty
    idx = np.tile(np.array([[3, 1]], np.int32), (5, 1))
    P = O.permute(idx, 16, 2)
    check_perm(idx, 16, 2, P)
    assert P["group_tok_offsets"][1] == P["group_tok_offsets"][2] == 5


# --------------------------------------------------------- expert and shared parts

def test_shared_in_columns_and_lora():
    sh = replace(S.TINY, lora_rank=8)
    W = S.make_layer(sh, 5, lora_seed=6)
    Ly = O.Layer(sh, W)
    Win = dense(W["W_in_q"], W["W_in_s"])  # [G][L][d]
    A, B = bf16_f(W["A_in"]), bf16_f(W["B_in"])
    for g in range(sh.G):
        for i in (0, 77, 255):
            x = np.zeros(sh.d)
            x[i] = 1.0
            h = O.shared_in(Ly, g, x)
            assert np.allclose(h, Win[g][:, i] + A[g][i] @ B[g], rtol=1e-13, atol=1e-15)
    # with the int4 base zeroed, only the low-rank branch remains (library matmul)
    W0 = dict(W, W_in_q=np.zeros_like(W["W_in_q"]))
    x = bf16_f(S.make_x(1, sh.d, 9))[0]
    assert np.allclose(O.shared_in(O.Layer(sh, W0), 1, x), (x @ A[1]) @ B[1], rtol=1e-12, atol=1e-15)


def test_shared_out_columns_and_lora():
    sh = replace(S.TINY, lora_rank=8)
    W = S.make_layer(sh, 5, lora_seed=6)
    Ly = O.Layer(sh, W)
    Wout = dense(W["W_out_q"], W["W_out_s"])  # [G][d][L]
    A, B = bf16_f(W["A_out"]), bf16_f(W["B_out"])
    for g in range(sh.G):
        for l in (0, 31, 63):
            u = np.zeros(sh.L)
            u[l] = 1.0
            assert np.allclose(O.shared_out(Ly, g, u), Wout[g][:, l] + A[g][l] @ B[g], rtol=1e-13, atol=1e-15)


def test_expert_swiglu_closed_form():
    """Gate = 1/2 I, Up = 2 I, Down = I (L = f = 32):  u = silu(h/2) * 2h.
    Swapping gate and up, or a sign error in silu, changes the result."""
    sh = S.LayerShape(d=64, E=4, G=2, k=1, L=32, f=32)
    W = blank_layer(sh)
    eye = pack_int4(np.eye(32, dtype=np.int64))
    e = 3
    W["gate_q"][e], W["gate_s"][e] = eye, HALF
    W["up_q"][e], W["up_s"][e] = eye, TWO
    W["down_q"][e] = eye
    h = np.linspace(-3, 3, 32)
    u = O.expert_latent(O.Layer(sh, W), e, h)
    assert np.allclose(u, silu(h / 2) * 2 * h, rtol=1e-15, atol=1e-300)
    assert not np.allclose(u, silu(2 * h) * h / 2)


# ----------------------------------------------------------------- whole layer

def test_zero_down_gives_exact_zero():
    sh = S.TINY
    W = S.make_layer(sh, 0)
    x = S.make_x(6, sh.d, 1)
    Wz = dict(W, down_q=np.zeros_like(W["down_q"]))
    y, idx, w, _ = O.layer_forward(O.Layer(sh, Wz), x)
    assert np.all(y == 0.0)
    # one expert's down zeroed -> its assignment contributes exactly nothing:
    # same result, bit for bit, as giving that assignment weight 0
    e0 = int(idx[0, 0])
    W1 = dict(W)
    W1["down_q"] = W["down_q"].copy()
    W1["down_q"][e0] = 0
    y1 = O.forward_routed(O.Layer(sh, W1), x[:1], idx[:1], w[:1])
    w0 = w[:1].copy()
    w0[0, 0] = 0.0
    y_ref = O.forward_routed(O.Layer(sh, W), x[:1], idx[:1], w0)
    assert np.array_equal(y1, y_ref)
    assert not np.array_equal(y1, O.forward_routed(O.Layer(sh, W), x[:1], idx[:1], w[:1]))


def test_group_homogeneous_reduces_to_shared_path():
    """All experts of group 1 share one SwiGLU and the bias sends every token
    into group 1: y = Wout[1] SwiGLU(Win[1] x) whatever the weights (they sum
    to 1). Checked against a numpy dense chain on independently unpacked
    matrices; expert 10 is in group 1 by e // (E/G) but in group 0 by e % G."""
    sh = replace(S.TINY, has_bias=True)
    W = S.make_layer(sh, 4, bias_seed=1)
    epg = sh.E // sh.G
    for e in range(epg, 2 * epg):
        for n in ("gate", "up", "down"):
            W[n + "_q"][e] = W[n + "_q"][epg + 2]
            W[n + "_s"][e] = W[n + "_s"][epg + 2]
    W["b_r"] = np.where(np.arange(sh.E) // epg == 1, 100.0, -100.0).astype(np.float32)
    x = S.make_x(5, sh.d, 3)
    y, idx, w, _ = O.layer_forward(O.Layer(sh, W), x)
    assert np.all(idx // epg == 1)
    Win = dense(W["W_in_q"][1], W["W_in_s"][1])
    Wout = dense(W["W_out_q"][1], W["W_out_s"][1])
    Gt = dense(W["gate_q"][epg + 2], W["gate_s"][epg + 2])
    Up = dense(W["up_q"][epg + 2], W["up_s"][epg + 2])
    Dn = dense(W["down_q"][epg + 2], W["down_s"][epg + 2])
    xf = bf16_f(x)
    h = xf @ Win.T
    ref = (Dn @ (silu(Gt @ h.T) * (Up @ h.T))).T @ Wout.T
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-18)


def test_identity_shared_matrices_reduce_to_weighted_expert_sum():
    """d = L, W_in = W_out = I (q = 1 on the diagonal, s = 1): the layer is
    sum_j w_j SwiGLU_{e_j}(x) -- a dropped routing weight or a wrong expert
    index shows up here."""
    sh = S.LayerShape(d=64, E=8, G=2, k=3, L=64, f=32)
    W = S.make_layer(sh, 8)
    eye = pack_int4(np.eye(64, dtype=np.int64))
    for g in range(sh.G):
        W["W_in_q"][g], W["W_in_s"][g] = eye, ONE
        W["W_out_q"][g], W["W_out_s"][g] = eye, ONE
    x = S.make_x(4, sh.d, 2)
    idx, w = S.routing(3, 4, sh.E, sh.k)
    w = w.astype(np.float64)
    y = O.forward_routed(O.Layer(sh, W), x, idx, w)
    xf = bf16_f(x)
    for t in range(4):
        ref = np.zeros(sh.d)
        for j in range(sh.k):
            e = idx[t, j]
            Gt, Up = dense(W["gate_q"][e], W["gate_s"][e]), dense(W["up_q"][e], W["up_s"][e])
            Dn = dense(W["down_q"][e], W["down_s"][e])
            ref += w[t, j] * (Dn @ (silu(Gt @ xf[t]) * (Up @ xf[t])))
        assert np.allclose(y[t], ref, rtol=1e-12, atol=1e-18)


def test_literal_equals_group_factored():
    for name, lora in (("tiny_t64", 0), ("tiny_t64", 16)):
        sh, T, W, x = S.make_workload(name)
        if lora:
            sh = replace(sh, lora_rank=lora)
            W = S.make_layer(sh, 0, lora_seed=3)
        Ly = O.Layer(sh, W)
        y, idx, w, _ = O.layer_forward(Ly, x[:16])
        yf = O.forward_routed(Ly, x[:16], idx, w, factored=True)
        assert np.allclose(y, yf, rtol=1e-12, atol=1e-18 * 0 + 1e-20)
        # group rows sum to the token output in ascending group order
        for t in (0, 7):
            rows = sum(O.group_row(Ly, g, x[t], idx[t], w[t]) for g in range(sh.G))
            assert np.allclose(rows, y[t], rtol=1e-12, atol=1e-20)


def test_residual_closed_forms():
    x = S.make_x(2, 64, 1)
    assert np.array_equal(O.residual(x, np.zeros((2, 64))), x)
    # y rounds to bf16 first, then the sum rounds once
    x1 = np.array([ONE], np.uint16)
    y = np.array([2 ** -8 + 2 ** -30])           # bf16(y) = 2^-8 exactly
    assert O.bf16_value(O.residual(x1, y))[0] == 1.0   # 1 + 2^-8 is a tie -> even (1.0)
    y = np.array([3 * 2 ** -9])
    assert O.bf16_value(O.residual(x1, y))[0] == 1 + 2 ** -7


def test_full_layer_against_numpy_chain_tiny():
    """End to end on the tiny workload: routing from library sorting of
    library matmul logits, experts from independently unpacked matrices."""
    sh, T, W, x = S.make_workload("tiny_t64")
    y, idx, w, lg = O.layer_forward(O.Layer(sh, W), x)
    xf = bf16_f(x)
    lg_ref = xf @ W["W_r"].astype(np.float64).T
    assert np.allclose(lg, lg_ref, rtol=1e-12, atol=1e-14)
    epg = sh.E // sh.G
    Win = dense(W["W_in_q"], W["W_in_s"])
    Wout = dense(W["W_out_q"], W["W_out_s"])
    for t in range(T):
        order = np.lexsort((np.arange(sh.E), -lg_ref[t].astype(np.float32)))[:sh.k]
        assert list(order) == list(idx[t])
        sel = lg_ref[t][order]
        wr = np.exp(sel - sel[0]) / np.exp(sel - sel[0]).sum()
        ref = np.zeros(sh.d)
        for e, wj in zip(order, wr):
            g = e // epg
            h = Win[g] @ xf[t]
            Gt, Up = dense(W["gate_q"][e], W["gate_s"][e]), dense(W["up_q"][e], W["up_s"][e])
            Dn = dense(W["down_q"][e], W["down_s"][e])
            ref += wj * (Wout[g] @ (Dn @ (silu(Gt @ h) * (Up @ h))))
        assert np.allclose(y[t], ref, rtol=1e-10, atol=1e-16)


def test_combine_closed_form():
    """Rows summed per token over its distinct groups (a group hit twice is
    counted once), plus the residual."""
    Y = np.arange(12, dtype=np.float32).reshape(3, 4)
    idx = np.array([[0, 3], [2, 1], [3, 2]], np.int32)        # E=4, G=2: groups 0,1 | 1,0 | 1,1
    ar = np.array([0, 1, 2, 0, 2, 2], np.int32)
    y = O.combine(Y, idx, ar, 4, 2)
    assert np.array_equal(y, np.stack([Y[0] + Y[1], Y[0] + Y[2], Y[2]]))
    res = np.full((3, 4), ONE, np.uint16)
    assert np.array_equal(O.combine(Y, idx, ar, 4, 2, residual=res), y + 1.0)


# ------------------------------------------------------------------ NVFP4
# NVFP4 ("Edge0-145B: Run a 145B Open-Source Model on Your Laptop", "What You
# Need to Run It": the checkpoint in NVIDIA's FP4 format): E2M1 elements, one
# E4M3 scale per 16 elements along K, one fp32 scale per weight tensor.

def minifloat(code: int, ebits: int, mbits: int, bias: int, nan_code=None) -> float:
    """Generic sign / exponent / mantissa decoder (exponent 0 subnormal), used
    only by the tests: checked against the library's E4M3 first, then applied
    to E2M1."""
    if nan_code is not None and (code & ((1 << (ebits + mbits)) - 1)) == nan_code:
        return float("nan")
    sgn = (code >> (ebits + mbits)) & 1
    e = (code >> mbits) & ((1 << ebits) - 1)
    m = code & ((1 << mbits) - 1)
    mag = (m / 2 ** mbits) * 2.0 ** (1 - bias) if e == 0 else (1 + m / 2 ** mbits) * 2.0 ** (e - bias)
    return -mag if sgn else mag


def e4m3_library(b) -> np.ndarray:
    import torch
    return torch.tensor(np.asarray(b, np.uint8)).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)


def test_e4m3_decode_matches_library_all_codes():
    lib = e4m3_library(np.arange(256))
    ours = np.array([O.e4m3_value(b) for b in range(256)])
    gen = np.array([minifloat(b, 4, 3, 7, nan_code=0x7F) for b in range(256)])
    assert np.array_equal(np.isnan(lib), np.isnan(ours)) and np.isnan(lib).sum() == 2
    fin = ~np.isnan(lib)
    assert np.array_equal(ours[fin], lib[fin])
    assert np.array_equal(gen[fin], lib[fin]) and np.array_equal(np.isnan(gen), np.isnan(lib))
    assert O.e4m3_value(0x7E) == 448.0 and O.e4m3_value(0x01) == 2.0 ** -9


def test_e2m1_decode_all_codes():
    """The generic decoder (pinned to the library on E4M3 above) at E2M1's
    parameters, and the format's invariants: 8 magnitudes strictly increasing
    from 0 to 6, the sign bit negating."""
    ours = [O.e2m1_value(c) for c in range(16)]
    assert ours == [minifloat(c, 2, 1, 1) for c in range(16)]
    mags = ours[:8]
    assert mags[0] == 0.0 and mags[-1] == 6.0 and all(a < b for a, b in zip(mags, mags[1:]))
    assert all(ours[c + 8] == -ours[c] for c in range(8))


def test_generator_e4m3_rounding_matches_library():
    import torch
    rng = np.random.default_rng(5)
    xs = np.concatenate([rng.uniform(0, 448, 4000), 2.0 ** rng.uniform(-12, 8.8, 4000),
                         [e4m3_library([b])[0] for b in range(1, 0x7F)]]).astype(np.float32)
    xs = xs[xs < 448]
    # exact midpoints between neighbouring E4M3 values (ties go to the even mantissa)
    vals = e4m3_library(np.arange(0, 0x7F))
    mids = ((vals[1:] + vals[:-1]) / 2).astype(np.float32)
    xs = np.concatenate([xs, mids[mids < 448]])
    lib = torch.tensor(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = np.array([S.e4m3_rne(v) for v in xs], np.uint8)
    assert np.array_equal(ours, lib)
    assert S.e4m3_rne(448.0) == 0x7E and S.e4m3_rne(1e6) == 0x7E and S.e4m3_rne(0.0) == 0


def unpack_codes(b: np.ndarray) -> np.ndarray:
    b = np.asarray(b, np.int64)
    return np.stack([b & 15, b >> 4], axis=-1).reshape(*b.shape[:-1], b.shape[-1] * 2)


def test_nvfp4_quantiser_is_nearest_level_and_dequant_exact():
    """The generator's NVFP4 matrices against brute force: the tensor scale is
    amax / (6 * 448), each block scale the library's E4M3 rounding of
    amax_block / 6 / gs, each code a nearest level; the oracle's dequantiser
    equals an independent unpack x decoder x library E4M3 x gs."""
    rows, K, rpt = 24, 64, 8
    q, s, gs = S.nvfp4_matrix(3, 11, rows, K, 0.02, rpt)
    w = S.int4_source(3, 11, rows, K, 0.02)  # the same draws
    table = np.array([minifloat(c, 2, 1, 1) for c in range(16)])
    codes = unpack_codes(q)
    for t in range(rows // rpt):
        wt = w[t * rpt:(t + 1) * rpt]
        assert gs[t] == np.float32(np.abs(wt).max()) / np.float32(6 * 448)
        blk = wt.reshape(rpt, K // 16, 16)
        amax = np.abs(blk).max(axis=-1).astype(np.float32)
        import torch
        sb = torch.tensor(amax / np.float32(6) / gs[t]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(s[t * rpt:(t + 1) * rpt], sb)
        scale = e4m3_library(sb).astype(np.float32) * gs[t]
        v = blk / scale[..., None]
        got = table[codes[t * rpt:(t + 1) * rpt].reshape(rpt, K // 16, 16)]
        err = np.abs(got - v)
        best = np.abs(table[None, None, None, :8] - np.abs(v)[..., None]).min(axis=-1)
        assert np.all(err <= best + 1e-6 * np.abs(v))
        dq = O.nvfp4_dequant(q[t * rpt:(t + 1) * rpt], s[t * rpt:(t + 1) * rpt], gs[t])
        ref = table[codes[t * rpt:(t + 1) * rpt]] * np.repeat(e4m3_library(s[t * rpt:(t + 1) * rpt]), 16, axis=-1) \
            * np.float64(gs[t])
        assert np.array_equal(dq, ref)


def nv_dense(q, s, gs):
    table = np.array([minifloat(c, 2, 1, 1) for c in range(16)])
    return table[unpack_codes(q)] * np.repeat(e4m3_library(s), 16, axis=-1) * np.float64(gs)


def test_full_layer_nvfp4_against_numpy_chain_tiny():
    """The NVFP4 layer end to end on the tiny workload, experts from the
    independently decoded matrices."""
    sh, T, W, x = S.make_workload("tiny_t64_nvfp4")
    y, idx, w, lg = O.layer_forward(O.Layer(sh, W), x)
    xf = bf16_f(x)
    epg = sh.E // sh.G
    for t in range(T):
        order = np.lexsort((np.arange(sh.E), -lg[t].astype(np.float32)))[:sh.k]
        assert list(order) == list(idx[t])
        sel = lg[t][order]
        wr = np.exp(sel - sel[0]) / np.exp(sel - sel[0]).sum()
        ref = np.zeros(sh.d)
        for e, wj in zip(order, wr):
            g = e // epg
            h = nv_dense(W["W_in_q"][g], W["W_in_s"][g], W["W_in_gs"][g]) @ xf[t]
            Gt = nv_dense(W["gate_q"][e], W["gate_s"][e], W["gate_gs"][e])
            Up = nv_dense(W["up_q"][e], W["up_s"][e], W["up_gs"][e])
            Dn = nv_dense(W["down_q"][e], W["down_s"][e], W["down_gs"][e])
            Wo = nv_dense(W["W_out_q"][g], W["W_out_s"][g], W["W_out_gs"][g])
            ref += wj * (Wo @ (Dn @ (silu(Gt @ h) * (Up @ h))))
        assert np.allclose(y[t], ref, rtol=1e-10, atol=1e-16)


def test_nvfp4_differs_from_int4_only_by_quantisation():
    """Same draws, two formats: both dequantised matrices stay within their
    own half-step of the source weights (a wrong scale or nibble order would
    not)."""
    q4, s4 = S.int4_matrix(0, 7, 16, 128, 0.02)
    qn, sn, gs = S.nvfp4_matrix(0, 7, 16, 128, 0.02, 16)
    w = S.int4_source(0, 7, 16, 128, 0.02).astype(np.float64)
    d4 = O.dequant(q4, s4)
    dn = O.nvfp4_dequant(qn, sn, gs[0])
    half4 = np.repeat(bf16_f(s4), 32, axis=-1) / 2
    assert np.all(np.abs(d4 - w) <= half4 * (1 + 1e-6))
    # NVFP4 level spacing is at most 2 (between 4 and 6) in units of the block scale
    stepn = np.repeat(e4m3_library(sn), 16, axis=-1) * gs[0]
    assert np.all(np.abs(dn - w) <= stepn * (1 + 1e-6) + 1e-12)
