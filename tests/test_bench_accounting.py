"""The algorithmic work bench.py divides by a kernel's time for its roofline
fraction, checked against independent counts: the bytes of the weight arrays
a routing touches (taken from the arrays themselves) and, for prefill, the
distinct (group, token) pairs by brute force."""
import os
import sys

import numpy as np

import lmoe_synth as S

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402

SH = S.TINY  # d=256, E=16, G=2 (8 experts a group), k=2, L=64, f=32


def test_decode_bytes_are_the_touched_weight_arrays():
    W = S.make_layer(SH, 5)
    T = 3
    idx = np.array([[0, 3], [3, 9], [1, 0]], np.int32)  # experts {0, 1, 3, 9}, groups {0, 1}
    b = bench.stage_bytes(SH, T, idx)
    epg = SH.E // SH.G
    experts = sorted({int(e) for e in idx.reshape(-1)})
    groups = sorted({e // epg for e in experts})
    act = 2 * T * SH.d  # bf16 x in or y out
    assert b["route"] == W["W_r"].nbytes + act
    assert b["win"] == sum(W["W_in_q"][g].nbytes + W["W_in_s"][g].nbytes for g in groups) + act
    assert b["gateup"] == sum(W[n][e].nbytes for e in experts for n in ("gate_q", "gate_s", "up_q", "up_s"))
    assert b["down"] == sum(W["down_q"][e].nbytes + W["down_s"][e].nbytes for e in experts)
    assert b["wout"] == sum(W["W_out_q"][g].nbytes + W["W_out_s"][g].nbytes for g in groups) + act
    assert b["decode_fused"] == sum(b[n] for n in ("route", "win", "gateup", "down", "wout"))


def test_prefill_flops_count_distinct_group_token_pairs():
    rng = np.random.default_rng(6)
    T = 40
    idx = np.stack([rng.choice(SH.E, SH.k, replace=False) for _ in range(T)]).astype(np.int32)
    f, rows = bench.stage_flops(SH, T, idx)
    epg = SH.E // SH.G
    pairs = {(int(e) // epg, t) for t in range(T) for e in idx[t]}
    assert rows == len(pairs)
    assert f["win"] == 2.0 * SH.d * SH.L * len(pairs) == f["wout"]
    assert f["route"] == 2.0 * T * SH.d * SH.E
    assert f["gateup"] == 2.0 * (2 * SH.f) * SH.L * T * SH.k
    assert f["down"] == 2.0 * SH.L * SH.f * T * SH.k


def test_prefill_flops_with_lora_by_brute_force():
    """With a rank-r branch: per distinct (group, token) pair, P = x . A_in
    (d x r), Q = Z . A_out (L x r), and the rank K blocks of W_in (r x L) and
    W_out (r x d); counted here pair by pair"""
    from dataclasses import replace
    sh = replace(SH, lora_rank=16)
    rng = np.random.default_rng(7)
    T = 33
    idx = np.stack([rng.choice(sh.E, sh.k, replace=False) for _ in range(T)]).astype(np.int32)
    f, rows = bench.stage_flops(sh, T, idx)
    f0, _ = bench.stage_flops(SH, T, idx)
    epg = sh.E // sh.G
    pairs = {(int(e) // epg, t) for t in range(T) for e in idx[t]}
    r = sh.lora_rank
    lp = lq = win = wout = 0.0
    for _ in pairs:
        lp += 2.0 * sh.d * r
        lq += 2.0 * sh.L * r
        win += 2.0 * sh.d * sh.L + 2.0 * r * sh.L
        wout += 2.0 * sh.L * sh.d + 2.0 * r * sh.d
    assert f["lora_p"] == lp and f["lora_q"] == lq
    assert f["win"] == win and f["wout"] == wout
    for n in ("route", "gateup", "down"):
        assert f[n] == f0[n]
