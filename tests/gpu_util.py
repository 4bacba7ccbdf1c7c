"""Shared helpers of the GPU parity tests: workloads, the oracle side, and
the comparison bars.

Bars (a bf16 output compared with an unrounded reference already shows
~1.4e-3 mean relative error from its final rounding alone, so outputs are
compared with bf16 of the oracle's value; fp16 intermediates with fp32
accumulation stay well inside 1e-3):
  - expert indices and the permutation: bit-exact; rows whose top-k is not
    unique at the logit tolerance (a near-tie between the k-th and (k+1)-th
    oracle logits) may differ and are counted, and their outputs excluded;
  - router logits: |l_gpu - l_ref| <= 1e-5 * max_e |l_ref| per token;
  - renormalised weights: relative 2 * (logit bar of the row) + 2e-6 (the
    weights depend on logit differences, each known to the logit bar, plus
    fp32 exp and sum);
  - layer outputs (bf16): compared with bf16(oracle): mean relative error
    sum|y - bf16(y_ref)| / sum|y_ref| <= 1e-3 and max-abs <= 2e-2.
"""
import numpy as np
import torch

import lmoe_synth as S
import oracle as O

LOGIT_RTOL = 1e-5
W_RTOL = 2e-6
MEAN_REL = 1e-3
MAX_ABS = 2e-2


def bf16_tensor(bits: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def ambiguous_rows(lg_ref: np.ndarray, k: int, tol: np.ndarray) -> np.ndarray:
    """Tokens whose top-k set is not unique within the logit tolerance:
    the gap between the k-th and (k+1)-th largest oracle logit is below
    2 * tol (both sides may err by tol)."""
    srt = -np.sort(-lg_ref, axis=1)
    if srt.shape[1] <= k:
        return np.zeros(lg_ref.shape[0], bool)
    return (srt[:, k - 1] - srt[:, k]) <= 2 * tol


def check_routing(lg_gpu, idx_gpu, w_gpu, lg_ref, idx_ref, w_ref, k):
    """Returns the boolean mask of tokens whose routing is unambiguous (and
    therefore compared bit-exactly)."""
    tol = LOGIT_RTOL * np.abs(lg_ref).max(axis=1)
    if lg_gpu is not None:
        err = np.abs(lg_gpu.astype(np.float64) - lg_ref).max(axis=1)
        assert np.all(err <= tol), f"logit error {err.max()} > {tol.min()}"
    amb = ambiguous_rows(lg_ref, k, tol)
    same_set = np.array([set(a) == set(b) for a, b in zip(idx_gpu, idx_ref)])
    bad = ~same_set & ~amb
    assert not bad.any(), f"expert sets differ on unambiguous tokens {np.nonzero(bad)[0][:10]}"
    # order within the set: descending logit, ties to the lower index; order
    # may legitimately differ only where two selected logits are within tol
    clean = same_set & ~amb
    for t in np.nonzero(clean)[0]:
        if list(idx_gpu[t]) != list(idx_ref[t]):
            sel = np.sort(lg_ref[t, idx_ref[t]])
            assert np.min(np.diff(sel)) <= 2 * tol[t], f"order differs on token {t}"
        else:
            rt = 2 * tol[t] + W_RTOL
            assert np.allclose(w_gpu[t], w_ref[t], rtol=rt, atol=1e-7), (t, w_gpu[t], w_ref[t], rt)
    return ~amb


def output_errors(y_gpu_bits: np.ndarray, y_ref: np.ndarray):
    ref16 = O.bf16_value(O.bf16_round(y_ref))
    got = O.bf16_value(y_gpu_bits)
    mean_rel = np.abs(got - ref16).sum() / max(np.abs(y_ref).sum(), 1e-300)
    max_abs = np.abs(got - ref16).max() if got.size else 0.0
    mean_rel_unrounded = np.abs(got - y_ref).sum() / max(np.abs(y_ref).sum(), 1e-300)
    return mean_rel, max_abs, mean_rel_unrounded


# Element-wise bound on fp32 rows of the expert FFN (Y[(g, t)] against the
# oracle's group row): every element within ROW_RTOL of its own row's largest
# magnitude. The GPU keeps H, V and Z in fp16 (relative rounding <= 2^-11 per
# element); the error each row reaches is a few times 2^-11 of the row's
# scale, so a wrong or misplaced row -- whose error is of the size of the row
# itself -- cannot pass, whatever its magnitude.
ROW_RTOL = 1e-2


def check_rows(Y_gpu: np.ndarray, Y_ref: np.ndarray, what=""):
    """Per-row max-abs check of fp32 rows; returns the largest relative
    error seen (max over rows of max|dY| / max|Y_ref row|)."""
    Y_gpu = np.asarray(Y_gpu, np.float64)
    scale = np.abs(Y_ref).max(axis=1)
    err = np.abs(Y_gpu - Y_ref).max(axis=1)
    rel = err / np.maximum(scale, 1e-30)
    worst = int(np.argmax(rel)) if rel.size else 0
    assert np.all(err <= ROW_RTOL * scale + 1e-12), (
        f"{what}: row {worst} max-abs error {err[worst]:.3e} > {ROW_RTOL} x row scale {scale[worst]:.3e}")
    return float(rel.max()) if rel.size else 0.0


def check_outputs(y_gpu_bits, y_ref, what=""):
    mr, ma, mru = output_errors(y_gpu_bits, y_ref)
    assert mr <= MEAN_REL, f"{what}: mean relative error {mr:.3e} > {MEAN_REL}"
    assert ma <= MAX_ABS, f"{what}: max-abs error {ma:.3e} > {MAX_ABS}"
    return mr, ma, mru
