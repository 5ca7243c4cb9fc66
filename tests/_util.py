"""Shared test helpers: tolerance checks and numpy/torch conversions (no layer arithmetic)."""
from __future__ import annotations

import numpy as np

# Tolerances for floating-point outputs (o, lse, dq, dk, dv): fp32 accumulation with bf16
# inputs and outputs.  The max-abs bound is applied on top of the rounding of the reference
# to bf16, which no bf16 output can avoid: |gpu - ref| <= MAX_ABS + BF16_HALF_ULP_REL * |ref|.
MAX_ABS = 2e-2
REL_L2 = 1e-2
BF16_HALF_ULP_REL = 2.0 ** -8
SELECT_SLACK = 1e-3     # every selected pool scores >= the oracle's k-th score - 1e-3


def bits_to_torch(bits: np.ndarray, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def torch_bf16_to_f64(t) -> np.ndarray:
    import torch
    return t.detach().to(torch.float32).cpu().numpy().astype(np.float64)


def assert_close(got: np.ndarray, ref: np.ndarray, name: str, max_abs=MAX_ABS, rel_l2=REL_L2, bf16_out=True):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    err = np.abs(got - ref)
    allow = max_abs + (BF16_HALF_ULP_REL * np.abs(ref) if bf16_out else 0.0)
    worst = np.argmax(err - allow)
    assert np.all(err <= allow), (f"{name}: |err| {err.flat[worst]:.3e} > {allow.flat[worst] if np.ndim(allow) else allow:.3e} "
                                  f"at {np.unravel_index(worst, err.shape)} (got {got.flat[worst]}, ref {ref.flat[worst]})")
    denom = np.linalg.norm(ref)
    rel = np.linalg.norm(got - ref) / (denom if denom > 0 else 1.0)
    assert rel <= rel_l2, f"{name}: rel-L2 {rel:.3e} > {rel_l2}"
    return float(err.max()), float(rel)


def check_selection_valid(pool_idx: np.ndarray, rows: np.ndarray, topk: int):
    """Structure every selected row must have: min(topk, floor(i/4)) distinct eligible pools,
    ascending, then -1 padding."""
    for r, i in enumerate(rows):
        n = int(i) // 4
        row = pool_idx[r]
        m = min(topk, n)
        sel = row[:m]
        assert np.all(row[m:] == -1), (i, row[m:])
        assert np.all(sel >= 0) and np.all(sel < n), (i, sel.min() if m else None, sel.max() if m else None, n)
        assert np.all(np.diff(sel) > 0), (i, "not strictly ascending")


def check_selection_scores(pool_idx: np.ndarray, rows: np.ndarray, scores: np.ndarray, kth: np.ndarray, topk: int,
                           slack=SELECT_SLACK):
    """Every selected pool's oracle score is >= the oracle's k-th score - slack."""
    for r, i in enumerate(rows):
        n = int(i) // 4
        m = min(topk, n)
        if m == 0:
            continue
        sel = pool_idx[r, :m]
        s = scores[r, sel].astype(np.float32)
        assert np.all(s >= np.float32(kth[r]) - slack), (int(i), float(s.min()), float(kth[r]))
