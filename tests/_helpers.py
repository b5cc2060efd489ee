"""Comparison helpers shared by the GPU parity tests.

Tolerances (derived from the arithmetic):
  * scores: |s_gpu - s_ref| <= 1e-3 * max(|s_ref|, 1e-2 * max_row |s_ref|)
    (the pages' 1e-3 relative agreement, with a floor for scores that cancel
    to near zero: f32 accumulation error scales with the row's magnitude, not
    with one score's);
  * selection: identical index sets, except that a key may be swapped only if
    its oracle score lies within 1e-3 * max(|s_k|, 1e-3 * max_row |s_ref|) of
    the oracle's k-th score s_k;
  * attention outputs: 2e-2 max-abs when the output is bf16, 1e-4 for f32
    (stated targets), compared on rows whose selected sets are identical.
"""

from __future__ import annotations

import numpy as np
import torch


def np64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def score_tol(ref_row: np.ndarray) -> np.ndarray:
    ref = np.asarray(ref_row, np.float64)
    floor = 1e-2 * (np.max(np.abs(ref)) if ref.size else 0.0)
    return 1e-3 * np.maximum(np.abs(ref), floor)


def assert_scores_close(gpu_row, ref_row, what=""):
    gpu = np.asarray(gpu_row, np.float64)
    ref = np.asarray(ref_row, np.float64)
    assert gpu.shape == ref.shape, what
    err = np.abs(gpu - ref)
    tol = score_tol(ref)
    bad = np.nonzero(err > tol)[0]
    assert bad.size == 0, f"{what}: {bad.size} scores off, first j={bad[:5]}, gpu={gpu[bad[:5]]}, ref={ref[bad[:5]]}"
    return float(np.max(err / np.maximum(np.abs(ref), 1e-30))) if ref.size else 0.0


def check_selection(gpu_sel, ref_sel, ref_scores, what=""):
    """True if the sets are identical; asserts that every difference is a
    near-tie swap under the tolerance rule.  Returns (identical, jaccard)."""
    a = set(int(x) for x in gpu_sel)
    b = set(int(x) for x in ref_sel)
    assert len(a) == len(gpu_sel), f"{what}: duplicate positions in GPU selection"
    assert len(a) == len(b), f"{what}: selection sizes differ {len(a)} vs {len(b)}"
    if a == b:
        return True, 1.0
    s = np.asarray(ref_scores, np.float64)
    kth = min(s[list(b)])
    tol = 1e-3 * max(abs(kth), 1e-3 * float(np.max(np.abs(s))))
    for j in a ^ b:
        assert abs(s[j] - kth) <= tol, f"{what}: swapped key {j} score {s[j]} vs k-th {kth} (tol {tol})"
    return False, len(a & b) / len(a | b)


def sorted_unique(row, n):
    v = [int(x) for x in row[:n]]
    assert v == sorted(v) and len(set(v)) == n, "selection must be ascending and unique"
    return v
