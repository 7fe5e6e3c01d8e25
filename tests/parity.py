"""Comparison helpers shared by the GPU parity tests (no arithmetic of the method).

Tolerances: floating-point scores must satisfy |gpu - oracle| <= rtol * A(t, s) with
A = k_scale * sum_h |w'| * sum_d |q k| the condition bound the oracle returns, rtol
1e-3 for bf16 and 2e-2 for FP8 inputs; integer-valued inputs must match exactly.
A top-k row is valid iff it has the right count of unique visible indices, -1
padding after them, every selected key scores at least the oracle's keep-th best
score minus tolerance, every unselected visible key at most that plus tolerance,
and (score order) the oracle scores along the row are non-increasing within
tolerance.
"""
from __future__ import annotations

import numpy as np

RTOL = {"bf16": 1e-3, "fp8_e4m3": 2e-2}


def assert_scores_close(gpu: np.ndarray, ref: np.ndarray, bound: np.ndarray, rtol: float, exact: bool):
    vis = np.isfinite(ref)
    g = gpu[vis].astype(np.float64)
    r = ref[vis]
    if exact:
        bad = np.nonzero(g != r)[0]
        assert bad.size == 0, f"{bad.size} scores differ, first: gpu {g[bad[0]]} oracle {r[bad[0]]}"
    else:
        err = np.abs(g - r)
        lim = rtol * bound[vis] + 1e-30
        worst = np.argmax(err / lim)
        assert np.all(err <= lim), f"score error {err[worst]:.3e} > {lim[worst]:.3e} (oracle {r[worst]})"


def check_topk_row(row: np.ndarray, ref_row: np.ndarray, o: np.ndarray, tol: np.ndarray, n: int, keep: int,
                   by_score: bool):
    """row: GPU output; ref_row: oracle output; o / tol: oracle scores and tolerances of the n visible keys."""
    k_out = row.shape[0]
    sel = row[:keep]
    assert np.all(row[keep:] == -1), "padding must be -1"
    assert np.all((sel >= 0) & (sel < n)), "index outside the visible keys"
    assert len(np.unique(sel)) == keep, "duplicate index"
    if keep == 0:
        return
    theta_idx = ref_row[keep - 1]
    theta = o[theta_idx]
    tt = tol[theta_idx]
    assert np.all(o[sel] >= theta - tol[sel] - tt), "a selected key scores below the k-th best"
    mask = np.ones(n, dtype=bool)
    mask[sel] = False
    un = np.nonzero(mask)[0]
    assert np.all(o[un] <= theta + tol[un] + tt), "an unselected key scores above the k-th best"
    if by_score:
        a, b = sel[:-1], sel[1:]
        assert np.all(o[a] >= o[b] - tol[a] - tol[b]), "row not in score order"
    else:
        assert np.all(np.diff(sel) > 0), "row not in index order"


def assert_topk_valid(gpu: np.ndarray, ref: np.ndarray, ref_scores: np.ndarray, bound: np.ndarray,
                      n_visible, topk_limit: int, rtol: float, exact: bool, by_score: bool = True):
    if exact:
        bad = np.nonzero(np.any(gpu != ref, axis=1))[0]
        assert bad.size == 0, f"{bad.size} rows differ; first row {bad[0]}: gpu {gpu[bad[0], :8]} oracle {ref[bad[0], :8]}"
        return
    for r in range(gpu.shape[0]):
        n = int(n_visible[r])
        keep = min(topk_limit, n, gpu.shape[1])
        o = ref_scores[r, :n]
        tol = rtol * bound[r, :n]
        check_topk_row(gpu[r], ref[r], o, tol, n, keep, by_score)
