"""Shared test helpers: oracle runs per unit and the tolerance contract.

Tolerances (fp32 accumulation, rel 1e-3 on scores):
  raw scores  |s - s_ref| <= 1e-3 * max(|s_ref|, std_h(s_ref))
  aggregated  |a - a_ref| <= 1e-3 * max(|a_ref|, 1)
  kept sets   equal, except slots whose a_ref lies within 1e-3 * max(|a_ref(B)|, 1)
              of a_ref(B), the B-th largest oracle score
  compaction  bit-exact
"""
import numpy as np

from oracle import tri_oracle as O

SCORE_RTOL = 1e-3


def unit_stats(center_all, R_all, m_all, g, G):
    """Oracle statistics of the G query heads of KV head g (arrays [Hq][F])."""
    sl = slice(g * G, (g + 1) * G)
    return center_all[sl], R_all[sl], m_all[sl]


def oracle_unit(w, stats_l, k_rows, v_rows, g, t, route="offsets"):
    """Runs the oracle on one unit.  stats_l = oracle (center, R, m) of the layer;
    k_rows/v_rows [N][d] float64 in logical slot order, positions 0..N-1.
    route: the oracle's per-offset route, or its closed form ("closed", pinned
    equal to it) for the many long units of the large workloads."""
    c, R, m = unit_stats(*stats_l, g, w.G)
    N = k_rows.shape[0]
    return O.compress_unit(c, R, m, k_rows, v_rows, np.arange(N, dtype=np.float64), t,
                           list(w.offsets), w.theta, w.budget, w.pairing, route=route)


def check_scores(s_gpu, s_ref):
    s_gpu = np.asarray(s_gpu, dtype=np.float64)
    sd = s_ref.std(axis=-1, keepdims=True)
    tol = SCORE_RTOL * np.maximum(np.abs(s_ref), sd)
    bad = np.abs(s_gpu - s_ref) > tol
    assert not bad.any(), f"{bad.sum()} raw scores out of tolerance; worst {np.abs(s_gpu - s_ref).max()}"


def check_agg(a_gpu, a_ref):
    a_gpu = np.asarray(a_gpu, dtype=np.float64)
    tol = SCORE_RTOL * np.maximum(np.abs(a_ref), 1.0)
    bad = np.abs(a_gpu - a_ref) > tol
    assert not bad.any(), f"{bad.sum()} aggregated scores out of tolerance; worst {np.abs(a_gpu - a_ref).max()}"


def check_kept(idx_gpu, idx_ref, a_ref, B):
    """Kept-set equality modulo the tie band around the B-th oracle score."""
    idx_gpu = np.asarray(idx_gpu)
    N = a_ref.shape[0]
    if N <= B:
        want = np.concatenate([np.arange(N), -np.ones(B - N, dtype=np.int64)])
        assert np.array_equal(idx_gpu, want)
        return 0
    assert idx_gpu.shape[0] == B
    assert np.all(np.diff(idx_gpu) > 0) and idx_gpu[0] >= 0 and idx_gpu[-1] < N
    aB = np.sort(np.where(np.isnan(a_ref), -np.inf, a_ref))[::-1][B - 1]
    band = np.abs(a_ref - aB) <= SCORE_RTOL * max(abs(aB), 1.0)
    diff = np.setxor1d(idx_gpu, idx_ref)
    assert band[diff].all(), f"kept sets differ outside the tie band at slots {diff[~band[diff]][:10]}"
    return diff.size


def check_compacted(k_after, k_before, idx_gpu, B):
    """Rows 0..B-1 after compaction equal the pristine rows at the GPU's idx."""
    np.testing.assert_array_equal(np.asarray(k_after)[:B], np.asarray(k_before)[np.asarray(idx_gpu)[:B]])
