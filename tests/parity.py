"""Parity gates between the CUDA path and the fp64 oracle.

Tolerances (the library's stated contract):
* Sum:     |a_gpu - a| <= 1e-4 * S,  S_ie = sum_j |k_ij b_je|   (relative to the absolute sum)
* LSE:     |L_gpu - L| <= 1e-4 + 2^-20 |L|: 1e-4 absolute, plus the fp32 rounding
           of an exponent of that magnitude (8 ulps of |L|; the distance itself is
           an fp32 sum, so |L| = 17000 carries ~5e-3 however it is reduced).  For
           the workloads (|L| < 10) the second term is below 1e-5.
* grad-x:  |gx_gpu - gx| <= 1e-4 * G, G_id = (2/sigma^2) sum_j k_ij |beta_ij| |x_id - y_jd|
* K-min:   indices bit-exact at every position k whose oracle distance is separated
           by more than 1e-5 (relative) from the distances at k-1 and k+1 (the
           (K+1)-th for k = K); other positions are near-ties: counted, and the
           GPU's index there must be a valid point whose exact distance is within
           1e-5 (relative) of the oracle's.  GPU distances within 2e-5 relative
           (fp32 rounding of a D-term sum) plus 1e-7 absolute.
"""
from __future__ import annotations

import numpy as np

SUM_RTOL = 1e-4
LSE_ATOL = 1e-4
LSE_RTOL = 2.0 ** -20
GRAD_RTOL = 1e-4
TIE_RTOL = 1e-5


def check_sum(a_gpu, a_ref, S_ref, what=""):
    a_gpu = np.asarray(a_gpu, dtype=np.float64)
    err = np.abs(a_gpu - a_ref)
    ok = err <= SUM_RTOL * S_ref + 1e-30
    worst = float(np.max(err / np.maximum(S_ref, 1e-300))) if err.size else 0.0
    assert ok.all(), f"Sum parity {what}: {int((~ok).sum())} bad, worst err/S {worst:.3e}"
    return worst


def check_lse(L_gpu, L_ref, what=""):
    L_gpu = np.asarray(L_gpu, dtype=np.float64)
    both_inf = np.isneginf(L_gpu) & np.isneginf(L_ref)
    with np.errstate(invalid="ignore"):
        err = np.where(both_inf, 0.0, np.abs(L_gpu - L_ref))
        ok = err <= LSE_ATOL + LSE_RTOL * np.where(np.isfinite(L_ref), np.abs(L_ref), 0.0)
    worst = float(np.max(err)) if err.size else 0.0
    assert ok.all(), f"LSE parity {what}: {int((~ok).sum())} bad, worst abs err {worst:.3e}"
    return worst


def check_grad(gx_gpu, gx_ref, G_ref, what=""):
    gx_gpu = np.asarray(gx_gpu, dtype=np.float64)
    err = np.abs(gx_gpu - gx_ref)
    ok = err <= GRAD_RTOL * G_ref + 1e-30
    worst = float(np.max(err / np.maximum(G_ref, 1e-300))) if err.size else 0.0
    assert ok.all(), f"grad parity {what}: {int((~ok).sum())} bad, worst err/G {worst:.3e}"
    return worst


def separated_positions(d_ref, next_ref):
    """Boolean (M, K): positions whose oracle distance is not a near-tie."""
    d = np.asarray(d_ref, dtype=np.float64)
    M, K = d.shape
    ext = np.concatenate([np.full((M, 1), -np.inf), d, np.asarray(next_ref, dtype=np.float64)[:, None]], axis=1)
    cur = ext[:, 1:K + 1]
    tol = TIE_RTOL * np.abs(cur)
    with np.errstate(invalid="ignore"):
        below = (cur - ext[:, 0:K]) > tol
        above = (ext[:, 2:K + 2] - cur) > tol
    return below & above


def check_knn(idx_gpu, dist_gpu, x, y, idx_ref, d_ref, next_ref, what=""):
    """Returns the number of near-tie positions (validated, not gated)."""
    idx_gpu = np.asarray(idx_gpu).astype(np.int64)
    idx_ref = np.asarray(idx_ref).astype(np.int64)
    sep = separated_positions(d_ref, next_ref)
    bad = sep & (idx_gpu != idx_ref)
    assert not bad.any(), (f"K-min parity {what}: {int(bad.sum())} separated positions differ; "
                           f"first at {np.argwhere(bad)[0].tolist()}")
    ties = ~sep
    x = np.asarray(x, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    for (i, k) in np.argwhere(ties):
        j = idx_gpu[i, k]
        if idx_ref[i, k] < 0:
            assert j == -1, f"K-min {what}: row {i} slot {k} should be empty"
            continue
        assert 0 <= j < y.shape[0], f"K-min {what}: row {i} slot {k} index {j} out of range"
        dj = float(np.sum((x[i] - y[j]) ** 2))
        assert abs(dj - d_ref[i, k]) <= TIE_RTOL * abs(d_ref[i, k]) + 1e-12, \
            f"K-min {what}: near-tie row {i} slot {k}: index {j} at {dj} vs {d_ref[i, k]}"
    for i in range(idx_gpu.shape[0]):
        row = idx_gpu[i][idx_gpu[i] >= 0]
        assert len(set(row.tolist())) == len(row), f"K-min {what}: duplicate index in row {i}"
    if dist_gpu is not None:
        dg = np.asarray(dist_gpu, dtype=np.float64)
        fin = np.isfinite(d_ref)
        assert (np.isinf(dg) == ~fin).all(), f"K-min {what}: empty slots differ"
        err = np.abs(dg[fin] - d_ref[fin])
        assert (err <= 2e-5 * np.abs(d_ref[fin]) + 1e-7).all(), \
            f"K-min {what}: distance error {np.max(err) if err.size else 0}"
    return int(ties.sum())


# ---------------------------------------------------------------------------
# Max / Min with Arg
# ---------------------------------------------------------------------------
MAX_RTOL = 1e-4
FLUSH = 2.0 ** -126   # ex2 / rcp / rsqrt flush results below this to zero (ftz)

# k as a function of the squared distance, used only to validate the index the GPU
# returns at a near-tie (its value must be within tolerance of the oracle's extreme).
_KFN = {
    "gaussian": lambda q, s: np.exp(-q / s ** 2),
    "laplace": lambda q, s: np.exp(-np.sqrt(q) / s),
    "cauchy": lambda q, s: 1.0 / (1.0 + q / s ** 2),
    "imq": lambda q, s: 1.0 / np.sqrt(1.0 + q / s ** 2),
}


def check_maxmin(val_gpu, idx_gpu, x, y, b, sigma, kernel, val_ref, idx_ref, second_ref, what=""):
    """Value: |v_gpu - v| <= 1e-4 |v| + 2^-126 max_j |b_je| (the flush-to-zero floor).
    Index: exact where the oracle's extreme and runner-up differ by more than 1e-5
    relative (plus the floor); at near-ties the GPU's index must be a valid point whose
    fp64 value is within the value tolerance of the extreme.  Returns the near-tie count."""
    b = np.asarray(b, dtype=np.float64)
    floor = FLUSH * (np.max(np.abs(b), axis=0)[None, :] if b.size else 0.0)
    if val_gpu is not None:
        v = np.asarray(val_gpu, dtype=np.float64)
        same_inf = np.isinf(v) & np.isinf(val_ref) & (np.sign(v) == np.sign(val_ref))
        with np.errstate(invalid="ignore"):
            err = np.where(same_inf, 0.0, np.abs(v - val_ref))
        ok = err <= MAX_RTOL * np.where(np.isfinite(val_ref), np.abs(val_ref), 0.0) + floor
        assert ok.all(), f"Max/Min value {what}: {int((~ok).sum())} bad, worst {np.max(err):.3e}"
    idx_gpu = np.asarray(idx_gpu).astype(np.int64)
    with np.errstate(invalid="ignore"):
        sep = np.abs(val_ref - second_ref) > TIE_RTOL * np.abs(val_ref) + floor
    sep |= idx_ref < 0
    bad = sep & (idx_gpu != idx_ref)
    assert not bad.any(), (f"Arg parity {what}: {int(bad.sum())} separated entries differ; "
                           f"first at {np.argwhere(bad)[0].tolist()}")
    x = np.asarray(x, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    kf = _KFN[kernel]
    ties = np.argwhere(~sep)
    for (i, e) in ties:
        j = idx_gpu[i, e]
        assert 0 <= j < y.shape[0], f"Arg {what}: row {i} column {e} index {j} out of range"
        f = kf(float(np.sum((x[i] - y[j]) ** 2)), sigma) * b[j, e]
        assert abs(f - val_ref[i, e]) <= MAX_RTOL * abs(val_ref[i, e]) + floor[0, e], \
            f"Arg {what}: near-tie row {i} column {e}: index {j} gives {f} vs {val_ref[i, e]}"
    return len(ties)
