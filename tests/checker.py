"""Tie-aware comparison of the CUDA path's output with the oracle's.

Tolerance (stated for the scores): a GPU score may differ from the oracle's fp32 score by at most
tau = 1e-5 * max_j |oracle score_j| of its row.  Index rule per row:

1. the same number of non-(-1) entries, min(k, n), followed only by -1;
2. no duplicates, every index visible (0 <= j < n);
3. the GPU's set may differ from the oracle's only by keys whose oracle score lies within tau of
   the oracle's last selected score (near-ties at the cut);
4. along the GPU order the oracle scores never rise by more than tau (swaps only among near-ties).

Rows where the oracle's selected keys are separated from the rest by more than tau, and whose
ordering has no near-ties, therefore have to match exactly.
"""
from __future__ import annotations

import numpy as np

REL_TOL = 1e-5


def row_tau(scores_row: np.ndarray, n: int) -> float:
    if n <= 0:
        return 0.0
    return REL_TOL * float(np.max(np.abs(scores_row[:n].astype(np.float64))))


def check_row(gpu: np.ndarray, ora: np.ndarray, scores_row, n: int, k: int):
    """Returns None when the row passes, else a message."""
    m = min(n, k)
    if m <= 0:
        return None if (gpu == -1).all() else "row should be all -1"
    g = gpu[:m]
    if (gpu[m:] != -1).any():
        return "padding is not -1"
    if (g < 0).any() or (g >= n).any():
        return "index outside [0, n)"
    if len(set(g.tolist())) != m:
        return "duplicate indices"
    if np.array_equal(g, ora[:m]):
        return None
    s = scores_row.astype(np.float64)
    tau = row_tau(scores_row, n)
    cut = s[ora[m - 1]]
    gs, os_ = set(g.tolist()), set(ora[:m].tolist())
    for j in gs - os_:
        if s[j] < cut - tau:
            return "GPU picked key %d (score %r) below the cut %r" % (j, s[j], cut)
    for j in os_ - gs:
        if s[j] > cut + tau:
            return "GPU missed key %d (score %r) above the cut %r" % (j, s[j], cut)
    sg = s[g]
    if (np.diff(sg) > tau).any():
        i = int(np.argmax(np.diff(sg)))
        return "order: score rises %r -> %r at %d" % (sg[i], sg[i + 1], i)
    return None


def check(gpu_idx, ora_idx, ora_scores, visible, k, rows=None):
    """Check every row (or the given rows).  ``visible[r]`` is the row's visible-key count.
    Returns (n_exact, n_checked, failures list)."""
    rows = range(gpu_idx.shape[0]) if rows is None else rows
    exact = 0
    checked = 0
    fails = []
    for r in rows:
        n = int(visible[r])
        msg = check_row(gpu_idx[r], ora_idx[r], ora_scores[r] if n > 0 else None, n, k)
        checked += 1
        if msg is not None:
            fails.append((r, msg))
        elif np.array_equal(gpu_idx[r], ora_idx[r]):
            exact += 1
    return exact, checked, fails


def check_scores(gpu_scores, ora_scores, visible, rows=None):
    """Largest |gpu - oracle| / tau over the visible keys of the given rows (must be <= 1)."""
    rows = range(ora_scores.shape[0]) if rows is None else rows
    worst = 0.0
    for r in rows:
        n = int(visible[r])
        if n <= 0:
            continue
        o = ora_scores[r, :n].astype(np.float64)
        g = gpu_scores[r, :n].astype(np.float64)
        tau = row_tau(ora_scores[r], n)
        if tau == 0:
            if not np.array_equal(o, g):
                return float("inf")
            continue
        worst = max(worst, float(np.max(np.abs(g - o)) / tau))
    return worst


def visible_counts(case, oracle_mod, complete_blocks_only=False):
    """Visible-key count of every output row (from the oracle's mask function)."""
    cb = complete_blocks_only
    rows = case.rows
    out = np.zeros(rows, dtype=np.int64)
    if case.layout_q == "BSND":
        for b in range(case.batch):
            sq = case.s1 if case.seq_lens_q is None else int(case.seq_lens_q[b])
            sk = int(case.seq_lens_k[b])
            for r in range(case.s1):
                out[b * case.s1 + r] = (oracle_mod.visible(case, sq, sk, r, complete_blocks_only=cb)
                                        if 0 <= sq <= case.s1 else 0)
    else:
        lo = 0
        for b in range(case.batch):
            hi = int(case.seq_lens_q[b])
            sk = int(case.seq_lens_k[b])
            for r in range(hi - lo):
                out[lo + r] = oracle_mod.visible(case, hi - lo, sk, r, complete_blocks_only=cb)
            lo = hi
    return out
