"""Per-(layer, KV head) top-k_l retention with a forced recent window.

Source: Novita AI, "How KV Sparsity achieves 1.5x acceleration for vLLM":
section "System model" (prune low-score KV pairs, keep the higher-scoring
and the nearer ones), section "Key techniques 1" (step-preparation phase:
the first three layers keep the full cache, later layers evict the
lowest-score KV), and section "Key techniques 2" (in each layer l and head h
the k_l tokens with the highest scores are kept; every other KV entry is
discarded for the rest of the generation).

Readings taken:
* the recent window of r tokens counts inside the budget k_l;
* ties in S go to the lower position;
* output indices are in ascending original position;
* k_l >= n keeps every token (identity).
"""
from __future__ import annotations

import numpy as np


def select_kept(scores, n, k, recent):
    """scores: [n] (any float type; compared as given).
    Returns int64 ascending indices of the kept tokens (length min(k, n)).
    """
    if k is None or k >= n:
        return np.arange(n, dtype=np.int64)
    if recent > k:
        raise ValueError("recent window larger than the budget")
    scores = np.asarray(scores)
    if np.isnan(scores[:n]).any():
        raise ValueError("NaN score")
    recent_idx = np.arange(n - recent, n)
    cand = np.arange(0, n - recent)
    # sort candidates by (-score, position): the highest score first, ties to
    # the lower position
    # (np.lexsort: the last key is the primary one)
    order = cand[np.lexsort((cand, -scores[cand].astype(np.float64)))]
    top = order[: k - recent].astype(np.int64)
    return np.sort(np.concatenate([top, recent_idx]).astype(np.int64))
