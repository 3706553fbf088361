"""Window scores S per (layer, KV head).

Source: Novita AI, "How KV Sparsity achieves 1.5x acceleration for vLLM",
section "Key techniques 2: attention modification" (the PyramidKV-style
score and the "online softmax" step).  The score formula itself was lost in
extraction; what survives: [n - alpha, n] is the instruction-token range, A
is the softmax probability, S sums the softmax values of the nearest alpha
queries, each probability is rebuilt as exp(k.q - rowmax) / l from the
prefill's stored row maximum and normaliser, and only query blocks inside the
window are visited.

Readings taken:
* the window is the alpha queries at 0-based positions n-alpha .. n-1;
* the exponent uses the same 1/sqrt(d) scale as the prefill, so m and l are
  in the scaled-logit domain;
* S is not pooled or smoothed;
* with grouped-query attention the per-KV-head score is the sum over that
  head's query group.

S[h][i] = sum over g in group(h), over q in [n-alpha, n) with i <= q, of
exp(scale * q_g.k_i - m[g][q]) / l[g][q].
"""
from __future__ import annotations

import numpy as np


def window_scores(q, k, m, l, alpha, scale):
    """q: [n, H_q, d]; k: [n, H_kv, d] (float64).
    m, l: [H_q, alpha] -- the prefill row max / normaliser of the window rows
    n-alpha .. n-1, in that order.
    Returns S: [H_kv, n] float64.
    """
    n, h_q, _ = q.shape
    h_kv = k.shape[1]
    group = h_q // h_kv
    win = np.arange(n - alpha, n)
    visible = np.arange(n)[None, :] <= win[:, None]           # [alpha, n]
    S = np.zeros((h_kv, n))
    for g in range(h_q):
        h = g // group
        s = (q[win, g, :] @ k[:, h, :].T) * scale              # [alpha, n]
        a = np.exp(np.where(visible, s, -np.inf) - m[g][:, None]) / l[g][:, None]
        S[h] += a.sum(axis=0)                                  # sum over window queries
    return S
