"""Causal prefill attention with per-row max and normaliser, and decode attention.

Source: Novita AI, "How KV Sparsity achieves 1.5x acceleration for vLLM",
section "Key techniques 2: attention modification".  The article's attention
formula was lost in extraction; it describes FlashAttention-2 (Figure 7)
computing softmax(QK^T)V in one pass while tracking a running row maximum and
a running normaliser l, and asks for that maximum and l as extra outputs.
Reading taken: standard scaled dot-product causal attention, scale 1/sqrt(d)
applied inside the exponent, natural exponent; query head g reads KV head
g // G (G = H_q / H_kv, contiguous groups).

Everything here is the definition written out: for each row, the full score
vector, its maximum, the exponentials, their sum, and the weighted sum of
values, all in float64.  No tiling, no online rescaling.
"""
from __future__ import annotations

import numpy as np


def prefill_rows(q, k, v, scale, rows=None, heads=None):
    """Causal attention for selected query rows of one sequence.

    q: [n, H_q, d] float64; k, v: [n, H_kv, d] float64.
    rows: query positions to evaluate (default: all n).
    heads: query heads to evaluate (default: all H_q).
    Returns O [len(rows), len(heads), d], m [len(heads), len(rows)],
    l [len(heads), len(rows)] where for row r and head g with s_i = scale*q.k_i
    over keys i <= r: m = max_i s_i, l = sum_i exp(s_i - m), and
    O = sum_i exp(s_i - m) / l * v_i.
    """
    n, h_q, d = q.shape
    h_kv = k.shape[1]
    group = h_q // h_kv
    rows = np.arange(n) if rows is None else np.asarray(rows, dtype=np.int64)
    heads = np.arange(h_q) if heads is None else np.asarray(heads, dtype=np.int64)
    out = np.zeros((rows.size, heads.size, d))
    m_out = np.zeros((heads.size, rows.size))
    l_out = np.zeros((heads.size, rows.size))
    # causal mask: key index i visible to row r iff i <= r
    visible = np.arange(n)[None, :] <= rows[:, None]
    for hi, g in enumerate(heads):
        h = g // group
        s = (q[rows, g, :] @ k[:, h, :].T) * scale          # [rows, n]
        s = np.where(visible, s, -np.inf)
        m = s.max(axis=1)                                     # row maximum
        e = np.exp(s - m[:, None])                            # masked -> 0
        l = e.sum(axis=1)                                     # normaliser
        out[:, hi, :] = (e / l[:, None]) @ v[:, h, :]
        m_out[hi] = m
        l_out[hi] = l
    return out, m_out, l_out


def decode_attention(q, k_cache, v_cache, scale):
    """One decode query against a gathered cache.

    q: [H_q, d]; k_cache, v_cache: [H_kv, T, d] (the kept prompt tokens in
    ascending position order followed by every appended token, the current
    one included, since the new token attends to itself).
    Returns out [H_q, d] = softmax(scale * K q) V per head, explicit softmax.
    """
    h_q, d = q.shape
    h_kv = k_cache.shape[0]
    group = h_q // h_kv
    out = np.zeros((h_q, d))
    for g in range(h_q):
        h = g // group
        s = (k_cache[h] @ q[g]) * scale
        m = s.max()
        e = np.exp(s - m)
        out[g] = (e / e.sum()) @ v_cache[h]
    return out
