"""Decode-time scoring and fixed-budget replacement: the decode side of the
layer-wise sparsification.

Source: Novita AI, "How KV Sparsity achieves 1.5x acceleration for vLLM",
section "Key techniques 1" (in the step-preparation phase the first three
layers keep a full cache while the later layers use a sliding-window strategy
that replaces the lowest-scoring KVs automatically) and section "Key
techniques 2" (the decode-side PagedAttention does work like the prefill's,
with the same goal: the score S).

The pages give no formula for the decode side.  Readings taken, the plainest
the rest supports:
* a budgeted layer's cache holds exactly k_l tokens per KV head from the end
  of the prefill on (the one-time selection leaves k_l); each decode step's
  new token takes the slot of one of them;
* the token replaced is, per KV head, the one with the lowest accumulated
  score among those outside the recent window -- the r most recent positions
  counting the new token's, so positions p_new - r + 1 .. p_new - 1 are kept;
  ties go to the lower position (as in the prefill's selection);
* a token's score starts at its prefill window score (prompt tokens) or 0 (a
  token generated during decode), and every step adds the attention
  probability the step's query heads give it, summed over the KV head's query
  group (the same per-key sum as the window score, the step's query being the
  window);
* the step attends over the k_l tokens after the replacement, the new token
  included.

Everything is float64 and written per head with explicit softmax.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Optional, Sequence

import numpy as np


@dataclass
class HeadCache:
    """One KV head of one (stream, layer) item: k_l slots."""
    k: np.ndarray        # [k_l, d] float64
    v: np.ndarray        # [k_l, d]
    score: np.ndarray    # [k_l] accumulated score
    pos: np.ndarray      # [k_l] int64 token position


def replace_slot(score, pos, new_pos, recent) -> Optional[int]:
    """Slot the token at position new_pos takes: the lowest score among the
    slots whose token lies outside the recent window (pos <= new_pos - recent),
    ties to the lower position.  None when every token is recent."""
    best = None
    for i in range(len(pos)):
        if pos[i] > new_pos - recent:
            continue
        if best is None or (score[i], pos[i]) < (score[best], pos[best]):
            best = i
    return best


def is_valid_choice(score, pos, new_pos, recent, chosen, rel, abs_tol=0.0) -> bool:
    """Whether `chosen` is an acceptable replacement when scores carry a
    relative error `rel`: an eligible slot whose score is within the error of
    the lowest eligible score."""
    if chosen is None or not (0 <= chosen < len(pos)) or pos[chosen] > new_pos - recent:
        return False
    lo = min(score[i] for i in range(len(pos)) if pos[i] <= new_pos - recent)
    return score[chosen] <= lo + rel * max(abs(lo), abs(score[chosen])) + abs_tol


def step(heads: List[HeadCache], q, k_new, v_new, new_pos, recent, scale,
         slots: Optional[Sequence[int]] = None):
    """One decode step of one item.

    q [H_q, d]; k_new, v_new [H_kv, d] (float64); heads[h] for h < H_kv.
    slots: per-head slots to use instead of replace_slot's (a caller checks
    them with is_valid_choice first, so that a run can follow another
    implementation's choices among near-equal scores).
    Returns (out [H_q, d], probs [H_kv, k_l] -- this step's per-slot sums over
    the query group --, the slots used)."""
    h_q, d = q.shape
    h_kv = len(heads)
    group = h_q // h_kv
    used = []
    for h, hc in enumerate(heads):
        s = replace_slot(hc.score, hc.pos, new_pos, recent) if slots is None else int(slots[h])
        if s is None:
            raise ValueError("no slot outside the recent window")
        hc.k[s] = k_new[h]
        hc.v[s] = v_new[h]
        hc.pos[s] = new_pos
        hc.score[s] = 0.0
        used.append(s)
    out = np.zeros((h_q, d))
    probs = np.zeros((h_kv, heads[0].k.shape[0]))
    for g in range(h_q):
        hc = heads[g // group]
        logits = (hc.k @ q[g]) * scale
        e = np.exp(logits - logits.max())
        p = e / e.sum()
        out[g] = p @ hc.v
        probs[g // group] += p
    for h, hc in enumerate(heads):
        hc.score += probs[h]
    return out, probs, used
