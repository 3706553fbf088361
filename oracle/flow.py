"""Step orders of the hot path, built from the oracle's pieces.

Sources: Novita AI, "How KV Sparsity achieves 1.5x acceleration for vLLM",
section "Key techniques 1" (three phases: service init, step preparation with
per-layer block-table strategies, sparsification after model execution;
continuous batching, Figure 4); Ultralytics glossary, "PagedAttention"
(sections "How paging works" and "Block sharing between sequences").

Orders fixed here (the pages leave them open; these are the plainest ones):
* prefill of a sequence visits layers 0..L-1; after selection, layer l pops
  ceil(k_eff / 16) blocks from the free list, in layer order;
* a decode step visits streams in order and, within a stream, layers
  0..L-1; for each (stream, layer) it pops a new block when the length is a
  multiple of 16, otherwise copies the last block first if it is shared, then
  appends the step's k/v at slot `len` and attends over len + 1 tokens;
* retiring a stream decrements every block of layer 0..L-1 in table order.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np

from .attention import prefill_rows, decode_attention
from .scoring import window_scores
from .selection import select_kept
from .paging import BLOCK, blocks_for, compact, gather_rows


def _f64(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@dataclass
class Stream:
    """One decoding stream (a sequence, or one parallel sample of it)."""
    tables: List[List[int]]
    lens: List[int]


@dataclass
class LayerRecord:
    budgeted: bool
    k_eff: int
    idx: np.ndarray                       # [H_kv, k_eff]
    scores: Optional[np.ndarray] = None   # [H_kv, n] when budgeted
    m_win: Optional[np.ndarray] = None    # [H_q, alpha]
    l_win: Optional[np.ndarray] = None
    rows: Optional[np.ndarray] = None     # rows whose O/m/l were evaluated
    o_rows: Optional[np.ndarray] = None
    m_rows: Optional[np.ndarray] = None
    l_rows: Optional[np.ndarray] = None
    table: List[int] = field(default_factory=list)
    hits: List[int] = field(default_factory=list)  # prefix blocks found, not written


def sparsify_layer(w, layer, q_bits, k_bits, v_bits, rows=None, scores_override=None):
    """Prefill + scoring + selection for one layer of one sequence.

    rows: extra prompt rows whose O, m, l are evaluated (the window rows are
    always evaluated since the scores need their m and l).
    scores_override: use these scores (e.g. another implementation's, or a
    precision-matched copy) for the selection instead of the oracle's own.
    """
    n = q_bits.shape[0]
    q, k, v = _f64(q_bits), _f64(k_bits), _f64(v_bits)
    budgeted = w.budgeted(layer, n)
    rec = LayerRecord(budgeted=budgeted, k_eff=w.k_eff(layer, n), idx=None)
    if rows is not None:
        rows = np.asarray(rows, dtype=np.int64)
        rec.rows = rows
        rec.o_rows, rec.m_rows, rec.l_rows = prefill_rows(q, k, v, w.scale, rows)
    if budgeted:
        alpha = min(w.alpha, n)
        win = np.arange(n - alpha, n)
        _, m_win, l_win = prefill_rows(q, k, v, w.scale, win)
        rec.m_win, rec.l_win = m_win, l_win
        rec.scores = window_scores(q, k, m_win, l_win, alpha, w.scale)
        sel = rec.scores if scores_override is None else scores_override
        rec.idx = np.stack([select_kept(sel[h], n, w.budget(layer, n), w.recent)
                            for h in range(w.h_kv)])
    else:
        rec.idx = np.tile(np.arange(n, dtype=np.int64), (w.h_kv, 1))
    return rec


def place_layer(rec, pool, k_bits, v_bits, pool_k, pool_v, layer=None, tokens=None):
    """Allocate ceil(k_eff/16) blocks and compact the kept rows into them.

    With the prompt's token ids given (and the layer's index), a layer that
    keeps every token looks its full blocks up as prefix blocks, in order,
    each chained to the one before; blocks found hold that prefix's rows
    already and are not written.  Its partial last block, and every block of a
    budgeted layer, come from the free list.  rec.hits lists the blocks found."""
    rec.hits = []
    if tokens is not None and not rec.budgeted:
        n_full = rec.k_eff // BLOCK
        parent, table = -1, []
        for i in range(n_full):
            b, hit = pool.prefix_block(layer, parent, tokens[i * BLOCK:(i + 1) * BLOCK])
            table.append(b)
            if hit:
                rec.hits.append(b)
            parent = b
        table += [pool.alloc() for _ in range(blocks_for(rec.k_eff) - n_full)]
        rec.table = table
    else:
        rec.table = [pool.alloc() for _ in range(blocks_for(rec.k_eff))]
    if pool_k is not None:
        if rec.hits:
            # only the blocks not found are written: compact into a scratch
            # copy, then take the written blocks from it
            sk, sv = pool_k.copy(), pool_v.copy()
            compact(k_bits, v_bits, rec.idx, rec.table, sk, sv)
            for b in rec.table:
                if b not in rec.hits:
                    pool_k[b], pool_v[b] = sk[b], sv[b]
        else:
            compact(k_bits, v_bits, rec.idx, rec.table, pool_k, pool_v)
    return rec.table


def new_stream(records) -> Stream:
    return Stream(tables=[list(r.table) for r in records], lens=[r.k_eff for r in records])


def share_stream(pool, stream: Stream) -> Stream:
    """Another stream over the same blocks (parallel sample): +1 on every block."""
    for t in stream.tables:
        for b in t:
            pool.incref(b)
    return Stream(tables=[list(t) for t in stream.tables], lens=list(stream.lens))


def prepare_append(pool, stream: Stream, layer, pool_k=None, pool_v=None):
    """Make slot `len` of (stream, layer) writable.  Returns (src, dst) of a
    copy-on-write block copy, or None."""
    L = stream.lens[layer]
    t = stream.tables[layer]
    if L % BLOCK == 0:
        t.append(pool.alloc())
        return None
    last = t[-1]
    nb, copied = pool.cow(last)
    if copied:
        if pool_k is not None:
            pool_k[nb] = pool_k[last]
            pool_v[nb] = pool_v[last]
        t[-1] = nb
        return (last, nb)
    return None


def append(stream: Stream, layer, k_bits, v_bits, pool_k, pool_v):
    """Write the step's k/v [H_kv, d] at slot len of (stream, layer); len + 1."""
    L = stream.lens[layer]
    t = stream.tables[layer]
    b, s = t[L // BLOCK], L % BLOCK
    pool_k[b, :, s] = k_bits
    pool_v[b, :, s] = v_bits
    stream.lens[layer] = L + 1


def attend(w, stream: Stream, layer, q_bits, pool_k, pool_v):
    """Decode attention of q [H_q, d] over the len tokens of (stream, layer),
    read back through its block table.  Returns out [H_q, d] float64."""
    L = stream.lens[layer]
    t = stream.tables[layer]
    kc = np.stack([gather_rows(pool_k, t, L, h) for h in range(w.h_kv)])
    vc = np.stack([gather_rows(pool_v, t, L, h) for h in range(w.h_kv)])
    return decode_attention(_f64(q_bits), _f64(kc), _f64(vc), w.scale)


def append_and_attend(w, stream: Stream, layer, q_bits, k_bits, v_bits, pool_k, pool_v):
    """Write the step's k/v at slot len, then attend over len + 1 tokens.
    q_bits [H_q, d], k_bits/v_bits [H_kv, d].  Returns out [H_q, d] float64."""
    append(stream, layer, k_bits, v_bits, pool_k, pool_v)
    return attend(w, stream, layer, q_bits, pool_k, pool_v)


def retire(pool, stream: Stream):
    for t in stream.tables:
        for b in t:
            pool.decref(b)
    stream.tables = [[] for _ in stream.tables]
