"""Pins of the CPU oracle against things other than itself.

Each test checks the oracle against what the pages or the mathematics fix:
the worked paging example (Ultralytics glossary "PagedAttention", section
"How paging works"), library routines (torch fp64 scaled_dot_product_attention
and softmax, numpy cumulative max, torch's bf16 rounding), closed forms
(softmax rows sum to one, equal keys), and brute force on tiny inputs.
"""
import itertools
import json
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import flow
from synth import bf16_bits, bf16_to_f64, tiny

RNG = np.random.default_rng(1234)


def _sdpa(q, k, v, causal=True):
    """torch fp64 SDPA on [n, H, d] arrays; GQA by repeating each KV head over
    its contiguous group of query heads."""
    h_q, h_kv = q.shape[1], k.shape[1]
    tq = torch.from_numpy(q).permute(1, 0, 2)
    tk = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(h_q // h_kv, dim=0)
    tv = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(h_q // h_kv, dim=0)
    if causal:
        o = F.scaled_dot_product_attention(tq, tk, tv, is_causal=True)
    else:
        o = F.scaled_dot_product_attention(tq, tk, tv)
    return o.permute(1, 0, 2).numpy()


def _sdpa_probs(q, k):
    """Causal attention probability matrices [H_q, n, n] via SDPA with V = I."""
    n, h_q, _ = q.shape
    eye = np.broadcast_to(np.eye(n)[:, None, :], (n, k.shape[1], n)).copy()
    return _sdpa(q, k, eye).transpose(1, 0, 2)


# ---------------------------------------------------------------------------
# paging: the worked example
# ---------------------------------------------------------------------------
def test_paging_worked_example(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "paging_worked_example.json")))
    pool = oracle.BlockPool(g["pool_blocks"], free=g["free_list"])
    n, bs, d = g["n_tokens"], g["block_size"], g["head_dim"]
    nb = oracle.blocks_for(n, bs)
    assert nb == g["expected_blocks"]
    table = [pool.alloc() for _ in range(nb)]
    assert table == g["expected_table"]
    keys = RNG.standard_normal((n, 1, d))
    pk = np.zeros((g["pool_blocks"], 1, bs, d))
    pv = np.zeros_like(pk)
    oracle.compact(keys, keys, np.arange(n)[None, :], table, pk, pv, block=bs)
    back = oracle.gather_rows(pk, table, n, 0, block=bs)
    assert np.array_equal(back, keys[:, 0]) == g["expected_keys_intact"]
    assert nb * bs - n == g["expected_unused_slots_paged"]
    assert g["reservation_tokens"] - n == g["expected_unused_slots_reserved"]
    # the two blocks left are still at the head of the free list, in order
    assert pool.free == g["free_list"][nb:]


def test_compaction_of_a_selected_set_follows_the_index_per_head():
    """Compaction of a selected (not identity) set, read back two ways.

    Every row carries its own coordinates (position and KV head in its first two
    entries), so each pool slot tells where its bytes came from.  The kept index
    differs per head, is not sorted by position, and 37 kept slots leave a
    partial last block.  The worked example's write and gather lines (Ultralytics
    glossary "PagedAttention", section "How paging works") fix what must hold:
    reading the table's blocks slot by slot gives the kept rows in index order,
    the gather returns exactly those rows, and nothing outside the table's
    blocks or past the last kept slot is touched."""
    n, h_kv, d, k_eff, nb_pool = 90, 3, 6, 37, 12
    k = RNG.standard_normal((n, h_kv, d))
    k[:, :, 0] = np.arange(n)[:, None]
    k[:, :, 1] = np.arange(h_kv)[None, :]
    v = k + 1000.0
    idx = np.stack([RNG.permutation(n)[:k_eff] for _ in range(h_kv)])
    assert not all(np.array_equal(idx[0], idx[h]) for h in range(1, h_kv))
    assert not (np.diff(idx, axis=1) > 0).all()
    table = [9, 2, 6]                                    # scattered, ceil(37/16) = 3
    sentinel = -7.0
    pk = np.full((nb_pool, h_kv, 16, d), sentinel)
    pv = np.full_like(pk, sentinel)
    oracle.compact(k, v, idx, table, pk, pv)
    for h in range(h_kv):
        slots = [pk[table[b], h, s] for b in range(len(table)) for s in range(16)]
        tags = [(int(r[0]), int(r[1])) for r in slots[:k_eff]]
        assert tags == [(int(p), h) for p in idx[h]]
        assert all((r == sentinel).all() for r in slots[k_eff:])
        np.testing.assert_array_equal(oracle.gather_rows(pk, table, k_eff, h), k[idx[h], h])
        np.testing.assert_array_equal(oracle.gather_rows(pv, table, k_eff, h), v[idx[h], h])
    untouched = [b for b in range(nb_pool) if b not in table]
    assert (pk[untouched] == sentinel).all() and (pv[untouched] == sentinel).all()


def test_pool_fifo_refcount_cow():
    pool = oracle.BlockPool(6)
    a, b, c = pool.alloc(), pool.alloc(), pool.alloc()
    assert (a, b, c) == (0, 1, 2)
    pool.decref(b)                       # returns to the tail
    assert pool.free == [3, 4, 5, 1]
    pool.incref(a)
    assert pool.ref[a] == 2
    nb, copied = pool.cow(a)             # shared -> copy into the head block
    assert copied and nb == 3 and pool.ref[a] == 1 and pool.ref[nb] == 1
    same, copied = pool.cow(a)           # sole owner -> in place
    assert not copied and same == a
    for blk in (a, c, nb):
        pool.decref(blk)
    assert sorted(pool.free) == list(range(6))
    with pytest.raises(ValueError):
        pool.decref(a)
    small = oracle.BlockPool(1)
    small.alloc()
    with pytest.raises(oracle.OutOfBlocks):
        small.alloc()


# ---------------------------------------------------------------------------
# prefix blocks (whole-block hashing across requests)
# ---------------------------------------------------------------------------
def _prefix_requests(rng, n_req, vocab=3):
    """Token sequences that share prefixes often: each request copies the
    start of an earlier one (or of a common root) and then diverges."""
    root = rng.integers(0, vocab, 200)
    reqs = []
    for _ in range(n_req):
        src = reqs[rng.integers(len(reqs))] if reqs and rng.random() < 0.7 else root
        cut = int(rng.integers(0, len(src) + 1))
        tail = rng.integers(0, vocab, int(rng.integers(0, 60)))
        reqs.append(np.concatenate([src[:cut], tail]).astype(np.int64))
    return reqs


def _place_prefix(pool, layer, toks):
    parent, table, hits = -1, [], []
    for i in range(len(toks) // 16):
        b, hit = pool.prefix_block(layer, parent, toks[i * 16:(i + 1) * 16])
        table.append(b)
        hits.append(hit)
        parent = b
    return table, hits


@pytest.mark.parametrize("seed", range(6))
def test_prefix_blocks_shared_iff_prefixes_equal_brute_force(seed):
    """Requests arrive and retire in a random order; every full block of a
    layer's prompt is a prefix block.  By brute force over the requests held
    at the time: block i of a new request is found iff some held request's
    first 16 (i + 1) tokens are the same (and that request's block i is full),
    and then it is that request's block i; the count of every block is the
    number of held requests whose table holds it."""
    rng = np.random.default_rng(seed)
    reqs = _prefix_requests(rng, 40, vocab=2 + seed % 3)
    pool = oracle.BlockPool(4000, free=rng.permutation(4000))
    held = {}                                         # request -> (tokens, table)
    order = list(range(len(reqs)))
    for r in order:
        if held and rng.random() < 0.35:              # retire someone first
            victim = list(held)[rng.integers(len(held))]
            for b in held.pop(victim)[1]:
                pool.decref(b)
        toks = reqs[r]
        table, hits = _place_prefix(pool, 0, toks)
        for i in range(len(table)):
            end = 16 * (i + 1)
            match = [q for q, (tq, bq) in held.items()
                     if len(tq) >= end and np.array_equal(tq[:end], toks[:end])]
            assert hits[i] == bool(match), (r, i)
            if match:
                assert all(held[q][1][i] == table[i] for q in match)
        held[r] = (toks, table)
        counts = {}
        for _, tbl in held.values():
            for b in tbl:
                counts[b] = counts.get(b, 0) + 1
        assert all(pool.ref[b] == c for b, c in counts.items())
        assert sum(1 for b in range(4000) if pool.ref[b] > 0) == len(counts)
        assert pool.num_free() + len(counts) == 4000


def test_prefix_blocks_forgotten_when_free_and_separate_per_layer():
    pool = oracle.BlockPool(64)
    toks = np.arange(48) % 5
    t0, h0 = _place_prefix(pool, 0, toks)
    assert h0 == [False] * 3 and t0 == [0, 1, 2]
    t1, h1 = _place_prefix(pool, 1, toks)             # another layer: its own blocks
    assert h1 == [False] * 3 and t1 == [3, 4, 5]
    t2, h2 = _place_prefix(pool, 0, toks)             # same layer, same prompt: all found
    assert h2 == [True] * 3 and t2 == t0 and all(pool.ref[b] == 2 for b in t0)
    other = toks.copy()
    other[20] += 1                                    # differs inside block 1
    t3, h3 = _place_prefix(pool, 0, other)
    assert h3 == [True, False, False] and t3[0] == t0[0]
    assert t3[2] != t0[2]                             # same tokens, another prefix: not found
    for t in (t0, t1, t2, t3):
        for b in t:
            pool.decref(b)
    assert pool.num_free() == 64 and not pool.prefix
    t4, h4 = _place_prefix(pool, 0, toks)             # nothing held: nothing found
    assert h4 == [False] * 3 and t4 == [8, 9, 10]     # the FIFO's head


def test_place_layer_writes_only_blocks_not_found():
    """A full-cache layer placed with its token ids: blocks found are left as
    they are; the rest hold the kept rows; a budgeted layer finds nothing."""
    w = tiny()
    n = 40
    qb, kb, vb = (bf16_bits(RNG.standard_normal(s).astype(np.float32))
                  for s in ((n, w.h_q, w.d), (n, w.h_kv, w.d), (n, w.h_kv, w.d)))
    toks = np.arange(n) % 7
    pool = oracle.BlockPool(32)
    pk = np.zeros((32, w.h_kv, 16, w.d), np.uint16)
    pv = np.zeros_like(pk)
    rec_a = flow.sparsify_layer(w, 0, qb, kb, vb)        # layer 0: full cache
    flow.place_layer(rec_a, pool, kb, vb, pk, pv, layer=0, tokens=toks)
    assert rec_a.hits == [] and len(rec_a.table) == 3
    marked = pk[rec_a.table[0]].copy()
    pk[rec_a.table[0]] ^= 0x1234                         # a write would restore it
    rec_b = flow.sparsify_layer(w, 0, qb, kb, vb)
    flow.place_layer(rec_b, pool, kb, vb, pk, pv, layer=0, tokens=toks)
    assert rec_b.hits == rec_a.table[:2] and rec_b.table[:2] == rec_a.table[:2]
    assert rec_b.table[2] != rec_a.table[2]              # the partial block is private
    np.testing.assert_array_equal(pk[rec_a.table[0]], marked ^ 0x1234)
    np.testing.assert_array_equal(oracle.gather_rows(pk, rec_b.table, n, 0)[32:], kb[32:, 0])
    n2 = 256
    qb2, kb2, vb2 = (bf16_bits(RNG.standard_normal(s).astype(np.float32))
                     for s in ((n2, w.h_q, w.d), (n2, w.h_kv, w.d), (n2, w.h_kv, w.d)))
    pool2 = oracle.BlockPool(64)
    recs = [flow.sparsify_layer(w, 1, qb2, kb2, vb2) for _ in range(2)]   # layer 1: budgeted
    assert recs[0].budgeted
    for r in recs:
        flow.place_layer(r, pool2, kb2, vb2, None, None, layer=1, tokens=np.zeros(n2, np.int64))
        assert r.hits == []


def test_pool_conservation_random_trace():
    pool = oracle.BlockPool(40, free=RNG.permutation(40))
    owned = []
    for _ in range(2000):
        op = RNG.integers(0, 4)
        if op == 0 and pool.num_free():
            owned.append(pool.alloc())
        elif op == 1 and owned:
            blk = owned[RNG.integers(len(owned))]
            pool.incref(blk)
            owned.append(blk)
        elif op == 2 and owned:
            pool.decref(owned.pop(RNG.integers(len(owned))))
        elif op == 3 and owned and pool.num_free():
            i = RNG.integers(len(owned))
            owned[i], _ = pool.cow(owned[i])
        in_use = {b for b in range(40) if pool.ref[b] > 0}
        assert pool.num_free() + len(in_use) == 40
        assert sorted(owned) == sorted(b for b in range(40) for _ in range(pool.ref[b]))


# ---------------------------------------------------------------------------
# prefill rows: O, m, l
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("n,h_q,h_kv,d", [(67, 4, 2, 16), (33, 6, 3, 8), (20, 2, 2, 32)])
def test_prefill_O_equals_sdpa(n, h_q, h_kv, d):
    q = RNG.standard_normal((n, h_q, d))
    k = RNG.standard_normal((n, h_kv, d))
    v = RNG.standard_normal((n, h_kv, d))
    o, m, l = oracle.prefill_rows(q, k, v, 1 / np.sqrt(d))
    np.testing.assert_allclose(o, _sdpa(q, k, v), atol=1e-12, rtol=0)


def test_prefill_l_is_inverse_max_probability():
    n, h_q, h_kv, d = 45, 4, 2, 16
    q = RNG.standard_normal((n, h_q, d)) * 2
    k = RNG.standard_normal((n, h_kv, d))
    _, _, l = oracle.prefill_rows(q, k, k, 1 / np.sqrt(d))
    p = _sdpa_probs(q, k)                       # [H_q, n, n]
    # the maximal logit contributes exp(0) = 1 to l, so max_i p = 1 / l
    np.testing.assert_allclose(l, 1.0 / p.max(axis=2), rtol=1e-12)


def test_prefill_m_one_hot_queries():
    n, h_q, h_kv, d = 50, 4, 2, 16
    k = RNG.standard_normal((n, h_kv, d))
    q = np.zeros((n, h_q, d))
    t = 3.0
    for g in range(h_q):
        q[:, g, g % d] = t
    scale = 1 / np.sqrt(d)
    _, m, _ = oracle.prefill_rows(q, k, k, scale)
    for g in range(h_q):
        h = g // (h_q // h_kv)
        expect = scale * t * np.maximum.accumulate(k[:, h, g % d])
        np.testing.assert_allclose(m[g], expect, rtol=1e-13, atol=1e-13)


def test_prefill_equal_keys_closed_form():
    n, h_q, h_kv, d = 40, 2, 1, 8
    k0 = RNG.standard_normal(d)
    k = np.broadcast_to(k0, (n, h_kv, d)).copy()
    q = RNG.standard_normal((n, h_q, d))
    v = RNG.standard_normal((n, h_kv, d))
    scale = 1 / np.sqrt(d)
    o, m, l = oracle.prefill_rows(q, k, v, scale)
    counts = np.arange(1, n + 1)
    for g in range(h_q):
        np.testing.assert_allclose(l[g], counts, rtol=1e-13)           # every logit equal
        np.testing.assert_allclose(m[g], scale * (q[:, g] @ k0), rtol=1e-13)
        np.testing.assert_allclose(o[:, g], np.cumsum(v[:, 0], axis=0) / counts[:, None],
                                   rtol=1e-11, atol=1e-12)


def test_prefill_row_subset_matches_full():
    n, h_q, h_kv, d = 70, 4, 2, 16
    q, k, v = (RNG.standard_normal((n, h, d)) for h in (h_q, h_kv, h_kv))
    o, m, l = oracle.prefill_rows(q, k, v, 0.3)
    rows = np.array([0, 5, 69, 33])
    o2, m2, l2 = oracle.prefill_rows(q, k, v, 0.3, rows)
    np.testing.assert_array_equal(o2, o[rows])
    np.testing.assert_array_equal(m2, m[:, rows])
    np.testing.assert_array_equal(l2, l[:, rows])


# ---------------------------------------------------------------------------
# window scores
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("n,h_q,h_kv,d,alpha", [(50, 4, 2, 16, 7), (33, 2, 1, 8, 33), (64, 8, 2, 16, 1)])
def test_window_scores_sum_to_alpha_times_group(n, h_q, h_kv, d, alpha):
    q, k = RNG.standard_normal((n, h_q, d)) * 1.5, RNG.standard_normal((n, h_kv, d))
    win = np.arange(n - alpha, n)
    _, m, l = oracle.prefill_rows(q, k, k, 1 / np.sqrt(d), win)
    S = oracle.window_scores(q, k, m, l, alpha, 1 / np.sqrt(d))
    # each causal softmax row sums to one: sum_i S[h][i] = alpha * G
    np.testing.assert_allclose(S.sum(axis=1), alpha * (h_q // h_kv), rtol=1e-12)
    assert (S >= 0).all()


def test_window_scores_equal_sdpa_probability_column_sums():
    n, h_q, h_kv, d, alpha = 48, 4, 2, 16, 9
    q, k = RNG.standard_normal((n, h_q, d)), RNG.standard_normal((n, h_kv, d))
    scale = 1 / np.sqrt(d)
    win = np.arange(n - alpha, n)
    _, m, l = oracle.prefill_rows(q, k, k, scale, win)
    S = oracle.window_scores(q, k, m, l, alpha, scale)
    p = _sdpa_probs(q, k)
    G = h_q // h_kv
    expect = np.stack([p[h * G:(h + 1) * G, n - alpha:, :].sum(axis=(0, 1)) for h in range(h_kv)])
    np.testing.assert_allclose(S, expect, rtol=1e-11, atol=1e-14)


def test_window_work_matches_article_estimate():
    # the article's example: n = 5000, window 256 -> ~5000*256 instead of
    # 5000*5000 (query, key) pairs.  Count the causal pairs inside the window.
    n, alpha = 5000, 256
    pairs = sum(q + 1 for q in range(n - alpha, n))
    assert pairs == alpha * n - alpha * (alpha - 1) // 2
    assert pairs <= n * alpha and pairs > 0.97 * n * alpha


# ---------------------------------------------------------------------------
# selection
# ---------------------------------------------------------------------------
def _brute_force_select(scores, n, k, r):
    cand = list(range(n - r))
    winners = []
    for sub in itertools.combinations(cand, k - r):
        rest = [i for i in cand if i not in sub]
        # every chosen key precedes every other one in (score desc, position asc)
        if all((scores[a] > scores[b]) or (scores[a] == scores[b] and a < b)
               for a in sub for b in rest):
            winners.append(sub)
    assert len(winners) == 1
    return sorted(list(winners[0]) + list(range(n - r, n)))


@pytest.mark.parametrize("trial", range(12))
def test_selection_brute_force(trial):
    n = int(RNG.integers(4, 11))
    scores = RNG.integers(0, 4, size=n).astype(np.float32)   # frequent ties
    for r in range(0, 3):
        for k in range(r, n + 2):
            got = oracle.select_kept(scores, n, k, r)
            if k >= n:
                assert got.tolist() == list(range(n))
            else:
                assert got.tolist() == _brute_force_select(scores, n, k, r)


def test_selection_all_equal_keeps_lowest_positions_and_recent():
    n, k, r = 100, 20, 5
    got = oracle.select_kept(np.ones(n, np.float32), n, k, r)
    assert got.tolist() == list(range(15)) + list(range(95, 100))


def test_selection_rejects_nan_and_oversized_recent():
    s = np.zeros(10, np.float32)
    s[3] = np.nan
    with pytest.raises(ValueError):
        oracle.select_kept(s, 10, 5, 2)
    with pytest.raises(ValueError):
        oracle.select_kept(np.zeros(10), 10, 3, 4)


# ---------------------------------------------------------------------------
# decode over the paged cache
# ---------------------------------------------------------------------------
def test_decode_full_cache_equals_dense_attention():
    """k_l >= n keeps every token, so paged decode must equal dense attention
    of each new query over prompt + appended tokens (itself included)."""
    w = tiny()
    n, steps = 37, 20
    qb, kb, vb = (bf16_bits(RNG.standard_normal(s).astype(np.float32))
                  for s in ((n, w.h_q, w.d), (n, w.h_kv, w.d), (n, w.h_kv, w.d)))
    dq, dk, dv = (bf16_bits(RNG.standard_normal(s).astype(np.float32))
                  for s in ((steps, w.h_q, w.d), (steps, w.h_kv, w.d), (steps, w.h_kv, w.d)))
    pool = oracle.BlockPool(16, free=RNG.permutation(16))
    pk = np.zeros((16, w.h_kv, 16, w.d), np.uint16)
    pv = np.zeros_like(pk)
    rec = flow.sparsify_layer(w, 1, qb, kb, vb)          # budget 64 >= n -> identity
    assert not rec.budgeted and rec.k_eff == n
    flow.place_layer(rec, pool, kb, vb, pk, pv)
    st = flow.new_stream([rec])
    allk, allv = bf16_to_f64(kb), bf16_to_f64(vb)
    for t in range(steps):
        flow.prepare_append(pool, st, 0, pk, pv)
        out = flow.append_and_attend(w, st, 0, dq[t], dk[t], dv[t], pk, pv)
        allk = np.concatenate([allk, bf16_to_f64(dk[t])[None]])
        allv = np.concatenate([allv, bf16_to_f64(dv[t])[None]])
        ref = _sdpa(bf16_to_f64(dq[t])[None], allk, allv, causal=False)[0]
        np.testing.assert_allclose(out, ref, atol=1e-12)
    assert st.lens[0] == n + steps
    assert len(st.tables[0]) == oracle.blocks_for(n + steps)


def test_copy_on_write_for_three_samples():
    w = tiny()
    n = 21                                              # partial last block
    qb, kb, vb = (bf16_bits(RNG.standard_normal(s).astype(np.float32))
                  for s in ((n, w.h_q, w.d), (n, w.h_kv, w.d), (n, w.h_kv, w.d)))
    pool = oracle.BlockPool(12)
    pk = np.zeros((12, w.h_kv, 16, w.d), np.uint16)
    pv = np.zeros_like(pk)
    rec = flow.sparsify_layer(w, 0, qb, kb, vb)
    flow.place_layer(rec, pool, kb, vb, pk, pv)
    s0 = flow.new_stream([rec])
    s1, s2 = flow.share_stream(pool, s0), flow.share_stream(pool, s0)
    assert pool.ref[s0.tables[0][1]] == 3
    copies = [flow.prepare_append(pool, s, 0, pk, pv) for s in (s0, s1, s2)]
    # the first two samples copy the shared partial block, the third writes in place
    assert copies[0] is not None and copies[1] is not None and copies[2] is None
    assert s2.tables[0][1] == rec.table[1]
    assert pool.ref[rec.table[0]] == 3                 # full prompt block still shared
    for s in (s0, s1, s2):
        np.testing.assert_array_equal(pk[s.tables[0][1], :, :5], pk[rec.table[1], :, :5])


# ---------------------------------------------------------------------------
# the generator's bf16 rounding against torch's
# ---------------------------------------------------------------------------
def test_bf16_rounding_matches_torch():
    x = np.concatenate([RNG.standard_normal(100000).astype(np.float32) * 7,
                        np.array([1.00390625, 1.01171875, -2.00781250, 0.0, -0.0], np.float32)])
    ours = bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)


# ---------------------------------------------------------------------------
# decode-time scoring and replacement (oracle/eviction.py)
# ---------------------------------------------------------------------------
def _heads(rng, h_kv, k_l, d, n_prompt):
    """k_l kept prompt tokens per head at distinct positions < n_prompt."""
    from oracle.eviction import HeadCache
    out = []
    for _ in range(h_kv):
        pos = np.sort(rng.choice(n_prompt, k_l, replace=False)).astype(np.int64)
        pos[-4:] = np.arange(n_prompt - 4, n_prompt)        # the recent prompt tokens
        out.append(HeadCache(rng.standard_normal((k_l, d)), rng.standard_normal((k_l, d)),
                             rng.uniform(0, 3, k_l), pos))
    return out


def test_eviction_step_attention_is_sdpa_over_the_cache():
    """The step's output is torch's fp64 SDPA of the query over the cache as it
    stands after the replacement (the new row in its slot, every other row
    unchanged), and its per-slot probabilities are softmax columns summed over
    the query group."""
    from oracle import eviction
    rng = np.random.default_rng(3)
    h_q, h_kv, d, k_l = 8, 2, 16, 12
    heads = _heads(rng, h_kv, k_l, d, 40)
    before = [(hc.k.copy(), hc.v.copy()) for hc in heads]
    q = rng.standard_normal((h_q, d))
    kn, vn = rng.standard_normal((h_kv, d)), rng.standard_normal((h_kv, d))
    out, probs, used = eviction.step(heads, q, kn, vn, 40, 4, 0.25)
    for h, hc in enumerate(heads):
        kb, vb = before[h]
        changed = [i for i in range(k_l) if not np.array_equal(kb[i], hc.k[i])]
        assert changed == [used[h]] and np.array_equal(hc.k[used[h]], kn[h])
        assert np.array_equal(np.delete(hc.v, used[h], 0), np.delete(vb, used[h], 0))
    kc = np.stack([hc.k for hc in heads], 1)    # [k_l, H_kv, d]
    vc = np.stack([hc.v for hc in heads], 1)
    tq = torch.from_numpy(q[:, None, :])        # [H_q, 1, d]
    tk = torch.from_numpy(kc).permute(1, 0, 2).repeat_interleave(h_q // h_kv, 0)
    tv = torch.from_numpy(vc).permute(1, 0, 2).repeat_interleave(h_q // h_kv, 0)
    ref = F.scaled_dot_product_attention(tq, tk, tv, scale=0.25)[:, 0].numpy()
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)
    sm = torch.softmax(torch.einsum("gd,gtd->gt", torch.from_numpy(q), tk) * 0.25, -1).numpy()
    np.testing.assert_allclose(probs, sm.reshape(h_kv, h_q // h_kv, k_l).sum(1), rtol=1e-12)
    np.testing.assert_allclose(probs.sum(1), h_q // h_kv, rtol=1e-12)   # softmax rows sum to 1


def test_eviction_replaces_lowest_outside_recent_window_brute_force():
    """Over a run of steps, every replaced token is (by exhaustive comparison)
    the lowest-scoring one among tokens older than the recent window, ties to
    the lower position; no token inside the window is ever replaced; scores
    grow by exactly the step's probabilities."""
    from oracle import eviction
    rng = np.random.default_rng(4)
    h_q, h_kv, d, k_l, recent = 4, 2, 8, 10, 4
    heads = _heads(rng, h_kv, k_l, d, 30)
    for h in range(h_kv):                                   # constructed ties
        heads[h].score[:3] = 0.5
    for t in range(25):
        new_pos = 30 + t
        snap = [(hc.score.copy(), hc.pos.copy()) for hc in heads]
        q = rng.standard_normal((h_q, d)) * (0.0 if t % 5 == 0 else 1.0)   # some uniform steps
        kn, vn = rng.standard_normal((h_kv, d)), rng.standard_normal((h_kv, d))
        _, probs, used = eviction.step(heads, q, kn, vn, new_pos, recent, 0.3)
        for h, hc in enumerate(heads):
            sc, ps = snap[h]
            elig = [i for i in range(k_l) if ps[i] <= new_pos - recent]
            assert all(ps[i] > new_pos - recent for i in range(k_l) if i not in elig)
            best = sorted(elig, key=lambda i: (sc[i], ps[i]))[0]
            assert used[h] == best
            assert ps[used[h]] <= new_pos - recent            # never a recent token
            expect = sc.copy()
            expect[used[h]] = 0.0
            np.testing.assert_allclose(hc.score, expect + probs[h], rtol=1e-12, atol=1e-15)
            assert hc.pos[used[h]] == new_pos
        if t % 5 == 0:                                       # q = 0: uniform attention
            np.testing.assert_allclose(probs, np.full((h_kv, k_l), (h_q // h_kv) / k_l))


def test_eviction_valid_choice_tolerance():
    from oracle.eviction import is_valid_choice
    score = np.array([1.0, 0.5, 0.5000001, 2.0])
    pos = np.array([0, 1, 2, 9])
    assert is_valid_choice(score, pos, 10, 2, 1, 1e-5)
    assert is_valid_choice(score, pos, 10, 2, 2, 1e-5)      # within the error of the lowest
    assert not is_valid_choice(score, pos, 10, 2, 0, 1e-5)
    assert not is_valid_choice(score, pos, 10, 2, 3, 1e-5)  # pos 9 > 10 - 2: recent


# ---------------------------------------------------------------------------
# FP8 (e4m3) storage of cached rows: pinned to torch's float8_e4m3fn casts and
# to the format's round-trip bound
# ---------------------------------------------------------------------------
def test_fp8_decode_matches_torch_for_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.fp8.e4m3_decode(codes)
    nan = np.isnan(ref)
    assert nan.sum() == 2 and np.array_equal(nan, np.isnan(got))
    np.testing.assert_array_equal(got[~nan], ref[~nan])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9


def test_fp8_encode_matches_torch_round_to_nearest_even():
    rng = np.random.default_rng(11)
    vals = oracle.fp8.e4m3_decode(np.arange(0x7F))
    mids = (vals[:-1] + vals[1:]) / 2            # every tie between neighbours
    rand = np.exp(rng.uniform(np.log(2.0 ** -12), np.log(448.0), 4000))
    x = np.concatenate([vals, mids, rand, np.nextafter(mids, 0), np.nextafter(mids, 1e9)])
    x = np.concatenate([x, -x]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(oracle.fp8.e4m3_encode(x), ref)


def test_fp8_encode_saturates_and_keeps_signed_zero():
    enc = oracle.fp8.e4m3_encode_one
    assert enc(448.0) == 0x7E and enc(460.0) == 0x7E and enc(1e9) == 0x7E
    assert enc(-500.0) == 0xFE
    assert enc(0.0) == 0x00 and enc(-0.0) == 0x80
    assert enc(2.0 ** -10) == 0x00        # a tie between 0 and the smallest subnormal: even


def test_fp8_row_quantisation_bounds():
    rng = np.random.default_rng(12)
    for scale in (1e-3, 0.5, 30.0):
        x = (rng.standard_normal((64, 128)) * scale).astype(np.float32)
        codes, s = oracle.fp8.quantize_rows(x)
        for i in range(x.shape[0]):
            v = oracle.fp8.dequantize_row(codes[i], s[i])
            # half a step of the format: 2^-4 relative (normals), 2^-10 s (subnormals)
            bound = np.maximum(np.abs(x[i]) * 2.0 ** -4, s[i] * 2.0 ** -10) * (1 + 1e-6)
            assert (np.abs(v - x[i]) <= bound).all()
            j = np.argmax(np.abs(x[i]))
            assert codes[i, j] & 0x7F == 0x7E            # the largest magnitude maps to 448
            assert s[i] == np.float32(np.float32(np.abs(x[i]).max()) / np.float32(448))
    codes, s = oracle.fp8.quantize_row(np.zeros(16, np.float32))
    assert (codes == 0).all() and s == 1.0


def test_fp8_vectorised_forms_match_the_scalar_ones():
    rng = np.random.default_rng(13)
    x = (rng.standard_normal((40, 128)) * np.exp(rng.uniform(-8, 6, (40, 1)))).astype(np.float32)
    x[3] = 0.0
    x[5, :7] = 1e6                                       # saturating values
    c1, s1 = oracle.fp8.quantize_rows(x)
    c2, s2 = oracle.fp8.quantize_rows_fast(x)
    np.testing.assert_array_equal(c1, c2)
    np.testing.assert_array_equal(s1, s2)
    enc1 = np.array([oracle.fp8.e4m3_encode_one(v) for v in x.ravel()[:2000]])
    np.testing.assert_array_equal(enc1, oracle.fp8.e4m3_encode(x.ravel()[:2000]))
    d1 = np.array([oracle.fp8.dequantize_row(c1[i], s1[i]) for i in range(40)])
    np.testing.assert_array_equal(d1, oracle.fp8.dequantize_rows(c1, s1))
