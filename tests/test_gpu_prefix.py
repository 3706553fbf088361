"""Prefix blocks across requests (prompt caching by whole-block hashing; the
Ultralytics glossary "PagedAttention", section "Block sharing between
sequences", last paragraph), on the GPU path against the oracle's flow.

Request A (600 prompt tokens) is prefilled and decodes a few steps; then
request B arrives, whose first 400 prompt tokens are A's (same token ids and,
as a causal model gives them, the same K/V rows), followed by 300 tokens of
its own.  In every layer that keeps all its tokens, B's first 25 full blocks
must be A's blocks (found, not written again), with two references each; the
budgeted layer shares nothing.  Tables, reference counts, the free list and
the recorded keys must match the oracle's allocator bit for bit, the shared
blocks' bytes must still be A's rows, and A and B then decode together
against the oracle's attention.  Retiring both frees every block and
forgets every key."""
import numpy as np
import pytest

import oracle
from oracle import flow
from synth import decode_qkv, llama3_8b, prefill_qkv
from gpu_helpers import ABS_O, bf16_f64, check_kept, dev_bf16, host_bits, kvs_lib, torch

pytestmark = pytest.mark.gpu

LAYERS = (0, 3, 31)          # full cache, full (k_3 = 2048 >= n), budgeted (k_31 = 256)
N_A, N_B, SHARED = 600, 700, 400


def _prompt(w, seq, n, layers):
    return {l: prefill_qkv(w, seq, l, n) for l in layers}


def test_prefix_blocks_shared_across_requests_vs_oracle():
    kvs_lib()
    from layer_wise_kv_gb300.pipeline import DecodeBatch, Engine, Shape
    w = llama3_8b()
    L = len(LAYERS)
    rng = np.random.default_rng(5)
    tok_a = rng.integers(0, 32000, N_A)
    tok_b = np.concatenate([tok_a[:SHARED], rng.integers(0, 32000, N_B - SHARED)])
    host_a = _prompt(w, 11, N_A, LAYERS)
    host_b = _prompt(w, 12, N_B, LAYERS)
    for l in LAYERS:                              # B's first SHARED rows are A's
        host_b[l] = tuple(np.concatenate([xa[:SHARED], xb[SHARED:]])
                          for xa, xb in zip(host_a[l], host_b[l]))
    N = 400
    eng = Engine(Shape(L, w.h_q, w.h_kv, w.d, w.alpha, w.recent), N, poison=True)
    pool = oracle.BlockPool(N)
    opk = np.zeros((N, w.h_kv, 16, w.d), np.uint16)
    opv = np.zeros_like(opk)

    def prefill(host, n, toks):
        ql, kl, vl = ([dev_bf16(host[l][i]) for l in LAYERS] for i in range(3))
        res = eng.prefill_sparsify(ql, kl, vl, [n], [[w.budget(l, n) for l in LAYERS]],
                                   prefix_tokens=[toks])
        torch.cuda.synchronize()
        eng.check_status()
        recs = []
        for li, l in enumerate(LAYERS):
            qb, kb, vb = host[l]
            rec = flow.sparsify_layer(w, l, qb, kb, vb)
            off = int(res.idx_off[0, li])
            gidx = res.kept_idx[off:off + w.h_kv * rec.k_eff].cpu().numpy().reshape(w.h_kv, -1)
            if rec.budgeted:
                for h in range(w.h_kv):
                    check_kept(gidx[h], rec.idx[h], rec.scores[h], n, w.budget(l, n), w.recent)
            rec.idx = gidx
            flow.place_layer(rec, pool, kb, vb, opk, opv, layer=li, tokens=toks)
            assert res.tables[0][li] == rec.table, l
            recs.append(rec)
        return res, recs

    res_a, recs_a = prefill(host_a, N_A, tok_a)
    assert res_a.prefix_hits == 0
    dec = DecodeBatch(eng, 2, N_B + 40)
    streams = [flow.new_stream(recs_a)]
    dec.set_stream(0, res_a.tables[0], res_a.k_eff[0])
    steps = 6
    dq = {(s, li): decode_qkv(w, 11 + s, l, 2 * steps) for s in range(2)
          for li, l in enumerate(LAYERS)}

    def decode_step(t, live):
        q, k, v = (dev_bf16(np.stack([dq[(s, li)][i][t] if s in live else
                                      np.zeros_like(dq[(0, li)][i][0])
                                      for s in range(2) for li in range(L)])) for i in range(3))
        out = bf16_f64(dec.step(q, k, v))
        for s in live:
            for li in range(L):
                flow.prepare_append(pool, streams[s], li, opk, opv)
                ref = flow.append_and_attend(w, streams[s], li, dq[(s, li)][0][t],
                                             dq[(s, li)][1][t], dq[(s, li)][2][t], opk, opv)
                assert np.abs(out[s * L + li] - ref).max() <= ABS_O, (t, s, LAYERS[li])

    # A alone: the second slot has length 0 and no blocks until B arrives
    dec_a = DecodeBatch(eng, 1, N_B + 40)
    dec_a.set_stream(0, res_a.tables[0], res_a.k_eff[0])
    for t in range(steps):
        qa, ka, va = (dev_bf16(np.stack([dq[(0, li)][i][t] for li in range(L)]))
                      for i in range(3))
        out = bf16_f64(dec_a.step(qa, ka, va))
        for li in range(L):
            flow.prepare_append(pool, streams[0], li, opk, opv)
            ref = flow.append_and_attend(w, streams[0], li, dq[(0, li)][0][t], dq[(0, li)][1][t],
                                         dq[(0, li)][2][t], opk, opv)
            assert np.abs(out[li] - ref).max() <= ABS_O, (t, LAYERS[li])
    torch.cuda.synchronize()
    a_tables = dec_a.stream_tables(0)
    assert a_tables == streams[0].tables

    # B arrives while A is held
    res_b, recs_b = prefill(host_b, N_B, tok_b)
    full = [li for li in range(L) if not recs_b[li].budgeted]
    assert [LAYERS[li] for li in full] == [0, 3]
    assert res_b.prefix_hits == (SHARED // 16) * len(full)
    for li in range(L):
        shared = res_b.tables[0][li][:SHARED // 16]
        if li in full:
            assert shared == a_tables[li][:SHARED // 16]
            assert recs_b[li].hits == shared
            assert all(eng.alloc.refcount(b) == 2 for b in shared)
        else:
            assert not set(res_b.tables[0][li]) & set(a_tables[li])
    assert eng.alloc.free_list() == pool.free
    assert [eng.alloc.refcount(b) for b in range(N)] == pool.ref
    assert eng.alloc.prefix_entries() == len(pool.prefix)
    # the shared blocks still hold A's rows (B's compaction skipped them)
    gk = host_bits(eng.k_pool)
    for li in full:
        for j in range(SHARED):
            b = res_b.tables[0][li][j // 16]
            np.testing.assert_array_equal(gk[b, :, j % 16], host_a[LAYERS[li]][1][j])

    # A and B decode together (A's state moved to slot 0 of a two-stream batch)
    dec.set_stream(0, a_tables, [streams[0].lens[li] for li in range(L)])
    dec.set_stream(1, res_b.tables[0], res_b.k_eff[0])
    streams.append(flow.new_stream(recs_b))
    for t in range(steps, 2 * steps):
        decode_step(t, live=(0, 1))
    torch.cuda.synchronize()
    eng.check_status()
    for s in range(2):
        assert dec.stream_tables(s) == streams[s].tables
    assert [eng.alloc.refcount(b) for b in range(N)] == pool.ref
    for s in range(2):
        dec.retire(s)
        flow.retire(pool, streams[s])
    assert eng.alloc.num_free() == pool.num_free() == N
    assert eng.alloc.prefix_entries() == 0 and not pool.prefix
