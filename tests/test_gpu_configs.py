"""Parity at the full sizes of the serving configurations: long contexts at
more than 10x compression, continuous batching at the serving point (20
concurrent sequences, 40 in total, blocks returned to a shuffled free pool),
and a shared prefix decoded as three parallel samples with copy-on-write.

Each test runs the GPU path through the C ABI (layer_wise_kv_gb300.pipeline)
at the configuration's prompt lengths, head shapes, budgets and decode
lengths, on a subset of the 32 layers that holds both kinds (full cache and
budgeted); every layer keeps its original index, which seeds its inputs and
decides its budget.  Checked against the oracle: block tables and the pool's
free list / reference counts bit-exact, compacted bytes bit-exact, kept sets
up to swaps inside the 1e-3 score band, scores and m / l within 1e-3, prefill
and decode outputs within 2e-2 max-abs on sampled rows and steps."""
import numpy as np
import pytest

import oracle
from oracle import flow
from synth import (continuous_batching, decode_qkv, long_context, prefill_qkv, shared_prefix,
                   shuffled_block_order)
from gpu_helpers import (ABS_O, REL_ML, REL_S, ABS_S, bf16_f64, check_kept, check_m, check_rel,
                         dev_bf16, host_bits, kvs_lib, torch)

pytestmark = pytest.mark.gpu


def _engine(w, layers, num_blocks, initial_free=None):
    from layer_wise_kv_gb300.pipeline import Engine, Shape
    sh = Shape(len(layers), w.h_q, w.h_kv, w.d, w.alpha, w.recent)
    return Engine(sh, num_blocks, initial_free=initial_free, poison=True)


def _prefill_inputs(w, seqs, lens, layers, keep_host=True):
    """Device Q/K/V of the packed sequences for each listed layer (original
    layer ids), as slices of one buffer per tensor; host bits per (seq, layer)."""
    T = int(sum(lens))
    nl = len(layers)
    qd = torch.empty((nl, T, w.h_q, w.d), dtype=torch.bfloat16, device="cuda")
    kd = torch.empty((nl, T, w.h_kv, w.d), dtype=torch.bfloat16, device="cuda")
    vd = torch.empty_like(kd)
    host = {}
    for li, lo in enumerate(layers):
        tok = 0
        for s, n in zip(seqs, lens):
            qb, kb, vb = prefill_qkv(w, s, lo, n)
            if keep_host:
                host[(s, lo)] = (qb, kb, vb)
            qd[li, tok:tok + n] = dev_bf16(qb)
            kd[li, tok:tok + n] = dev_bf16(kb)
            vd[li, tok:tok + n] = dev_bf16(vb)
            tok += n
    return [qd[i] for i in range(nl)], [kd[i] for i in range(nl)], \
        [vd[i] for i in range(nl)], host


def _gpu_idx(res, b, li, h_kv, k_eff):
    off = int(res.idx_off[b, li])
    return res.kept_idx[off:off + h_kv * k_eff].cpu().numpy().reshape(h_kv, k_eff)


def _check_layer(w, res, b, li, lo, tok0, n, qb, kb, vb, rows=None):
    """Oracle sparsification of (sequence b, layer lo) against the GPU's
    outputs; returns the oracle record with the GPU's kept set (the GPU path
    selects on its own fp32 scores) and the number of band swaps."""
    rec = flow.sparsify_layer(w, lo, qb, kb, vb, rows=rows)
    swaps = 0
    if rows is not None:
        o = bf16_f64(res.o[li][tok0 + rows])
        assert np.abs(o - rec.o_rows).max() <= ABS_O, (b, lo)
        check_m(res.m[li][:, tok0 + rows].cpu().numpy(), rec.m_rows)
        check_rel(res.l[li][:, tok0 + rows].cpu().numpy(), rec.l_rows, REL_ML, what="l rows")
    gidx = _gpu_idx(res, b, li, w.h_kv, rec.k_eff)
    if rec.budgeted:
        if res.m is not None:
            win = np.arange(tok0 + n - w.alpha, tok0 + n)
            check_m(res.m[li][:, win].cpu().numpy(), rec.m_win)
            check_rel(res.l[li][:, win].cpu().numpy(), rec.l_win, REL_ML, what="l win")
        sc = res.scores[li][:, tok0:tok0 + n].cpu().numpy().astype(np.float64)
        check_rel(sc, rec.scores, REL_S, ABS_S, what=f"S seq {b} layer {lo}")
        for h in range(w.h_kv):
            swaps += check_kept(gidx[h], rec.idx[h], rec.scores[h], n, w.budget(lo, n),
                                w.recent)
    else:
        np.testing.assert_array_equal(gidx, rec.idx)
    rec.idx = gidx
    return rec, swaps


def _check_compacted(gk, gv, rec, kb, vb, h_kv):
    """The pool read back through the table equals K[idx] / V[idx], bit for bit."""
    t = np.array(rec.table, dtype=np.int64)
    j = np.arange(rec.k_eff)
    for h in range(h_kv):
        np.testing.assert_array_equal(gk[t[j // 16], h, j % 16], kb[rec.idx[h], h])
        np.testing.assert_array_equal(gv[t[j // 16], h, j % 16], vb[rec.idx[h], h])


# ---------------------------------------------------------------------------
def test_long_context_sampled():
    """Four prompts of 7000, 12000, 20000 and 30000 tokens in one packed
    prefill; layers 0-2 full, later layers keep floor(n / 12) including the 32
    most recent; 64 decode steps over every (sequence, layer) item."""
    kvs_lib()
    from layer_wise_kv_gb300.pipeline import DecodeBatch
    w = long_context()
    layers = (0, 1, 2, 3, 17, 31)
    lens = [int(x) for x in w.prompt_lens]
    B, nl, steps = len(lens), len(layers), w.decode_steps
    N = sum(oracle.blocks_for(w.k_eff(lo, n) + steps) for n in lens for lo in layers) + 64
    eng = _engine(w, layers, N)
    seqs = list(range(B))
    ql, kl, vl, host = _prefill_inputs(w, seqs, lens, layers)
    budgets = [[w.budget(lo, n) for lo in layers] for n in lens]
    res = eng.prefill_sparsify(ql, kl, vl, lens, budgets, keep_outputs=True)
    torch.cuda.synchronize()
    eng.check_status()
    assert all(w.budget(lo, n) == n // 12 for lo in layers[3:] for n in lens)

    rng = np.random.default_rng(11)
    pool = oracle.BlockPool(N)
    gk, gv = host_bits(eng.k_pool), host_bits(eng.v_pool)
    recs, swaps, tok0 = [], 0, 0
    for b, n in enumerate(lens):
        rows = np.unique(np.concatenate([np.arange(16), np.arange(n - 16, n),
                                         rng.integers(0, n, 32)]))
        per = []
        for li, lo in enumerate(layers):
            qb, kb, vb = host[(b, lo)]
            rec, sw = _check_layer(w, res, b, li, lo, tok0, n, qb, kb, vb,
                                   rows=rows if lo in (0, 17) else None)
            swaps += sw
            flow.place_layer(rec, pool, kb, vb, None, None)
            assert res.tables[b][li] == rec.table, (b, lo)
            _check_compacted(gk, gv, rec, kb, vb, w.h_kv)
            per.append(rec)
        recs.append(per)
        tok0 += n

    # decode: every step writes the new rows; outputs checked on four steps
    dec = DecodeBatch(eng, B, max(lens) + steps)
    streams = []
    for b in range(B):
        dec.set_stream(b, res.tables[b], res.k_eff[b])
        streams.append(flow.new_stream(recs[b]))
    opk, opv = gk.copy(), gv.copy()
    dq = {(b, lo): decode_qkv(w, b, lo, steps) for b in range(B) for lo in layers}
    check_steps = {0, 1, steps // 2, steps - 1}
    for t in range(steps):
        q = dev_bf16(np.stack([dq[(b, lo)][0][t] for b in range(B) for lo in layers]))
        k = dev_bf16(np.stack([dq[(b, lo)][1][t] for b in range(B) for lo in layers]))
        v = dev_bf16(np.stack([dq[(b, lo)][2][t] for b in range(B) for lo in layers]))
        out = dec.step(q, k, v)
        got = bf16_f64(out) if t in check_steps else None
        for b in range(B):
            for li, lo in enumerate(layers):
                flow.prepare_append(pool, streams[b], li, opk, opv)
                flow.append(streams[b], li, dq[(b, lo)][1][t], dq[(b, lo)][2][t], opk, opv)
                if got is not None:
                    ref = flow.attend(w, streams[b], li, dq[(b, lo)][0][t], opk, opv)
                    assert np.abs(got[b * nl + li] - ref).max() <= ABS_O, (t, b, lo)
    torch.cuda.synchronize()
    eng.check_status()
    for b in range(B):
        assert dec.stream_tables(b) == streams[b].tables
    print(f"long context: kept-set swaps within the 1e-3 band: {swaps}")


# ---------------------------------------------------------------------------
def test_continuous_batching_serving_point():
    """20 concurrent 4000-token sequences, 40 in total, output lengths drawn in
    [400, 600]; a finished sequence's blocks return to the free list (which
    starts as a seeded shuffle) and its slot is refilled at once.  Tables are
    compared at every admission, kept sets and compacted bytes of every
    admitted sequence, decode outputs of every live item on sampled steps, and
    the free list and reference counts at the end."""
    kvs_lib()
    from layer_wise_kv_gb300.pipeline import DecodeBatch
    w = continuous_batching()
    layers = (0, 3, 31)
    nl = len(layers)
    conc = w.concurrency
    prompts = [int(x) for x in w.prompt_lens]
    outs = [int(x) for x in w.out_lens]
    per_seq = max(sum(oracle.blocks_for(w.k_eff(lo, n) + o) for lo in layers)
                  for n, o in zip(prompts, outs))
    N = conc * per_seq + 64
    order = shuffled_block_order(N, 1)
    eng = _engine(w, layers, N, initial_free=order)
    pool = oracle.BlockPool(N, free=order)
    opk = np.zeros((N, w.h_kv, 16, w.d), np.uint16)
    opv = np.zeros_like(opk)
    dec = DecodeBatch(eng, conc, max(prompts) + max(outs) + 1)
    live = {}          # slot -> [seq, produced, oracle stream, decode q/k/v per layer]
    swaps = 0

    def admit(slot_seqs):
        nonlocal swaps
        seqs = [q for _, q in slot_seqs]
        lens = [prompts[q] for q in seqs]
        ql, kl, vl, host = _prefill_inputs(w, seqs, lens, layers)
        budgets = [[w.budget(lo, n) for lo in layers] for n in lens]
        res = eng.prefill_sparsify(ql, kl, vl, lens, budgets)
        torch.cuda.synchronize()
        gk, gv = host_bits(eng.k_pool), host_bits(eng.v_pool)
        tok0 = 0
        for b, (slot, q) in enumerate(slot_seqs):
            n = lens[b]
            recs = []
            for li, lo in enumerate(layers):
                qb, kb, vb = host[(q, lo)]
                rec, sw = _check_layer(w, res, b, li, lo, tok0, n, qb, kb, vb)
                swaps += sw
                flow.place_layer(rec, pool, kb, vb, None, None)
                assert res.tables[b][li] == rec.table, (q, lo)
                _check_compacted(gk, gv, rec, kb, vb, w.h_kv)
                t = np.array(rec.table, dtype=np.int64)
                opk[t], opv[t] = gk[t], gv[t]
                recs.append(rec)
            dec.set_stream(slot, res.tables[b], res.k_eff[b])
            dq = [decode_qkv(w, q, lo, outs[q]) for lo in layers]
            live[slot] = [q, 0, flow.new_stream(recs), dq]
            tok0 += n

    admit([(s, s) for s in range(conc)])       # the first 20 in one packed prefill
    nxt = conc
    step = 0
    while live:
        check = step % 97 == 0 or any(v[1] == 0 for v in live.values())
        qs, ks, vs = [], [], []
        for s in range(conc):
            for li in range(nl):
                dq, t = live[s][3][li], live[s][1]
                qs.append(dq[0][t]), ks.append(dq[1][t]), vs.append(dq[2][t])
        out = dec.step(dev_bf16(np.stack(qs)), dev_bf16(np.stack(ks)), dev_bf16(np.stack(vs)))
        got = bf16_f64(out) if check else None
        for s in sorted(live):
            q, t, st, dq = live[s]
            for li in range(nl):
                flow.prepare_append(pool, st, li, opk, opv)
                flow.append(st, li, dq[li][1][t], dq[li][2][t], opk, opv)
                if got is not None:
                    ref = flow.attend(w, st, li, dq[li][0][t], opk, opv)
                    assert np.abs(got[s * nl + li] - ref).max() <= ABS_O, (step, q, layers[li])
            live[s][1] += 1
        step += 1
        refill = []
        for s in sorted(live):
            if live[s][1] >= outs[live[s][0]]:
                flow.retire(pool, live[s][2])
                dec.retire(s)
                del live[s]
                if nxt < len(prompts):
                    refill.append((s, nxt))
                    nxt += 1
        for pair in refill:                        # one sequence per admission
            admit([pair])
        if len(live) < conc:
            break                                  # all 40 admitted; the batch drains
    torch.cuda.synchronize()
    eng.check_status()
    assert nxt == len(prompts)
    for s in sorted(live):                         # retire what is still running
        flow.retire(pool, live[s][2])
        dec.retire(s)
    assert eng.alloc.free_list() == pool.free
    assert [eng.alloc.refcount(b) for b in range(N)] == pool.ref
    print(f"continuous batching: {step} steps, kept-set swaps within the band: {swaps}")


# ---------------------------------------------------------------------------
def test_shared_prefix_three_samples():
    """16 prompts of 512 .. 16384 tokens, each compacted once and decoded as
    three parallel samples that share its blocks through reference counts; the
    partially filled last block of a layer is copied on a sample's first write
    while others still hold it.  256 decode steps per sample."""
    kvs_lib()
    from layer_wise_kv_gb300.pipeline import DecodeBatch
    w = shared_prefix()
    layers = (0, 3, 31)
    nl = len(layers)
    lens = [int(x) for x in w.prompt_lens]
    P, S, steps = len(lens), w.samples, w.decode_steps
    base_blocks = sum(oracle.blocks_for(w.k_eff(lo, n)) for n in lens for lo in layers)
    growth = sum(oracle.blocks_for(w.k_eff(lo, n) + steps) - oracle.blocks_for(w.k_eff(lo, n)) + 1
                 for n in lens for lo in layers)
    N = base_blocks + S * growth + 64
    eng = _engine(w, layers, N)
    ql, kl, vl, host = _prefill_inputs(w, list(range(P)), lens, layers)
    budgets = [[w.budget(lo, n) for lo in layers] for n in lens]
    res = eng.prefill_sparsify(ql, kl, vl, lens, budgets)
    torch.cuda.synchronize()
    eng.check_status()
    del ql, kl, vl

    pool = oracle.BlockPool(N)
    gk, gv = host_bits(eng.k_pool), host_bits(eng.v_pool)
    recs, swaps, tok0 = [], 0, 0
    for b, n in enumerate(lens):
        per = []
        for li, lo in enumerate(layers):
            qb, kb, vb = host[(b, lo)]
            rec, sw = _check_layer(w, res, b, li, lo, tok0, n, qb, kb, vb)
            swaps += sw
            flow.place_layer(rec, pool, kb, vb, None, None)
            assert res.tables[b][li] == rec.table, (b, lo)
            _check_compacted(gk, gv, rec, kb, vb, w.h_kv)
            per.append(rec)
        recs.append(per)
        tok0 += n
    host.clear()

    dec = DecodeBatch(eng, P * S, max(lens) + steps)
    streams = {}
    for b in range(P):
        streams[(b, 0)] = flow.new_stream(recs[b])
        dec.set_stream(b * S, res.tables[b], res.k_eff[b])
        for s in range(1, S):
            streams[(b, s)] = flow.share_stream(pool, streams[(b, 0)])
            for t in res.tables[b]:
                for blk in t:
                    eng.alloc.incref(blk)
            dec.set_stream(b * S + s, res.tables[b], res.k_eff[b])
    opk, opv = gk.copy(), gv.copy()
    dq = {(b, s, lo): decode_qkv(w, b, lo, steps, sample=s)
          for b in range(P) for s in range(S) for lo in layers}
    check_steps = {0, 1, steps // 2, steps - 1}
    for t in range(steps):
        order = [(b, s, lo) for b in range(P) for s in range(S) for lo in layers]
        q = dev_bf16(np.stack([dq[key][0][t] for key in order]))
        k = dev_bf16(np.stack([dq[key][1][t] for key in order]))
        v = dev_bf16(np.stack([dq[key][2][t] for key in order]))
        out = dec.step(q, k, v)
        got = bf16_f64(out) if t in check_steps else None
        copies = 0
        for i, (b, s, lo) in enumerate(order):
            li = i % nl
            st = streams[(b, s)]
            copies += flow.prepare_append(pool, st, li, opk, opv) is not None
            flow.append(st, li, dq[(b, s, lo)][1][t], dq[(b, s, lo)][2][t], opk, opv)
            if got is not None:
                ref = flow.attend(w, st, li, dq[(b, s, lo)][0][t], opk, opv)
                assert np.abs(got[i] - ref).max() <= ABS_O, (t, b, s, lo)
        if t == 0:
            partial = sum(w.k_eff(lo, n) % 16 != 0 for n in lens for lo in layers)
            assert copies == (S - 1) * partial > 0
    torch.cuda.synchronize()
    eng.check_status()
    for b in range(P):
        for s in range(S):
            assert dec.stream_tables(b * S + s) == streams[(b, s)].tables
    assert [eng.alloc.refcount(blk) for blk in range(N)] == pool.ref
    for b in range(P):
        for s in range(S):
            flow.retire(pool, streams[(b, s)])
            dec.retire(b * S + s)
    assert eng.alloc.free_list() == pool.free
    print(f"shared prefix: kept-set swaps within the band: {swaps}")
