"""End-to-end parity of the hot path (prefill attention + m/l, window scores,
selection, allocation + compaction, paged decode) against the oracle's flow,
on the seeded workloads.  The GPU path runs through the C ABI via
layer_wise_kv_gb300.pipeline; the oracle runs the same step orders on CPU."""
import numpy as np
import pytest

import oracle
from oracle import flow
from synth import (bf16_to_f64, continuous_batching, decode_qkv, llama3_8b, prefill_qkv,
                   shuffled_block_order, tiny)
from gpu_helpers import (ABS_O, REL_ML, REL_S, ABS_S, bf16_f64, check_kept, check_m, check_rel,
                         dev_bf16, host_bits, kvs_lib, torch)

pytestmark = pytest.mark.gpu


def _shape(w):
    from layer_wise_kv_gb300.pipeline import Shape
    return Shape(w.n_layers, w.h_q, w.h_kv, w.d, w.alpha, w.recent)


def _layers_to_device(w, seqs, lens, layers=None):
    """Per-layer Q/K/V of the packed sequences, as slices of one buffer each."""
    layers = list(range(w.n_layers)) if layers is None else layers
    T = sum(lens)
    qd = torch.empty((len(layers), T, w.h_q, w.d), dtype=torch.bfloat16, device="cuda")
    kd = torch.empty((len(layers), T, w.h_kv, w.d), dtype=torch.bfloat16, device="cuda")
    vd = torch.empty_like(kd)
    host = {}
    for li, l in enumerate(layers):
        tok = 0
        for s, n in zip(seqs, lens):
            qb, kb, vb = prefill_qkv(w, s, l, n)
            host[(s, l)] = (qb, kb, vb)
            qd[li, tok:tok + n] = dev_bf16(qb)
            kd[li, tok:tok + n] = dev_bf16(kb)
            vd[li, tok:tok + n] = dev_bf16(vb)
            tok += n
    return [qd[i] for i in range(len(layers))], [kd[i] for i in range(len(layers))], \
        [vd[i] for i in range(len(layers))], host


def _gpu_idx(res, b, l, h_kv, k_eff):
    off = int(res.idx_off[b, l])
    return res.kept_idx[off:off + h_kv * k_eff].cpu().numpy().reshape(h_kv, k_eff)


# ---------------------------------------------------------------------------
def test_tiny_workload_end_to_end():
    kvs_lib()
    from layer_wise_kv_gb300.pipeline import DecodeBatch, Engine
    w = tiny()
    n = w.prompt_lens[0]
    L = w.n_layers
    eng = Engine(_shape(w), 64, poison=True)
    ql, kl, vl, host = _layers_to_device(w, [0], [n])
    budgets = [[w.budget(l, n) for l in range(L)]]
    res = eng.prefill_sparsify(ql, kl, vl, [n], budgets, keep_outputs=True)
    torch.cuda.synchronize()
    eng.check_status()

    pool = oracle.BlockPool(64)
    opk = np.zeros((64, w.h_kv, 16, w.d), np.uint16)
    opv = np.zeros_like(opk)
    recs = []
    for l in range(L):
        qb, kb, vb = host[(0, l)]
        rec = flow.sparsify_layer(w, l, qb, kb, vb, rows=np.arange(n))
        recs.append(rec)
        # prefill O, m, l on every row
        assert np.abs(bf16_f64(res.o[l]) - rec.o_rows).max() <= ABS_O
        check_m(res.m[l].cpu().numpy(), rec.m_rows)
        check_rel(res.l[l].cpu().numpy(), rec.l_rows, REL_ML, what="l")
        gidx = _gpu_idx(res, 0, l, w.h_kv, rec.k_eff)
        if rec.budgeted:
            S = res.scores[l].cpu().numpy().astype(np.float64)
            check_rel(S, rec.scores, REL_S, ABS_S, what=f"S layer {l}")
            for h in range(w.h_kv):
                check_kept(gidx[h], rec.idx[h], rec.scores[h], n, w.budget(l, n), w.recent)
        else:
            np.testing.assert_array_equal(gidx, rec.idx)
        # tables: same allocator order, bit-exact
        rec.idx = gidx                               # compact what the GPU kept
        flow.place_layer(rec, pool, kb, vb, opk, opv)
        assert res.tables[0][l] == rec.table
    # compacted bytes, valid slots only
    gk, gv = host_bits(eng.k_pool), host_bits(eng.v_pool)
    for l in range(L):
        for j in range(recs[l].k_eff):
            b, s = recs[l].table[j // 16], j % 16
            np.testing.assert_array_equal(gk[b, :, s], opk[b, :, s])
            np.testing.assert_array_equal(gv[b, :, s], opv[b, :, s])

    # selection on the oracle's scores (cast to fp32): bit-exact
    sel = torch.zeros_like(res.scores)
    for l in range(L):
        if recs[l].budgeted:
            sel[l] = torch.from_numpy(recs[l].scores.astype(np.float32))
    eng2 = Engine(_shape(w), 64, poison=True)
    res2 = eng2.prefill_sparsify(ql, kl, vl, [n], budgets, select_scores=sel)
    torch.cuda.synchronize()
    for l in range(L):
        want = np.stack([oracle.select_kept(sel[l, h].cpu().numpy(), n, w.budget(l, n), w.recent)
                         for h in range(w.h_kv)]) if recs[l].budgeted else recs[l].idx
        np.testing.assert_array_equal(_gpu_idx(res2, 0, l, w.h_kv, recs[l].k_eff), want)

    # decode steps over the paged cache
    steps = w.decode_steps
    dec = DecodeBatch(eng, 1, n + steps)
    dec.set_stream(0, res.tables[0], res.k_eff[0])
    st = flow.new_stream(recs)
    dq = [decode_qkv(w, 0, l, steps) for l in range(L)]
    for t in range(steps):
        q = dev_bf16(np.stack([dq[l][0][t] for l in range(L)]))
        k = dev_bf16(np.stack([dq[l][1][t] for l in range(L)]))
        v = dev_bf16(np.stack([dq[l][2][t] for l in range(L)]))
        out = bf16_f64(dec.step(q, k, v))
        for l in range(L):
            flow.prepare_append(pool, st, l, opk, opv)
            ref = flow.append_and_attend(w, st, l, dq[l][0][t], dq[l][1][t], dq[l][2][t], opk, opv)
            assert np.abs(out[l] - ref).max() <= ABS_O, (t, l)
    torch.cuda.synchronize()
    eng.check_status()
    assert dec.stream_tables(0) == st.tables


# ---------------------------------------------------------------------------
def test_shared_prefix_copy_on_write():
    """n = 3 parallel samples share a prompt's blocks; the partial last block
    of a full-cache layer is copied on each sample's first write (the first
    two samples copy, the third writes in place)."""
    kvs_lib()
    from layer_wise_kv_gb300.pipeline import DecodeBatch, Engine
    w = tiny()
    n = 100                                  # layer 0: 100 tokens (partial block); layer 1: 64
    L = w.n_layers
    N = 64
    eng = Engine(_shape(w), N, poison=True)
    ql, kl, vl, host = _layers_to_device(w, [3], [n])
    budgets = [[w.budget(l, n) for l in range(L)]]
    res = eng.prefill_sparsify(ql, kl, vl, [n], budgets)
    torch.cuda.synchronize()
    pool = oracle.BlockPool(N)
    opk = np.zeros((N, w.h_kv, 16, w.d), np.uint16)
    opv = np.zeros_like(opk)
    recs = []
    for l in range(L):
        qb, kb, vb = host[(3, l)]
        rec = flow.sparsify_layer(w, l, qb, kb, vb)
        rec.idx = _gpu_idx(res, 0, l, w.h_kv, rec.k_eff)
        flow.place_layer(rec, pool, kb, vb, opk, opv)
        assert res.tables[0][l] == rec.table
        recs.append(rec)
    S = 3
    dec = DecodeBatch(eng, S, n + 40)
    streams = [flow.new_stream(recs)]
    dec.set_stream(0, res.tables[0], res.k_eff[0])
    for s in range(1, S):
        streams.append(flow.share_stream(pool, streams[0]))
        for t in res.tables[0]:
            for b in t:
                eng.alloc.incref(b)
        dec.set_stream(s, res.tables[0], res.k_eff[0])
    assert eng.alloc.refcount(res.tables[0][0][-1]) == 3
    steps = 20
    dq = {(s, l): decode_qkv(w, 3, l, steps, sample=s) for s in range(S) for l in range(L)}
    for t in range(steps):
        q = dev_bf16(np.stack([dq[(s, l)][0][t] for s in range(S) for l in range(L)]))
        k = dev_bf16(np.stack([dq[(s, l)][1][t] for s in range(S) for l in range(L)]))
        v = dev_bf16(np.stack([dq[(s, l)][2][t] for s in range(S) for l in range(L)]))
        out = bf16_f64(dec.step(q, k, v))
        copies = 0
        for s in range(S):
            for l in range(L):
                c = flow.prepare_append(pool, streams[s], l, opk, opv)
                copies += c is not None
                ref = flow.append_and_attend(w, streams[s], l, dq[(s, l)][0][t], dq[(s, l)][1][t],
                                             dq[(s, l)][2][t], opk, opv)
                assert np.abs(out[s * L + l] - ref).max() <= ABS_O, (t, s, l)
        if t == 0:
            assert copies == 2                        # samples 0 and 1 copy layer 0's block
    torch.cuda.synchronize()
    eng.check_status()
    for s in range(S):
        assert dec.stream_tables(s) == streams[s].tables
    assert [eng.alloc.refcount(b) for b in range(N)] == pool.ref


# ---------------------------------------------------------------------------
def test_continuous_batching_small():
    """Slots are refilled as sequences finish; finished sequences' blocks go
    back to a seed-shuffled free pool.  Tables must match the oracle's pool
    bit-exactly at every admission; outputs are checked on every step."""
    kvs_lib()
    from layer_wise_kv_gb300.pipeline import DecodeBatch, Engine
    w = tiny()
    L = w.n_layers
    N = 96
    order = shuffled_block_order(N, 1)
    eng = Engine(_shape(w), N, initial_free=order, poison=True)
    pool = oracle.BlockPool(N, free=order)
    opk = np.zeros((N, w.h_kv, 16, w.d), np.uint16)
    opv = np.zeros_like(opk)
    rng = np.random.default_rng(5)
    prompt = [int(x) for x in rng.integers(40, 140, size=5)]
    outs = [int(x) for x in rng.integers(3, 12, size=5)]
    slots = 2
    dec = DecodeBatch(eng, slots, 140 + 12)
    live = {}                                  # slot -> (seq, produced, oracle stream)

    def admit(slot, seq):
        n = prompt[seq]
        ql, kl, vl, host = _layers_to_device(w, [10 + seq], [n])
        res = eng.prefill_sparsify(ql, kl, vl, [n], [[w.budget(l, n) for l in range(L)]])
        recs = []
        for l in range(L):
            qb, kb, vb = host[(10 + seq, l)]
            rec = flow.sparsify_layer(w, l, qb, kb, vb)
            rec.idx = _gpu_idx(res, 0, l, w.h_kv, rec.k_eff)
            flow.place_layer(rec, pool, kb, vb, opk, opv)
            assert res.tables[0][l] == rec.table
            recs.append(rec)
        dec.set_stream(slot, res.tables[0], res.k_eff[0])
        live[slot] = [seq, 0, flow.new_stream(recs)]

    nxt = 0
    for s in range(slots):
        admit(s, nxt)
        nxt += 1
    step = 0
    while live:
        qs, ks, vs = [], [], []
        for s in range(slots):
            seq = live[s][0]
            for l in range(L):
                dq = decode_qkv(w, 50 + seq, l, step + 1)
                qs.append(dq[0][step]), ks.append(dq[1][step]), vs.append(dq[2][step])
        out = bf16_f64(dec.step(dev_bf16(np.stack(qs)), dev_bf16(np.stack(ks)),
                                dev_bf16(np.stack(vs))))
        for s in sorted(live):
            seq, made, st = live[s]
            for l in range(L):
                flow.prepare_append(pool, st, l, opk, opv)
                ref = flow.append_and_attend(w, st, l, qs[s * L + l], ks[s * L + l],
                                             vs[s * L + l], opk, opv)
                assert np.abs(out[s * L + l] - ref).max() <= ABS_O
            live[s][1] += 1
        step += 1
        for s in sorted(live):
            if live[s][1] >= outs[live[s][0]]:
                flow.retire(pool, live[s][2])
                dec.retire(s)
                del live[s]
                if nxt < len(prompt):
                    admit(s, nxt)
                    nxt += 1
        if len(live) < slots and nxt >= len(prompt):
            break                               # the batch drains with one slot idle
    torch.cuda.synchronize()
    eng.check_status()
    assert eng.alloc.free_list() == pool.free
    assert [eng.alloc.refcount(b) for b in range(N)] == pool.ref


# ---------------------------------------------------------------------------
def test_llama3_8b_full_size_sampled():
    """The bench's launch configuration (32 layers, 32/8 heads, d=128, one 4000
    token prompt): prefill O/m/l on sampled rows of four layers, every window
    score, the kept sets of every budgeted layer, compacted bytes of every
    layer and three decode steps over all 32 layers."""
    kvs_lib()
    from layer_wise_kv_gb300.pipeline import DecodeBatch, Engine
    w = llama3_8b()
    n = w.prompt_lens[0]
    L = w.n_layers
    N = 4096
    eng = Engine(_shape(w), N, poison=True)
    ql, kl, vl, host = _layers_to_device(w, [0], [n])
    budgets = [[w.budget(l, n) for l in range(L)]]
    res = eng.prefill_sparsify(ql, kl, vl, [n], budgets, keep_outputs=True)
    torch.cuda.synchronize()
    eng.check_status()
    rng = np.random.default_rng(8)
    rows = np.unique(np.concatenate([np.arange(128), np.arange(n - 128, n),
                                     rng.integers(0, n, 64)]))
    pool = oracle.BlockPool(N)
    swaps = 0
    recs = []
    for l in range(L):
        qb, kb, vb = host[(0, l)]
        sample = rows if l in (0, 3, 17, 31) else None
        rec = flow.sparsify_layer(w, l, qb, kb, vb, rows=sample)
        if sample is not None:
            assert np.abs(bf16_f64(res.o[l])[rows] - rec.o_rows).max() <= ABS_O
            check_m(res.m[l].cpu().numpy()[:, rows], rec.m_rows)
            check_rel(res.l[l].cpu().numpy()[:, rows], rec.l_rows, REL_ML, what="l")
        gidx = _gpu_idx(res, 0, l, w.h_kv, rec.k_eff)
        if rec.budgeted:
            check_m(res.m[l].cpu().numpy()[:, n - w.alpha:], rec.m_win)
            check_rel(res.l[l].cpu().numpy()[:, n - w.alpha:], rec.l_win, REL_ML, what="l win")
            check_rel(res.scores[l].cpu().numpy().astype(np.float64), rec.scores, REL_S, ABS_S,
                      what=f"S layer {l}")
            for h in range(w.h_kv):
                swaps += check_kept(gidx[h], rec.idx[h], rec.scores[h], n, w.budget(l, n),
                                    w.recent)
        else:
            np.testing.assert_array_equal(gidx, rec.idx)
        rec.idx = gidx
        flow.place_layer(rec, pool, kb, vb, None, None)
        assert res.tables[0][l] == rec.table
        recs.append(rec)
    # compacted bytes: gather back through the tables equals K[idx], bit for bit
    gk, gv = host_bits(eng.k_pool), host_bits(eng.v_pool)
    for l in range(L):
        _, kb, vb = host[(0, l)]
        t = np.array(recs[l].table)
        j = np.arange(recs[l].k_eff)
        for h in range(w.h_kv):
            np.testing.assert_array_equal(gk[t[j // 16], h, j % 16], kb[recs[l].idx[h], h])
            np.testing.assert_array_equal(gv[t[j // 16], h, j % 16], vb[recs[l].idx[h], h])
    # decode: three steps over all 32 layers in one launch per step
    steps = 3
    dec = DecodeBatch(eng, 1, n + w.decode_steps)
    dec.set_stream(0, res.tables[0], res.k_eff[0])
    opk, opv = gk.copy(), gv.copy()
    st = flow.new_stream(recs)
    dq = [decode_qkv(w, 0, l, steps) for l in range(L)]
    for t in range(steps):
        out = bf16_f64(dec.step(dev_bf16(np.stack([dq[l][0][t] for l in range(L)])),
                                dev_bf16(np.stack([dq[l][1][t] for l in range(L)])),
                                dev_bf16(np.stack([dq[l][2][t] for l in range(L)]))))
        for l in range(L):
            flow.prepare_append(pool, st, l, opk, opv)
            ref = flow.append_and_attend(w, st, l, dq[l][0][t], dq[l][1][t], dq[l][2][t], opk, opv)
            assert np.abs(out[l] - ref).max() <= ABS_O, (t, l)
    torch.cuda.synchronize()
    eng.check_status()
    print(f"kept-set swaps within the 1e-3 band: {swaps}")


def test_layerwise_upload_matches_resident_inputs():
    """prefill_sparsify(ready=upload_layers(...)): the prompt's Q/K/V start in
    pinned host memory and reach the device layer by layer on a copy stream
    while earlier layers compute.  Every kept index, block table entry and
    compacted pool byte equals the run on inputs already on the device."""
    kvs_lib()
    from layer_wise_kv_gb300.pipeline import Engine, upload_layers
    w = tiny()
    n = w.prompt_lens[0]
    L = w.n_layers
    budgets = [[w.budget(l, n) for l in range(L)]]
    ql, kl, vl, _ = _layers_to_device(w, [0], [n])
    eng_a = Engine(_shape(w), 64, poison=True)
    res_a = eng_a.prefill_sparsify(ql, kl, vl, [n], budgets)
    hq = [x.cpu().pin_memory() for x in ql]
    hk = [x.cpu().pin_memory() for x in kl]
    hv = [x.cpu().pin_memory() for x in vl]
    dq = [torch.full_like(x, float("nan")) for x in ql]
    dk = [torch.full_like(x, float("nan")) for x in kl]
    dv = [torch.full_like(x, float("nan")) for x in vl]
    eng_b = Engine(_shape(w), 64, poison=True)
    ready = upload_layers((hq, hk, hv), (dq, dk, dv), [torch.cuda.Stream()])
    res_b = eng_b.prefill_sparsify(dq, dk, dv, [n], budgets, ready=ready)
    torch.cuda.synchronize()
    eng_a.check_status()
    eng_b.check_status()
    assert res_a.tables == res_b.tables
    assert torch.equal(res_a.kept_idx, res_b.kept_idx)
    np.testing.assert_array_equal(host_bits(eng_a.k_pool), host_bits(eng_b.k_pool))
    np.testing.assert_array_equal(host_bits(eng_a.v_pool), host_bits(eng_b.v_pool))


def test_decode_graphs_match_eager():
    """DecodeBatch.capture_graphs(): steps replayed from CUDA graphs give, bit
    for bit, the outputs, block tables, lengths, refcounts and pool bytes of
    eager steps, and every replayed step's outputs match the oracle's flow
    (its allocator, copy-on-write and decode attention) within the output
    tolerance.  Three samples share a prompt's blocks, so the first step
    copies blocks on write (launched eagerly), and later steps cross block
    boundaries (graphs that upload a table patch) and stay inside blocks
    (graphs without one)."""
    kvs_lib()
    from layer_wise_kv_gb300.pipeline import DecodeBatch, Engine
    w = tiny()
    n, L, N, S, steps = 100, w.n_layers, 64, 3, 24
    ql, kl, vl, host = _layers_to_device(w, [3], [n])
    budgets = [[w.budget(l, n) for l in range(L)]]
    dq = {(s, l): decode_qkv(w, 3, l, steps, sample=s) for s in range(S) for l in range(L)}
    runs = []
    for graphs in (False, True):
        eng = Engine(_shape(w), N, poison=True)
        res = eng.prefill_sparsify(ql, kl, vl, [n], budgets)
        dec = DecodeBatch(eng, S, n + 40)
        dec.set_stream(0, res.tables[0], res.k_eff[0])
        for s in range(1, S):
            for t in res.tables[0]:
                for b in t:
                    eng.alloc.incref(b)
            dec.set_stream(s, res.tables[0], res.k_eff[0])
        if graphs:
            dec.capture_graphs()
            # the oracle's flow over the same kept sets: allocator, pools, streams
            torch.cuda.synchronize()
            pool = oracle.BlockPool(N)
            opk = np.zeros((N, w.h_kv, 16, w.d), np.uint16)
            opv = np.zeros_like(opk)
            recs = []
            for l in range(L):
                qb, kb, vb = host[(3, l)]
                rec = flow.sparsify_layer(w, l, qb, kb, vb)
                rec.idx = _gpu_idx(res, 0, l, w.h_kv, rec.k_eff)
                flow.place_layer(rec, pool, kb, vb, opk, opv)
                assert res.tables[0][l] == rec.table
                recs.append(rec)
            streams = [flow.new_stream(recs)]
            streams += [flow.share_stream(pool, streams[0]) for _ in range(1, S)]
        outs = []
        for t in range(steps):
            q = dev_bf16(np.stack([dq[(s, l)][0][t] for s in range(S) for l in range(L)]))
            k = dev_bf16(np.stack([dq[(s, l)][1][t] for s in range(S) for l in range(L)]))
            v = dev_bf16(np.stack([dq[(s, l)][2][t] for s in range(S) for l in range(L)]))
            outs.append(dec.step(q, k, v).clone())
            if graphs:
                got = bf16_f64(outs[-1])
                for s in range(S):
                    for l in range(L):
                        flow.prepare_append(pool, streams[s], l, opk, opv)
                        ref = flow.append_and_attend(w, streams[s], l, dq[(s, l)][0][t],
                                                     dq[(s, l)][1][t], dq[(s, l)][2][t], opk, opv)
                        assert np.abs(got[s * L + l] - ref).max() <= ABS_O, (t, s, l)
        torch.cuda.synchronize()
        eng.check_status()
        runs.append((eng, dec, outs))
    (ea, da, oa), (eb, db, ob) = runs
    for t in range(steps):
        assert torch.equal(oa[t].view(torch.int16), ob[t].view(torch.int16)), t
    for s in range(S):
        assert da.stream_tables(s) == db.stream_tables(s) == streams[s].tables
    assert torch.equal(da.tables_d, db.tables_d)
    assert torch.equal(da.lens_d[da.cur], db.lens_d[db.cur])
    assert [ea.alloc.refcount(b) for b in range(N)] == [eb.alloc.refcount(b) for b in range(N)] \
        == pool.ref
    np.testing.assert_array_equal(host_bits(ea.k_pool), host_bits(eb.k_pool))
    np.testing.assert_array_equal(host_bits(ea.v_pool), host_bits(eb.v_pool))


@pytest.mark.parametrize("mode", ["layers", "layers_graphs", "interleave"])
def test_decode_layer_order_vs_oracle(mode):
    """DecodeBatch(layer_order=True): items numbered layer-major, one host
    preparation per step, then one decode launch per layer (the launch
    sequence of a model), eager or replayed from CUDA graphs; and
    DecodeBatch(interleave=True): the same numbering with one launch over
    every item.  Three samples share a prompt's blocks, so copy-on-write
    happens on the first step.  The oracle's flow prepares the items in the
    same layer-major order: tables, reference counts and every step's outputs
    must match it."""
    kvs_lib()
    from layer_wise_kv_gb300.pipeline import DecodeBatch, Engine
    w = tiny()
    n, L, N, S, steps = 100, w.n_layers, 64, 3, 24
    ql, kl, vl, host = _layers_to_device(w, [3], [n])
    budgets = [[w.budget(l, n) for l in range(L)]]
    eng = Engine(_shape(w), N, poison=True)
    res = eng.prefill_sparsify(ql, kl, vl, [n], budgets)
    torch.cuda.synchronize()
    pool = oracle.BlockPool(N)
    opk = np.zeros((N, w.h_kv, 16, w.d), np.uint16)
    opv = np.zeros_like(opk)
    recs = []
    for l in range(L):
        qb, kb, vb = host[(3, l)]
        rec = flow.sparsify_layer(w, l, qb, kb, vb)
        rec.idx = _gpu_idx(res, 0, l, w.h_kv, rec.k_eff)
        flow.place_layer(rec, pool, kb, vb, opk, opv)
        recs.append(rec)
    dec = DecodeBatch(eng, S, n + steps + 1, layer_order=mode != "interleave",
                      interleave=mode == "interleave")
    streams = [flow.new_stream(recs)]
    dec.set_stream(0, res.tables[0], res.k_eff[0])
    for s in range(1, S):
        streams.append(flow.share_stream(pool, streams[0]))
        for t in res.tables[0]:
            for b in t:
                eng.alloc.incref(b)
        dec.set_stream(s, res.tables[0], res.k_eff[0])
    if mode == "layers_graphs":
        dec.capture_graphs()
    dq = {(s, l): decode_qkv(w, 3, l, steps, sample=s) for s in range(S) for l in range(L)}
    for t in range(steps):
        # layer-major inputs: item l * S + s
        q, k, v = (dev_bf16(np.stack([dq[(s, l)][i][t] for l in range(L) for s in range(S)]))
                   for i in range(3))
        got = bf16_f64(dec.step(q, k, v))
        for l in range(L):
            for s in range(S):
                flow.prepare_append(pool, streams[s], l, opk, opv)
        for l in range(L):
            for s in range(S):
                ref = flow.append_and_attend(w, streams[s], l, dq[(s, l)][0][t], dq[(s, l)][1][t],
                                             dq[(s, l)][2][t], opk, opv)
                assert np.abs(got[l * S + s] - ref).max() <= ABS_O, (t, s, l)
    torch.cuda.synchronize()
    eng.check_status()
    for s in range(S):
        assert dec.stream_tables(s) == streams[s].tables
    assert [eng.alloc.refcount(b) for b in range(N)] == pool.ref
    for s in range(S):
        dec.retire(s)
        flow.retire(pool, streams[s])
    assert eng.alloc.num_free() == pool.num_free()


@pytest.mark.parametrize("fused", [True, False])
def test_evicting_decode_vs_oracle(fused):
    """Decode-time replacement in the tiny workload's budgeted layer (k = 64,
    recent window 16): every step, each KV head's replaced slot must be a
    valid choice for the oracle's fp64 scores (the lowest outside the recent
    window, up to fp32 rounding; the oracle then follows it), the attention
    output must match the oracle's, and the accumulated scores and positions
    must track the oracle's through 48 steps -- long enough for decode tokens
    to age out of the window and be replaced in turn."""
    kvs_lib()
    from oracle import eviction
    from layer_wise_kv_gb300.pipeline import EvictingDecode, Engine
    w = tiny()
    n, L, layer, steps = w.prompt_lens[0], w.n_layers, 1, 48
    eng = Engine(_shape(w), 64, poison=True)
    ql, kl, vl, host = _layers_to_device(w, [0], [n])
    res = eng.prefill_sparsify(ql, kl, vl, [n], [[w.budget(l, n) for l in range(L)]])
    torch.cuda.synchronize()
    qb, kb, vb = host[(0, layer)]
    rec = flow.sparsify_layer(w, layer, qb, kb, vb)
    ke = rec.k_eff
    gidx = _gpu_idx(res, 0, layer, w.h_kv, ke)
    heads = [eviction.HeadCache(bf16_to_f64(kb[gidx[h], h]), bf16_to_f64(vb[gidx[h], h]),
                                rec.scores[h][gidx[h]].astype(np.float64),
                                gidx[h].astype(np.int64)) for h in range(w.h_kv)]
    ev = EvictingDecode(eng, res, 0, 0, n, [layer], fused=fused)
    dq, dk, dv = decode_qkv(w, 0, layer, steps)
    scale = 1 / np.sqrt(w.d)
    replaced_decode_token = False
    for t in range(steps):
        new_pos = n + t
        out = ev.step(dev_bf16(dq[t][None]), dev_bf16(dk[t][None]), dev_bf16(dv[t][None]))
        torch.cuda.synchronize()
        pos_g = ev.pos[0, :, :ke].cpu().numpy()
        slots = []
        for h, hc in enumerate(heads):
            where = np.nonzero(pos_g[h] == new_pos)[0]
            assert where.size == 1, (t, h)
            s = int(where[0])
            assert eviction.is_valid_choice(hc.score, hc.pos, new_pos, w.recent, s, 1e-3, 1e-6), \
                (t, h, s, hc.score[s], hc.score.min())
            replaced_decode_token |= hc.pos[s] >= n
            slots.append(s)
        ref, _, _ = eviction.step(heads, bf16_to_f64(dq[t]), bf16_to_f64(dk[t]), bf16_to_f64(dv[t]),
                                  new_pos, w.recent, scale, slots=slots)
        assert np.abs(bf16_f64(out)[0] - ref).max() <= ABS_O, t
        sc_g = ev.score[0, :, :ke].cpu().numpy().astype(np.float64)
        for h, hc in enumerate(heads):
            np.testing.assert_array_equal(pos_g[h], hc.pos)
            np.testing.assert_allclose(sc_g[h], hc.score, rtol=1e-3, atol=1e-5)
    eng.check_status()
    assert replaced_decode_token            # the window moved past some decode tokens
    assert int(ev.new_pos[0]) == n + steps


@pytest.mark.parametrize("fused", [True, False])
def test_evicting_decode_llama_shapes(fused):
    """The same at Llama-3-8B shapes (32/8 heads, d = 128, recent window 32,
    one 4000-token prompt) for layers 3 and 31 (budgets 2048 and 256), two
    items in one launch each step."""
    kvs_lib()
    from oracle import eviction
    from layer_wise_kv_gb300.pipeline import EvictingDecode, Engine, Shape
    w = llama3_8b()
    n, steps, real = w.prompt_lens[0], 12, [3, 31]
    shape = Shape(len(real), w.h_q, w.h_kv, w.d, w.alpha, w.recent)
    eng = Engine(shape, 512, poison=True)
    ql, kl, vl, host = _layers_to_device(w, [0], [n], layers=real)
    res = eng.prefill_sparsify(ql, kl, vl, [n], [[w.budget(l, n) for l in real]])
    torch.cuda.synchronize()
    heads, kes = [], []
    for li, l in enumerate(real):
        qb, kb, vb = host[(0, l)]
        rec = flow.sparsify_layer(w, l, qb, kb, vb)
        gidx = _gpu_idx(res, 0, li, w.h_kv, rec.k_eff)
        kes.append(rec.k_eff)
        heads.append([eviction.HeadCache(bf16_to_f64(kb[gidx[h], h]), bf16_to_f64(vb[gidx[h], h]),
                                         rec.scores[h][gidx[h]].astype(np.float64),
                                         gidx[h].astype(np.int64)) for h in range(w.h_kv)])
    ev = EvictingDecode(eng, res, 0, 0, n, [0, 1], fused=fused)
    dqkv = [decode_qkv(w, 0, l, steps) for l in real]
    scale = 1 / np.sqrt(w.d)
    for t in range(steps):
        new_pos = n + t
        q = dev_bf16(np.stack([dqkv[i][0][t] for i in range(2)]))
        k = dev_bf16(np.stack([dqkv[i][1][t] for i in range(2)]))
        v = dev_bf16(np.stack([dqkv[i][2][t] for i in range(2)]))
        out = bf16_f64(ev.step(q, k, v))
        torch.cuda.synchronize()
        for i in range(2):
            pos_g = ev.pos[i, :, :kes[i]].cpu().numpy()
            slots = []
            for h, hc in enumerate(heads[i]):
                s = int(np.nonzero(pos_g[h] == new_pos)[0][0])
                assert eviction.is_valid_choice(hc.score, hc.pos, new_pos, w.recent, s, 1e-3,
                                                1e-6), (t, i, h)
                slots.append(s)
            ref, _, _ = eviction.step(heads[i], bf16_to_f64(dqkv[i][0][t]),
                                      bf16_to_f64(dqkv[i][1][t]), bf16_to_f64(dqkv[i][2][t]),
                                      new_pos, w.recent, scale, slots=slots)
            assert np.abs(out[i] - ref).max() <= ABS_O, (t, i)
            sc_g = ev.score[i, :, :kes[i]].cpu().numpy().astype(np.float64)
            for h, hc in enumerate(heads[i]):
                np.testing.assert_array_equal(pos_g[h], hc.pos)
                np.testing.assert_allclose(sc_g[h], hc.score, rtol=1e-3, atol=1e-5)
    eng.check_status()
