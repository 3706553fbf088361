"""FP8 (e4m3, per-row scale) KV pools: compaction and paged decode through the
C ABI against the oracle (oracle/fp8.py for the codes, the oracle's decode
attention over the values the codes stand for)."""
import numpy as np
import pytest

import oracle
from synth import bf16_bits, bf16_to_f64
from gpu_helpers import ABS_O, bf16_f64, dev_bf16, kvs_lib, torch

pytestmark = pytest.mark.gpu

D = 128


def _randn_bits(rng, shape, scale=1.0):
    return bf16_bits((rng.standard_normal(shape) * scale).astype(np.float32))


# the library's FP8 pool layout (per block and KV head), written out from its
# description: K rows token-major with the 16-byte chunks of odd rows swapped
# (chunk c at position c ^ 4), V transposed (row = element, byte = slot)
_K_CHUNKS_ODD = np.array([4, 5, 6, 7, 0, 1, 2, 3])


def k_physical(kc):
    """[..., 16, 128] codes in logical order -> the stored byte order."""
    ph = kc.copy()
    odd = kc[..., 1::2, :].reshape(kc.shape[:-2] + (8, 8, 16))
    ph[..., 1::2, :] = odd[..., _K_CHUNKS_ODD, :].reshape(odd.shape[:-2] + (128,))
    return ph


def v_physical(vc):
    """[..., 16, 128] codes -> [..., 128, 16]."""
    return np.ascontiguousarray(np.swapaxes(vc, -1, -2))


def test_pool_layout_helpers_match_the_documented_offsets():
    rng = np.random.default_rng(0)
    kc = rng.integers(0, 256, (16, D), dtype=np.uint8)
    ph = k_physical(kc).reshape(-1)
    for r in range(16):
        for e in range(D):
            off = r * 128 + (((e >> 4) ^ ((r & 1) << 2)) << 4) + (e & 15)
            assert ph[off] == kc[r, e]
    pv = v_physical(kc).reshape(-1)
    for r in range(16):
        for e in range(D):
            assert pv[e * 16 + r] == kc[r, e]


def _cuda(t):
    return torch.from_numpy(np.ascontiguousarray(t)).cuda()


@pytest.mark.parametrize("h_kv", [8, 2])
def test_compact_fp8_bit_exact(h_kv):
    """Codes and scales bit for bit against the oracle's quantiser (fp32
    divisions, round to nearest even): ragged items, partial last blocks
    (zero codes and scales past k_eff), blocks outside every table untouched."""
    kvs = kvs_lib()
    from layer_wise_kv_gb300.pipeline import _u8 as pack_items
    rng = np.random.default_rng(21 + h_kv)
    lens = [100, 37, 300, 1, 64]
    keff = [64, 37, 201, 1, 48]
    T = sum(lens)
    # rows of very different magnitudes, one all-zero row
    kb = bf16_bits((rng.standard_normal((T, h_kv, D)) *
                    np.exp(rng.uniform(-6, 4, (T, h_kv, 1)))).astype(np.float32))
    vb = _randn_bits(rng, (T, h_kv, D), 3.0)
    kb[5, 0] = 0
    N = 64
    pool = oracle.BlockPool(N, free=rng.permutation(N))
    items = np.zeros(len(lens), dtype=kvs.COMPACT_ITEM)
    ref_kc = np.full((N, h_kv, 16, D), 0xAB, np.uint8)
    ref_vc = ref_kc.copy()
    ref_ks = np.full((N, h_kv, 16), -7.0, np.float32)
    ref_vs = ref_ks.copy()
    idx_all, tab_all = [], []
    tok = row = ioff = toff = 0
    for i, (n, ke) in enumerate(zip(lens, keff)):
        idx = np.stack([np.sort(rng.choice(n, ke, replace=False)) for _ in range(h_kv)])
        if i == 0:
            idx[0, 3] = 5 - tok                          # the all-zero row is kept
        table = [pool.alloc() for _ in range(oracle.blocks_for(ke))]
        for b in table:
            ref_kc[b] = 0
            ref_vc[b] = 0
            ref_ks[b] = 0
            ref_vs[b] = 0
        for h in range(h_kv):
            rows_k = bf16_to_f64(kb[tok + idx[h], h]).astype(np.float32)
            rows_v = bf16_to_f64(vb[tok + idx[h], h]).astype(np.float32)
            ck, sk = oracle.fp8.quantize_rows_fast(rows_k)
            cv, sv = oracle.fp8.quantize_rows_fast(rows_v)
            for j in range(ke):
                b, r = table[j // 16], j % 16
                ref_kc[b, h, r], ref_ks[b, h, r] = ck[j], sk[j]
                ref_vc[b, h, r], ref_vs[b, h, r] = cv[j], sv[j]
        items[i] = (tok, ioff, row, n, ke, toff, 0)
        idx_all.append(idx.reshape(-1))
        tab_all.extend(table)
        tok += n
        row += ke
        ioff += idx.size
        toff += len(table)
    k_pool = _cuda(np.full((N, h_kv, 16 * D), 0xAB, np.uint8))
    v_pool = k_pool.clone()
    k_scale = torch.full((N, h_kv, 16), -7.0, dtype=torch.float32, device="cuda")
    v_scale = k_scale.clone()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvs.kvs_compact_blocks_fp8(dev_bf16(kb), dev_bf16(vb), pack_items(items, "cuda"), len(lens),
                               row, h_kv, D,
                               torch.from_numpy(np.concatenate(idx_all).astype(np.int32)).cuda(),
                               torch.tensor(tab_all, dtype=torch.int32).cuda(), k_pool, v_pool,
                               k_scale, v_scale, N, status)
    torch.cuda.synchronize()
    assert status.item() == 0
    used = np.zeros(N, bool)
    used[tab_all] = True
    got_k = k_pool.cpu().numpy().reshape(N, h_kv, 16, D)
    got_v = v_pool.cpu().numpy().reshape(N, h_kv, D, 16)
    np.testing.assert_array_equal(got_k[used], k_physical(ref_kc[used]))
    np.testing.assert_array_equal(got_v[used], v_physical(ref_vc[used]))
    np.testing.assert_array_equal(got_k[~used], ref_kc[~used])
    np.testing.assert_array_equal(k_scale.cpu().numpy(), ref_ks)
    np.testing.assert_array_equal(v_scale.cpu().numpy(), ref_vs)


@pytest.mark.parametrize("h_q,h_kv", [(32, 8), (6, 2), (16, 1)])
def test_paged_decode_fp8_vs_oracle(h_q, h_kv):
    """Several decode steps with appends over FP8 pools: every step's output
    against the oracle's decode attention over the stored values (codes times
    scales), the appended rows' codes and scales bit for bit against the
    oracle's quantiser, lengths and table patches as in the bf16 decode.
    Lengths 0, 1, 15, 16, 17, 255 .. 1100: empty, partial and full blocks,
    items split across warps and items that are one piece."""
    kvs = kvs_lib()
    rng = np.random.default_rng(h_q * 7 + h_kv)
    start_lens = [0, 1, 15, 16, 17, 255, 256, 257, 700, 1100]
    steps = 6
    n_items = len(start_lens)
    max_blocks = oracle.blocks_for(max(start_lens) + steps)
    N = n_items * max_blocks + 8
    a = kvs.BlockAllocator(N, rng.permutation(N))
    # logical codes (NaN patterns everywhere no row was written) and scales
    kc = np.full((N, h_kv, 16, D), 0x7F, np.uint8)
    vc = kc.copy()
    ks = np.full((N, h_kv, 16), np.nan, np.float32)
    vs = ks.copy()
    tables = np.full((n_items, max_blocks), -1, np.int32)
    for i, L0 in enumerate(start_lens):
        ids = a.alloc_many(oracle.blocks_for(L0))
        tables[i, :len(ids)] = ids
        for h in range(h_kv):
            rk = bf16_to_f64(_randn_bits(rng, (L0, D), 2.0)).astype(np.float32)
            rv = bf16_to_f64(_randn_bits(rng, (L0, D))).astype(np.float32)
            ck, sk = oracle.fp8.quantize_rows_fast(rk)
            cv, sv = oracle.fp8.quantize_rows_fast(rv)
            for j in range(L0):
                b, r = ids[j // 16], j % 16
                kc[b, h, r], ks[b, h, r], vc[b, h, r], vs[b, h, r] = ck[j], sk[j], cv[j], sv[j]
    k_pool = _cuda(k_physical(kc).reshape(N, h_kv, 16 * D))
    v_pool = _cuda(v_physical(vc).reshape(N, h_kv, 16 * D))
    k_scale, v_scale = _cuda(ks), _cuda(vs)
    tables_d = torch.from_numpy(tables).cuda()
    lens_h = np.array(start_lens, np.int32)
    lens_d = [torch.from_numpy(lens_h.copy()).cuda(),
              torch.zeros(n_items, dtype=torch.int32, device="cuda")]
    ws_bytes = kvs.kvs_paged_decode_workspace_size(n_items, h_q, h_kv, D)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    out = torch.empty((n_items, h_q, D), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    patch = np.zeros(n_items, np.int32)
    cs, cd = np.zeros(n_items, np.int32), np.zeros(n_items, np.int32)
    for step in range(steps):
        a.decode_prepare(tables, lens_h, patch, cs, cd)
        q = _randn_bits(rng, (n_items, h_q, D))
        kn = _randn_bits(rng, (n_items, h_kv, D), 2.0)
        vn = _randn_bits(rng, (n_items, h_kv, D))
        cur = step % 2
        kvs.kvs_paged_decode_fp8(dev_bf16(q), dev_bf16(kn), dev_bf16(vn), k_pool, v_pool,
                                 k_scale, v_scale, N, tables_d, max_blocks,
                                 torch.from_numpy(patch).cuda(), lens_d[cur], lens_d[1 - cur],
                                 n_items, h_q, h_kv, D, 1 / np.sqrt(D), out, ws, ws_bytes, status)
        torch.cuda.synchronize()
        assert status.item() == 0
        for i in range(n_items):
            L0 = lens_h[i]
            b, r = tables[i, L0 // 16], L0 % 16
            ck, sk = oracle.fp8.quantize_rows_fast(bf16_to_f64(kn[i]).astype(np.float32))
            cv, sv = oracle.fp8.quantize_rows_fast(bf16_to_f64(vn[i]).astype(np.float32))
            kc[b, :, r], ks[b, :, r], vc[b, :, r], vs[b, :, r] = ck, sk, cv, sv
        lens_h += 1
        np.testing.assert_array_equal(tables_d.cpu().numpy(), tables)
        np.testing.assert_array_equal(lens_d[1 - cur].cpu().numpy(), lens_h)
        kval = oracle.fp8.dequantize_rows(kc, ks)
        vval = oracle.fp8.dequantize_rows(vc, vs)
        got = bf16_f64(out)
        for i in range(n_items):
            L1 = lens_h[i]
            kk = np.stack([oracle.gather_rows(kval, tables[i], L1, h) for h in range(h_kv)])
            vv = np.stack([oracle.gather_rows(vval, tables[i], L1, h) for h in range(h_kv)])
            ref = oracle.decode_attention(bf16_to_f64(q[i]), kk, vv, 1 / np.sqrt(D))
            err = np.abs(got[i] - ref).max()
            assert err <= ABS_O, (step, i, err)
    # every written row's codes and scales, bit for bit
    used = np.isfinite(ks)
    got_k = k_pool.cpu().numpy().reshape(N, h_kv, 16, D)
    got_v = v_pool.cpu().numpy().reshape(N, h_kv, D, 16)
    exp_k, exp_v = k_physical(kc), v_physical(vc)
    for b, h, r in zip(*np.nonzero(used)):
        np.testing.assert_array_equal(got_k[b, h].reshape(-1)[r * 128:(r + 1) * 128],
                                      exp_k[b, h].reshape(-1)[r * 128:(r + 1) * 128])
        np.testing.assert_array_equal(got_v[b, h][:, r], exp_v[b, h][:, r])
    np.testing.assert_array_equal(k_scale.cpu().numpy()[used], ks[used])
    np.testing.assert_array_equal(v_scale.cpu().numpy()[used], vs[used])
    a.close()


def test_engine_fp8_prefill_and_decode_vs_oracle_flow():
    """The engine with FP8 pools, end to end: prefill + sparsify of a
    600-token prompt at the Llama-3-8B head shapes over layers 0, 30 and 31
    (one full-cache layer, two budgeted ones), the compaction into FP8 pools
    and six eager decode steps.  Tables and kept sets against the oracle's
    flow, every kept row's codes and scales bit for bit against the oracle's
    quantiser, each step's outputs against the oracle's decode attention over
    the stored values (the appended rows quantised the same way)."""
    kvs_lib()
    from layer_wise_kv_gb300.pipeline import DecodeBatch, Engine, Shape
    from oracle import flow
    from synth import decode_qkv, llama3_8b, prefill_qkv
    from gpu_helpers import check_kept
    w = llama3_8b()
    n, steps, layers = 600, 6, [0, 30, 31]
    shape = Shape(len(layers), w.h_q, w.h_kv, w.d, w.alpha, w.recent)
    N = 256
    eng = Engine(shape, N, poison=True, kv_dtype="fp8")
    host = {l: prefill_qkv(w, 0, l, n) for l in layers}
    ql, kl, vl = ([dev_bf16(host[l][i]) for l in layers] for i in range(3))
    budgets = [[w.budget(l, n) for l in layers]]
    res = eng.prefill_sparsify(ql, kl, vl, [n], budgets)
    torch.cuda.synchronize()
    eng.check_status()

    pool = oracle.BlockPool(N)
    recs, kdq, vdq = [], [], []
    got_k = eng.k_pool.cpu().numpy().reshape(N, w.h_kv, 16, D)
    got_v = eng.v_pool.cpu().numpy().reshape(N, w.h_kv, D, 16)
    got_ks, got_vs = eng.k_scale.cpu().numpy(), eng.v_scale.cpu().numpy()
    for li, l in enumerate(layers):
        qb, kb, vb = host[l]
        rec = flow.sparsify_layer(w, l, qb, kb, vb)
        off = int(res.idx_off[0, li])
        gidx = res.kept_idx[off:off + w.h_kv * rec.k_eff].cpu().numpy().reshape(w.h_kv, rec.k_eff)
        if rec.budgeted:
            for h in range(w.h_kv):
                check_kept(gidx[h], rec.idx[h], rec.scores[h], n, w.budget(l, n), w.recent)
        else:
            np.testing.assert_array_equal(gidx, rec.idx)
        rec.idx = gidx
        flow.place_layer(rec, pool, kb, vb, None, None)
        assert res.tables[0][li] == rec.table
        recs.append(rec)
        ks_l, vs_l = [], []
        for h in range(w.h_kv):
            ck, sk = oracle.fp8.quantize_rows_fast(bf16_to_f64(kb[gidx[h], h]).astype(np.float32))
            cv, sv = oracle.fp8.quantize_rows_fast(bf16_to_f64(vb[gidx[h], h]).astype(np.float32))
            for j in range(rec.k_eff):
                b, r = rec.table[j // 16], j % 16
                # the row as stored: row r of a 16-row tile (chunks swapped on odd rows)
                phys = k_physical(np.pad(ck[j:j + 1], ((r, 15 - r), (0, 0))))[r]
                np.testing.assert_array_equal(got_k[b, h, r], phys)
                np.testing.assert_array_equal(got_v[b, h][:, r], cv[j])
                assert got_ks[b, h, r] == sk[j] and got_vs[b, h, r] == sv[j]
            ks_l.append(list(oracle.fp8.dequantize_rows(ck, sk)))
            vs_l.append(list(oracle.fp8.dequantize_rows(cv, sv)))
        kdq.append(ks_l)
        vdq.append(vs_l)

    dec = DecodeBatch(eng, 1, n + steps)
    dec.set_stream(0, res.tables[0], res.k_eff[0])
    st = flow.new_stream(recs)
    dq = [decode_qkv(w, 0, l, steps) for l in layers]
    for t in range(steps):
        q = dev_bf16(np.stack([dq[li][0][t] for li in range(len(layers))]))
        k = dev_bf16(np.stack([dq[li][1][t] for li in range(len(layers))]))
        v = dev_bf16(np.stack([dq[li][2][t] for li in range(len(layers))]))
        out = bf16_f64(dec.step(q, k, v))
        for li in range(len(layers)):
            flow.prepare_append(pool, st, li)
            st.lens[li] += 1
            for h in range(w.h_kv):
                ck, sk = oracle.fp8.quantize_rows_fast(
                    bf16_to_f64(dq[li][1][t][h:h + 1]).astype(np.float32))
                cv, sv = oracle.fp8.quantize_rows_fast(
                    bf16_to_f64(dq[li][2][t][h:h + 1]).astype(np.float32))
                kdq[li][h].append(oracle.fp8.dequantize_rows(ck, sk)[0])
                vdq[li][h].append(oracle.fp8.dequantize_rows(cv, sv)[0])
            kk = np.stack([np.stack(kdq[li][h]) for h in range(w.h_kv)])
            vv = np.stack([np.stack(vdq[li][h]) for h in range(w.h_kv)])
            ref = oracle.decode_attention(bf16_to_f64(dq[li][0][t]), kk, vv, w.scale)
            err = np.abs(out[li] - ref).max()
            assert err <= ABS_O, (t, layers[li], err)
    torch.cuda.synchronize()
    eng.check_status()
    assert dec.stream_tables(0) == st.tables


def test_copy_blocks_fp8_bit_exact():
    kvs = kvs_lib()
    rng = np.random.default_rng(5)
    N, h_kv = 12, 8
    kp = rng.integers(0, 256, (N, h_kv, 16 * D), dtype=np.uint8)
    vp = rng.integers(0, 256, (N, h_kv, 16 * D), dtype=np.uint8)
    ks = rng.standard_normal((N, h_kv, 16)).astype(np.float32)
    vs = rng.standard_normal((N, h_kv, 16)).astype(np.float32)
    dev = [_cuda(x) for x in (kp, vp, ks, vs)]
    src, dst = np.array([3, 7, 0], np.int32), np.array([9, 1, 11], np.int32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvs.kvs_copy_blocks_fp8(_cuda(src), _cuda(dst), 3, *dev, N, h_kv, D, status)
    torch.cuda.synchronize()
    assert status.item() == 0
    for x in (kp, vp, ks, vs):
        x[dst] = x[src]
    for got, want in zip(dev, (kp, vp, ks, vs)):
        np.testing.assert_array_equal(got.cpu().numpy(), want)


def test_engine_fp8_shared_prefix_copy_on_write():
    """Three parallel samples share a 600-token prompt's FP8 blocks (Llama-3-8B
    head shapes, layers 0 and 31): the partial last block of the full-cache
    layer is copied, codes and scales, on the first write of samples 0 and 1;
    every sample's outputs against the oracle's attention over its own stored
    values; tables and reference counts against the oracle's allocator."""
    kvs_lib()
    from layer_wise_kv_gb300.pipeline import DecodeBatch, Engine, Shape
    from oracle import flow
    from synth import decode_qkv, llama3_8b, prefill_qkv
    w = llama3_8b()
    n, steps, layers, S = 600, 8, [0, 31], 3
    L = len(layers)
    N = 160
    eng = Engine(Shape(L, w.h_q, w.h_kv, w.d, w.alpha, w.recent), N, poison=True,
                 kv_dtype="fp8")
    host = {l: prefill_qkv(w, 0, l, n) for l in layers}
    ql, kl, vl = ([dev_bf16(host[l][i]) for l in layers] for i in range(3))
    res = eng.prefill_sparsify(ql, kl, vl, [n], [[w.budget(l, n) for l in layers]])
    torch.cuda.synchronize()
    eng.check_status()
    pool = oracle.BlockPool(N)
    recs, rows_k, rows_v = [], [], []
    for li, l in enumerate(layers):
        qb, kb, vb = host[l]
        rec = flow.sparsify_layer(w, l, qb, kb, vb)
        off = int(res.idx_off[0, li])
        rec.idx = res.kept_idx[off:off + w.h_kv * rec.k_eff].cpu().numpy().reshape(w.h_kv, -1)
        flow.place_layer(rec, pool, kb, vb, None, None)
        assert res.tables[0][li] == rec.table
        recs.append(rec)
        kq = [oracle.fp8.quantize_rows_fast(bf16_to_f64(kb[rec.idx[h], h]).astype(np.float32))
              for h in range(w.h_kv)]
        vq = [oracle.fp8.quantize_rows_fast(bf16_to_f64(vb[rec.idx[h], h]).astype(np.float32))
              for h in range(w.h_kv)]
        rows_k.append([list(oracle.fp8.dequantize_rows(*x)) for x in kq])
        rows_v.append([list(oracle.fp8.dequantize_rows(*x)) for x in vq])
    assert recs[0].k_eff % 16 != 0          # the full-cache layer ends in a partial block
    dec = DecodeBatch(eng, S, n + steps)
    streams = [flow.new_stream(recs)]
    dec.set_stream(0, res.tables[0], res.k_eff[0])
    for s in range(1, S):
        streams.append(flow.share_stream(pool, streams[0]))
        for t in res.tables[0]:
            for b in t:
                eng.alloc.incref(b)
        dec.set_stream(s, res.tables[0], res.k_eff[0])
    # per sample, per layer, per head: the stored values the sample attends over
    kval = [[[list(r) for r in rows_k[li]] for li in range(L)] for _ in range(S)]
    vval = [[[list(r) for r in rows_v[li]] for li in range(L)] for _ in range(S)]
    dq = {(s, li): decode_qkv(w, 0, l, steps, sample=s) for s in range(S)
          for li, l in enumerate(layers)}
    for t in range(steps):
        q, k, v = (dev_bf16(np.stack([dq[(s, li)][i][t] for s in range(S) for li in range(L)]))
                   for i in range(3))
        out = bf16_f64(dec.step(q, k, v))
        copies = 0
        for s in range(S):
            for li in range(L):
                copies += flow.prepare_append(pool, streams[s], li) is not None
                streams[s].lens[li] += 1
                for h in range(w.h_kv):
                    kval[s][li][h].append(oracle.fp8.dequantize_rows(*oracle.fp8.quantize_rows_fast(
                        bf16_to_f64(dq[(s, li)][1][t][h:h + 1]).astype(np.float32)))[0])
                    vval[s][li][h].append(oracle.fp8.dequantize_rows(*oracle.fp8.quantize_rows_fast(
                        bf16_to_f64(dq[(s, li)][2][t][h:h + 1]).astype(np.float32)))[0])
                kk = np.stack([np.stack(kval[s][li][h]) for h in range(w.h_kv)])
                vv = np.stack([np.stack(vval[s][li][h]) for h in range(w.h_kv)])
                ref = oracle.decode_attention(bf16_to_f64(dq[(s, li)][0][t]), kk, vv, w.scale)
                err = np.abs(out[s * L + li] - ref).max()
                assert err <= ABS_O, (t, s, layers[li], err)
        if t == 0:
            assert copies == 2
    torch.cuda.synchronize()
    eng.check_status()
    for s in range(S):
        assert dec.stream_tables(s) == streams[s].tables
    assert [eng.alloc.refcount(b) for b in range(N)] == pool.ref


class _Fp8SampleOracle:
    """The oracle's side of S samples sharing one FP8-compacted prompt: its
    allocator and streams (flow), and per sample, layer and KV head the stored
    values (dequantised e4m3 codes times row scales) the sample attends over."""

    def __init__(self, w, res, host, layers, S, N):
        from oracle import flow
        self.w, self.S, self.L = w, S, len(layers)
        self.pool = oracle.BlockPool(N)
        recs, rows_k, rows_v = [], [], []
        for li, l in enumerate(layers):
            qb, kb, vb = host[l]
            rec = flow.sparsify_layer(w, l, qb, kb, vb)
            off = int(res.idx_off[0, li])
            rec.idx = res.kept_idx[off:off + w.h_kv * rec.k_eff].cpu().numpy().reshape(w.h_kv, -1)
            flow.place_layer(rec, self.pool, kb, vb, None, None)
            assert res.tables[0][li] == rec.table
            recs.append(rec)
            for rows, x in ((rows_k, kb), (rows_v, vb)):
                rows.append([list(oracle.fp8.dequantize_rows(*oracle.fp8.quantize_rows_fast(
                    bf16_to_f64(x[rec.idx[h], h]).astype(np.float32)))) for h in range(w.h_kv)])
        self.streams = [flow.new_stream(recs)]
        self.streams += [flow.share_stream(self.pool, self.streams[0]) for _ in range(1, S)]
        self.kval = [[[list(r) for r in rows_k[li]] for li in range(self.L)] for _ in range(S)]
        self.vval = [[[list(r) for r in rows_v[li]] for li in range(self.L)] for _ in range(S)]

    def step(self, qs, ks, vs):
        """One decode step of every (sample, layer): qs[(s, li)] etc. are the
        step's bf16 rows.  Returns the expected outputs [(S * L), h_q, d]."""
        from oracle import flow
        w, outs = self.w, []
        for s in range(self.S):
            for li in range(self.L):
                flow.prepare_append(self.pool, self.streams[s], li)
                self.streams[s].lens[li] += 1
                for h in range(w.h_kv):
                    for vals, x in ((self.kval, ks), (self.vval, vs)):
                        vals[s][li][h].append(oracle.fp8.dequantize_rows(
                            *oracle.fp8.quantize_rows_fast(
                                bf16_to_f64(x[(s, li)][h:h + 1]).astype(np.float32)))[0])
                kk = np.stack([np.stack(self.kval[s][li][h]) for h in range(w.h_kv)])
                vv = np.stack([np.stack(self.vval[s][li][h]) for h in range(w.h_kv)])
                outs.append(oracle.decode_attention(bf16_to_f64(qs[(s, li)]), kk, vv, w.scale))
        return np.stack(outs)


def test_engine_fp8_graphs_match_eager():
    """DecodeBatch.capture_graphs() over FP8 pools: steps replayed from CUDA
    graphs give, bit for bit, the outputs, tables, lengths, reference counts,
    codes and scales of eager steps, and every replayed step's outputs match
    the oracle's attention over the stored values within the output
    tolerance.  Three samples share a prompt (the first step copies blocks on
    write, launched eagerly); later steps cross block boundaries (graphs that
    upload a table patch) and stay inside blocks."""
    kvs_lib()
    from layer_wise_kv_gb300.pipeline import DecodeBatch, Engine, Shape
    from synth import decode_qkv, llama3_8b, prefill_qkv
    w = llama3_8b()
    n, steps, layers, S, N = 600, 24, [0, 31], 3, 160
    L = len(layers)
    host = {l: prefill_qkv(w, 0, l, n) for l in layers}
    ql, kl, vl = ([dev_bf16(host[l][i]) for l in layers] for i in range(3))
    dq = {(s, li): decode_qkv(w, 0, l, steps, sample=s) for s in range(S)
          for li, l in enumerate(layers)}
    runs = []
    for graphs in (False, True):
        eng = Engine(Shape(L, w.h_q, w.h_kv, w.d, w.alpha, w.recent), N, poison=True,
                     kv_dtype="fp8")
        res = eng.prefill_sparsify(ql, kl, vl, [n], [[w.budget(l, n) for l in layers]])
        dec = DecodeBatch(eng, S, n + steps)
        dec.set_stream(0, res.tables[0], res.k_eff[0])
        for s in range(1, S):
            for t in res.tables[0]:
                for b in t:
                    eng.alloc.incref(b)
            dec.set_stream(s, res.tables[0], res.k_eff[0])
        if graphs:
            dec.capture_graphs()
            torch.cuda.synchronize()
            orc = _Fp8SampleOracle(w, res, host, layers, S, N)
        outs = []
        for t in range(steps):
            q, k, v = (dev_bf16(np.stack([dq[(s, li)][i][t] for s in range(S) for li in range(L)]))
                       for i in range(3))
            outs.append(dec.step(q, k, v).clone())
            if graphs:
                ref = orc.step(*({key: val[i][t] for key, val in dq.items()} for i in range(3)))
                err = np.abs(bf16_f64(outs[-1]) - ref).max()
                assert err <= ABS_O, (t, err)
        torch.cuda.synchronize()
        eng.check_status()
        runs.append((eng, dec, outs))
    (ea, da, oa), (eb, db, ob) = runs
    for t in range(steps):
        assert torch.equal(oa[t].view(torch.int16), ob[t].view(torch.int16)), t
    for s in range(S):
        assert da.stream_tables(s) == db.stream_tables(s) == orc.streams[s].tables
    assert torch.equal(da.tables_d, db.tables_d)
    assert torch.equal(da.lens_d[da.cur], db.lens_d[db.cur])
    assert [ea.alloc.refcount(b) for b in range(N)] == [eb.alloc.refcount(b) for b in range(N)] \
        == orc.pool.ref
    for x, y in ((ea.k_pool, eb.k_pool), (ea.v_pool, eb.v_pool), (ea.k_scale, eb.k_scale),
                 (ea.v_scale, eb.v_scale)):
        assert torch.equal(x.view(torch.uint8), y.view(torch.uint8))


@pytest.mark.parametrize("n,layers,N", [(600, [30, 31], 128), (4000, [3, 31], 512)])
def test_evicting_decode_fp8_vs_oracle(n, layers, N):
    """Decode-time replacement over FP8 pools at the Llama-3-8B head shapes:
    a 600-token prompt with the budgeted layers 30 and 31 (320 and 256 slots
    per KV head), and the full 4000-token prompt with layers 3 and 31 (2048
    and 256 slots); recent window 32, both items in one launch per step, 24
    steps, each step reading the rows placed by the steps before it.  Every
    step, for every KV head: the replaced slot must be a valid choice for the
    oracle's fp64 scores (the oracle then follows it); the codes and scales
    written into it must match the oracle's quantiser bit for bit; the output
    must match the oracle's attention over the stored values; scores and
    positions must track the oracle's."""
    kvs_lib()
    from layer_wise_kv_gb300.pipeline import Engine, EvictingDecode, Shape
    from oracle import eviction, flow
    from synth import decode_qkv, llama3_8b, prefill_qkv
    w = llama3_8b()
    steps = 24
    shape = Shape(len(layers), w.h_q, w.h_kv, w.d, w.alpha, w.recent)
    eng = Engine(shape, N, poison=True, kv_dtype="fp8")
    host = {l: prefill_qkv(w, 0, l, n) for l in layers}
    ql, kl, vl = ([dev_bf16(host[l][i]) for l in layers] for i in range(3))
    res = eng.prefill_sparsify(ql, kl, vl, [n], [[w.budget(l, n) for l in layers]])
    torch.cuda.synchronize()
    eng.check_status()
    heads, kes = [], []
    for li, l in enumerate(layers):
        qb, kb, vb = host[l]
        rec = flow.sparsify_layer(w, l, qb, kb, vb)
        off = int(res.idx_off[0, li])
        gidx = res.kept_idx[off:off + w.h_kv * rec.k_eff].cpu().numpy().reshape(w.h_kv, rec.k_eff)
        kes.append(rec.k_eff)
        hl = []
        for h in range(w.h_kv):
            ck, sk = oracle.fp8.quantize_rows_fast(bf16_to_f64(kb[gidx[h], h]).astype(np.float32))
            cv, sv = oracle.fp8.quantize_rows_fast(bf16_to_f64(vb[gidx[h], h]).astype(np.float32))
            hl.append(eviction.HeadCache(oracle.fp8.dequantize_rows(ck, sk),
                                         oracle.fp8.dequantize_rows(cv, sv),
                                         rec.scores[h][gidx[h]].astype(np.float64),
                                         gidx[h].astype(np.int64)))
        heads.append(hl)
    ev = EvictingDecode(eng, res, 0, 0, n, [0, 1])
    dqkv = [decode_qkv(w, 0, l, steps) for l in layers]
    for t in range(steps):
        new_pos = n + t
        q = dev_bf16(np.stack([dqkv[i][0][t] for i in range(2)]))
        k = dev_bf16(np.stack([dqkv[i][1][t] for i in range(2)]))
        v = dev_bf16(np.stack([dqkv[i][2][t] for i in range(2)]))
        out = bf16_f64(ev.step(q, k, v))
        torch.cuda.synchronize()
        got_k = eng.k_pool.cpu().numpy().reshape(N, w.h_kv, 16, D)
        got_v = eng.v_pool.cpu().numpy().reshape(N, w.h_kv, D, 16)
        got_ks, got_vs = eng.k_scale.cpu().numpy(), eng.v_scale.cpu().numpy()
        for i in range(2):
            pos_g = ev.pos[i, :, :kes[i]].cpu().numpy()
            slots, kval, vval = [], [], []
            for h, hc in enumerate(heads[i]):
                where = np.nonzero(pos_g[h] == new_pos)[0]
                assert where.size == 1, (t, i, h)
                s = int(where[0])
                assert eviction.is_valid_choice(hc.score, hc.pos, new_pos, w.recent, s, 1e-3,
                                                1e-6), (t, i, h, hc.score[s], hc.score.min())
                slots.append(s)
                ck, sk = oracle.fp8.quantize_rows_fast(
                    bf16_to_f64(dqkv[i][1][t][h:h + 1]).astype(np.float32))
                cv, sv = oracle.fp8.quantize_rows_fast(
                    bf16_to_f64(dqkv[i][2][t][h:h + 1]).astype(np.float32))
                b, r = int(ev.tables_h[i][s // 16]), s % 16
                phys = k_physical(np.pad(ck, ((r, 15 - r), (0, 0))))[r]
                np.testing.assert_array_equal(got_k[b, h, r], phys)
                np.testing.assert_array_equal(got_v[b, h][:, r], cv[0])
                assert got_ks[b, h, r] == sk[0] and got_vs[b, h, r] == sv[0], (t, i, h)
                kval.append(oracle.fp8.dequantize_rows(ck, sk)[0])
                vval.append(oracle.fp8.dequantize_rows(cv, sv)[0])
            ref, _, _ = eviction.step(heads[i], bf16_to_f64(dqkv[i][0][t]), np.stack(kval),
                                      np.stack(vval), new_pos, w.recent, w.scale, slots=slots)
            assert np.abs(out[i] - ref).max() <= ABS_O, (t, i, np.abs(out[i] - ref).max())
            sc_g = ev.score[i, :, :kes[i]].cpu().numpy().astype(np.float64)
            for h, hc in enumerate(heads[i]):
                np.testing.assert_array_equal(pos_g[h], hc.pos)
                np.testing.assert_allclose(sc_g[h], hc.score, rtol=1e-3, atol=1e-5)
    eng.check_status()
