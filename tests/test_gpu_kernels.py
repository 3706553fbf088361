"""Per-kernel parity of the CUDA path (through the C ABI) against the CPU
oracle, on seeded inputs spanning several tiles and a ragged tail."""
import numpy as np
import pytest

import oracle
from synth import bf16_bits, bf16_to_f64, uniform_scores
from gpu_helpers import (ABS_O, ABS_S, REL_ML, REL_S, bf16_f64, check_m, check_rel, dev_bf16,
                         host_bits, kvs_lib, torch)

pytestmark = pytest.mark.gpu


def _randn_bits(rng, shape, scale=1.0):
    return bf16_bits((rng.standard_normal(shape) * scale).astype(np.float32))


# ---------------------------------------------------------------------------
# compaction and block copies: bit-exact
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("h_kv,d", [(8, 128), (2, 64)])
def test_compact_bit_exact(h_kv, d):
    kvs = kvs_lib()
    from layer_wise_kv_gb300.pipeline import _u8
    rng = np.random.default_rng(11)
    lens = [100, 37, 300, 1]
    keff = [64, 37, 201, 1]
    T = sum(lens)
    kb = _randn_bits(rng, (T, h_kv, d))
    vb = _randn_bits(rng, (T, h_kv, d))
    N = 64
    pool = oracle.BlockPool(N, free=rng.permutation(N))
    items = np.zeros(len(lens), dtype=kvs.COMPACT_ITEM)
    idx_all, tab_all = [], []
    ref_k = np.full((N, h_kv, 16, d), 0xFFFF, dtype=np.uint16)
    ref_v = ref_k.copy()
    tok = row = ioff = toff = 0
    tables = []
    for i, (n, ke) in enumerate(zip(lens, keff)):
        idx = np.stack([np.sort(rng.choice(n, ke, replace=False)) for _ in range(h_kv)])
        table = [pool.alloc() for _ in range(oracle.blocks_for(ke))]
        tables.append(table)
        oracle.compact(kb[tok:tok + n], vb[tok:tok + n], idx, table, ref_k, ref_v)
        items[i] = (tok, ioff, row, n, ke, toff, 0)
        idx_all.append(idx.reshape(-1))
        tab_all.extend(table)
        tok += n
        row += ke
        ioff += idx.size
        toff += len(table)
    k_pool = dev_bf16(np.full((N, h_kv, 16, d), 0xFFFF, dtype=np.uint16))
    v_pool = k_pool.clone()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvs.kvs_compact_blocks(dev_bf16(kb), dev_bf16(vb), _u8(items, "cuda"), len(lens), row, h_kv,
                           d, torch.from_numpy(np.concatenate(idx_all).astype(np.int32)).cuda(),
                           torch.tensor(tab_all, dtype=torch.int32).cuda(), k_pool, v_pool, N,
                           status)
    torch.cuda.synchronize()
    assert status.item() == 0
    np.testing.assert_array_equal(host_bits(k_pool), ref_k)
    np.testing.assert_array_equal(host_bits(v_pool), ref_v)

    # whole-block copies (copy-on-write payload)
    src = np.array(tables[2][:3], dtype=np.int32)
    dst = np.array([pool.alloc() for _ in range(3)], dtype=np.int32)
    kvs.kvs_copy_blocks(torch.from_numpy(src).cuda(), torch.from_numpy(dst).cuda(), 3, k_pool,
                        v_pool, N, h_kv, d, status)
    torch.cuda.synchronize()
    ref_k[dst] = ref_k[src]
    ref_v[dst] = ref_v[src]
    np.testing.assert_array_equal(host_bits(k_pool), ref_k)
    np.testing.assert_array_equal(host_bits(v_pool), ref_v)


def test_compact_flags_bad_block_id():
    kvs = kvs_lib()
    from layer_wise_kv_gb300.pipeline import _u8
    h_kv, d = 2, 64
    items = np.zeros(1, dtype=kvs.COMPACT_ITEM)
    items[0] = (0, 0, 0, 16, 16, 0, 0)
    k = dev_bf16(np.zeros((16, h_kv, d), np.uint16))
    pool = dev_bf16(np.zeros((4, h_kv, 16, d), np.uint16))
    pool2 = pool.clone()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    idx = torch.arange(16, dtype=torch.int32).repeat(h_kv).cuda()
    kvs.kvs_compact_blocks(k, k, _u8(items, "cuda"), 1, 16, h_kv, d, idx,
                           torch.tensor([7], dtype=torch.int32).cuda(), pool, pool2, 4, status)
    torch.cuda.synchronize()
    assert status.item() == kvs.KVS_ERR_INVALID
    assert int(pool.view(torch.int16).abs().sum()) == 0   # nothing written


# ---------------------------------------------------------------------------
# selection on identical fp32 scores: bit-exact
# ---------------------------------------------------------------------------
SEL_CASES = [  # (n, k, recent, levels)
    (1, 1, 0, 0), (17, 64, 16, 0), (100, 64, 16, 0), (100, 64, 16, 3), (4000, 2048, 32, 0),
    (4000, 256, 32, 7), (4001, 2048, 32, 0), (30000, 2500, 32, 0), (30000, 2500, 32, 50),
    (500, 32, 32, 0), (500, 33, 32, 1), (64, 63, 0, 2), (5000, 5000, 32, 0), (300, 1000, 16, 0),
]


def test_select_bit_exact_on_identical_scores():
    kvs = kvs_lib()
    from layer_wise_kv_gb300.pipeline import _u8
    h_kv = 3
    T = sum(c[0] for c in SEL_CASES)
    scores = np.zeros((h_kv, T), dtype=np.float32)
    items = np.zeros(len(SEL_CASES), dtype=kvs.SELECT_ITEM)
    tok = off = 0
    offs = []
    for i, (n, k, r, lv) in enumerate(SEL_CASES):
        scores[:, tok:tok + n] = uniform_scores((h_kv, n), 5, (i,), levels=lv)
        items[i] = (tok, n, k, off)
        offs.append((tok, off))
        tok += n
        off += h_kv * min(k, n)
    kept = torch.full((off,), -7, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    # recent differs per case: one launch per distinct recent value
    for r in sorted({c[2] for c in SEL_CASES}):
        sel = items.copy()
        mask = np.array([c[2] == r for c in SEL_CASES])
        kvs.kvs_select_topk(torch.from_numpy(scores).cuda(), T, _u8(sel[mask], "cuda"),
                            int(mask.sum()), h_kv, r, kept, status)
    torch.cuda.synchronize()
    assert status.item() == 0
    got = kept.cpu().numpy()
    for i, (n, k, r, lv) in enumerate(SEL_CASES):
        tok, off = offs[i]
        ke = min(k, n)
        for h in range(h_kv):
            ref = oracle.select_kept(scores[h, tok:tok + n], n, k, r)
            np.testing.assert_array_equal(got[off + h * ke: off + (h + 1) * ke], ref,
                                          err_msg=f"case {SEL_CASES[i]} head {h}")


# ---------------------------------------------------------------------------
# prefill attention with m and l
# ---------------------------------------------------------------------------
PREFILL_CASES = [  # (lens, h_q, h_kv, d)
    ([256], 4, 2, 64),                     # the tiny workload's shape
    ([1, 127, 128, 129, 300], 8, 2, 128),  # ragged varlen batch
    ([700], 8, 8, 128),                    # no grouping, several diagonal rows
    ([0, 130, 0, 1], 4, 2, 128),           # empty sequences inside the batch
]


@pytest.mark.parametrize("lens,h_q,h_kv,d", PREFILL_CASES)
def test_prefill_vs_oracle(lens, h_q, h_kv, d):
    kvs = kvs_lib()
    rng = np.random.default_rng(sum(lens) + d)
    T = sum(lens)
    qb = _randn_bits(rng, (T, h_q, d), 1.5)
    kb = _randn_bits(rng, (T, h_kv, d))
    vb = _randn_bits(rng, (T, h_kv, d))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    o = torch.empty((T, h_q, d), dtype=torch.bfloat16, device="cuda")
    m = torch.empty((h_q, T), dtype=torch.float32, device="cuda")
    l = torch.empty_like(m)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    scale = 1 / np.sqrt(d)
    kvs.kvs_prefill_attn_lse(dev_bf16(qb), dev_bf16(kb), dev_bf16(vb), o, m, l,
                             torch.from_numpy(cu).cuda(), len(lens), max(lens), T, h_q, h_kv, d,
                             scale, status)
    torch.cuda.synchronize()
    assert status.item() == 0
    go, gm, gl = bf16_f64(o), m.cpu().numpy(), l.cpu().numpy()
    for b, n in enumerate(lens):
        if n == 0:
            continue                       # an empty sequence owns no rows
        s0 = cu[b]
        ro, rm, rl = oracle.prefill_rows(bf16_to_f64(qb[s0:s0 + n]), bf16_to_f64(kb[s0:s0 + n]),
                                         bf16_to_f64(vb[s0:s0 + n]), scale)
        assert np.abs(go[s0:s0 + n] - ro).max() <= ABS_O
        check_m(gm[:, s0:s0 + n], rm)
        check_rel(gl[:, s0:s0 + n], rl, REL_ML, what="l")


@pytest.mark.parametrize("lens,h_q,h_kv,d", [([1, 127, 128, 129, 300], 8, 2, 128),
                                              ([256], 4, 2, 64)])
def test_prefill_layers_match_per_layer_launches(lens, h_q, h_kv, d):
    """kvs_prefill_attn_lse_layers over layers stacked in one buffer gives, bit
    for bit, the O, m and l that kvs_prefill_attn_lse gives layer by layer
    (whose values the test above checks against the oracle); its work items
    of all layers share one persistent grid."""
    kvs = kvs_lib()
    rng = np.random.default_rng(5 * sum(lens) + d)
    n_layers, T = 3, sum(lens)
    cu = torch.from_numpy(np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)).cuda()
    q = dev_bf16(_randn_bits(rng, (n_layers, T, h_q, d), 1.5))
    k = dev_bf16(_randn_bits(rng, (n_layers, T, h_kv, d)))
    v = dev_bf16(_randn_bits(rng, (n_layers, T, h_kv, d)))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    scale = 1 / np.sqrt(d)
    outs = []
    for one_launch in (False, True):
        o = torch.full((n_layers, T, h_q, d), float("nan"), dtype=torch.bfloat16, device="cuda")
        m = torch.full((n_layers, h_q, T), float("nan"), dtype=torch.float32, device="cuda")
        l = torch.full_like(m, float("nan"))
        if one_launch:
            kvs.kvs_prefill_attn_lse_layers(q, k, v, o, m, l, cu, len(lens), max(lens), T, h_q,
                                            h_kv, d, scale, n_layers, status)
        else:
            for li in range(n_layers):
                kvs.kvs_prefill_attn_lse(q[li], k[li], v[li], o[li], m[li], l[li], cu, len(lens),
                                         max(lens), T, h_q, h_kv, d, scale, status)
        outs.append((o, m, l))
    torch.cuda.synchronize()
    assert status.item() == 0
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a.view(torch.int32),
                           b.view(torch.int16) if b.dtype == torch.bfloat16 else b.view(torch.int32))
    assert not torch.isnan(outs[1][0]).any() and not torch.isnan(outs[1][1]).any()


# ---------------------------------------------------------------------------
# window scores, given the oracle's m and l
# ---------------------------------------------------------------------------
SCORE_CASES = [  # (lens, h_q, h_kv, d, alpha)
    ([256], 4, 2, 64, 16),
    ([300, 129, 20], 8, 2, 128, 32),       # the last sequence is shorter than alpha
    ([1000], 32, 8, 128, 32),
    ([0, 40, 0, 7], 8, 2, 64, 16),         # empty sequences; one shorter than alpha
    ([600, 200, 31], 64, 8, 128, 32),      # alpha * G = 256 columns (sixteen chunks)
    ([500, 33, 9], 12, 4, 64, 16),         # 48 columns: a width without its own kernel
    ([300, 77], 32, 2, 64, 16),            # d = 64, 256 columns
    ([129, 1000], 16, 2, 64, 16),          # d = 64, 128 columns
]


@pytest.mark.parametrize("lens,h_q,h_kv,d,alpha", SCORE_CASES)
def test_window_scores_vs_oracle(lens, h_q, h_kv, d, alpha):
    kvs = kvs_lib()
    rng = np.random.default_rng(sum(lens) * 3 + alpha)
    T = sum(lens)
    qb = _randn_bits(rng, (T, h_q, d), 1.5)
    kb = _randn_bits(rng, (T, h_kv, d))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    scale = 1 / np.sqrt(d)
    m_in = np.zeros((h_q, T), np.float32)
    l_in = np.ones((h_q, T), np.float32)
    refs = []
    for b, n in enumerate(lens):
        if n == 0:
            refs.append(None)              # an empty sequence has no keys
            continue
        s0 = cu[b]
        w = min(alpha, n)
        win = np.arange(n - w, n)
        q64, k64 = bf16_to_f64(qb[s0:s0 + n]), bf16_to_f64(kb[s0:s0 + n])
        _, mw, lw = oracle.prefill_rows(q64, k64, k64, scale, win)
        m_in[:, s0 + n - w:s0 + n] = mw
        l_in[:, s0 + n - w:s0 + n] = lw
        # the oracle sees the same fp32 m and l the kernel reads
        refs.append(oracle.window_scores(q64, k64, m_in[:, s0 + n - w:s0 + n].astype(np.float64),
                                         l_in[:, s0 + n - w:s0 + n].astype(np.float64), w, scale))
    scores = torch.full((h_kv, T), -1.0, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvs.kvs_window_scores(dev_bf16(qb), dev_bf16(kb), torch.from_numpy(m_in).cuda(),
                          torch.from_numpy(l_in).cuda(), scores, torch.from_numpy(cu).cuda(),
                          len(lens), max(lens), T, h_q, h_kv, d, alpha, scale, status)
    torch.cuda.synchronize()
    assert status.item() == 0
    got = scores.cpu().numpy().astype(np.float64)
    for b, n in enumerate(lens):
        if n == 0:
            continue
        s0 = cu[b]
        check_rel(got[:, s0:s0 + n], refs[b], REL_S, ABS_S, what=f"S seq {b}")
        w = min(alpha, n)
        np.testing.assert_allclose(got[:, s0:s0 + n].sum(axis=1), w * (h_q // h_kv), rtol=1e-4)


def test_window_scores_beyond_the_persistent_batch_limit_vs_oracle():
    """More sequences than the persistent form takes (2100 > 2048) go to the
    one-CTA-per-tile form: lengths 1..48 (many shorter than the window), a
    sample of sequences against the oracle, every sequence's total against
    alpha * G (each window row's probabilities sum to one)."""
    kvs = kvs_lib()
    rng = np.random.default_rng(2100)
    h_q, h_kv, d, alpha = 8, 2, 64, 16
    lens = [int(x) for x in rng.integers(1, 49, 2100)]
    T = sum(lens)
    qb = _randn_bits(rng, (T, h_q, d), 1.5)
    kb = _randn_bits(rng, (T, h_kv, d))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    scale = 1 / np.sqrt(d)
    m_in = np.zeros((h_q, T), np.float32)
    l_in = np.ones((h_q, T), np.float32)
    for b, n in enumerate(lens):
        s0, w = cu[b], min(alpha, n)
        q64, k64 = bf16_to_f64(qb[s0:s0 + n]), bf16_to_f64(kb[s0:s0 + n])
        _, mw, lw = oracle.prefill_rows(q64, k64, k64, scale, np.arange(n - w, n))
        m_in[:, s0 + n - w:s0 + n] = mw
        l_in[:, s0 + n - w:s0 + n] = lw
    scores = torch.full((h_kv, T), -1.0, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvs.kvs_window_scores(dev_bf16(qb), dev_bf16(kb), torch.from_numpy(m_in).cuda(),
                          torch.from_numpy(l_in).cuda(), scores, torch.from_numpy(cu).cuda(),
                          len(lens), max(lens), T, h_q, h_kv, d, alpha, scale, status)
    torch.cuda.synchronize()
    assert status.item() == 0
    got = scores.cpu().numpy().astype(np.float64)
    for b in rng.choice(len(lens), 150, replace=False):
        n, s0 = lens[b], cu[b]
        w = min(alpha, n)
        q64, k64 = bf16_to_f64(qb[s0:s0 + n]), bf16_to_f64(kb[s0:s0 + n])
        ref = oracle.window_scores(q64, k64, m_in[:, s0 + n - w:s0 + n].astype(np.float64),
                                   l_in[:, s0 + n - w:s0 + n].astype(np.float64), w, scale)
        check_rel(got[:, s0:s0 + n], ref, REL_S, ABS_S, what=f"S seq {b}")
    tot = np.add.reduceat(got, cu[:-1], axis=1)
    want = np.array([min(alpha, n) * (h_q // h_kv) for n in lens], np.float64)
    np.testing.assert_allclose(tot, np.broadcast_to(want, tot.shape), rtol=1e-4)


def test_window_scores_layers_match_per_layer_launches():
    """kvs_window_scores_layers over layers stacked in one buffer gives, bit
    for bit, what kvs_window_scores gives layer by layer (whose values the
    test above checks against the oracle): ragged sequences, one shorter than
    the window."""
    kvs = kvs_lib()
    rng = np.random.default_rng(77)
    lens, h_q, h_kv, d, alpha, n_layers = [300, 129, 20], 8, 2, 128, 32, 3
    T = sum(lens)
    cu = torch.from_numpy(np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)).cuda()
    q = dev_bf16(_randn_bits(rng, (n_layers, T, h_q, d), 1.5))
    k = dev_bf16(_randn_bits(rng, (n_layers, T, h_kv, d)))
    # any finite m and positive l exercise the same arithmetic
    m = torch.from_numpy(rng.uniform(8.0, 12.0, (n_layers, h_q, T)).astype(np.float32)).cuda()
    l = torch.from_numpy(rng.uniform(0.5, 4.0, (n_layers, h_q, T)).astype(np.float32)).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    scale = 1 / np.sqrt(d)
    one = torch.full((n_layers, h_kv, T), -1.0, dtype=torch.float32, device="cuda")
    for li in range(n_layers):
        kvs.kvs_window_scores(q[li], k[li], m[li], l[li], one[li], cu, len(lens), max(lens), T,
                              h_q, h_kv, d, alpha, scale, status)
    many = torch.full_like(one, -2.0)
    kvs.kvs_window_scores_layers(q, k, m, l, many, cu, len(lens), max(lens), T, h_q, h_kv, d,
                                 alpha, scale, n_layers, status)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert torch.equal(one, many)
    assert (one >= 0).all()


# ---------------------------------------------------------------------------
# paged decode with appends, several splits, copy-on-write blocks
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("h_q,h_kv,d", [(32, 8, 128), (4, 2, 64), (16, 1, 128), (6, 2, 128),
                                        (4, 4, 64)])
def test_paged_decode_vs_oracle(h_q, h_kv, d):
    kvs = kvs_lib()
    rng = np.random.default_rng(h_q * d)
    start_lens = [0, 1, 15, 16, 17, 255, 256, 257, 700, 1100]
    steps = 18
    n_items = len(start_lens)
    max_len = max(start_lens) + steps
    max_blocks = oracle.blocks_for(max_len)
    N = n_items * max_blocks + 8
    a = kvs.BlockAllocator(N, rng.permutation(N))
    # every slot starts as a bf16 NaN pattern; only slots below each item's
    # length hold data, so a read of an unwritten slot poisons the output
    pk = np.full((N, h_kv, 16, d), 0xFFFF, np.uint16)
    pv = pk.copy()
    tables = np.full((n_items, max_blocks), -1, np.int32)
    for i, L0 in enumerate(start_lens):
        ids = a.alloc_many(oracle.blocks_for(L0))
        tables[i, :len(ids)] = ids
        for j in range(L0):
            pk[ids[j // 16], :, j % 16] = _randn_bits(rng, (h_kv, d))
            pv[ids[j // 16], :, j % 16] = _randn_bits(rng, (h_kv, d))
    k_pool, v_pool = dev_bf16(pk), dev_bf16(pv)
    tables_d = torch.from_numpy(tables).cuda()
    lens_h = np.array(start_lens, np.int32)
    lens_d = [torch.from_numpy(lens_h.copy()).cuda(), torch.zeros(n_items, dtype=torch.int32,
                                                                  device="cuda")]
    ws_bytes = kvs.kvs_paged_decode_workspace_size(n_items, h_q, h_kv, d)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    kvs.kvs_workspace_zero(ws, ws_bytes)
    out = torch.empty((n_items, h_q, d), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    patch = np.zeros(n_items, np.int32)
    cs, cd = np.zeros(n_items, np.int32), np.zeros(n_items, np.int32)
    # host-side oracle cache: per item, the gathered rows so far
    for step in range(steps):
        a.decode_prepare(tables, lens_h, patch, cs, cd)
        q = _randn_bits(rng, (n_items, h_q, d))
        kn = _randn_bits(rng, (n_items, h_kv, d))
        vn = _randn_bits(rng, (n_items, h_kv, d))
        cur = step % 2
        if step == 5:
            # leftovers of some other call in the partial slots: every slot a
            # call reads must be one it wrote
            ws.fill_(0xAB)
        kvs.kvs_paged_decode(dev_bf16(q), dev_bf16(kn), dev_bf16(vn), k_pool, v_pool, N,
                             tables_d, max_blocks, torch.from_numpy(patch).cuda(), lens_d[cur],
                             lens_d[1 - cur], n_items, h_q, h_kv, d, 1 / np.sqrt(d), out,
                             ws, ws_bytes, status)
        torch.cuda.synchronize()
        assert status.item() == 0
        # oracle: write the new rows into the host pools through the host tables
        for i in range(n_items):
            L0 = lens_h[i]
            b = tables[i, L0 // 16]
            pk[b, :, L0 % 16] = kn[i]
            pv[b, :, L0 % 16] = vn[i]
        lens_h += 1
        np.testing.assert_array_equal(tables_d.cpu().numpy(), tables)
        np.testing.assert_array_equal(lens_d[1 - cur].cpu().numpy(), lens_h)
        got = bf16_f64(out)
        for i in range(n_items):
            L1 = lens_h[i]
            kc = np.stack([oracle.gather_rows(pk, tables[i], L1, h) for h in range(h_kv)])
            vc = np.stack([oracle.gather_rows(pv, tables[i], L1, h) for h in range(h_kv)])
            ref = oracle.decode_attention(bf16_to_f64(q[i]), bf16_to_f64(kc), bf16_to_f64(vc),
                                          1 / np.sqrt(d))
            assert np.abs(got[i] - ref).max() <= ABS_O, (step, i, np.abs(got[i] - ref).max())
    # pool bytes hold every appended row
    np.testing.assert_array_equal(host_bits(k_pool), pk)
    np.testing.assert_array_equal(host_bits(v_pool), pv)
    a.close()



def test_paged_decode_large_batch_in_chunks_vs_oracle():
    """1400 items at the Llama-3-8B head shape: their length and prefix arrays
    leave a one-launch plan a single stage per warp, so the call decodes
    consecutive chunks of items.  Two steps with appends (lengths 0 .. 70,
    block boundaries crossed); every output against the oracle, the pools
    and the next lengths exact."""
    kvs = kvs_lib()
    rng = np.random.default_rng(1400)
    h_q, h_kv, d = 32, 8, 128
    n_items, steps = 1400, 2
    start_lens = [int(x) for x in rng.integers(0, 70, n_items)]
    max_blocks = oracle.blocks_for(max(start_lens) + steps)
    N = n_items * max_blocks + 8
    a = kvs.BlockAllocator(N, rng.permutation(N))
    pk = np.full((N, h_kv, 16, d), 0xFFFF, np.uint16)
    pv = pk.copy()
    tables = np.full((n_items, max_blocks), -1, np.int32)
    for i, L0 in enumerate(start_lens):
        ids = a.alloc_many(oracle.blocks_for(L0))
        tables[i, :len(ids)] = ids
        if L0:
            rows_k = _randn_bits(rng, (L0, h_kv, d))
            rows_v = _randn_bits(rng, (L0, h_kv, d))
            for j in range(L0):
                pk[ids[j // 16], :, j % 16] = rows_k[j]
                pv[ids[j // 16], :, j % 16] = rows_v[j]
    k_pool, v_pool = dev_bf16(pk), dev_bf16(pv)
    tables_d = torch.from_numpy(tables).cuda()
    lens_h = np.array(start_lens, np.int32)
    lens_d = [torch.from_numpy(lens_h.copy()).cuda(), torch.zeros(n_items, dtype=torch.int32,
                                                                  device="cuda")]
    ws_bytes = kvs.kvs_paged_decode_workspace_size(n_items, h_q, h_kv, d)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    out = torch.empty((n_items, h_q, d), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    patch = np.zeros(n_items, np.int32)
    cs, cd = np.zeros(n_items, np.int32), np.zeros(n_items, np.int32)
    for step in range(steps):
        a.decode_prepare(tables, lens_h, patch, cs, cd)
        q = _randn_bits(rng, (n_items, h_q, d))
        kn = _randn_bits(rng, (n_items, h_kv, d))
        vn = _randn_bits(rng, (n_items, h_kv, d))
        cur = step % 2
        kvs.kvs_paged_decode(dev_bf16(q), dev_bf16(kn), dev_bf16(vn), k_pool, v_pool, N,
                             tables_d, max_blocks, torch.from_numpy(patch).cuda(), lens_d[cur],
                             lens_d[1 - cur], n_items, h_q, h_kv, d, 1 / np.sqrt(d), out,
                             ws, ws_bytes, status)
        torch.cuda.synchronize()
        assert status.item() == 0
        for i in range(n_items):
            L0 = lens_h[i]
            b = tables[i, L0 // 16]
            pk[b, :, L0 % 16] = kn[i]
            pv[b, :, L0 % 16] = vn[i]
        lens_h += 1
        np.testing.assert_array_equal(tables_d.cpu().numpy(), tables)
        np.testing.assert_array_equal(lens_d[1 - cur].cpu().numpy(), lens_h)
        got = bf16_f64(out)
        for i in range(n_items):
            L1 = lens_h[i]
            kc = np.stack([oracle.gather_rows(pk, tables[i], L1, h) for h in range(h_kv)])
            vc = np.stack([oracle.gather_rows(pv, tables[i], L1, h) for h in range(h_kv)])
            ref = oracle.decode_attention(bf16_to_f64(q[i]), bf16_to_f64(kc), bf16_to_f64(vc),
                                          1 / np.sqrt(d))
            assert np.abs(got[i] - ref).max() <= ABS_O, (step, i, np.abs(got[i] - ref).max())
    np.testing.assert_array_equal(host_bits(k_pool), pk)
    np.testing.assert_array_equal(host_bits(v_pool), pv)
    a.close()


# ---------------------------------------------------------------------------
# decode that also writes its logits and softmax denominators, and the score
# update that reads them (decode-time replacement)
# ---------------------------------------------------------------------------
def _oracle_probs(q, kc, d, scale):
    """Per query head, the softmax probabilities over the cache, from the
    oracle's decode attention with one-hot value rows: with v_j = e_(j - c*d)
    for the slots j of column chunk c (zero elsewhere), the output row is
    that chunk's probabilities."""
    h_kv, n, _ = kc.shape
    out = np.zeros((q.shape[0], n))
    for c0 in range(0, n, d):
        w = min(d, n - c0)
        vc = np.zeros((h_kv, n, d))
        vc[:, np.arange(c0, c0 + w), np.arange(w)] = 1.0
        out[:, c0:c0 + w] = oracle.decode_attention(q, kc, vc, scale)[:, :w]
    return out


@pytest.mark.parametrize("h_q,h_kv,d", [(32, 8, 128), (6, 2, 128), (4, 4, 64)])
def test_paged_decode_logits_and_score_update_vs_oracle(h_q, h_kv, d):
    """kvs_paged_decode_logits: the same output as kvs_paged_decode, bit for
    bit, and per slot exp2(logit - lse) equal to the oracle's softmax
    probability, for items short enough to be one decode piece (their
    denominators written by the decode kernel) and long enough to be split
    (written by the merge).  kvs_decode_scores_from_logits then adds the
    group's probabilities to each slot's score; an empty item is left alone."""
    kvs = kvs_lib()
    rng = np.random.default_rng(7 * h_q + d)
    lens = [1, 0, 15, 16, 17, 200, 700, 2048, 3001]
    n_items, G = len(lens), h_q // h_kv
    max_blocks = oracle.blocks_for(max(lens))
    N = n_items * max_blocks + 4
    perm = rng.permutation(N).astype(np.int32)
    pk = np.full((N, h_kv, 16, d), 0xFFFF, np.uint16)
    pv = pk.copy()
    tables = np.full((n_items, max_blocks), -1, np.int32)
    at = 0
    for i, n in enumerate(lens):
        nb = oracle.blocks_for(n)
        tables[i, :nb] = perm[at:at + nb]
        at += nb
        for j in range(n):
            pk[tables[i, j // 16], :, j % 16] = _randn_bits(rng, (h_kv, d))
            pv[tables[i, j // 16], :, j % 16] = _randn_bits(rng, (h_kv, d))
    k_pool, v_pool = dev_bf16(pk), dev_bf16(pv)
    tables_d = torch.from_numpy(tables).cuda()
    lens_d = torch.tensor(lens, dtype=torch.int32, device="cuda")
    q = _randn_bits(rng, (n_items, h_q, d), 2.0)
    scale = 1 / np.sqrt(d)
    ws_bytes = kvs.kvs_paged_decode_workspace_size(n_items, h_q, h_kv, d)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = [torch.zeros((n_items, h_q, d), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    kvs.kvs_paged_decode(dev_bf16(q), None, None, k_pool, v_pool, N, tables_d, max_blocks, None,
                         lens_d, None, n_items, h_q, h_kv, d, scale, outs[0], ws, ws_bytes, status)
    max_slots = max(lens)
    ld = (max_slots + 3) // 4 * 4
    logits = torch.full((n_items, h_kv, G, ld), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((n_items, h_q), float("nan"), dtype=torch.float32, device="cuda")
    kvs.kvs_paged_decode_logits(dev_bf16(q), None, None, k_pool, v_pool, N, tables_d, max_blocks,
                                None, lens_d, None, n_items, h_q, h_kv, d, scale, outs[1], ws,
                                ws_bytes, logits, ld, lse, status)
    score0 = rng.uniform(0.0, 3.0, (n_items, h_kv, max_slots)).astype(np.float32)
    score = torch.from_numpy(score0).cuda()
    new_pos = torch.arange(n_items, dtype=torch.int32, device="cuda")
    kvs.kvs_decode_scores_from_logits(logits, ld, lse, lens_d, score, new_pos, max_slots, n_items,
                                      h_q, h_kv, status)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert torch.equal(outs[0], outs[1])
    lg = logits.cpu().numpy().astype(np.float64)
    ls = lse.cpu().numpy().astype(np.float64)
    sc = score.cpu().numpy().astype(np.float64)
    np.testing.assert_array_equal(new_pos.cpu().numpy(), np.arange(n_items) + 1)
    for i, n in enumerate(lens):
        if n == 0:
            np.testing.assert_array_equal(sc[i], score0[i])
            continue
        kc = np.stack([oracle.gather_rows(pk, tables[i], n, h) for h in range(h_kv)])
        ref = _oracle_probs(bf16_to_f64(q[i]), bf16_to_f64(kc), d, scale)
        got = np.exp2(lg[i, :, :, :n].reshape(h_q, n) - ls[i][:, None])
        check_rel(got, ref, REL_S, ABS_S, what=f"probabilities item {i} (n={n})")
        want = score0[i].astype(np.float64)
        want[:, :n] += ref.reshape(h_kv, G, n).sum(axis=1)
        check_rel(sc[i], want, REL_S, ABS_S, what=f"scores item {i}")
