"""The C ABI library on the host: it loads without a GPU, exports every
function include/kvs.h declares, and its block allocator (host code) agrees
with the oracle's list-based pool on the worked example and on random traces.
No compute call is made here."""
import os
import re
import shutil

import numpy as np
import pytest

import oracle
from oracle import flow
from synth import tiny

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def kvs():
    from layer_wise_kv_gb300 import kvs as k
    if shutil.which("nvcc") is not None or os.path.exists("/usr/local/cuda/bin/nvcc"):
        from layer_wise_kv_gb300 import build
        build.build()          # incremental: a no-op when the library is current
    elif not os.path.exists(k.LIB_PATH):
        pytest.skip("libkvs.so not built and nvcc unavailable")
    k.library()
    return k


def _declared():
    text = open(os.path.join(ROOT, "include", "kvs.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvs_[a-z0-9_]+)\s*\(", text)))


def test_header_symbols_exported(kvs):
    lib = kvs.library()
    names = _declared()
    assert len(names) >= 20
    for name in names:
        assert hasattr(lib, name), name
    # the binding wraps every declared function
    assert sorted(names) == sorted(kvs.exported_symbols())


def test_last_error_and_version(kvs):
    assert kvs.library().kvs_version() >= 100
    with pytest.raises(kvs.KvsError) as e:
        kvs.BlockAllocator(0)
    assert e.value.code == kvs.KVS_ERR_INVALID
    assert "num_blocks" in kvs.last_error()


def test_invalid_arguments_rejected_before_launch(kvs):
    lib = kvs.library()
    # NULL pointers and unsupported shapes return an error without touching a GPU
    assert lib.kvs_compact_blocks(None, None, None, 1, 1, 8, 128, None, None, None, None, 4,
                                  None, None) == kvs.KVS_ERR_INVALID
    rc = lib.kvs_paged_decode(1, None, None, 1, 1, 4, 1, 4, None, 1, None, 1, 8, 8, 96,
                              0.1, 1, 1, 1 << 20, None, None)
    assert rc == kvs.KVS_ERR_UNSUPPORTED and "d = 96" in kvs.last_error()
    rc = lib.kvs_paged_decode(256, None, None, 256, 256, 4, 256, 4, None, 256, None, 1, 32, 8,
                              128, 0.1, 256, 264, 1 << 20, None, None)  # workspace at 8 mod 16
    assert rc == kvs.KVS_ERR_INVALID and "workspace" in kvs.last_error()
    assert lib.kvs_window_scores(1, 1, 1, 1, 1, 1, 1, 64, 64, 32, 8, 128, 128, 0.1, None,
                                 None) == kvs.KVS_ERR_UNSUPPORTED  # alpha * G > 256
    assert lib.kvs_prefill_attn_lse(1, 1, 1, 1, 1, 1, 1, 1, 16, 16, 6, 4, 128, 0.1, None,
                                    None) == kvs.KVS_ERR_INVALID  # 6 % 4 != 0
    assert kvs.kvs_paged_decode_workspace_size(0, 32, 8, 128) == 0
    # block counts beyond 32-bit prefix sums (batch x max_blocks x h_kv >= 2^31)
    rc = lib.kvs_paged_decode(256, None, None, 256, 256, 4, 256, 1 << 20, None, 256, None, 2048,
                              32, 8, 128, 0.1, 256, 256, 1 << 40, None, None)
    assert rc == kvs.KVS_ERR_INVALID and "2^31" in kvs.last_error()
    # the allocation-free decode: 625 items at the Llama-3-8B head shapes exceed
    # its built-in array and are refused before any CUDA call
    rc = lib.kvs_paged_decode_static(None, None, None, None, None, 1, None, 1, None, None, None,
                                     625, 32, 8, 128, 0.1, None, None, None)
    assert rc == kvs.KVS_ERR_UNSUPPORTED and "built-in array" in kvs.last_error()
    # the stalled-decode test hook checks its wait limit first
    for wait_ns in (0, 2_000_000_000):
        assert lib.kvs_test_paged_decode_stalled(256, 256, 256, 4, 256, 1, 256, 1, 32, 8, 128,
                                                 0.1, 256, 256, 1 << 20, wait_ns, None,
                                                 None) == kvs.KVS_ERR_INVALID
    # the multi-layer entries: zero layers is a no-op, a negative count an error,
    # both before any launch
    assert lib.kvs_prefill_attn_lse_layers(256, 256, 256, 256, 256, 256, 256, 1, 16, 16, 8, 2,
                                           128, 0.1, 0, None, None) == kvs.KVS_OK
    assert lib.kvs_prefill_attn_lse_layers(256, 256, 256, 256, 256, 256, 256, 1, 16, 16, 8, 2,
                                           128, 0.1, -1, None, None) == kvs.KVS_ERR_INVALID
    assert lib.kvs_window_scores_layers(256, 256, 256, 256, 256, 256, 1, 16, 16, 8, 2, 128, 16,
                                        0.1, 0, None, None) == kvs.KVS_OK
    assert lib.kvs_window_scores_layers(256, 256, 256, 256, 256, 256, 1, 16, 16, 8, 2, 128, 16,
                                        0.1, -2, None, None) == kvs.KVS_ERR_INVALID
    assert lib.kvs_window_scores_layers(256, 256, 256, 256, 256, 256, 1, 16, 16, 8, 2, 128, 16,
                                        0.1, 70000, None, None) == kvs.KVS_ERR_UNSUPPORTED
    # decode-time replacement: zero items are a no-op; bad arguments fail before
    # any launch
    assert lib.kvs_evict_place(256, 256, 256, 256, 4, 256, 1, 256, 256, 256, 256, 16, 0, 8, 128,
                               32, None, None) == kvs.KVS_OK
    assert lib.kvs_evict_place(256, 256, 256, 256, 4, 256, 1, 256, 256, 256, 256, 16, 2, 8, 96,
                               32, None, None) == kvs.KVS_ERR_UNSUPPORTED
    assert lib.kvs_evict_place(None, 256, 256, 256, 4, 256, 1, 256, 256, 256, 256, 16, 2, 8, 128,
                               32, None, None) == kvs.KVS_ERR_INVALID
    assert lib.kvs_decode_scores(256, 256, 4, 256, 1, 256, 256, 256, 16, 0, 32, 8, 128, 0.1,
                                 256, 1 << 20, None, None) == kvs.KVS_OK
    assert lib.kvs_decode_scores(256, 256, 4, 256, 1, 256, 256, 256, 2048, 2, 32, 8, 128, 0.1,
                                 256, 1024, None, None) == kvs.KVS_ERR_INVALID   # workspace short
    assert lib.kvs_decode_scores(256, 256, 4, 256, 1, 256, 256, 256, 16, 2, 32, 6, 128, 0.1,
                                 256, 1 << 20, None, None) == kvs.KVS_ERR_INVALID  # 32 % 6 != 0
    assert kvs.kvs_decode_scores_workspace_size(2, 32, 8, 2048) == 2 * 8 * 4 * (2048 + 8) * 4
    # FP8 pools: d = 128 only, scales required, zero work is a no-op
    assert lib.kvs_compact_blocks_fp8(256, 256, 256, 0, 0, 8, 128, 256, 256, 256, 256, 256, 256,
                                      4, None, None) == kvs.KVS_OK
    assert lib.kvs_compact_blocks_fp8(256, 256, 256, 2, 64, 8, 64, 256, 256, 256, 256, 256, 256,
                                      4, None, None) == kvs.KVS_ERR_UNSUPPORTED
    assert lib.kvs_compact_blocks_fp8(256, 256, 256, 2, 64, 8, 128, 256, 256, 256, 256, None, 256,
                                      4, None, None) == kvs.KVS_ERR_INVALID
    assert lib.kvs_copy_blocks_fp8(256, 256, 0, 256, 256, 256, 256, 4, 8, 128, None,
                                   None) == kvs.KVS_OK
    assert lib.kvs_copy_blocks_fp8(256, 256, 2, 256, 256, None, 256, 4, 8, 128, None,
                                   None) == kvs.KVS_ERR_INVALID
    assert lib.kvs_copy_blocks_fp8(256, 256, 2, 256, 256, 256, 256, 4, 8, 64, None,
                                   None) == kvs.KVS_ERR_UNSUPPORTED
    df = [256, None, None, 256, 256, 256, 256, 4, 256, 1, None, 256, None, 2, 32, 8, 128, 0.1, 256,
          256, 1 << 26, None, None]
    df[16] = 64
    assert lib.kvs_paged_decode_fp8(*df) == kvs.KVS_ERR_UNSUPPORTED
    df[16], df[5] = 128, None
    assert lib.kvs_paged_decode_fp8(*df) == kvs.KVS_ERR_INVALID
    df[5], df[13] = 256, 0
    assert lib.kvs_paged_decode_fp8(*df) == kvs.KVS_OK
    # decode-time replacement over FP8 pools (d = 128 only; k_new / v_new 8-byte
    # aligned): placement, then the FP8 decode that writes logits and lse
    ef = [256, 256, 256, 256, 256, 256, 4, 256, 1, 256, 256, 256, 256, 16, 0, 8, 128, 32, None,
          None]
    assert lib.kvs_evict_place_fp8(*ef) == kvs.KVS_OK
    ef[14] = 2
    ef[16] = 64
    assert lib.kvs_evict_place_fp8(*ef) == kvs.KVS_ERR_UNSUPPORTED
    ef[16], ef[4] = 128, None
    assert lib.kvs_evict_place_fp8(*ef) == kvs.KVS_ERR_INVALID
    ef[4], ef[0] = 256, 260
    assert lib.kvs_evict_place_fp8(*ef) == kvs.KVS_ERR_INVALID
    dlf = [256, None, None, 256, 256, 256, 256, 4, 256, 1, None, 256, None, 0, 32, 8, 128, 0.1,
           256, 256, 1 << 26, 256, 16, 256, None, None]
    assert lib.kvs_paged_decode_logits_fp8(*dlf) == kvs.KVS_OK
    dlf[21] = None
    assert lib.kvs_paged_decode_logits_fp8(*dlf) == kvs.KVS_ERR_INVALID
    dlf[21], dlf[13], dlf[16] = 256, 2, 64
    assert lib.kvs_paged_decode_logits_fp8(*dlf) == kvs.KVS_ERR_UNSUPPORTED
    dlf[16], dlf[5] = 128, None
    assert lib.kvs_paged_decode_logits_fp8(*dlf) == kvs.KVS_ERR_INVALID
    # decode that writes its logits and denominators: both buffers are required
    dl = [256, None, None, 256, 256, 4, 256, 1, None, 256, None, 0, 32, 8, 128, 0.1, 256, 256,
          1 << 20, 256, 16, 256, None, None]
    assert lib.kvs_paged_decode_logits(*dl) == kvs.KVS_OK
    dl[21] = None
    assert lib.kvs_paged_decode_logits(*dl) == kvs.KVS_ERR_INVALID
    assert lib.kvs_decode_scores_from_logits(256, 16, 256, 256, 256, 256, 16, 0, 32, 8, None,
                                             None) == kvs.KVS_OK
    assert lib.kvs_decode_scores_from_logits(256, 16, None, 256, 256, 256, 16, 2, 32, 8, None,
                                             None) == kvs.KVS_ERR_INVALID
    assert lib.kvs_decode_scores_from_logits(256, 16, 256, 256, 256, 256, 16, 2, 32, 6, None,
                                             None) == kvs.KVS_ERR_INVALID    # 32 % 6 != 0
    assert lib.kvs_decode_scores_from_logits(256, 16, 256, 256, 256, 256, 16, 2, 64, 2, None,
                                             None) == kvs.KVS_ERR_UNSUPPORTED  # group 32 > 16
    # the native decode step: nothing to do for zero items; NULL staging and a
    # step without an append are rejected before the allocator is touched
    args = [None] * 29
    for i in (12, 14, 17, 18, 19, 20, 24):           # the integer arguments
        args[i] = 0
    args[21] = 0.0                                  # scale
    args[17] = 0                                    # n_items
    assert lib.kvs_decode_step(*args) == kvs.KVS_OK
    args[17] = 4
    assert lib.kvs_decode_step(*args) == kvs.KVS_ERR_INVALID
    # the FP8 step: the same checks, with the two scale arrays after the pools
    args8 = args[:12] + [None, None] + args[12:]
    args8[19] = 0                                   # n_items
    assert lib.kvs_decode_step_fp8(*args8) == kvs.KVS_OK
    args8[19] = 4
    assert lib.kvs_decode_step_fp8(*args8) == kvs.KVS_ERR_INVALID


def test_worked_example_allocator(kvs, golden_dir):
    import json
    g = json.load(open(os.path.join(golden_dir, "paging_worked_example.json")))
    a = kvs.BlockAllocator(g["pool_blocks"], g["free_list"])
    table = a.alloc_many(g["expected_blocks"]).tolist()
    assert table == g["expected_table"]
    assert a.free_list() == g["free_list"][len(table):]
    a.close()


def test_allocator_matches_oracle_random_trace(kvs):
    rng = np.random.default_rng(7)
    N = 50
    order = rng.permutation(N)
    a = kvs.BlockAllocator(N, order)
    o = oracle.BlockPool(N, free=order)
    owned = []
    for step in range(5000):
        op = rng.integers(0, 5)
        if op == 0:
            if o.num_free():
                b1, b2 = a.alloc(), o.alloc()
                assert b1 == b2
                owned.append(b1)
            else:
                with pytest.raises(kvs.KvsError) as e:
                    a.alloc()
                assert e.value.code == kvs.KVS_ERR_OOM_BLOCKS
        elif op == 1 and owned:
            b = owned[rng.integers(len(owned))]
            a.incref(b)
            o.incref(b)
            owned.append(b)
        elif op == 2 and owned:
            b = owned.pop(rng.integers(len(owned)))
            a.decref(b)
            o.decref(b)
        elif op == 3 and owned and o.num_free():
            i = rng.integers(len(owned))
            r1 = a.cow(owned[i])
            r2 = o.cow(owned[i])
            assert r1 == r2
            owned[i] = r1[0]
        elif op == 4:
            k = int(rng.integers(0, 4))
            if k <= o.num_free():
                got = a.alloc_many(k).tolist()
                assert got == [o.alloc() for _ in range(k)]
                owned.extend(got)
        assert a.num_free() == o.num_free()
        if step % 97 == 0:
            assert a.free_list() == o.free
            assert [a.refcount(b) for b in range(N)] == o.ref
    a.close()


def test_decode_prepare_matches_oracle_flow(kvs):
    """kvs_decode_prepare (host) against the oracle's prepare_append, with
    shared blocks so that copy-on-write happens."""
    w = tiny()
    rng = np.random.default_rng(3)
    N = 64
    a = kvs.BlockAllocator(N)
    o = oracle.BlockPool(N)
    # three streams of one layer sharing a prompt of 21 tokens (partial last block)
    prompt = [o.alloc(), o.alloc()]
    assert a.alloc_many(2).tolist() == prompt
    streams = [flow.Stream(tables=[list(prompt)], lens=[21])]
    for _ in range(2):
        streams.append(flow.share_stream(o, streams[0]))
        for b in prompt:
            a.incref(b)
    max_blocks = 8
    tables = np.full((3, max_blocks), -1, dtype=np.int32)
    tables[:, :2] = prompt
    lens = np.full(3, 21, dtype=np.int32)
    patch = np.zeros(3, dtype=np.int32)
    cs, cd = np.zeros(3, dtype=np.int32), np.zeros(3, dtype=np.int32)
    for step in range(40):
        n_cow, n_patch = a.decode_prepare(tables, lens, patch, cs, cd, with_patch_count=True)
        assert n_patch == int((patch >= 0).sum())
        copies = []
        for s in streams:
            c = flow.prepare_append(o, s, 0)
            copies.append(c)
            s.lens[0] += 1
        exp_pairs = [c for c in copies if c is not None]
        assert n_cow == len(exp_pairs)
        assert list(zip(cs[:n_cow].tolist(), cd[:n_cow].tolist())) == exp_pairs
        for i, s in enumerate(streams):
            assert tables[i, :len(s.tables[0])].tolist() == s.tables[0]
        lens += 1
        assert [a.refcount(b) for b in range(N)] == o.ref
    assert step == 39
    a.close()


@pytest.mark.parametrize("seed", range(4))
def test_prefix_blocks_match_the_oracle(kvs, seed):
    """kvs_alloc_prefix_blocks against the oracle's prefix blocks over a random
    trace of requests (shared prefixes, several layers, retirements): the same
    blocks, hits, counts, free list order and number of recorded keys at every
    step."""
    rng = np.random.default_rng(100 + seed)
    N = 3000
    free = rng.permutation(N).astype(np.int32)
    a = kvs.BlockAllocator(N, free)
    pool = oracle.BlockPool(N, free=free)
    root = rng.integers(0, 3, 300)
    reqs, held = [], {}
    for r in range(50):
        if held and rng.random() < 0.4:
            victim = list(held)[rng.integers(len(held))]
            for b in held.pop(victim):
                a.decref(b)
                pool.decref(b)
        src = reqs[rng.integers(len(reqs))] if reqs and rng.random() < 0.7 else root
        toks = np.concatenate([src[:rng.integers(0, len(src) + 1)],
                               rng.integers(0, 3, rng.integers(0, 50))]).astype(np.int32)
        reqs.append(toks)
        taken = []
        for layer in range(3):
            blocks, hits = a.prefix_blocks(layer, toks)
            parent, want_b, want_h = -1, [], []
            for i in range(len(toks) // 16):
                b, hit = pool.prefix_block(layer, parent, toks[16 * i:16 * i + 16])
                want_b.append(b)
                want_h.append(hit)
                parent = b
            assert blocks.tolist() == want_b and hits.tolist() == want_h, (r, layer)
            taken += want_b
        held[r] = taken
        assert a.free_list() == pool.free
        assert [a.refcount(b) for b in range(N)] == pool.ref
        assert a.prefix_entries() == len(pool.prefix)
    a.close()


def test_prefix_blocks_out_of_blocks_changes_nothing(kvs):
    a = kvs.BlockAllocator(4)
    toks = np.arange(64, dtype=np.int32)                  # 4 full blocks
    blocks, hits = a.prefix_blocks(0, toks)
    assert not hits.any() and a.num_free() == 0
    longer = np.arange(80, dtype=np.int32)                # 4 found + 1 new: no room
    with pytest.raises(kvs.KvsError) as e:
        a.prefix_blocks(0, longer)
    assert e.value.code == kvs.KVS_ERR_OOM_BLOCKS
    assert [a.refcount(b) for b in range(4)] == [1, 1, 1, 1] and a.prefix_entries() == 4
    again, hits2 = a.prefix_blocks(0, toks[:40])           # 2 full blocks, both found
    assert hits2.all() and again.tolist() == blocks[:2].tolist()
    a.close()
