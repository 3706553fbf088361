"""Failure detection on the GPU, without a fault.

* A bounded wait that runs out: the decode's copy-issuing lane arms each
  stage's barrier but starts none of the copies (the test hook
  kvs_test_paged_decode_stalled), so every consumer wait gives up after a short
  limit.  The kernel must store KVS_ERR_DEVICE_TIMEOUT and return, the context
  must stay usable, and the next ordinary call on the same stream must match
  the oracle.
* Corrupt inputs that the kernels catch: a block-table entry outside the pool,
  a negative length and a length beyond the item's table row.  The decode
  substitutes an in-range block or clamps the length, stores KVS_ERR_INVALID,
  and the other items' outputs still match the oracle.
None of these cases makes an access outside the buffers: the substitutions and
clamps happen before any address is formed.
"""
import numpy as np
import pytest

import oracle
from gpu_helpers import ABS_O, bf16_f64, dev_bf16, kvs_lib, torch
from synth import bf16_bits, bf16_to_f64

pytestmark = pytest.mark.gpu

H_Q, H_KV, D = 8, 2, 128


def _setup(lens, seed, spare_blocks=0):
    """Pools filled with N(0,1) bf16 rows, one scattered table row per item
    covering its length (plus spare_blocks more)."""
    rng = np.random.default_rng(seed)
    max_blocks = max(oracle.blocks_for(n) for n in lens) + spare_blocks
    num_blocks = len(lens) * max_blocks + 4
    pk = bf16_bits(rng.standard_normal((num_blocks, H_KV, 16, D)).astype(np.float32))
    pv = bf16_bits(rng.standard_normal((num_blocks, H_KV, 16, D)).astype(np.float32))
    perm = rng.permutation(num_blocks)
    tables = np.full((len(lens), max_blocks), -1, np.int32)
    used = 0
    for i, n in enumerate(lens):
        nb = oracle.blocks_for(n) + spare_blocks
        tables[i, :nb] = perm[used:used + nb]
        used += nb
    q = bf16_bits(rng.standard_normal((len(lens), H_Q, D)).astype(np.float32))
    return pk, pv, tables, q, max_blocks, num_blocks


def _oracle_out(pk, pv, table, n, q):
    kc = np.stack([oracle.gather_rows(pk, table, n, h) for h in range(H_KV)])
    vc = np.stack([oracle.gather_rows(pv, table, n, h) for h in range(H_KV)])
    return oracle.decode_attention(bf16_to_f64(q), bf16_to_f64(kc), bf16_to_f64(vc), D ** -0.5)


def _decode(kvs, pk_d, pv_d, num_blocks, tables, max_blocks, lens, q, status, stream=None):
    batch = len(lens)
    ws_bytes = kvs.kvs_paged_decode_workspace_size(batch, H_Q, H_KV, D)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    out = torch.zeros((batch, H_Q, D), dtype=torch.bfloat16, device="cuda")
    kvs.kvs_paged_decode(dev_bf16(q), None, None, pk_d, pv_d, num_blocks,
                         torch.from_numpy(tables).cuda(), max_blocks, None,
                         torch.tensor(lens, dtype=torch.int32, device="cuda"), None, batch, H_Q,
                         H_KV, D, D ** -0.5, out, ws, ws_bytes, status, stream=stream)
    return out


def test_decode_wait_runs_out_then_next_call_is_correct():
    kvs = kvs_lib()
    lens = [300, 50, 1000, 17]
    pk, pv, tables, q, max_blocks, num_blocks = _setup(lens, 1)
    pk_d, pv_d = dev_bf16(pk), dev_bf16(pv)
    stream = torch.cuda.Stream()
    batch = len(lens)
    ws_bytes = kvs.kvs_paged_decode_workspace_size(batch, H_Q, H_KV, D)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    out = torch.zeros((batch, H_Q, D), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    tables_d = torch.from_numpy(tables).cuda()
    lens_d = torch.tensor(lens, dtype=torch.int32, device="cuda")
    with torch.cuda.stream(stream):
        kvs.kvs_test_paged_decode_stalled(dev_bf16(q), pk_d, pv_d, num_blocks, tables_d,
                                          max_blocks, lens_d, batch, H_Q, H_KV, D, D ** -0.5,
                                          out, ws, ws_bytes, 200_000, status, stream=stream)
    stream.synchronize()                        # returns: the waits gave up
    assert status.item() == kvs.KVS_ERR_DEVICE_TIMEOUT
    # the pools were not written
    assert torch.equal(pk_d.view(torch.int16).cpu(), torch.from_numpy(pk.view(np.int16)))
    # the same stream, an ordinary call: status clean, results match the oracle
    status2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    with torch.cuda.stream(stream):
        got = _decode(kvs, pk_d, pv_d, num_blocks, tables, max_blocks, lens, q, status2,
                      stream=stream)
    stream.synchronize()
    assert status2.item() == 0
    got = bf16_f64(got)
    for i, n in enumerate(lens):
        assert np.abs(got[i] - _oracle_out(pk, pv, tables[i], n, q[i])).max() <= ABS_O


def test_decode_flags_out_of_range_block_id():
    kvs = kvs_lib()
    lens = [300, 50, 1000, 17]
    pk, pv, tables, q, max_blocks, num_blocks = _setup(lens, 2)
    bad = tables.copy()
    bad[2, 20] = num_blocks + 5                 # item 2's 21st block: outside the pool
    pk_d, pv_d = dev_bf16(pk), dev_bf16(pv)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = _decode(kvs, pk_d, pv_d, num_blocks, bad, max_blocks, lens, q, status)
    torch.cuda.synchronize()
    assert status.item() == kvs.KVS_ERR_INVALID
    got = bf16_f64(got)
    for i, n in enumerate(lens):
        if i != 2:                              # item 2's output is undefined
            assert np.abs(got[i] - _oracle_out(pk, pv, tables[i], n, q[i])).max() <= ABS_O
    assert torch.equal(pk_d.view(torch.int16).cpu(), torch.from_numpy(pk.view(np.int16)))


def test_decode_clamps_negative_and_oversized_lengths():
    kvs = kvs_lib()
    lens = [300, 50, 1000, 17, 64]
    pk, pv, tables, q, max_blocks, num_blocks = _setup(lens, 3)
    bad_lens = list(lens)
    bad_lens[1] = -40                           # clamped to 0: no output row
    bad_lens[3] = 1 << 30                       # clamped to the table row: max_blocks * 16
    pk_d, pv_d = dev_bf16(pk), dev_bf16(pv)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = _decode(kvs, pk_d, pv_d, num_blocks, tables, max_blocks, bad_lens, q, status)
    torch.cuda.synchronize()
    assert status.item() == kvs.KVS_ERR_INVALID
    got = bf16_f64(got)
    for i, n in enumerate(lens):
        if i not in (1, 3):
            assert np.abs(got[i] - _oracle_out(pk, pv, tables[i], n, q[i])).max() <= ABS_O
    assert np.all(got[1] == 0.0)                # untouched: the output buffer's zeros
