"""The allocation-free decode entry point, kvs_paged_decode_static.

Callers that may not allocate on the decode path (a server that reserved all
device memory for its block pool up front, or a C host without a device
allocator) use this entry point: it keeps its split partials in a device
array built into the library instead of a caller workspace.  The test checks
it against kvs_paged_decode (caller workspace) on the same inputs, for two
calls in a row with different queries, so a result left over from the first
call cannot pass for the second.  This file is collected last so that a run
stopping at the first failure has already run every other test.
"""
import numpy as np
import pytest

from gpu_helpers import ABS_O, bf16_f64, kvs_lib, torch

pytestmark = pytest.mark.gpu


def test_static_scratch_matches_workspace_entry_point():
    kvs = kvs_lib()
    torch.manual_seed(7)
    h_q, h_kv, d = 32, 8, 128
    lens_l = [4000, 4000, 4000] + [2048 - 64 * i for i in range(29)]  # one 32-layer sequence
    batch = len(lens_l)
    max_blocks = -(-max(lens_l) // 16)
    num_blocks = sum(-(-n // 16) for n in lens_l) + 16
    k_pool = torch.randn(num_blocks, h_kv, 16, d, device="cuda").bfloat16()
    v_pool = torch.randn_like(k_pool)
    perm = torch.randperm(num_blocks, dtype=torch.int32)
    tables = torch.full((batch, max_blocks), -1, dtype=torch.int32)
    used = 0
    for i, n in enumerate(lens_l):
        nb = -(-n // 16)
        tables[i, :nb] = perm[used:used + nb]
        used += nb
    tables = tables.cuda()
    lens = torch.tensor(lens_l, dtype=torch.int32, device="cuda")
    ws_bytes = kvs.kvs_paged_decode_workspace_size(batch, h_q, h_kv, d)
    assert ws_bytes <= (16 << 20)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call in range(2):                           # two calls in a row
        q = torch.randn(batch, h_q, d, device="cuda").bfloat16()
        ref = torch.empty(batch, h_q, d, dtype=torch.bfloat16, device="cuda")
        got = torch.full_like(ref, float("nan"))
        kvs.kvs_paged_decode(q, None, None, k_pool, v_pool, num_blocks, tables, max_blocks,
                             None, lens, None, batch, h_q, h_kv, d, d ** -0.5, ref, ws, ws_bytes,
                             status)
        kvs.kvs_paged_decode_static(q, None, None, k_pool, v_pool, num_blocks, tables,
                                    max_blocks, None, lens, None, batch, h_q, h_kv, d, d ** -0.5,
                                    got, status)
        torch.cuda.synchronize()
        assert status.item() == 0
        diff = np.abs(bf16_f64(got) - bf16_f64(ref))
        assert np.isfinite(diff).all()
        assert diff.max() <= ABS_O, (call, diff.max())


def test_static_scratch_rejects_oversized_batch():
    kvs = kvs_lib()
    h_q, h_kv, d = 32, 8, 128
    batch = 700                                     # needs more than the 16 MiB array
    assert kvs.kvs_paged_decode_workspace_size(batch, h_q, h_kv, d) > (16 << 20)
    t = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    i = torch.zeros(batch, dtype=torch.int32, device="cuda")
    with pytest.raises(kvs.KvsError) as e:
        kvs.kvs_paged_decode_static(t, None, None, t, t, 1, i, 1, None, i, None, batch, h_q,
                                    h_kv, d, 0.1, t)
    assert e.value.code == kvs.KVS_ERR_UNSUPPORTED
    assert "built-in array" in kvs.last_error()
