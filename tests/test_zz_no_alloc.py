"""The allocation-free decode entry point, kvs_paged_decode_static.

Callers that may not allocate on the decode path (a server that reserved all
device memory for its block pool up front, or a C host without a device
allocator) use this entry point: it keeps its split partials in a device
array built into the library instead of a caller workspace.  It launches the
same kernels with the same split as kvs_paged_decode, so its outputs must be
bit-identical to that entry point's on the same inputs: a partial left over
in the shared array from an earlier call would show up as a difference.  The
tests run two calls in a row with different queries, one call that appends
the step's k/v (checked against the oracle's decode attention as well), and
the size limit of the array.  This file is collected last so that a run
stopping at the first failure has already run every other test.
"""
import numpy as np
import pytest

from gpu_helpers import ABS_O, bf16_f64, kvs_lib, torch

import oracle

H_Q, H_KV, D = 32, 8, 128
LENS = [4000, 4000, 4000] + [2048 - 64 * i for i in range(29)]   # one 32-layer sequence


def _paged_setup(seed, spare_slots=0):
    torch.manual_seed(seed)
    batch = len(LENS)
    max_blocks = -(-(max(LENS) + spare_slots) // 16)
    num_blocks = sum(-(-(n + spare_slots) // 16) for n in LENS) + 16
    k_pool = torch.randn(num_blocks, H_KV, 16, D, device="cuda").bfloat16()
    v_pool = torch.randn_like(k_pool)
    perm = torch.randperm(num_blocks, dtype=torch.int32)
    tables = torch.full((batch, max_blocks), -1, dtype=torch.int32)
    used = 0
    for i, n in enumerate(LENS):
        nb = -(-(n + spare_slots) // 16)
        tables[i, :nb] = perm[used:used + nb]
        used += nb
    lens = torch.tensor(LENS, dtype=torch.int32, device="cuda")
    return batch, max_blocks, num_blocks, k_pool, v_pool, tables.cuda(), lens


@pytest.mark.gpu
def test_static_scratch_is_bit_identical_to_the_workspace_entry_point():
    kvs = kvs_lib()
    batch, max_blocks, num_blocks, k_pool, v_pool, tables, lens = _paged_setup(7)
    ws_bytes = kvs.kvs_paged_decode_workspace_size(batch, H_Q, H_KV, D)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call in range(2):                           # two calls in a row
        q = torch.randn(batch, H_Q, D, device="cuda").bfloat16()
        ref = torch.empty(batch, H_Q, D, dtype=torch.bfloat16, device="cuda")
        got = torch.full_like(ref, float("nan"))
        kvs.kvs_paged_decode(q, None, None, k_pool, v_pool, num_blocks, tables, max_blocks,
                             None, lens, None, batch, H_Q, H_KV, D, D ** -0.5, ref, ws, ws_bytes,
                             status)
        kvs.kvs_paged_decode_static(q, None, None, k_pool, v_pool, num_blocks, tables,
                                    max_blocks, None, lens, None, batch, H_Q, H_KV, D, D ** -0.5,
                                    got, status)
        torch.cuda.synchronize()
        assert status.item() == 0
        assert torch.isfinite(got.float()).all()
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), call


@pytest.mark.gpu
def test_static_scratch_with_append_matches_workspace_entry_point_and_oracle():
    kvs = kvs_lib()
    batch, max_blocks, num_blocks, k_pool, v_pool, tables, lens = _paged_setup(8, spare_slots=1)
    q = torch.randn(batch, H_Q, D, device="cuda").bfloat16()
    k_new = torch.randn(batch, H_KV, D, device="cuda").bfloat16()
    v_new = torch.randn(batch, H_KV, D, device="cuda").bfloat16()
    ws_bytes = kvs.kvs_paged_decode_workspace_size(batch, H_Q, H_KV, D)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kp_ref, vp_ref = k_pool.clone(), v_pool.clone()
    kp_got, vp_got = k_pool.clone(), v_pool.clone()
    ref = torch.empty(batch, H_Q, D, dtype=torch.bfloat16, device="cuda")
    got = torch.full_like(ref, float("nan"))
    nxt_ref = torch.zeros_like(lens)
    nxt_got = torch.zeros_like(lens)
    kvs.kvs_paged_decode(q, k_new, v_new, kp_ref, vp_ref, num_blocks, tables, max_blocks, None,
                         lens, nxt_ref, batch, H_Q, H_KV, D, D ** -0.5, ref, ws, ws_bytes, status)
    kvs.kvs_paged_decode_static(q, k_new, v_new, kp_got, vp_got, num_blocks, tables, max_blocks,
                                None, lens, nxt_got, batch, H_Q, H_KV, D, D ** -0.5, got, status)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16))
    assert torch.equal(kp_got.view(torch.int16), kp_ref.view(torch.int16))
    assert torch.equal(vp_got.view(torch.int16), vp_ref.view(torch.int16))
    assert nxt_got.tolist() == [n + 1 for n in LENS] == nxt_ref.tolist()
    # the oracle: each item's kept rows gathered through its table, the new row
    # appended, explicit fp64 softmax attention of the step's query
    kp, vp = bf16_f64(kp_got), bf16_f64(vp_got)
    qh, kn, vn, out = bf16_f64(q), bf16_f64(k_new), bf16_f64(v_new), bf16_f64(got)
    tab = tables.cpu().numpy()
    worst = 0.0
    for i, n in enumerate(LENS):
        kc = np.stack([np.concatenate([oracle.gather_rows(kp, tab[i], n, h), kn[i, h][None]])
                       for h in range(H_KV)])
        vc = np.stack([np.concatenate([oracle.gather_rows(vp, tab[i], n, h), vn[i, h][None]])
                       for h in range(H_KV)])
        expect = oracle.decode_attention(qh[i], kc, vc, D ** -0.5)
        worst = max(worst, float(np.abs(out[i] - expect).max()))
        # the pool's slot n of each head now holds the appended row
        np.testing.assert_array_equal(oracle.gather_rows(kp, tab[i], n + 1, 0)[n], kn[i, 0])
    assert worst <= ABS_O, worst


@pytest.mark.gpu
def test_static_scratch_size_limit_on_the_device():
    kvs = kvs_lib()
    lib = kvs.library()
    # 624 items at the Llama-3-8B head shapes fit the array: the call gets past
    # the size check and fails on its NULL pointers instead
    assert lib.kvs_paged_decode_static(None, None, None, None, None, 1, None, 1, None, None,
                                       None, 624, H_Q, H_KV, D, 0.1, None, None, None) \
        == kvs.KVS_ERR_INVALID
    t = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    i = torch.zeros(625, dtype=torch.int32, device="cuda")
    with pytest.raises(kvs.KvsError) as e:
        kvs.kvs_paged_decode_static(t, None, None, t, t, 1, i, 1, None, i, None, 625, H_Q,
                                    H_KV, D, 0.1, t)
    assert e.value.code == kvs.KVS_ERR_UNSUPPORTED
    assert "built-in array" in kvs.last_error()
