"""Thin Python binding of the kvs C ABI (include/kvs.h).

Argument marshalling only: every step of the hot path runs in the CUDA
library.  Functions keep the C names; tensors are torch tensors whose data
pointers are passed through, host-side arrays are numpy arrays.  If the
library has not been built, importing works but the first call raises
``KvsLibraryMissing`` -- there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libkvs.so")

KVS_OK, KVS_ERR_INVALID, KVS_ERR_OOM_BLOCKS, KVS_ERR_CUDA, KVS_ERR_UNSUPPORTED, \
    KVS_ERR_DEVICE_TIMEOUT = range(6)
BLOCK_TOKENS = 16
KVS_BLOCK_SKIP = -2

SELECT_ITEM = np.dtype([("score_off", "<i8"), ("n", "<i4"), ("k", "<i4"), ("idx_off", "<i8")])
COMPACT_ITEM = np.dtype([("src_tok", "<i8"), ("idx_off", "<i8"), ("row_off", "<i8"),
                         ("n", "<i4"), ("k_eff", "<i4"), ("table_off", "<i4"),
                         ("reserved", "<i4")])
assert SELECT_ITEM.itemsize == 24 and COMPACT_ITEM.itemsize == 40


class KvsLibraryMissing(RuntimeError):
    pass


class KvsError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"kvs status {code}: {msg}")
        self.code = code


_VP, _I32, _I64, _F32, _SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, \
    ctypes.c_size_t
_P32 = ctypes.POINTER(ctypes.c_int32)

_SIGS = {
    "kvs_last_error": (ctypes.c_char_p, []),
    "kvs_version": (_I32, []),
    "kvs_prefill_attn_lse": (_I32, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _I32, _I32, _I32, _I32,
                                    _I32, _I32, _F32, _VP, _VP]),
    "kvs_prefill_attn_lse_layers": (_I32, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _I32, _I32, _I32,
                                           _I32, _I32, _I32, _F32, _I32, _VP, _VP]),
    "kvs_window_scores": (_I32, [_VP, _VP, _VP, _VP, _VP, _VP, _I32, _I32, _I32, _I32, _I32,
                                 _I32, _I32, _F32, _VP, _VP]),
    "kvs_window_scores_layers": (_I32, [_VP, _VP, _VP, _VP, _VP, _VP, _I32, _I32, _I32, _I32,
                                        _I32, _I32, _I32, _F32, _I32, _VP, _VP]),
    "kvs_select_topk": (_I32, [_VP, _I64, _VP, _I32, _I32, _I32, _VP, _VP, _VP]),
    "kvs_evict_place": (_I32, [_VP, _VP, _VP, _VP, _I32, _VP, _I32, _VP, _VP, _VP, _VP, _I32,
                               _I32, _I32, _I32, _I32, _VP, _VP]),
    "kvs_evict_place_fp8": (_I32, [_VP, _VP, _VP, _VP, _VP, _VP, _I32, _VP, _I32, _VP, _VP, _VP,
                                   _VP, _I32, _I32, _I32, _I32, _I32, _VP, _VP]),
    "kvs_paged_decode_logits_fp8": (_I32, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _I32, _VP, _I32,
                                           _VP, _VP, _VP, _I32, _I32, _I32, _I32, _F32, _VP, _VP,
                                           _SZ, _VP, _I32, _VP, _VP, _VP]),
    "kvs_decode_scores_workspace_size": (_SZ, [_I32, _I32, _I32, _I32]),
    "kvs_paged_decode_logits": (_I32, [_VP, _VP, _VP, _VP, _VP, _I32, _VP, _I32, _VP, _VP, _VP,
                                       _I32, _I32, _I32, _I32, _F32, _VP, _VP, _SZ, _VP, _I32,
                                       _VP, _VP, _VP]),
    "kvs_decode_scores_from_logits": (_I32, [_VP, _I32, _VP, _VP, _VP, _VP, _I32, _I32, _I32,
                                             _I32, _VP, _VP]),
    "kvs_decode_scores": (_I32, [_VP, _VP, _I32, _VP, _I32, _VP, _VP, _VP, _I32, _I32, _I32,
                                 _I32, _I32, _F32, _VP, _SZ, _VP, _VP]),
    "kvs_decode_step": (_I32, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _I32,
                               _VP, _I32, _VP, _VP, _I32, _I32, _I32, _I32, _F32, _VP, _VP, _SZ,
                               _VP, _VP, _VP, _VP]),
    "kvs_decode_step_fp8": (_I32, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                   _VP, _VP, _I32, _VP, _I32, _VP, _VP, _I32, _I32, _I32, _I32,
                                   _F32, _VP, _VP, _SZ, _VP, _VP, _VP, _VP]),
    "kvs_compact_blocks": (_I32, [_VP, _VP, _VP, _I32, _I64, _I32, _I32, _VP, _VP, _VP, _VP,
                                  _I32, _VP, _VP]),
    "kvs_compact_blocks_fp8": (_I32, [_VP, _VP, _VP, _I32, _I64, _I32, _I32, _VP, _VP, _VP, _VP,
                                      _VP, _VP, _I32, _VP, _VP]),
    "kvs_paged_decode_fp8": (_I32, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _I32, _VP, _I32, _VP, _VP,
                                    _VP, _I32, _I32, _I32, _I32, _F32, _VP, _VP, _SZ, _VP, _VP]),
    "kvs_copy_blocks": (_I32, [_VP, _VP, _I32, _VP, _VP, _I32, _I32, _I32, _VP, _VP]),
    "kvs_copy_blocks_fp8": (_I32, [_VP, _VP, _I32, _VP, _VP, _VP, _VP, _I32, _I32, _I32, _VP,
                                   _VP]),
    "kvs_paged_decode_workspace_size": (_SZ, [_I32, _I32, _I32, _I32]),
    "kvs_workspace_zero": (_I32, [_VP, _SZ, _VP]),
    "kvs_paged_decode": (_I32, [_VP, _VP, _VP, _VP, _VP, _I32, _VP, _I32, _VP, _VP, _VP, _I32,
                                _I32, _I32, _I32, _F32, _VP, _VP, _SZ, _VP, _VP]),
    "kvs_paged_decode_static": (_I32, [_VP, _VP, _VP, _VP, _VP, _I32, _VP, _I32, _VP, _VP, _VP,
                                       _I32, _I32, _I32, _I32, _F32, _VP, _VP, _VP]),
    "kvs_test_paged_decode_stalled": (_I32, [_VP, _VP, _VP, _I32, _VP, _I32, _VP, _I32, _I32,
                                             _I32, _I32, _F32, _VP, _VP, _SZ, ctypes.c_uint32,
                                             _VP, _VP]),
    "kvs_alloc_create": (_I32, [_I32, _VP, _I32, ctypes.POINTER(_VP)]),
    "kvs_alloc_destroy": (None, [_VP]),
    "kvs_alloc_block": (_I32, [_VP, _P32]),
    "kvs_alloc_blocks": (_I32, [_VP, _I32, _VP]),
    "kvs_alloc_incref": (_I32, [_VP, _I32]),
    "kvs_alloc_decref": (_I32, [_VP, _I32]),
    "kvs_alloc_cow": (_I32, [_VP, _I32, _P32, _P32]),
    "kvs_alloc_refcount": (_I32, [_VP, _I32]),
    "kvs_alloc_num_free": (_I32, [_VP]),
    "kvs_alloc_free_list": (_I32, [_VP, _VP, _I32]),
    "kvs_alloc_prefix_blocks": (_I32, [_VP, _I32, _VP, _I32, _VP, _VP, _P32]),
    "kvs_alloc_prefix_entries": (_I32, [_VP]),
    "kvs_decode_prepare": (_I32, [_VP, _VP, _I32, _VP, _I32, _VP, _VP, _VP, _P32, _P32, _P32]),
}

_lib = None


def library():
    """Load libkvs.so (built by layer_wise_kv_gb300.build); raise if absent."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise KvsLibraryMissing(
                f"{LIB_PATH} is missing: build the CUDA library first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def exported_symbols():
    return list(_SIGS)


def last_error() -> str:
    return library().kvs_last_error().decode()


def _check(code):
    if code != KVS_OK:
        raise KvsError(code, last_error())


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dev(t, dtype_name, what):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{what} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    want = {"bf16": torch.bfloat16, "f32": torch.float32, "i32": torch.int32,
            "u8": torch.uint8}[dtype_name]
    if t.dtype != want:
        raise TypeError(f"{what} must be {want}, got {t.dtype}")
    return t.data_ptr()


# ---------------------------------------------------------------------------
# the five hot-path calls
# ---------------------------------------------------------------------------
def kvs_prefill_attn_lse_layers(q, k, v, o, m, l, cu_seqlens, batch, max_n, total_tokens, h_q,
                                h_kv, d, scale, n_layers, status=None, stream=None):
    """q, k, v, o, m, l: n_layers layers stacked in one buffer each (leading
    dimension n_layers)."""
    for t, what in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (m, "m"), (l, "l")):
        if t.shape[0] != n_layers:
            raise ValueError(f"{what} must have n_layers = {n_layers} as its leading dimension")
    _check(library().kvs_prefill_attn_lse_layers(
        _dev(q, "bf16", "q"), _dev(k, "bf16", "k"), _dev(v, "bf16", "v"), _dev(o, "bf16", "o"),
        _dev(m, "f32", "m"), _dev(l, "f32", "l"), _dev(cu_seqlens, "i32", "cu_seqlens"),
        batch, max_n, total_tokens, h_q, h_kv, d, float(scale), n_layers,
        None if status is None else _dev(status, "i32", "status"), _stream(stream)))


def kvs_prefill_attn_lse(q, k, v, o, m, l, cu_seqlens, batch, max_n, total_tokens, h_q, h_kv,
                         d, scale, status=None, stream=None):
    _check(library().kvs_prefill_attn_lse(
        _dev(q, "bf16", "q"), _dev(k, "bf16", "k"), _dev(v, "bf16", "v"), _dev(o, "bf16", "o"),
        _dev(m, "f32", "m"), _dev(l, "f32", "l"), _dev(cu_seqlens, "i32", "cu_seqlens"),
        batch, max_n, total_tokens, h_q, h_kv, d, float(scale),
        None if status is None else _dev(status, "i32", "status"), _stream(stream)))


def kvs_window_scores_layers(q, k, m, l, scores, cu_seqlens, batch, max_n, total_tokens, h_q,
                             h_kv, d, alpha, scale, n_layers, status=None, stream=None):
    """q, k, m, l, scores: n_layers layers stacked in one buffer each (leading
    dimension n_layers)."""
    for t, what in ((q, "q"), (k, "k"), (m, "m"), (l, "l"), (scores, "scores")):
        if t.shape[0] != n_layers:
            raise ValueError(f"{what} must have n_layers = {n_layers} as its leading dimension")
    _check(library().kvs_window_scores_layers(
        _dev(q, "bf16", "q"), _dev(k, "bf16", "k"), _dev(m, "f32", "m"), _dev(l, "f32", "l"),
        _dev(scores, "f32", "scores"), _dev(cu_seqlens, "i32", "cu_seqlens"), batch, max_n,
        total_tokens, h_q, h_kv, d, alpha, float(scale), n_layers,
        None if status is None else _dev(status, "i32", "status"), _stream(stream)))


def kvs_window_scores(q, k, m, l, scores, cu_seqlens, batch, max_n, total_tokens, h_q, h_kv, d,
                      alpha, scale, status=None, stream=None):
    _check(library().kvs_window_scores(
        _dev(q, "bf16", "q"), _dev(k, "bf16", "k"), _dev(m, "f32", "m"), _dev(l, "f32", "l"),
        _dev(scores, "f32", "scores"), _dev(cu_seqlens, "i32", "cu_seqlens"), batch, max_n,
        total_tokens, h_q, h_kv, d, alpha, float(scale),
        None if status is None else _dev(status, "i32", "status"), _stream(stream)))


def kvs_select_topk(scores, head_stride, items, n_items, h_kv, recent, kept_idx, status=None,
                    stream=None):
    _check(library().kvs_select_topk(
        _dev(scores, "f32", "scores"), int(head_stride), _dev(items, "u8", "items"), n_items,
        h_kv, recent, _dev(kept_idx, "i32", "kept_idx"),
        None if status is None else _dev(status, "i32", "status"), _stream(stream)))


def kvs_compact_blocks(k, v, items, n_items, total_rows, h_kv, d, kept_idx, block_tables,
                       k_pool, v_pool, num_blocks, status=None, stream=None):
    _check(library().kvs_compact_blocks(
        _dev(k, "bf16", "k"), _dev(v, "bf16", "v"), _dev(items, "u8", "items"), n_items,
        int(total_rows), h_kv, d, _dev(kept_idx, "i32", "kept_idx"),
        _dev(block_tables, "i32", "block_tables"), _dev(k_pool, "bf16", "k_pool"),
        _dev(v_pool, "bf16", "v_pool"), num_blocks,
        None if status is None else _dev(status, "i32", "status"), _stream(stream)))


def kvs_compact_blocks_fp8(k, v, items, n_items, total_rows, h_kv, d, kept_idx, block_tables,
                           k_pool, v_pool, k_scale, v_scale, num_blocks, status=None,
                           stream=None):
    """kvs_compact_blocks into FP8 pools: k_pool, v_pool uint8 [num_blocks][h_kv][16 * d] (V
    transposed per block and head), k_scale, v_scale float32 [num_blocks][h_kv][16]."""
    _check(library().kvs_compact_blocks_fp8(
        _dev(k, "bf16", "k"), _dev(v, "bf16", "v"), _dev(items, "u8", "items"), n_items,
        int(total_rows), h_kv, d, _dev(kept_idx, "i32", "kept_idx"),
        _dev(block_tables, "i32", "block_tables"), _dev(k_pool, "u8", "k_pool"),
        _dev(v_pool, "u8", "v_pool"), _dev(k_scale, "f32", "k_scale"),
        _dev(v_scale, "f32", "v_scale"), num_blocks,
        None if status is None else _dev(status, "i32", "status"), _stream(stream)))


def kvs_paged_decode_fp8(q, k_new, v_new, k_pool, v_pool, k_scale, v_scale, num_blocks,
                         block_tables, max_blocks, table_patch, lens, lens_next, batch, h_q, h_kv,
                         d, scale, out, workspace, workspace_bytes, status=None, stream=None):
    _check(library().kvs_paged_decode_fp8(
        _dev(q, "bf16", "q"), None if k_new is None else _dev(k_new, "bf16", "k_new"),
        None if v_new is None else _dev(v_new, "bf16", "v_new"), _dev(k_pool, "u8", "k_pool"),
        _dev(v_pool, "u8", "v_pool"), _dev(k_scale, "f32", "k_scale"),
        _dev(v_scale, "f32", "v_scale"), num_blocks, _dev(block_tables, "i32", "block_tables"),
        max_blocks, None if table_patch is None else _dev(table_patch, "i32", "table_patch"),
        _dev(lens, "i32", "lens"), None if lens_next is None else _dev(lens_next, "i32", "lens_next"),
        batch, h_q, h_kv, d, float(scale), _dev(out, "bf16", "out"),
        _dev(workspace, "u8", "workspace"), workspace_bytes,
        None if status is None else _dev(status, "i32", "status"), _stream(stream)))


def kvs_copy_blocks_fp8(src, dst, count, k_pool, v_pool, k_scale, v_scale, num_blocks, h_kv, d,
                        status=None, stream=None):
    _check(library().kvs_copy_blocks_fp8(
        _dev(src, "i32", "src"), _dev(dst, "i32", "dst"), count, _dev(k_pool, "u8", "k_pool"),
        _dev(v_pool, "u8", "v_pool"), _dev(k_scale, "f32", "k_scale"),
        _dev(v_scale, "f32", "v_scale"), num_blocks, h_kv, d,
        None if status is None else _dev(status, "i32", "status"), _stream(stream)))


def kvs_copy_blocks(src, dst, count, k_pool, v_pool, num_blocks, h_kv, d, status=None,
                    stream=None):
    _check(library().kvs_copy_blocks(
        _dev(src, "i32", "src"), _dev(dst, "i32", "dst"), count, _dev(k_pool, "bf16", "k_pool"),
        _dev(v_pool, "bf16", "v_pool"), num_blocks, h_kv, d,
        None if status is None else _dev(status, "i32", "status"), _stream(stream)))


def kvs_paged_decode_workspace_size(batch, h_q, h_kv, d) -> int:
    return int(library().kvs_paged_decode_workspace_size(batch, h_q, h_kv, d))


def kvs_workspace_zero(workspace, nbytes, stream=None):
    _check(library().kvs_workspace_zero(_dev(workspace, "u8", "workspace"), nbytes,
                                        _stream(stream)))


def kvs_paged_decode(q, k_new, v_new, k_pool, v_pool, num_blocks, block_tables, max_blocks,
                     table_patch, lens, lens_next, batch, h_q, h_kv, d, scale, out,
                     workspace, workspace_bytes, status=None, stream=None):
    _check(library().kvs_paged_decode(
        _dev(q, "bf16", "q"), None if k_new is None else _dev(k_new, "bf16", "k_new"),
        None if v_new is None else _dev(v_new, "bf16", "v_new"),
        _dev(k_pool, "bf16", "k_pool"), _dev(v_pool, "bf16", "v_pool"), num_blocks,
        _dev(block_tables, "i32", "block_tables"), max_blocks,
        None if table_patch is None else _dev(table_patch, "i32", "table_patch"),
        _dev(lens, "i32", "lens"), None if lens_next is None else _dev(lens_next, "i32", "lens_next"),
        batch, h_q, h_kv, d, float(scale), _dev(out, "bf16", "out"),
        _dev(workspace, "u8", "workspace"), workspace_bytes,
        None if status is None else _dev(status, "i32", "status"), _stream(stream)))


def kvs_test_paged_decode_stalled(q, k_pool, v_pool, num_blocks, block_tables, max_blocks, lens,
                                  batch, h_q, h_kv, d, scale, out, workspace, workspace_bytes,
                                  wait_ns, status=None, stream=None):
    _check(library().kvs_test_paged_decode_stalled(
        _dev(q, "bf16", "q"), _dev(k_pool, "bf16", "k_pool"), _dev(v_pool, "bf16", "v_pool"),
        num_blocks, _dev(block_tables, "i32", "block_tables"), max_blocks,
        _dev(lens, "i32", "lens"), batch, h_q, h_kv, d, float(scale), _dev(out, "bf16", "out"),
        _dev(workspace, "u8", "workspace"), workspace_bytes, int(wait_ns),
        None if status is None else _dev(status, "i32", "status"), _stream(stream)))


def kvs_paged_decode_static(q, k_new, v_new, k_pool, v_pool, num_blocks, block_tables,
                            max_blocks, table_patch, lens, lens_next, batch, h_q, h_kv, d, scale,
                            out, status=None, stream=None):
    """kvs_paged_decode for callers that cannot pass a workspace: the library's
    built-in device scratch holds the split partials (see include/kvs.h)."""
    _check(library().kvs_paged_decode_static(
        _dev(q, "bf16", "q"), None if k_new is None else _dev(k_new, "bf16", "k_new"),
        None if v_new is None else _dev(v_new, "bf16", "v_new"),
        _dev(k_pool, "bf16", "k_pool"), _dev(v_pool, "bf16", "v_pool"), num_blocks,
        _dev(block_tables, "i32", "block_tables"), max_blocks,
        None if table_patch is None else _dev(table_patch, "i32", "table_patch"),
        _dev(lens, "i32", "lens"), None if lens_next is None else _dev(lens_next, "i32", "lens_next"),
        batch, h_q, h_kv, d, float(scale), _dev(out, "bf16", "out"),
        None if status is None else _dev(status, "i32", "status"), _stream(stream)))


# ---------------------------------------------------------------------------
# block allocator (host)
# ---------------------------------------------------------------------------
def kvs_decode_step(alloc, tables_h, lens_h, patch_h, cow_h, patch_d, cow_d, q, k_new, v_new,
                    k_pool, v_pool, num_blocks, block_tables, max_blocks, lens, lens_next,
                    n_items, h_q, h_kv, d, scale, out, workspace, workspace_bytes, status=None,
                    stream=None):
    """One decode step in one native call (host preparation, uploads, paged
    decode).  tables_h [n_items][max_blocks], lens_h [n_items]: host int32
    numpy mirrors (updated in place); patch_h [n_items], cow_h [2 n_items]:
    pinned host int32 staging tensors; the rest as for kvs_paged_decode.
    Returns (n_cow, n_patch)."""
    assert tables_h.dtype == np.int32 and tables_h.flags.c_contiguous
    assert lens_h.dtype == np.int32 and lens_h.flags.c_contiguous
    for t, what in ((patch_h, "patch_h"), (cow_h, "cow_h")):
        if t.is_cuda or t.dtype != __import__("torch").int32 or not t.is_contiguous():
            raise TypeError(f"{what} must be a contiguous host int32 tensor")
    n_cow, n_patch = ctypes.c_int32(), ctypes.c_int32()
    _check(library().kvs_decode_step(
        alloc._h, tables_h.ctypes.data, lens_h.ctypes.data, patch_h.data_ptr(), cow_h.data_ptr(),
        _dev(patch_d, "i32", "patch_d"), _dev(cow_d, "i32", "cow_d"), _dev(q, "bf16", "q"),
        _dev(k_new, "bf16", "k_new"), _dev(v_new, "bf16", "v_new"), _dev(k_pool, "bf16", "k_pool"),
        _dev(v_pool, "bf16", "v_pool"), num_blocks, _dev(block_tables, "i32", "block_tables"),
        max_blocks, _dev(lens, "i32", "lens"), _dev(lens_next, "i32", "lens_next"), n_items, h_q,
        h_kv, d, float(scale), _dev(out, "bf16", "out"), _dev(workspace, "u8", "workspace"),
        workspace_bytes, None if status is None else _dev(status, "i32", "status"),
        ctypes.byref(n_cow), ctypes.byref(n_patch), _stream(stream)))
    return n_cow.value, n_patch.value


def kvs_evict_place(k_new, v_new, k_pool, v_pool, num_blocks, block_tables, max_blocks, lens,
                    new_pos, score, pos, max_slots, n_items, h_kv, d, recent, status=None,
                    stream=None):
    _check(library().kvs_evict_place(
        _dev(k_new, "bf16", "k_new"), _dev(v_new, "bf16", "v_new"), _dev(k_pool, "bf16", "k_pool"),
        _dev(v_pool, "bf16", "v_pool"), num_blocks, _dev(block_tables, "i32", "block_tables"),
        max_blocks, _dev(lens, "i32", "lens"), _dev(new_pos, "i32", "new_pos"),
        _dev(score, "f32", "score"), _dev(pos, "i32", "pos"), max_slots, n_items, h_kv, d, recent,
        None if status is None else _dev(status, "i32", "status"), _stream(stream)))


def kvs_evict_place_fp8(k_new, v_new, k_pool, v_pool, k_scale, v_scale, num_blocks, block_tables,
                        max_blocks, lens, new_pos, score, pos, max_slots, n_items, h_kv, d, recent,
                        status=None, stream=None):
    _check(library().kvs_evict_place_fp8(
        _dev(k_new, "bf16", "k_new"), _dev(v_new, "bf16", "v_new"), _dev(k_pool, "u8", "k_pool"),
        _dev(v_pool, "u8", "v_pool"), _dev(k_scale, "f32", "k_scale"),
        _dev(v_scale, "f32", "v_scale"), num_blocks, _dev(block_tables, "i32", "block_tables"),
        max_blocks, _dev(lens, "i32", "lens"), _dev(new_pos, "i32", "new_pos"),
        _dev(score, "f32", "score"), _dev(pos, "i32", "pos"), max_slots, n_items, h_kv, d, recent,
        None if status is None else _dev(status, "i32", "status"), _stream(stream)))


def kvs_paged_decode_logits_fp8(q, k_new, v_new, k_pool, v_pool, k_scale, v_scale, num_blocks,
                                block_tables, max_blocks, table_patch, lens, lens_next, batch, h_q,
                                h_kv, d, scale, out, workspace, workspace_bytes, logits, logit_ld,
                                lse, status=None, stream=None):
    if logits.numel() < batch * h_kv * (h_q // h_kv) * logit_ld:
        raise ValueError("logits must hold batch x h_kv x G x logit_ld floats")
    if lse.numel() < batch * h_q:
        raise ValueError("lse must hold batch x h_q floats")
    _check(library().kvs_paged_decode_logits_fp8(
        _dev(q, "bf16", "q"), None if k_new is None else _dev(k_new, "bf16", "k_new"),
        None if v_new is None else _dev(v_new, "bf16", "v_new"), _dev(k_pool, "u8", "k_pool"),
        _dev(v_pool, "u8", "v_pool"), _dev(k_scale, "f32", "k_scale"),
        _dev(v_scale, "f32", "v_scale"), num_blocks, _dev(block_tables, "i32", "block_tables"),
        max_blocks, None if table_patch is None else _dev(table_patch, "i32", "table_patch"),
        _dev(lens, "i32", "lens"), None if lens_next is None else _dev(lens_next, "i32", "lens_next"),
        batch, h_q, h_kv, d, float(scale), _dev(out, "bf16", "out"),
        _dev(workspace, "u8", "workspace"), workspace_bytes, _dev(logits, "f32", "logits"),
        logit_ld, _dev(lse, "f32", "lse"), None if status is None else _dev(status, "i32", "status"),
        _stream(stream)))


def kvs_paged_decode_logits(q, k_new, v_new, k_pool, v_pool, num_blocks, block_tables,
                            max_blocks, table_patch, lens, lens_next, batch, h_q, h_kv, d, scale,
                            out, workspace, workspace_bytes, logits, logit_ld, lse, status=None,
                            stream=None):
    if logits.numel() < batch * h_kv * (h_q // h_kv) * logit_ld:
        raise ValueError("logits must hold batch x h_kv x G x logit_ld floats")
    if lse.numel() < batch * h_q:
        raise ValueError("lse must hold batch x h_q floats")
    _check(library().kvs_paged_decode_logits(
        _dev(q, "bf16", "q"), None if k_new is None else _dev(k_new, "bf16", "k_new"),
        None if v_new is None else _dev(v_new, "bf16", "v_new"), _dev(k_pool, "bf16", "k_pool"),
        _dev(v_pool, "bf16", "v_pool"), num_blocks, _dev(block_tables, "i32", "block_tables"),
        max_blocks, None if table_patch is None else _dev(table_patch, "i32", "table_patch"),
        _dev(lens, "i32", "lens"), None if lens_next is None else _dev(lens_next, "i32", "lens_next"),
        batch, h_q, h_kv, d, float(scale), _dev(out, "bf16", "out"),
        _dev(workspace, "u8", "workspace"), workspace_bytes, _dev(logits, "f32", "logits"),
        logit_ld, _dev(lse, "f32", "lse"), None if status is None else _dev(status, "i32", "status"),
        _stream(stream)))


def kvs_decode_scores_from_logits(logits, logit_ld, lse, lens, score, new_pos, max_slots, n_items,
                                  h_q, h_kv, status=None, stream=None):
    _check(library().kvs_decode_scores_from_logits(
        _dev(logits, "f32", "logits"), logit_ld, _dev(lse, "f32", "lse"), _dev(lens, "i32", "lens"),
        _dev(score, "f32", "score"), _dev(new_pos, "i32", "new_pos"), max_slots, n_items, h_q,
        h_kv, None if status is None else _dev(status, "i32", "status"), _stream(stream)))


def kvs_decode_scores_workspace_size(n_items, h_q, h_kv, max_slots) -> int:
    return int(library().kvs_decode_scores_workspace_size(n_items, h_q, h_kv, max_slots))


def kvs_decode_scores(q, k_pool, num_blocks, block_tables, max_blocks, lens, score, new_pos,
                      max_slots, n_items, h_q, h_kv, d, scale, workspace, workspace_bytes,
                      status=None, stream=None):
    _check(library().kvs_decode_scores(
        _dev(q, "bf16", "q"), _dev(k_pool, "bf16", "k_pool"), num_blocks,
        _dev(block_tables, "i32", "block_tables"), max_blocks, _dev(lens, "i32", "lens"),
        _dev(score, "f32", "score"), _dev(new_pos, "i32", "new_pos"), max_slots, n_items, h_q,
        h_kv, d, float(scale), _dev(workspace, "u8", "workspace"), workspace_bytes,
        None if status is None else _dev(status, "i32", "status"), _stream(stream)))


class BlockAllocator:
    """kvs_alloc_*: FIFO free list, reference counts, copy-on-write."""

    def __init__(self, num_blocks: int, initial_free=None):
        lib = library()
        h = _VP()
        if initial_free is None:
            _check(lib.kvs_alloc_create(num_blocks, None, 0, ctypes.byref(h)))
        else:
            arr = np.ascontiguousarray(initial_free, dtype=np.int32)
            _check(lib.kvs_alloc_create(num_blocks, arr.ctypes.data, arr.size, ctypes.byref(h)))
        self._h = h
        self._lib = lib
        self.num_blocks = num_blocks

    def close(self):
        if self._h:
            self._lib.kvs_alloc_destroy(self._h)
            self._h = _VP()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def alloc(self) -> int:
        out = ctypes.c_int32()
        _check(self._lib.kvs_alloc_block(self._h, ctypes.byref(out)))
        return out.value

    def alloc_many(self, count: int) -> np.ndarray:
        out = np.empty(count, dtype=np.int32)
        _check(self._lib.kvs_alloc_blocks(self._h, count, out.ctypes.data if count else None))
        return out

    def incref(self, b: int):
        _check(self._lib.kvs_alloc_incref(self._h, int(b)))

    def decref(self, b: int):
        _check(self._lib.kvs_alloc_decref(self._h, int(b)))

    def cow(self, b: int):
        out, copied = ctypes.c_int32(), ctypes.c_int32()
        _check(self._lib.kvs_alloc_cow(self._h, int(b), ctypes.byref(out), ctypes.byref(copied)))
        return out.value, bool(copied.value)

    def refcount(self, b: int) -> int:
        return int(self._lib.kvs_alloc_refcount(self._h, int(b)))

    def num_free(self) -> int:
        return int(self._lib.kvs_alloc_num_free(self._h))

    def prefix_blocks(self, layer: int, tokens):
        """kvs_alloc_prefix_blocks: the blocks of the full 16-token blocks of a
        prompt's token ids in one full-cache layer, found (hit) or new.
        Returns (blocks int32, hits bool) arrays of len(tokens) // 16."""
        toks = np.ascontiguousarray(tokens, dtype=np.int32)
        n_full = toks.size // BLOCK_TOKENS
        blocks = np.empty(max(n_full, 1), dtype=np.int32)
        hits = np.empty(max(n_full, 1), dtype=np.int32)
        _check(self._lib.kvs_alloc_prefix_blocks(self._h, int(layer),
                                                 toks.ctypes.data if toks.size else None,
                                                 toks.size, blocks.ctypes.data, hits.ctypes.data,
                                                 None))
        return blocks[:n_full], hits[:n_full].astype(bool)

    def prefix_entries(self) -> int:
        return int(self._lib.kvs_alloc_prefix_entries(self._h))

    def free_list(self) -> list:
        n = self.num_free()
        buf = np.empty(max(n, 1), dtype=np.int32)
        got = self._lib.kvs_alloc_free_list(self._h, buf.ctypes.data, n)
        return buf[:got].tolist()

    def decode_prepare(self, tables: np.ndarray, lens: np.ndarray, patch: np.ndarray,
                       cow_src: np.ndarray, cow_dst: np.ndarray, with_patch_count=False):
        """kvs_decode_prepare on host int32 arrays (tables [n_items, max_blocks],
        updated in place).  Returns the number of copy-on-write pairs (and the
        number of patched table entries with with_patch_count)."""
        assert tables.dtype == np.int32 and tables.flags.c_contiguous
        n_items, max_blocks = tables.shape
        n_cow, n_patch, n_done = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
        _check(self._lib.kvs_decode_prepare(
            self._h, tables.ctypes.data, max_blocks, lens.ctypes.data, n_items,
            patch.ctypes.data, cow_src.ctypes.data, cow_dst.ctypes.data, ctypes.byref(n_cow),
            ctypes.byref(n_patch), ctypes.byref(n_done)))
        if with_patch_count:
            return n_cow.value, n_patch.value
        return n_cow.value
