"""The hot path as a sequence of kvs C-ABI calls: prefill+sparsify of a batch
of prompts over all layers, then decode steps over the paged cache.

Step orders (the same ones the CPU oracle uses):
* prefill: for each layer, prefill attention (+ m, l) -- one launch over all
  layers when every layer's inputs are resident in one buffer; then the window scores
  of the layers with a budget below the prompt length (one launch per run of
  consecutive such layers: a layer's scores read only its own q, k, m, l;
  while the layers' inputs are still being copied in, each layer's scores
  follow its prefill instead); then one selection launch over every
  (sequence, layer) item; then, sequence by sequence and layer by
  layer, ceil(k_eff / 16) blocks from the allocator; then one compaction
  launch over all items.
* decode step: the host allocator prepares every (stream, layer) item in order
  (new block when the length is a multiple of 16, copy-on-write of a shared
  last block), the copies run, then one paged-decode launch covers all items
  -- or, in layer order (the launches a model issues, since layer l + 1's
  query depends on layer l's output), one launch per layer over that layer's
  items.

Sources: Novita AI, "How KV Sparsity achieves 1.5x acceleration for vLLM"
(sections "Key techniques 1" and "Key techniques 2"); Ultralytics glossary
"PagedAttention" (sections "How paging works", "Block sharing between
sequences").
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import numpy as np
import torch

from . import kvs

BLOCK = kvs.BLOCK_TOKENS


def blocks_for(tokens: int) -> int:
    return -(-tokens // BLOCK)


def _u8(arr: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(arr).view(np.uint8).reshape(-1)).to(device)


@dataclass
class Shape:
    n_layers: int
    h_q: int
    h_kv: int
    d: int
    alpha: int
    recent: int

    @property
    def group(self):
        return self.h_q // self.h_kv

    @property
    def scale(self):
        return 1.0 / float(np.sqrt(self.d))


@dataclass
class PrefillResult:
    """Per-sequence, per-layer block tables (host) and kept-token counts."""
    tables: List[List[List[int]]]        # [seq][layer] -> block ids
    k_eff: List[List[int]]               # [seq][layer]
    kept_idx: torch.Tensor               # device int32, all items
    idx_off: np.ndarray                  # [seq][layer] element offsets into kept_idx
    scores: Optional[torch.Tensor] = None  # [L][h_kv][T] fp32 (budgeted layers filled)
    m: Optional[List[torch.Tensor]] = None  # per layer [h_q][T] when kept
    l: Optional[List[torch.Tensor]] = None
    o: Optional[List[torch.Tensor]] = None
    prefix_hits: int = 0                 # prefix blocks found (not written again)


class Engine:
    """Device pools, the host block allocator and scratch for one workload."""

    def __init__(self, shape: Shape, num_blocks: int, device="cuda", initial_free=None,
                 poison=False, kv_dtype: str = "bf16"):
        """poison: fill the pools with NaN patterns (bf16 0xFFFF, e4m3 0xFF)
        so that any read of an unwritten slot shows up in the outputs (tests).
        kv_dtype "fp8": the pools hold e4m3 codes with per-row fp32 scales
        (k_scale, v_scale; layout of kvs_compact_blocks_fp8, d = 128); the
        prefill compacts into them and DecodeBatch decodes from them."""
        self.shape = shape
        self.device = torch.device(device)
        self.num_blocks = num_blocks
        self.alloc = kvs.BlockAllocator(num_blocks, initial_free)
        s = shape
        if kv_dtype not in ("bf16", "fp8"):
            raise ValueError("kv_dtype is 'bf16' or 'fp8'")
        self.kv_fp8 = kv_dtype == "fp8"
        self.k_scale = self.v_scale = None
        if self.kv_fp8:
            if s.d != 128:
                raise ValueError("FP8 pools need d = 128")
            self.k_pool = torch.empty((num_blocks, s.h_kv, BLOCK * s.d), dtype=torch.uint8,
                                      device=self.device)
            self.k_scale = torch.zeros((num_blocks, s.h_kv, BLOCK), dtype=torch.float32,
                                       device=self.device)
            self.v_scale = torch.zeros_like(self.k_scale)
        else:
            self.k_pool = torch.empty((num_blocks, s.h_kv, BLOCK, s.d), dtype=torch.bfloat16,
                                      device=self.device)
        self.v_pool = torch.empty_like(self.k_pool)
        if poison:
            self.k_pool.view(torch.uint8).fill_(0xFF)
            self.v_pool.view(torch.uint8).fill_(0xFF)
        self.status = torch.zeros(1, dtype=torch.int32, device=self.device)
        self._plans = {}

    # ------------------------------------------------------------------ checks
    def check_status(self):
        code = int(self.status.item())
        if code != 0:
            raise kvs.KvsError(code, "a kernel reported a device-side error")

    # ------------------------------------------------------------------ prefill
    def _plan(self, lens, budgets):
        """Descriptors that depend only on the prompt lengths and budgets, built
        once and kept on the device (selection and compaction items, offsets)."""
        s = self.shape
        L = s.n_layers
        key = (tuple(lens), tuple(tuple(b) for b in budgets))
        plan = self._plans.get(key)
        if plan is not None:
            return plan
        dev = self.device
        B = len(lens)
        T = int(sum(lens))
        cu = np.zeros(B + 1, dtype=np.int32)
        cu[1:] = np.cumsum(lens)
        keff = [[(n if budgets[b][l] is None else min(int(budgets[b][l]), n))
                 for l in range(L)] for b, n in enumerate(lens)]
        budgeted = [[budgets[b][l] is not None and budgets[b][l] < lens[b] for l in range(L)]
                    for b in range(B)]
        sel = np.zeros(B * L, dtype=kvs.SELECT_ITEM)
        comp = np.zeros(B * L, dtype=kvs.COMPACT_ITEM)
        idx_off = np.zeros((B, L), dtype=np.int64)
        off = row = toff = 0
        for b in range(B):
            for l in range(L):
                i = b * L + l
                sel[i] = (l * s.h_kv * T + cu[b], lens[b],
                          lens[b] if not budgeted[b][l] else int(budgets[b][l]), off)
                comp[i] = (l * T + cu[b], off, row, lens[b], keff[b][l], toff, 0)
                idx_off[b, l] = off
                off += s.h_kv * keff[b][l]
                row += keff[b][l]
                toff += blocks_for(keff[b][l])
        plan = {"T": T, "max_n": max(lens), "keff": keff, "budgeted": budgeted,
                "any_budget": [any(budgeted[b][l] for b in range(B)) for l in range(L)],
                "cu_d": torch.from_numpy(cu).to(dev), "sel_d": _u8(sel, dev),
                "comp_d": _u8(comp, dev), "idx_off": idx_off, "n_kept": off,
                "total_rows": row, "n_tables": toff}
        if len(self._plans) > 64:
            self._plans.clear()
        self._plans[key] = plan
        return plan

    def prefill_sparsify(self, q_layers: Sequence[torch.Tensor], k_layers: Sequence[torch.Tensor],
                         v_layers: Sequence[torch.Tensor], seq_lens: Sequence[int],
                         budgets: Sequence[Sequence[Optional[int]]], keep_outputs=False,
                         o_buf=None, ml_buf=None, select_scores: Optional[torch.Tensor] = None,
                         stream=None, timing=None, timing_layers=None,
                         ready: Optional[Sequence[Sequence[torch.cuda.Event]]] = None,
                         prefix_tokens: Optional[Sequence[Optional[np.ndarray]]] = None
                         ) -> PrefillResult:
        """q_layers[l]: [T][h_q][d] bf16, k/v_layers[l]: [T][h_kv][d] (T = sum of
        seq_lens, sequences packed).  budgets[b][l]: k_l for sequence b (None =
        full cache).  select_scores: optional [L][h_kv][T] scores to select on
        instead of the ones computed here.  o_buf: optional [L][T][h_q][d]
        buffer for every layer's attention output, or one [T][h_q][d] buffer
        that each layer overwrites (which rules out the single launch over
        all layers).  ml_buf: optional pair of [L][h_q][T] fp32 buffers for
        every layer's m and l.  timing: optional
        dict of lists "attn" / "scores" that receive a (start, end) CUDA event
        pair around the prefill-attention launches of the layers in
        timing_layers (every layer when None; the one launch over all layers
        when inputs are resident and stacked, "attn_layers" receiving the
        layers each timed launch covers) / around each window-score
        launch (one per run of consecutive budgeted layers; per layer when
        `ready` is given).  An event
        recorded between two launches ends the overlap of the second one's
        start with the first one's tail, so timing a few layers disturbs the
        stream less.
        ready: optional per-layer lists of CUDA events (see upload_layers);
        layer l's launches wait for every event in ready[l], so the layers'
        inputs may still be on their way to the device when this is called.
        prefix_tokens: optional per-sequence host arrays of the prompt's token
        ids (None for a sequence: no prefix lookup): the full blocks of every
        layer that keeps all its tokens are looked up as prefix blocks
        (kvs_alloc_prefix_blocks, the layer's index as key); blocks found are
        shared, not written again by the compaction."""
        s = self.shape
        dev = self.device
        L = s.n_layers
        lens = [int(x) for x in seq_lens]
        B = len(lens)
        plan = self._plan(lens, budgets)
        T, cu_d, max_n = plan["T"], plan["cu_d"], plan["max_n"]
        keff, budgeted, any_budget = plan["keff"], plan["budgeted"], plan["any_budget"]

        # O of every layer ([L][T][h_q][d]) unless the caller passes one
        # [T][h_q][d] buffer that every layer overwrites
        o_all = None
        if keep_outputs or o_buf is None:
            o_all = torch.empty((L, T, s.h_q, s.d), dtype=torch.bfloat16, device=dev)
        elif o_buf.dim() == 4:
            if tuple(o_buf.shape) != (L, T, s.h_q, s.d):
                raise ValueError(f"o_buf must be [{L}][{T}][{s.h_q}][{s.d}] or [{T}][{s.h_q}][{s.d}]")
            o_all = o_buf
        # scores of layers without a budget are never read (their selection is
        # the identity), so the buffer needs no clearing
        scores = torch.empty((L, s.h_kv, T), dtype=torch.float32, device=dev)
        # every layer's m and l stay until the window scores read them after
        # the prefill loop
        if ml_buf is None or keep_outputs:
            m_all = torch.empty((L, s.h_q, T), dtype=torch.float32, device=dev)
            l_all = torch.empty_like(m_all)
        else:
            m_all, l_all = ml_buf
            if tuple(m_all.shape) != (L, s.h_q, T) or tuple(l_all.shape) != (L, s.h_q, T):
                raise ValueError(f"ml_buf must be two [{L}][{s.h_q}][{T}] fp32 tensors")
        # inputs resident and every layer's Q, K, V (and O) slices of one
        # buffer each: one persistent launch over all layers' work items, so
        # the launch, start-up and uneven tail are paid once, not per layer
        qa, ka, va = _stacked_view(q_layers), _stacked_view(k_layers), _stacked_view(v_layers)
        one_launch = (ready is None and o_all is not None and qa is not None and ka is not None
                      and va is not None)
        if one_launch:
            ev = _events(timing, "attn", stream)
            kvs.kvs_prefill_attn_lse_layers(qa, ka, va, o_all, m_all, l_all, cu_d, B, max_n, T,
                                            s.h_q, s.h_kv, s.d, s.scale, L, self.status, stream)
            _close(ev, stream)
            if timing is not None:
                timing.setdefault("attn_layers", []).append(L)
        for l in range(L if not one_launch else 0):
            m, lsum = m_all[l], l_all[l]
            o = o_all[l] if o_all is not None else o_buf
            if ready is not None:
                for e in ready[l]:
                    (torch.cuda.current_stream() if stream is None else stream).wait_event(e)
            tl = timing if (timing_layers is None or l in timing_layers) else None
            ev = _events(tl, "attn", stream)
            kvs.kvs_prefill_attn_lse(q_layers[l], k_layers[l], v_layers[l], o, m, lsum, cu_d, B,
                                     max_n, T, s.h_q, s.h_kv, s.d, s.scale, self.status, stream)
            _close(ev, stream)
            if tl is not None:
                timing.setdefault("attn_layers", []).append(1)
            if ready is not None and any_budget[l]:
                # inputs still arriving: the GPU waits for the next layer's
                # copies anyway, so this layer's scores go in that gap
                ev = _events(timing, "scores", stream)
                kvs.kvs_window_scores(q_layers[l], k_layers[l], m, lsum, scores[l], cu_d, B, max_n,
                                      T, s.h_q, s.h_kv, s.d, s.alpha, s.scale, self.status, stream)
                _close(ev, stream)

        # inputs resident: the window scores of every budgeted layer after the
        # prefill loop.  A layer's scores need only its own q, k, m and l, so
        # each run of consecutive budgeted layers is one launch (when their q
        # and k are slices of one buffer) instead of a latency-bound launch
        # between every two prefills
        l0 = 0 if ready is None else L
        while l0 < L:
            if not any_budget[l0]:
                l0 += 1
                continue
            l1 = l0
            while l1 < L and any_budget[l1]:
                l1 += 1
            qs, ks = _stacked_view(q_layers[l0:l1]), _stacked_view(k_layers[l0:l1])
            ev = _events(timing, "scores", stream)
            if qs is not None and ks is not None:
                kvs.kvs_window_scores_layers(qs, ks, m_all[l0:l1], l_all[l0:l1], scores[l0:l1],
                                             cu_d, B, max_n, T, s.h_q, s.h_kv, s.d, s.alpha,
                                             s.scale, l1 - l0, self.status, stream)
            else:
                for l in range(l0, l1):
                    kvs.kvs_window_scores(q_layers[l], k_layers[l], m_all[l], l_all[l], scores[l],
                                          cu_d, B, max_n, T, s.h_q, s.h_kv, s.d, s.alpha, s.scale,
                                          self.status, stream)
            _close(ev, stream)
            l0 = l1

        # selection over every (sequence, layer) item
        kept = torch.empty(max(plan["n_kept"], 1), dtype=torch.int32, device=dev)
        src_scores = scores if select_scores is None else select_scores
        kvs.kvs_select_topk(src_scores, T, plan["sel_d"], B * L, s.h_kv, s.recent, kept,
                            self.status, stream)

        # host allocator: sequence by sequence, layer by layer
        tables: List[List[List[int]]] = []
        flat = np.empty(max(plan["n_tables"], 1), dtype=np.int32)
        toff = 0
        n_hits = 0
        for b in range(B):
            per_layer = []
            toks = None if prefix_tokens is None else prefix_tokens[b]
            for l in range(L):
                nb = blocks_for(keff[b][l])
                if toks is not None and not budgeted[b][l]:
                    n_full = keff[b][l] // BLOCK
                    pre, hit = self.alloc.prefix_blocks(l, np.asarray(toks)[:n_full * BLOCK])
                    ids = np.concatenate([pre, self.alloc.alloc_many(nb - n_full)])
                    # blocks found already hold these rows: the compaction skips them
                    flat[toff:toff + ids.size] = ids
                    flat[toff:toff + n_full][hit] = kvs.KVS_BLOCK_SKIP
                    n_hits += int(hit.sum())
                else:
                    ids = self.alloc.alloc_many(nb)
                    flat[toff:toff + ids.size] = ids
                toff += ids.size
                per_layer.append(ids.tolist())
            tables.append(per_layer)
        tab_d = torch.from_numpy(flat).pin_memory().to(dev, non_blocking=True)

        k_all = _stacked(k_layers)
        v_all = _stacked(v_layers)
        if self.kv_fp8:
            kvs.kvs_compact_blocks_fp8(k_all, v_all, plan["comp_d"], B * L, plan["total_rows"],
                                       s.h_kv, s.d, kept, tab_d, self.k_pool, self.v_pool,
                                       self.k_scale, self.v_scale, self.num_blocks, self.status,
                                       stream)
        else:
            kvs.kvs_compact_blocks(k_all, v_all, plan["comp_d"], B * L, plan["total_rows"],
                                   s.h_kv, s.d, kept, tab_d, self.k_pool, self.v_pool,
                                   self.num_blocks, self.status, stream)
        idx_off = plan["idx_off"]
        res = PrefillResult(tables=tables, k_eff=keff, kept_idx=kept, idx_off=idx_off,
                            scores=scores, prefix_hits=n_hits)
        if keep_outputs:
            res.m, res.l, res.o = list(m_all), list(l_all), list(o_all)
        return res


def upload_layers(host: Sequence[Sequence[torch.Tensor]], dev: Sequence[Sequence[torch.Tensor]],
                  streams: Sequence[torch.cuda.Stream]) -> List[List[torch.cuda.Event]]:
    """Layer-wise upload of a prompt's inputs: host[i][l] (pinned host memory)
    is copied into dev[i][l] for every tensor kind i (e.g. Q, K, V), layer by
    layer, kind i on streams[i % len(streams)].  Returns, per layer, one event
    per copy stream that carried part of it; prefill_sparsify(ready=...)
    starts layer l once they have completed, so layer l computes while layers
    l+1, ... are still being copied.  Each copy stream first waits for the
    work already queued on the current stream."""
    cur = torch.cuda.current_stream()
    for st in streams:
        st.wait_stream(cur)
    events = []
    for l in range(len(dev[0])):
        used = []
        for i, (h, d) in enumerate(zip(host, dev)):
            st = streams[i % len(streams)]
            with torch.cuda.stream(st):
                d[l].copy_(h[l], non_blocking=True)
            if st not in used:
                used.append(st)
        # one event per copy stream that carried a part of this layer
        per_layer = []
        for st in used:
            e = torch.cuda.Event()
            e.record(st)
            per_layer.append(e)
        events.append(per_layer)
    return events


def _raw_stream(stream, device_index):
    """cudaStream_t of `stream`, else of the current stream (the cheapest
    lookup torch offers, with the public one as the fallback)."""
    if stream is not None:
        return stream.cuda_stream
    get = getattr(torch._C, "_cuda_getCurrentRawStream", None)
    if get is not None:
        return get(device_index)
    return torch.cuda.current_stream().cuda_stream


def _events(timing, key, stream):
    if timing is None:
        return None
    st = torch.cuda.current_stream() if stream is None else stream
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(st)
    timing.setdefault(key, []).append((a, b))
    return b


def _close(ev, stream):
    if ev is not None:
        ev.record(torch.cuda.current_stream() if stream is None else stream)


def _stacked_view(layers):
    """[n][T][h][d] view of per-layer tensors that are consecutive slices of
    one contiguous buffer, else None."""
    first = layers[0]
    n = len(layers)
    base = first.data_ptr()
    step = first.numel() * first.element_size()
    storage = first.untyped_storage().data_ptr()
    if (first.is_contiguous()
            and all(t.untyped_storage().data_ptr() == storage and t.is_contiguous()
                    and t.shape == first.shape and t.data_ptr() == base + i * step
                    for i, t in enumerate(layers))):
        return torch.as_strided(first, (n, *first.shape), (first.numel(), *first.stride()))
    return None


def _stacked(layers):
    """View per-layer [T][h][d] tensors as one [L*T][h][d] tensor when they are
    consecutive slices of one contiguous buffer (one storage: separate
    allocations that merely sit next to each other do not count); otherwise
    concatenate."""
    first = layers[0]
    T = first.shape[0]
    n = len(layers)
    base = first.data_ptr()
    step = first.numel() * first.element_size()
    storage = first.untyped_storage().data_ptr()
    if (first.is_contiguous()
            and all(t.untyped_storage().data_ptr() == storage and t.is_contiguous()
                    and t.data_ptr() == base + i * step for i, t in enumerate(layers))):
        return torch.as_strided(first, (n * T, *first.shape[1:]),
                                (first.stride(0), first.stride(1), first.stride(2)))
    return torch.cat(list(layers), dim=0)


class DecodeBatch:
    """Decode items (one per (stream, layer)) over an Engine's pools."""

    def __init__(self, eng: Engine, n_streams: int, max_len: int, n_layers: Optional[int] = None,
                 layer_order: bool = False, interleave: bool = False):
        """n_layers: layers per stream (default: the engine's), e.g. only the
        full-cache layers when the budgeted ones run in an EvictingDecode.
        layer_order: items are numbered layer-major (item = layer * n_streams
        + stream; the step's q / k_new / v_new and its output follow that
        order) and each step issues one decode launch per layer over that
        layer's n_streams items, in layer order, after one host preparation
        of every item (which therefore allocates blocks layer by layer).  This
        is the launch sequence of a model, whose layer l + 1 query depends on
        layer l's output; without it, one launch covers every item of the
        step (stream-major numbering).
        interleave: the layer-major numbering with one launch over every item:
        streams that share blocks (parallel samples of one prompt, in
        consecutive slots) then have their items next to one another in the
        launch's split, so their reads of the shared blocks fall together and
        hit L2."""
        s = eng.shape
        self.eng = eng
        self.n_streams = n_streams
        self.n_layers = s.n_layers if n_layers is None else int(n_layers)
        self.n_items = n_streams * self.n_layers
        self.layer_order = bool(layer_order)
        self.item_major = self.layer_order or bool(interleave)
        self.shape_ = s
        self.max_len = max_len
        self.max_blocks = blocks_for(max_len)
        dev = eng.device
        self.tables_h = np.full((self.n_items, self.max_blocks), -1, dtype=np.int32)
        self.lens_h = np.zeros(self.n_items, dtype=np.int32)
        self.tables_d = torch.zeros((self.n_items, self.max_blocks), dtype=torch.int32, device=dev)
        self.lens_d = [torch.zeros(self.n_items, dtype=torch.int32, device=dev) for _ in range(2)]
        self.cur = 0
        # pinned staging for the per-step table patches and copy-on-write pairs:
        # a ring, each slot guarded by an event so the host never rewrites a
        # buffer whose upload has not run yet
        self._ring = 4
        self.patch_h = [torch.empty(self.n_items, dtype=torch.int32).pin_memory()
                        for _ in range(self._ring)]
        self.cow_h = [torch.empty(2 * self.n_items, dtype=torch.int32).pin_memory()
                      for _ in range(self._ring)]
        self._ev = [None] * self._ring
        self._slot = 0
        self._patch_np = [t.numpy() for t in self.patch_h]
        self._cow_np = [t.numpy() for t in self.cow_h]
        self.patch_d = torch.empty(self.n_items, dtype=torch.int32, device=dev)
        self.cow_src = np.zeros(self.n_items, dtype=np.int32)
        self.cow_dst = np.zeros(self.n_items, dtype=np.int32)
        self.cow_d = torch.empty(2 * self.n_items, dtype=torch.int32, device=dev)
        self.ws_bytes = kvs.kvs_paged_decode_workspace_size(self.n_items, s.h_q, s.h_kv, s.d)
        self.ws = torch.zeros(max(self.ws_bytes, 256), dtype=torch.uint8, device=dev)
        kvs.kvs_workspace_zero(self.ws, self.ws_bytes)
        self.out = torch.empty((self.n_items, s.h_q, s.d), dtype=torch.bfloat16, device=dev)
        self._graphs = None
        # the native step's fixed arguments, looked up once (raw addresses of
        # buffers this object owns for its whole life)
        self._nat = (eng.alloc._h, self.tables_h.ctypes.data, self.lens_h.ctypes.data,
                     [t.data_ptr() for t in self.patch_h], [t.data_ptr() for t in self.cow_h],
                     self.patch_d.data_ptr(), self.cow_d.data_ptr(), eng.k_pool.data_ptr(),
                     eng.v_pool.data_ptr(), self.tables_d.data_ptr(),
                     [t.data_ptr() for t in self.lens_d], self.out.data_ptr(),
                     self.ws.data_ptr(), eng.status.data_ptr())
        self._counts = (ctypes.c_int32(), ctypes.c_int32())
        self._count_refs = tuple(ctypes.byref(c) for c in self._counts)
        self._lib = kvs.library()
        self._dev_index = self.eng.device.index if self.eng.device.index is not None \
            else torch.cuda.current_device()

    def _native_step(self, q, k_new, v_new, stream):
        s = self.shape_
        for t, shape in ((q, (self.n_items, s.h_q, s.d)), (k_new, (self.n_items, s.h_kv, s.d)),
                         (v_new, (self.n_items, s.h_kv, s.d))):
            if (not t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous()
                    or tuple(t.shape) != shape):
                raise ValueError(f"decode inputs must be contiguous CUDA bf16 {shape} tensors")
        slot = self._slot
        if self._ev[slot] is not None:
            # the copies that last read this slot's staging have run; once
            # seen, the slot needs no further wait
            self._ev[slot].synchronize()
            self._ev[slot] = None
        (alloc, tables_h, lens_h, patch_h, cow_h, patch_d, cow_d, k_pool, v_pool, tables_d,
         lens_d, out, ws, status) = self._nat
        raw_stream = _raw_stream(stream, self._dev_index)
        n_cow, n_patch = self._counts
        if self.eng.kv_fp8:
            kvs._check(self._lib.kvs_decode_step_fp8(
                alloc, tables_h, lens_h, patch_h[slot], cow_h[slot], patch_d, cow_d,
                q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(), k_pool, v_pool,
                self.eng.k_scale.data_ptr(), self.eng.v_scale.data_ptr(), self.eng.num_blocks,
                tables_d, self.max_blocks, lens_d[self.cur], lens_d[1 - self.cur], self.n_items,
                s.h_q, s.h_kv, s.d, s.scale, out, ws, self.ws_bytes, status,
                self._count_refs[0], self._count_refs[1], raw_stream))
        else:
            kvs._check(self._lib.kvs_decode_step(
                alloc, tables_h, lens_h, patch_h[slot], cow_h[slot], patch_d, cow_d,
                q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(), k_pool, v_pool,
                self.eng.num_blocks, tables_d, self.max_blocks, lens_d[self.cur],
                lens_d[1 - self.cur], self.n_items, s.h_q, s.h_kv, s.d, s.scale, out, ws,
                self.ws_bytes, status, self._count_refs[0], self._count_refs[1], raw_stream))
        if n_patch.value or n_cow.value:
            # this slot's staging buffers are read by copies queued above
            ev = torch.cuda.Event()
            ev.record(torch.cuda.current_stream() if stream is None else stream)
            self._ev[slot] = ev
            self._slot = (slot + 1) % self._ring
        self.cur = 1 - self.cur
        return self.out

    # ------------------------------------------------------------ CUDA graphs
    def _item(self, slot: int, layer: int) -> int:
        return layer * self.n_streams + slot if self.item_major else slot * self.n_layers + layer

    def _decode_launch(self, q, k_new, v_new, patch, lens, lens_next, stream=None):
        """The step's decode over every item, on the engine's pool type: one
        call, or in layer order one call per layer over its rows (each call
        reuses the workspace; the calls are ordered on the stream)."""
        eng, s = self.eng, self.eng.shape
        groups = ([slice(l * self.n_streams, (l + 1) * self.n_streams)
                   for l in range(self.n_layers)] if self.layer_order else [slice(None)])

        def part(t, r):
            return None if t is None else t[r]

        for r in groups:
            n = self.n_streams if self.layer_order else self.n_items
            if eng.kv_fp8:
                kvs.kvs_paged_decode_fp8(q[r], part(k_new, r), part(v_new, r), eng.k_pool,
                                         eng.v_pool, eng.k_scale, eng.v_scale, eng.num_blocks,
                                         self.tables_d[r], self.max_blocks, part(patch, r),
                                         lens[r], part(lens_next, r), n, s.h_q, s.h_kv, s.d,
                                         s.scale, self.out[r], self.ws, self.ws_bytes, eng.status,
                                         stream)
            else:
                kvs.kvs_paged_decode(q[r], part(k_new, r), part(v_new, r), eng.k_pool, eng.v_pool,
                                     eng.num_blocks, self.tables_d[r], self.max_blocks,
                                     part(patch, r), lens[r], part(lens_next, r), n, s.h_q,
                                     s.h_kv, s.d, s.scale, self.out[r], self.ws, self.ws_bytes,
                                     eng.status, stream)

    def capture_graphs(self):
        """Capture the decode step as CUDA graphs, so that a step costs the host
        one graph launch instead of the library's launches (the method's
        serving loop runs in CUDA-graph mode).  Four graphs: the two
        directions of the length ping-pong, each with and without the upload
        of the allocator's table patch.  Afterwards step() replays the
        matching graph, and launches eagerly only on a step where a block
        needs copy-on-write (its count of copies varies).  The graphs read
        the step's inputs from the fixed buffers self.q_in, self.k_in,
        self.v_in (step() copies other tensors into them) and the patch from
        two pinned buffers, one per direction."""
        s, dev = self.eng.shape, self.eng.device
        n = self.n_items
        self.q_in = torch.zeros((n, s.h_q, s.d), dtype=torch.bfloat16, device=dev)
        self.k_in = torch.zeros((n, s.h_kv, s.d), dtype=torch.bfloat16, device=dev)
        self.v_in = torch.zeros_like(self.k_in)
        self._patch_g = [torch.full((n,), -1, dtype=torch.int32).pin_memory() for _ in range(2)]
        self._patch_g_np = [t.numpy() for t in self._patch_g]
        self._gev = [None, None]
        # one-time library set-up (kernel attributes, tensor maps) outside the
        # capture: a call that appends nothing and writes only out and the
        # workspace leaves the caches as they are
        self._decode_launch(self.q_in, None, None, None, self.lens_d[self.cur], None)
        torch.cuda.synchronize()
        graphs = {}
        for cur in (0, 1):
            for with_patch in (False, True):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    if with_patch:
                        self.patch_d.copy_(self._patch_g[cur], non_blocking=True)
                    self._decode_launch(self.q_in, self.k_in, self.v_in,
                                        self.patch_d if with_patch else None, self.lens_d[cur],
                                        self.lens_d[1 - cur])
                graphs[(cur, with_patch)] = g
        self._graphs = graphs

    def set_stream(self, slot: int, tables: List[List[int]], lens: List[int]):
        """Install a stream's per-layer tables (host copy + device rows)."""
        L = self.n_layers
        rows = [self._item(slot, l) for l in range(L)]
        for l, i in enumerate(rows):
            self.tables_h[i, :] = -1
            self.tables_h[i, :len(tables[l])] = tables[l]
            self.lens_h[i] = lens[l]
        if self.item_major:
            idx = torch.tensor(rows, dtype=torch.long, device=self.eng.device)
            self.tables_d[idx] = torch.from_numpy(self.tables_h[rows]).to(self.eng.device)
            self.lens_d[self.cur][idx] = torch.from_numpy(self.lens_h[rows]).to(self.eng.device)
        else:
            r = slice(slot * L, (slot + 1) * L)
            self.tables_d[r] = torch.from_numpy(self.tables_h[r]).to(self.eng.device)
            self.lens_d[self.cur][r] = torch.from_numpy(self.lens_h[r]).to(self.eng.device)

    def stream_tables(self, slot: int) -> List[List[int]]:
        out = []
        for l in range(self.n_layers):
            i = self._item(slot, l)
            nb = blocks_for(int(self.lens_h[i]))
            out.append(self.tables_h[i, :nb].tolist())
        return out

    def retire(self, slot: int):
        for t in self.stream_tables(slot):
            for b in t:
                self.eng.alloc.decref(b)
        rows = [self._item(slot, l) for l in range(self.n_layers)]
        self.tables_h[rows] = -1
        self.lens_h[rows] = 0

    def step(self, q, k_new, v_new, stream=None, timing=None):
        """One decode step for every item: q [n_items][h_q][d], k_new/v_new
        [n_items][h_kv][d] bf16 on the device.  Returns the output tensor.
        timing: optional list receiving a (start, end) event pair around the
        decode kernel(s).  Without graphs or timing, and not in layer order,
        the step is one native call (kvs_decode_step: host preparation,
        uploads and decode)."""
        if self._graphs is None and timing is None and not self.layer_order:
            return self._native_step(q, k_new, v_new, stream)
        eng, s = self.eng, self.eng.shape
        n = self.n_items
        slot = self._slot
        patch_t, cow_t = self.patch_h[slot], self.cow_h[slot]
        patch_np = self._patch_np[slot]
        if self._graphs is not None:
            # the patch goes to this direction's fixed pinned buffer, last read
            # by the replay two steps ago
            if self._gev[self.cur] is not None:
                self._gev[self.cur].synchronize()
            patch_t, patch_np = self._patch_g[self.cur], self._patch_g_np[self.cur]
        if self._ev[slot] is not None:
            self._ev[slot].synchronize()
        n_cow, n_patch = eng.alloc.decode_prepare(self.tables_h, self.lens_h, patch_np,
                                                  self.cow_src, self.cow_dst,
                                                  with_patch_count=True)
        cur_stream = torch.cuda.current_stream() if stream is None else stream
        nxt = 1 - self.cur
        if self._graphs is not None and n_cow == 0:
            with torch.cuda.stream(cur_stream):
                for src, dst in ((q, self.q_in), (k_new, self.k_in), (v_new, self.v_in)):
                    if src is not dst:
                        dst.copy_(src, non_blocking=True)
                if timing is not None:
                    a = torch.cuda.Event(enable_timing=True)
                    b = torch.cuda.Event(enable_timing=True)
                    a.record(cur_stream)
                self._graphs[(self.cur, bool(n_patch))].replay()
                if timing is not None:
                    b.record(cur_stream)
                    timing.append((a, b))
                if n_patch:
                    ev = torch.cuda.Event()
                    ev.record(cur_stream)
                    self._gev[self.cur] = ev
            self.cur = nxt
            self.lens_h += 1
            return self.out
        patch_arg = None
        if n_patch or n_cow:
            self._slot = (slot + 1) % self._ring
            with torch.cuda.stream(cur_stream):
                self.patch_d.copy_(patch_t, non_blocking=True)
                patch_arg = self.patch_d
                if n_cow:
                    cow = self._cow_np[slot]
                    cow[:n_cow] = self.cow_src[:n_cow]
                    cow[n_cow:2 * n_cow] = self.cow_dst[:n_cow]
                    self.cow_d[:2 * n_cow].copy_(cow_t[:2 * n_cow], non_blocking=True)
                    if eng.kv_fp8:
                        kvs.kvs_copy_blocks_fp8(self.cow_d[:n_cow], self.cow_d[n_cow:2 * n_cow],
                                                n_cow, eng.k_pool, eng.v_pool, eng.k_scale,
                                                eng.v_scale, eng.num_blocks, s.h_kv, s.d,
                                                eng.status, cur_stream)
                    else:
                        kvs.kvs_copy_blocks(self.cow_d[:n_cow], self.cow_d[n_cow:2 * n_cow],
                                            n_cow, eng.k_pool, eng.v_pool, eng.num_blocks,
                                            s.h_kv, s.d, eng.status, cur_stream)
                ev = torch.cuda.Event()
                ev.record(cur_stream)
                self._ev[slot] = ev
                if self._graphs is not None:
                    self._gev[self.cur] = ev
        if timing is not None:
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(cur_stream)
        self._decode_launch(q, k_new, v_new, patch_arg, self.lens_d[self.cur],
                            self.lens_d[nxt], cur_stream)
        if timing is not None:
            b.record(cur_stream)
            timing.append((a, b))
        self.cur = nxt
        self.lens_h += 1
        return self.out


class EvictingDecode:
    """Decode of budgeted (stream, layer) items with a fixed budget: the cache
    of each keeps exactly its k_l slots per KV head; each step's new token
    takes the slot of the lowest-scoring token outside the recent window, the
    step attends over the k_l slots, and its attention probabilities are added
    to the scores (kvs_evict_place, then kvs_paged_decode_logits and
    kvs_decode_scores_from_logits; or kvs_paged_decode and kvs_decode_scores,
    which recompute the logits from K).

    Sources: Novita AI, "How KV Sparsity achieves 1.5x acceleration for vLLM",
    section "Key techniques 1" (later layers replace their lowest-scoring KVs
    with a sliding-window strategy) and section "Key techniques 2" (the
    decode-side PagedAttention works toward the same score).  The score of a
    prompt token starts at its prefill window score; a decode token's at 0.
    Layers without a budget keep growing through DecodeBatch."""

    def __init__(self, eng: Engine, res: PrefillResult, seq: int, seq_start: int, prompt_len: int,
                 layers: Sequence[int], fused: bool = True):
        """fused: the decode launch writes the slots' logits and each query
        head's softmax denominator, and the score update reads them
        (kvs_paged_decode_logits); otherwise the update recomputes the logits
        from K (kvs_decode_scores).  Over FP8 pools only the fused form is
        built (kvs_evict_place_fp8, kvs_paged_decode_logits_fp8)."""
        s = eng.shape
        if eng.kv_fp8 and not fused:
            raise NotImplementedError("over FP8 pools the score update reads the decode's logits "
                                      "(fused=True)")
        self.fused = fused
        dev = eng.device
        self.eng, self.layers = eng, list(layers)
        n = len(self.layers)
        self.n_items = n
        keff = [int(res.k_eff[seq][l]) for l in self.layers]
        if any(k >= prompt_len for k in keff):
            raise ValueError("every layer of an EvictingDecode needs a budget below the prompt")
        if any(k < s.recent for k in keff):
            raise ValueError("a budget below the recent window leaves nothing to replace")
        self.max_slots = max(keff)
        self.max_blocks = blocks_for(self.max_slots)
        tables = np.full((n, self.max_blocks), -1, dtype=np.int32)
        for i, l in enumerate(self.layers):
            t = res.tables[seq][l]
            tables[i, :len(t)] = t
        self.tables_h = tables
        self.tables_d = torch.from_numpy(tables).to(dev)
        self.lens_d = torch.tensor(keff, dtype=torch.int32, device=dev)
        self.new_pos = torch.full((n,), prompt_len, dtype=torch.int32, device=dev)
        self.score = torch.zeros((n, s.h_kv, self.max_slots), dtype=torch.float32, device=dev)
        self.pos = torch.full((n, s.h_kv, self.max_slots), -1, dtype=torch.int32, device=dev)
        for i, l in enumerate(self.layers):
            off, ke = int(res.idx_off[seq, l]), keff[i]
            idx = res.kept_idx[off:off + s.h_kv * ke].view(s.h_kv, ke).long()
            self.pos[i, :, :ke] = idx.int()
            self.score[i, :, :ke] = res.scores[l].gather(1, seq_start + idx)
        self.out = torch.empty((n, s.h_q, s.d), dtype=torch.bfloat16, device=dev)
        self.ws_bytes = kvs.kvs_paged_decode_workspace_size(n, s.h_q, s.h_kv, s.d)
        self.ws = torch.zeros(max(self.ws_bytes, 256), dtype=torch.uint8, device=dev)
        self.sws_bytes = kvs.kvs_decode_scores_workspace_size(n, s.h_q, s.h_kv, self.max_slots)
        self.sws = torch.empty(max(self.sws_bytes, 256), dtype=torch.uint8, device=dev)
        self.logit_ld = (self.max_slots + 3) // 4 * 4
        self.logits = torch.empty((n, s.h_kv, s.h_q // s.h_kv, self.logit_ld), dtype=torch.float32,
                                  device=dev)
        self.lse = torch.empty((n, s.h_q), dtype=torch.float32, device=dev)

    def step(self, q, k_new, v_new, stream=None):
        """q [n_items][h_q][d], k_new / v_new [n_items][h_kv][d] bf16 (items in
        the order of `layers`).  Returns the attention output."""
        eng, s = self.eng, self.eng.shape
        n = self.n_items
        if eng.kv_fp8:
            kvs.kvs_evict_place_fp8(k_new, v_new, eng.k_pool, eng.v_pool, eng.k_scale, eng.v_scale,
                                    eng.num_blocks, self.tables_d, self.max_blocks, self.lens_d,
                                    self.new_pos, self.score, self.pos, self.max_slots, n, s.h_kv,
                                    s.d, s.recent, eng.status, stream)
            kvs.kvs_paged_decode_logits_fp8(q, None, None, eng.k_pool, eng.v_pool, eng.k_scale,
                                            eng.v_scale, eng.num_blocks, self.tables_d,
                                            self.max_blocks, None, self.lens_d, None, n, s.h_q,
                                            s.h_kv, s.d, s.scale, self.out, self.ws, self.ws_bytes,
                                            self.logits, self.logit_ld, self.lse, eng.status,
                                            stream)
            kvs.kvs_decode_scores_from_logits(self.logits, self.logit_ld, self.lse, self.lens_d,
                                              self.score, self.new_pos, self.max_slots, n, s.h_q,
                                              s.h_kv, eng.status, stream)
            return self.out
        kvs.kvs_evict_place(k_new, v_new, eng.k_pool, eng.v_pool, eng.num_blocks, self.tables_d,
                            self.max_blocks, self.lens_d, self.new_pos, self.score, self.pos,
                            self.max_slots, n, s.h_kv, s.d, s.recent, eng.status, stream)
        if self.fused:
            kvs.kvs_paged_decode_logits(q, None, None, eng.k_pool, eng.v_pool, eng.num_blocks,
                                        self.tables_d, self.max_blocks, None, self.lens_d, None, n,
                                        s.h_q, s.h_kv, s.d, s.scale, self.out, self.ws,
                                        self.ws_bytes, self.logits, self.logit_ld, self.lse,
                                        eng.status, stream)
            kvs.kvs_decode_scores_from_logits(self.logits, self.logit_ld, self.lse, self.lens_d,
                                              self.score, self.new_pos, self.max_slots, n, s.h_q,
                                              s.h_kv, eng.status, stream)
            return self.out
        kvs.kvs_paged_decode(q, None, None, eng.k_pool, eng.v_pool, eng.num_blocks, self.tables_d,
                             self.max_blocks, None, self.lens_d, None, n, s.h_q, s.h_kv, s.d,
                             s.scale, self.out, self.ws, self.ws_bytes, eng.status, stream)
        kvs.kvs_decode_scores(q, eng.k_pool, eng.num_blocks, self.tables_d, self.max_blocks,
                              self.lens_d, self.score, self.new_pos, self.max_slots, n, s.h_q,
                              s.h_kv, s.d, s.scale, self.sws, self.sws_bytes, eng.status, stream)
        return self.out

    def release(self):
        """Give the items' blocks back to the allocator."""
        for i in range(self.n_items):
            for b in self.tables_h[i]:
                if b >= 0:
                    self.eng.alloc.decref(int(b))
