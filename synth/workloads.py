"""Workload shapes and seeded bf16 draws.

Every tensor is identified by a tuple ``(workload id, sequence, layer, kind,
sample)`` and drawn from its own counter-based Philox stream, in fixed-size
chunks so that the bytes do not depend on how many threads draw them.  Values
are N(0, 1) in fp32, shifted by the sink construction below, then rounded to
bf16 (round-to-nearest-even) and returned as raw ``uint16`` bit patterns.

Sink construction (all workloads): a seeded unit vector ``u`` of length d;
the keys at sequence positions 0 and 37 get ``+6 u`` and every prompt query
gets ``+0.5 u``, added in fp32 before rounding.  Decode-step q/k/v are fresh
N(0, 1) draws without the sink shift.

The five workloads follow the shapes the Novita article ("How KV Sparsity
achieves 1.5x acceleration for vLLM") reports on: 4000/500 in/out tokens
(section "Inference performance"), concurrency 20 (same section), 7k-30k
inputs at >10x compression (section "Model accuracy", Table 3), Llama3-8B
attention shapes, the first three layers on full cache (section "Key
techniques 1", step-preparation phase), and parallel samples sharing prompt
blocks (Ultralytics glossary "PagedAttention", section "Block sharing").
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
from typing import Callable, Optional, Tuple

import numpy as np

KIND_Q, KIND_K, KIND_V, KIND_DQ, KIND_DK, KIND_DV, KIND_U, KIND_MISC = range(8)
SINK_POSITIONS = (0, 37)
SINK_KEY_GAIN = 6.0
SINK_QUERY_GAIN = 0.5
_CHUNK = 1 << 22  # elements per Philox stream chunk


# ----------------------------------------------------------------------------
# bf16 bit helpers (pure representation changes, no method arithmetic)
# ----------------------------------------------------------------------------
def bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even (inputs are finite)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    u = u + (((u >> 16) & 1) + np.uint32(0x7FFF))
    return (u >> 16).astype(np.uint16)


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def bf16_to_f64(b: np.ndarray) -> np.ndarray:
    return bf16_to_f32(b).astype(np.float64)


# ----------------------------------------------------------------------------
# workloads
# ----------------------------------------------------------------------------
@dataclass(frozen=True)
class Workload:
    name: str
    wid: int
    n_layers: int
    h_q: int
    h_kv: int
    d: int
    alpha: int
    recent: int
    prompt_lens: Tuple[int, ...]
    decode_steps: int
    budget_fn: Callable[[int, int], Optional[int]] = field(compare=False, repr=False)
    block: int = 16
    seed: int = 0
    concurrency: int = 0          # continuous batching: live sequences
    out_lens: Tuple[int, ...] = ()  # continuous batching: per-sequence outputs
    samples: int = 1              # shared prefix: parallel samples per prompt

    @property
    def group(self) -> int:
        return self.h_q // self.h_kv

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.d))

    def budget(self, layer: int, n: int) -> Optional[int]:
        """Kept-token budget k_l for a prompt of n tokens; None = full cache."""
        return self.budget_fn(layer, n)

    def k_eff(self, layer: int, n: int) -> int:
        k = self.budget(layer, n)
        return n if k is None else min(k, n)

    def budgeted(self, layer: int, n: int) -> bool:
        k = self.budget(layer, n)
        return k is not None and k < n


def _tiny_budget(layer, n):
    return None if layer == 0 else 64


def _linear_budget(layer, n):
    # layers 0-2 full; then 2048 falling by 64 per layer to 256 at layer 31
    return None if layer < 3 else 2048 - 64 * (layer - 3)


def _twelfth_budget(layer, n):
    return None if layer < 3 else n // 12


def tiny(seed: int = 0) -> Workload:
    return Workload("tiny", 0, 2, 4, 2, 64, 16, 16, (256,), 8, _tiny_budget, seed=seed)


def llama3_8b(seed: int = 0) -> Workload:
    return Workload("llama3-8b-4000/500", 1, 32, 32, 8, 128, 32, 32, (4000,), 500,
                    _linear_budget, seed=seed)


def continuous_batching(seed: int = 0) -> Workload:
    rng = _rng(seed, (2, 0, 0, KIND_MISC, 0))
    outs = tuple(int(x) for x in rng.integers(400, 601, size=40))
    return Workload("continuous-batching-20x", 2, 32, 32, 8, 128, 32, 32, (4000,) * 40, 0,
                    _linear_budget, seed=seed, concurrency=20, out_lens=outs)


def long_context(seed: int = 0) -> Workload:
    return Workload("long-context-7k-30k", 3, 32, 32, 8, 128, 32, 32,
                    (7000, 12000, 20000, 30000), 64, _twelfth_budget, seed=seed)


def shared_prefix(seed: int = 0) -> Workload:
    rng = _rng(seed, (4, 0, 0, KIND_MISC, 0))
    lens = tuple(int(x) for x in rng.integers(512, 16385, size=16))
    return Workload("shared-prefix-n3", 4, 32, 32, 8, 128, 32, 32, lens, 256,
                    _linear_budget, seed=seed, samples=3)


WORKLOADS = {
    "tiny": tiny,
    "llama3-8b": llama3_8b,
    "continuous-batching": continuous_batching,
    "long-context": long_context,
    "shared-prefix": shared_prefix,
}


# ----------------------------------------------------------------------------
# seeded draws
# ----------------------------------------------------------------------------
def _rng(seed: int, tid: Tuple[int, ...], chunk: int = 0) -> np.random.Generator:
    ss = np.random.SeedSequence([int(seed) & 0xFFFFFFFF, *[int(t) for t in tid], int(chunk)])
    return np.random.Generator(np.random.Philox(ss))


_POOL: Optional[ThreadPoolExecutor] = None


def _pool() -> ThreadPoolExecutor:
    global _POOL
    if _POOL is None:
        _POOL = ThreadPoolExecutor(max(1, min(16, os.cpu_count() or 1)))
    return _POOL


def _normal_f32(seed: int, tid: Tuple[int, ...], count: int) -> np.ndarray:
    out = np.empty(count, dtype=np.float32)
    starts = list(range(0, count, _CHUNK))

    def fill(ci: int):
        s = starts[ci]
        e = min(count, s + _CHUNK)
        out[s:e] = _rng(seed, tid, ci).standard_normal(e - s, dtype=np.float32)

    if len(starts) <= 1:
        for ci in range(len(starts)):
            fill(ci)
    else:
        list(_pool().map(fill, range(len(starts))))
    return out


def sink_direction(w: Workload) -> np.ndarray:
    """The seeded unit vector u (fp32, length d)."""
    g = _rng(w.seed, (w.wid, 0, 0, KIND_U, 0)).standard_normal(w.d)
    return (g / np.sqrt(np.sum(g * g))).astype(np.float32)


def _to_bits_threaded(x: np.ndarray) -> np.ndarray:
    flat = x.reshape(-1)
    out = np.empty(flat.shape, dtype=np.uint16)
    starts = list(range(0, flat.size, _CHUNK))

    def conv(s):
        out[s:s + _CHUNK] = bf16_bits(flat[s:s + _CHUNK])

    if len(starts) <= 1:
        for s in starts:
            conv(s)
    else:
        list(_pool().map(conv, starts))
    return out.reshape(x.shape)


def prefill_qkv(w: Workload, seq: int, layer: int, n: int):
    """Prompt Q [n, h_q, d], K and V [n, h_kv, d] as bf16 bit patterns."""
    u = sink_direction(w)
    q = _normal_f32(w.seed, (w.wid, seq, layer, KIND_Q, 0), n * w.h_q * w.d).reshape(n, w.h_q, w.d)
    k = _normal_f32(w.seed, (w.wid, seq, layer, KIND_K, 0), n * w.h_kv * w.d).reshape(n, w.h_kv, w.d)
    v = _normal_f32(w.seed, (w.wid, seq, layer, KIND_V, 0), n * w.h_kv * w.d).reshape(n, w.h_kv, w.d)
    q += np.float32(SINK_QUERY_GAIN) * u
    for p in SINK_POSITIONS:
        if p < n:
            k[p] += np.float32(SINK_KEY_GAIN) * u
    return _to_bits_threaded(q), _to_bits_threaded(k), _to_bits_threaded(v)


def decode_qkv(w: Workload, seq: int, layer: int, steps: int, sample: int = 0):
    """Decode-step q [steps, h_q, d], k and v [steps, h_kv, d] as bf16 bits."""
    q = _normal_f32(w.seed, (w.wid, seq, layer, KIND_DQ, sample), steps * w.h_q * w.d)
    k = _normal_f32(w.seed, (w.wid, seq, layer, KIND_DK, sample), steps * w.h_kv * w.d)
    v = _normal_f32(w.seed, (w.wid, seq, layer, KIND_DV, sample), steps * w.h_kv * w.d)
    return (_to_bits_threaded(q).reshape(steps, w.h_q, w.d),
            _to_bits_threaded(k).reshape(steps, w.h_kv, w.d),
            _to_bits_threaded(v).reshape(steps, w.h_kv, w.d))


def shuffled_block_order(num_blocks: int, seed: int = 0) -> np.ndarray:
    """A seeded permutation of physical block ids, used as an initial free list."""
    return _rng(seed, (99, 0, 0, KIND_MISC, num_blocks)).permutation(num_blocks).astype(np.int32)


def uniform_scores(shape, seed: int, tid: Tuple[int, ...], levels: int = 0) -> np.ndarray:
    """Seeded non-negative fp32 scores; with ``levels`` > 0 they take only that
    many distinct values, so that ties are frequent."""
    g = _rng(seed, (98, *tid))
    if levels > 0:
        return (g.integers(0, levels, size=shape).astype(np.float32) / np.float32(levels))
    return g.random(size=shape, dtype=np.float32)
