"""CPU oracle for layer-wise KV-cache sparsification over a paged KV cache.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, single-threaded
restatement in float64 numpy of what the hot path computes, written from the
two sources the method is described in:

* Novita AI, "How KV Sparsity achieves 1.5x acceleration for vLLM"
  (sections "System model", "Key techniques 1: layer-wise sparsity and tensor
  parallelism", "Key techniques 2: attention modification"), and
* Ultralytics glossary, "PagedAttention" (sections "How paging works",
  including its worked example, "Block sharing between sequences" and
  "Related techniques").

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` import it.  It shares no code with the CUDA library and
imports nothing from it; its only shared dependency is the seeded input
generator in ``synth/``.

Modules
-------
attention : prefill rows (O, m, l) and decode attention, explicit softmax.
scoring   : window scores S over the last alpha queries.
selection : per-(layer, KV head) top-k_l with a forced recent window.
paging    : list-based block pool (FIFO free list, ref counts, copy-on-write),
            compaction into 16-token blocks and table gathers.
flow      : the step orders that tie these together (prefill+sparsify of a
            sequence, one decode step, retirement).
eviction  : decode-time scores and fixed-budget replacement in budgeted layers.
fp8       : the 8-bit (e4m3, per-row scale) storage of cached keys and values.

Every function is pinned by a ``-m "not gpu"`` test against something other
than itself (closed forms, library routines, brute force, the worked paging
example); none is "parity unpinned".
"""
from .attention import prefill_rows, decode_attention  # noqa: F401
from .scoring import window_scores  # noqa: F401
from .selection import select_kept  # noqa: F401
from .paging import BlockPool, OutOfBlocks, compact, gather_rows, blocks_for  # noqa: F401
from . import flow  # noqa: F401
from . import eviction  # noqa: F401
from . import fp8  # noqa: F401
