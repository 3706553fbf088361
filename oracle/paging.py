"""List-based paged block pool, compaction into fixed blocks, table gathers.

Source: Ultralytics glossary, "PagedAttention":
* section "How paging works": the cache is cut into blocks of a fixed number
  of tokens (16 by default); a request gets a new block only when its last
  one is full, taken from wherever a free block is; a per-request block table
  records the order; attention follows the table block by block.  The worked
  example pops free blocks from the front of a scattered free list and writes
  token p to slot p % block_size of block table[p // block_size].
* section "Block sharing between sequences": sequences may point at the same
  physical blocks, with a reference count per block; a sequence that must
  write into a block others still use copies it first (copy-on-write).
* section "Related techniques" (continuous batching): a finished sequence's
  blocks return to the free pool at once.
* section "Block sharing between sequences", last paragraph: the sharing
  extends across requests by hashing whole blocks (prompt caching): a request
  whose prompt starts like one already held reuses that one's full blocks.

Readings taken: allocation pops the head of the free list (as in the worked
example), a block whose count drops to zero is appended to the tail; copy on
write happens iff the block's count is above one at write time.  Pool layout
is [num_blocks][H_kv][block][d]; the unused tail slots of a last block have
undefined contents.

Prefix blocks (whole-block hashing), readings taken: a full block of 16
prompt tokens of one layer is identified by (layer, the physical block of
the previous 16 tokens of that prefix or -1, the 16 token ids); since a
request holding a block also holds its parent, the parent block stands for
the whole prefix before it, so equal keys mean equal prefixes.  A block can
be found while some request holds it; when its count drops to zero its key
is forgotten.  A lookup that finds the key adds a reference to that block;
one that does not pops a new block and records the key.  The hash of the key
is only how an implementation finds it; equality of keys decides.
"""
from __future__ import annotations

import numpy as np

BLOCK = 16


class OutOfBlocks(RuntimeError):
    pass


def blocks_for(tokens: int, block: int = BLOCK) -> int:
    return -(-tokens // block)


class BlockPool:
    """Free list (a Python list), reference counts, copy-on-write."""

    def __init__(self, num_blocks, free=None):
        self.num_blocks = int(num_blocks)
        self.free = list(range(self.num_blocks)) if free is None else [int(b) for b in free]
        self.ref = [0] * self.num_blocks
        self.prefix = {}          # (layer, parent, tokens) -> block, for held prefix blocks
        self.prefix_key = {}      # block -> its key

    def alloc(self):
        if not self.free:
            raise OutOfBlocks("no free block")
        b = self.free.pop(0)
        self.ref[b] = 1
        return b

    def incref(self, b):
        if self.ref[b] <= 0:
            raise ValueError("incref of a free block")
        self.ref[b] += 1

    def decref(self, b):
        if self.ref[b] <= 0:
            raise ValueError("decref of a free block")
        self.ref[b] -= 1
        if self.ref[b] == 0:
            key = self.prefix_key.pop(b, None)
            if key is not None:
                del self.prefix[key]
            self.free.append(b)

    def prefix_block(self, layer, parent, tokens):
        """The block for 16 prompt tokens of `layer` after the prefix ending in
        block `parent` (-1: none): (block, hit)."""
        key = (int(layer), int(parent), tuple(int(t) for t in tokens))
        if len(key[2]) != BLOCK:
            raise ValueError("a prefix block holds exactly one block of tokens")
        b = self.prefix.get(key)
        if b is not None:
            self.ref[b] += 1
            return b, True
        b = self.alloc()
        self.prefix[key] = b
        self.prefix_key[b] = key
        return b, False

    def cow(self, b):
        """Returns (block to write into, copied?)."""
        if self.ref[b] > 1:
            nb = self.alloc()
            self.decref(b)
            return nb, True
        return b, False

    def num_free(self):
        return len(self.free)


def compact(k, v, idx, table, pool_k, pool_v, block=BLOCK):
    """Copy the kept rows into the pool through a block table.

    k, v: [n, H_kv, d]; idx: [H_kv, k_eff] ascending kept positions;
    table: physical block ids, len >= ceil(k_eff / block);
    pool_k, pool_v: [num_blocks, H_kv, block, d], written in place.
    Kept slot j of head h lands in block table[j // block], slot j % block.
    """
    h_kv, k_eff = idx.shape
    for h in range(h_kv):
        for j in range(k_eff):
            b = table[j // block]
            pool_k[b, h, j % block] = k[idx[h, j], h]
            pool_v[b, h, j % block] = v[idx[h, j], h]


def gather_rows(pool, table, length, h, block=BLOCK):
    """Read slots 0..length-1 of head h back through the table: [length, d].
    Slot j is slot j % block of block table[j // block]."""
    j = np.arange(length)
    return pool[np.asarray(table, dtype=np.int64)[j // block], h, j % block]
