// Host-only parts of the C ABI: error reporting, the block allocator and the
// per-step decode preparation.
//
// Block allocator: Ultralytics glossary "PagedAttention", sections "How paging
// works" (fixed 16-token blocks handed out from wherever one is free; the
// worked example pops the front of a scattered free list) and "Block sharing
// between sequences" (one reference count per block; a writer copies a block
// that other sequences still use).  The free list is a FIFO ring: a block
// appears in it at most once, so a ring of num_blocks entries never
// overflows, and pop-head / push-tail are O(1).
//
// Prefix blocks: the same glossary section's last paragraph (sharing extends
// across requests by hashing whole blocks).  A held full block of a
// full-cache layer's prompt is recorded under (layer, parent block, its 16
// token ids) in a hash map; a lookup hits only on an equal key, so a hash
// collision never aliases two prefixes.  The key is forgotten when the
// block's count reaches zero.
#include <cstdlib>
#include <cstring>
#include <new>
#include <unordered_map>
#include <vector>

#include "host_common.h"

namespace kvs {

namespace {
thread_local std::string g_last_error;
}

void set_error(const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error.assign(buf);
}

void clear_error() { g_last_error.clear(); }

kvs_status fail(kvs_status code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error.assign(buf);
  return code;
}

const char* last_error_cstr() { return g_last_error.c_str(); }

}  // namespace kvs

namespace {

struct PrefixKey {
  int32_t layer;
  int32_t parent;
  int32_t tok[KVS_BLOCK_TOKENS];
  bool operator==(const PrefixKey& o) const {
    return layer == o.layer && parent == o.parent &&
           std::memcmp(tok, o.tok, sizeof(tok)) == 0;
  }
};

// FNV-1a (64-bit) over the key's words, as bytes.
struct PrefixKeyHash {
  size_t operator()(const PrefixKey& k) const {
    uint64_t h = 14695981039346656037ull;
    auto mix = [&h](int32_t word) {
      const uint32_t u = static_cast<uint32_t>(word);
      for (int i = 0; i < 4; ++i) {
        h ^= (u >> (8 * i)) & 0xFFu;
        h *= 1099511628211ull;
      }
    };
    mix(k.layer);
    mix(k.parent);
    for (int i = 0; i < KVS_BLOCK_TOKENS; ++i) mix(k.tok[i]);
    return static_cast<size_t>(h);
  }
};

}  // namespace

struct kvs_allocator {
  int32_t num_blocks = 0;
  std::vector<int32_t> ring;  // free list, FIFO
  int32_t head = 0;           // index of the next block to hand out
  int32_t count = 0;          // blocks in the free list
  std::vector<int32_t> ref;   // reference count per block
  std::vector<uint8_t> managed;
  std::unordered_map<PrefixKey, int32_t, PrefixKeyHash> prefix;  // held prefix blocks
  std::vector<PrefixKey> key_of;  // per block: its prefix key, if keyed[b]
  std::vector<uint8_t> keyed;

  bool valid(int32_t b) const { return b >= 0 && b < num_blocks; }

  void push_tail(int32_t b) {
    ring[(head + count) % num_blocks] = b;
    ++count;
  }

  int32_t pop_head() {
    const int32_t b = ring[head];
    head = (head + 1) % num_blocks;
    --count;
    return b;
  }
};

extern "C" {

const char* kvs_last_error(void) { return kvs::last_error_cstr(); }

int32_t kvs_version(void) { return 100; }

kvs_status kvs_alloc_create(int32_t num_blocks, const int32_t* initial_free, int32_t n_initial,
                            kvs_allocator** out) {
  KVS_REQUIRE(out != nullptr, "kvs_alloc_create: out is NULL");
  *out = nullptr;
  KVS_REQUIRE(num_blocks > 0, "kvs_alloc_create: num_blocks must be > 0 (got %d)", num_blocks);
  auto* a = new (std::nothrow) kvs_allocator();
  if (a == nullptr) return kvs::fail(KVS_ERR_INVALID, "kvs_alloc_create: out of host memory");
  a->num_blocks = num_blocks;
  a->ring.assign(num_blocks, -1);
  a->ref.assign(num_blocks, 0);
  a->managed.assign(num_blocks, 0);
  a->keyed.assign(num_blocks, 0);
  a->key_of.resize(num_blocks);
  if (initial_free == nullptr) {
    for (int32_t b = 0; b < num_blocks; ++b) {
      a->managed[b] = 1;
      a->push_tail(b);
    }
  } else {
    if (n_initial < 0 || n_initial > num_blocks) {
      delete a;
      return kvs::fail(KVS_ERR_INVALID, "kvs_alloc_create: n_initial %d outside [0, %d]",
                       n_initial, num_blocks);
    }
    for (int32_t i = 0; i < n_initial; ++i) {
      const int32_t b = initial_free[i];
      if (!a->valid(b) || a->managed[b]) {
        delete a;
        return kvs::fail(KVS_ERR_INVALID,
                         "kvs_alloc_create: initial_free[%d] = %d is out of range or repeated",
                         i, b);
      }
      a->managed[b] = 1;
      a->push_tail(b);
    }
  }
  *out = a;
  return KVS_OK;
}

void kvs_alloc_destroy(kvs_allocator* a) { delete a; }

kvs_status kvs_alloc_block(kvs_allocator* a, int32_t* out) {
  KVS_REQUIRE(a != nullptr && out != nullptr, "kvs_alloc_block: NULL argument");
  if (a->count == 0) return kvs::fail(KVS_ERR_OOM_BLOCKS, "kvs_alloc_block: no free block");
  const int32_t b = a->pop_head();
  a->ref[b] = 1;
  *out = b;
  return KVS_OK;
}

kvs_status kvs_alloc_blocks(kvs_allocator* a, int32_t count, int32_t* out) {
  KVS_REQUIRE(a != nullptr && (out != nullptr || count == 0) && count >= 0,
              "kvs_alloc_blocks: bad argument");
  if (count > a->count)
    return kvs::fail(KVS_ERR_OOM_BLOCKS, "kvs_alloc_blocks: %d requested, %d free", count,
                     a->count);
  for (int32_t i = 0; i < count; ++i) {
    const int32_t b = a->pop_head();
    a->ref[b] = 1;
    out[i] = b;
  }
  return KVS_OK;
}

kvs_status kvs_alloc_incref(kvs_allocator* a, int32_t block) {
  KVS_REQUIRE(a != nullptr, "kvs_alloc_incref: NULL allocator");
  KVS_REQUIRE(a->valid(block), "kvs_alloc_incref: block %d out of range", block);
  KVS_REQUIRE(a->ref[block] > 0, "kvs_alloc_incref: block %d is not in use", block);
  ++a->ref[block];
  return KVS_OK;
}

kvs_status kvs_alloc_decref(kvs_allocator* a, int32_t block) {
  KVS_REQUIRE(a != nullptr, "kvs_alloc_decref: NULL allocator");
  KVS_REQUIRE(a->valid(block), "kvs_alloc_decref: block %d out of range", block);
  KVS_REQUIRE(a->ref[block] > 0, "kvs_alloc_decref: block %d is not in use", block);
  if (--a->ref[block] == 0) {
    if (a->keyed[block]) {
      a->prefix.erase(a->key_of[block]);
      a->keyed[block] = 0;
    }
    a->push_tail(block);
  }
  return KVS_OK;
}

kvs_status kvs_alloc_prefix_blocks(kvs_allocator* a, int32_t layer, const int32_t* tokens,
                                   int32_t n_tokens, int32_t* blocks, int32_t* hits,
                                   int32_t* n_hits) {
  KVS_REQUIRE(a != nullptr && n_tokens >= 0 && (tokens != nullptr || n_tokens == 0),
              "kvs_alloc_prefix_blocks: bad argument");
  const int32_t n_full = n_tokens / KVS_BLOCK_TOKENS;
  KVS_REQUIRE(n_full == 0 || (blocks != nullptr && hits != nullptr),
              "kvs_alloc_prefix_blocks: NULL output");
  // the blocks found form a run from the start (the key after a new block
  // names that block as its parent, which no key can hold yet): count it, so
  // that a shortage of free blocks is known before anything changes
  PrefixKey key;
  key.layer = layer;
  key.parent = -1;
  int32_t run = 0;
  for (; run < n_full; ++run) {
    std::memcpy(key.tok, tokens + static_cast<int64_t>(run) * KVS_BLOCK_TOKENS, sizeof(key.tok));
    const auto it = a->prefix.find(key);
    if (it == a->prefix.end()) break;
    key.parent = it->second;
  }
  if (n_full - run > a->count)
    return kvs::fail(KVS_ERR_OOM_BLOCKS, "kvs_alloc_prefix_blocks: %d new blocks needed, %d free",
                     n_full - run, a->count);
  key.parent = -1;
  for (int32_t i = 0; i < n_full; ++i) {
    std::memcpy(key.tok, tokens + static_cast<int64_t>(i) * KVS_BLOCK_TOKENS, sizeof(key.tok));
    int32_t b;
    if (i < run) {
      b = a->prefix.find(key)->second;
      ++a->ref[b];
      hits[i] = 1;
    } else {
      b = a->pop_head();
      a->ref[b] = 1;
      a->prefix.emplace(key, b);
      a->key_of[b] = key;
      a->keyed[b] = 1;
      hits[i] = 0;
    }
    blocks[i] = b;
    key.parent = b;
  }
  if (n_hits != nullptr) *n_hits = run;
  return KVS_OK;
}

int32_t kvs_alloc_prefix_entries(const kvs_allocator* a) {
  return a == nullptr ? -1 : static_cast<int32_t>(a->prefix.size());
}

kvs_status kvs_alloc_cow(kvs_allocator* a, int32_t block, int32_t* out, int32_t* copied) {
  KVS_REQUIRE(a != nullptr && out != nullptr && copied != nullptr, "kvs_alloc_cow: NULL argument");
  KVS_REQUIRE(a->valid(block), "kvs_alloc_cow: block %d out of range", block);
  KVS_REQUIRE(a->ref[block] > 0, "kvs_alloc_cow: block %d is not in use", block);
  if (a->ref[block] > 1) {
    if (a->count == 0) return kvs::fail(KVS_ERR_OOM_BLOCKS, "kvs_alloc_cow: no free block");
    const int32_t nb = a->pop_head();
    a->ref[nb] = 1;
    --a->ref[block];
    *out = nb;
    *copied = 1;
  } else {
    *out = block;
    *copied = 0;
  }
  return KVS_OK;
}

int32_t kvs_alloc_refcount(const kvs_allocator* a, int32_t block) {
  if (a == nullptr || !a->valid(block)) return -1;
  return a->ref[block];
}

int32_t kvs_alloc_num_free(const kvs_allocator* a) { return a == nullptr ? -1 : a->count; }

int32_t kvs_alloc_free_list(const kvs_allocator* a, int32_t* buf, int32_t cap) {
  if (a == nullptr || buf == nullptr || cap <= 0) return 0;
  const int32_t n = cap < a->count ? cap : a->count;
  for (int32_t i = 0; i < n; ++i) buf[i] = a->ring[(a->head + i) % a->num_blocks];
  return n;
}

kvs_status kvs_decode_prepare(kvs_allocator* a, int32_t* tables, int32_t max_blocks,
                              const int32_t* lens, int32_t n_items, int32_t* patch,
                              int32_t* cow_src, int32_t* cow_dst, int32_t* n_cow,
                              int32_t* n_patch, int32_t* n_done) {
  KVS_REQUIRE(a != nullptr && tables != nullptr && lens != nullptr && patch != nullptr &&
                  cow_src != nullptr && cow_dst != nullptr && n_cow != nullptr,
              "kvs_decode_prepare: NULL argument");
  KVS_REQUIRE(n_items >= 0 && max_blocks > 0, "kvs_decode_prepare: bad sizes");
  *n_cow = 0;
  if (n_patch) *n_patch = 0;
  if (n_done) *n_done = 0;
  for (int32_t i = 0; i < n_items; ++i) {
    const int32_t len = lens[i];
    KVS_REQUIRE(len >= 0, "kvs_decode_prepare: lens[%d] = %d", i, len);
    const int32_t slot = len / KVS_BLOCK_TOKENS;
    KVS_REQUIRE(slot < max_blocks, "kvs_decode_prepare: item %d needs block %d >= max_blocks %d",
                i, slot, max_blocks);
    int32_t* row = tables + static_cast<int64_t>(i) * max_blocks;
    if (len % KVS_BLOCK_TOKENS == 0) {
      if (a->count == 0)
        return kvs::fail(KVS_ERR_OOM_BLOCKS, "kvs_decode_prepare: no free block for item %d", i);
      const int32_t b = a->pop_head();
      a->ref[b] = 1;
      row[slot] = b;
      patch[i] = b;
      if (n_patch) ++*n_patch;
    } else {
      const int32_t last = row[slot];
      KVS_REQUIRE(a->valid(last) && a->ref[last] > 0,
                  "kvs_decode_prepare: item %d last block %d is not in use", i, last);
      if (a->ref[last] > 1) {
        if (a->count == 0)
          return kvs::fail(KVS_ERR_OOM_BLOCKS, "kvs_decode_prepare: no free block for item %d",
                           i);
        const int32_t nb = a->pop_head();
        a->ref[nb] = 1;
        --a->ref[last];
        row[slot] = nb;
        patch[i] = nb;
        if (n_patch) ++*n_patch;
        cow_src[*n_cow] = last;
        cow_dst[*n_cow] = nb;
        ++*n_cow;
      } else {
        patch[i] = -1;
      }
    }
    if (n_done) *n_done = i + 1;
  }
  return KVS_OK;
}

}  // extern "C"
