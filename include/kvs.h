/*
 * kvs.h -- C ABI of the layer-wise KV-cache sparsification hot path over a
 * paged KV cache, for one NVIDIA GB300 (sm_103a).
 *
 * The method (Novita AI, "How KV Sparsity achieves 1.5x acceleration for
 * vLLM"; Ultralytics glossary, "PagedAttention"):
 *   1. causal prefill attention that also returns each query row's maximum
 *      logit m and softmax normaliser l          -> kvs_prefill_attn_lse
 *   2. window scores S summed over the last alpha queries -> kvs_window_scores
 *   3. per-(layer, KV head) top-k_l with a recent window  -> kvs_select_topk
 *   4. compaction of the kept K/V into 16-token blocks    -> kvs_compact_blocks
 *      tracked by a block allocator (free list, reference counts,
 *      copy-on-write)                                   -> kvs_alloc_*, kvs_copy_blocks
 *   5. decode attention gathering K/V through block tables -> kvs_paged_decode
 *      (one whole step with the host allocator's work   -> kvs_decode_step)
 * Beyond them:
 *   - decode-time replacement in budgeted layers -> kvs_evict_place,
 *     kvs_paged_decode_logits, kvs_decode_scores_from_logits (section 7)
 *   - FP8 (e4m3, per-row scale) pools -> kvs_compact_blocks_fp8,
 *     kvs_copy_blocks_fp8, kvs_paged_decode_fp8, kvs_decode_step_fp8;
 *     decode-time replacement over them -> kvs_evict_place_fp8,
 *     kvs_paged_decode_logits_fp8, kvs_decode_scores_from_logits
 *
 * Conventions (all entry points)
 *   - bf16 tensors are passed as raw 16-bit patterns (kvs_bf16).
 *   - Every tensor pointer is a DEVICE pointer owned by the caller unless the
 *     argument says "host".  The library never allocates device memory; scratch
 *     is a caller-provided workspace whose size a *_workspace_size call gives.
 *   - Launching calls are asynchronous on `stream` (a cudaStream_t; NULL = the
 *     legacy default stream).  Arguments are validated on the host before any
 *     launch: a bad argument returns KVS_ERR_INVALID (or KVS_ERR_UNSUPPORTED
 *     for a shape outside the supported set) and launches nothing.  A launch
 *     failure returns KVS_ERR_CUDA.  Faults inside kernels surface at the
 *     caller's next synchronisation.
 *   - `status` (nullable device int32): kernels that meet a corrupt index
 *     (block id outside the pool, kept index outside the sequence) skip that
 *     access and store KVS_ERR_INVALID there; a kernel whose bounded wait on
 *     an mbarrier gives up stores KVS_ERR_DEVICE_TIMEOUT and returns.  The
 *     word is only ever set, never cleared, by the library.
 *   - kvs_last_error() returns a thread-local message for the last failure.
 *   - Supported: d in {64, 128}; h_q % h_kv == 0; G = h_q / h_kv <= 16;
 *     block size fixed at 16 tokens.
 *   - Layouts: prompt Q is [T][h_q][d], prompt K and V are [T][h_kv][d]
 *     (token-major, sequences packed back to back, T = total tokens); the
 *     paged pools are [num_blocks][h_kv][16][d].
 */
#ifndef KVS_H_
#define KVS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t kvs_bf16;  /* raw bf16 bit pattern */
typedef void* kvs_stream;   /* cudaStream_t */

typedef enum {
  KVS_OK = 0,
  KVS_ERR_INVALID = 1,
  KVS_ERR_OOM_BLOCKS = 2,
  KVS_ERR_CUDA = 3,
  KVS_ERR_UNSUPPORTED = 4,
  KVS_ERR_DEVICE_TIMEOUT = 5
} kvs_status;

#define KVS_BLOCK_TOKENS 16

/* Message describing the last failed call on this thread ("" if none). */
const char* kvs_last_error(void);

/* Library ABI version (major * 100 + minor). */
int32_t kvs_version(void);

/* ------------------------------------------------------------------------
 * 1. Prefill attention with row max and normaliser.
 * Source: Novita article, section "Key techniques 2: attention
 * modification" -- FlashAttention-2 (Figure 7) already computes the running
 * row maximum and l; the modification returns them.  Computes, per query
 * head g (KV head g / G) and query row r of each sequence,
 *     s_i = scale * q_r . k_i  for keys i <= r of the same sequence,
 *     m = max_i s_i,  l = sum_i exp(s_i - m),  O_r = sum_i exp(s_i - m)/l v_i
 *   q      [T][h_q][d] bf16, k/v [T][h_kv][d] bf16
 *   o      [T][h_q][d] bf16 (output)
 *   m, l   [h_q][T] fp32 (output; natural-exponent, scaled-logit domain)
 *   cu_seqlens [batch + 1] int32 (device): sequence b owns tokens
 *          cu_seqlens[b] .. cu_seqlens[b+1]-1; cu_seqlens[batch] == T.
 *   max_n  host upper bound of the sequence lengths (sizes the grid).
 * Row blocks of 128 queries run on the 5th-generation tensor cores
 * (tcgen05, TMEM accumulators, TMA-fed shared memory).
 * ---------------------------------------------------------------------- */
kvs_status kvs_prefill_attn_lse(const kvs_bf16* q, const kvs_bf16* k, const kvs_bf16* v,
                                kvs_bf16* o, float* m, float* l,
                                const int32_t* cu_seqlens, int32_t batch, int32_t max_n,
                                int32_t total_tokens, int32_t h_q, int32_t h_kv, int32_t d,
                                float scale, int32_t* status, kvs_stream stream);

/* The same attention for n_layers layers in one launch.  Layer j's tensors
 * follow layer j-1's in the same buffers: q [n_layers][T][h_q][d], k, v
 * [n_layers][T][h_kv][d], o [n_layers][T][h_q][d], m, l [n_layers][h_q][T]
 * (one cu_seqlens for all layers).  Given every layer's Q, K and V at once,
 * the layers are independent: the persistent CTAs take the work items of all
 * layers, longest first, so the launch, start-up and uneven end of a launch
 * are paid once instead of per layer.  Results are bit-identical to
 * kvs_prefill_attn_lse per layer.  n_layers x T < 2^31; n_layers = 0 is a
 * no-op.  (The batching over layers is this library's, not a step of the
 * method: a model whose layer l+1 inputs come from layer l's output calls
 * kvs_prefill_attn_lse layer by layer.)
 */
kvs_status kvs_prefill_attn_lse_layers(const kvs_bf16* q, const kvs_bf16* k, const kvs_bf16* v,
                                       kvs_bf16* o, float* m, float* l,
                                       const int32_t* cu_seqlens, int32_t batch, int32_t max_n,
                                       int32_t total_tokens, int32_t h_q, int32_t h_kv,
                                       int32_t d, float scale, int32_t n_layers,
                                       int32_t* status, kvs_stream stream);

/* ------------------------------------------------------------------------
 * 2. Window scores.
 * Source: Novita article, section "Key techniques 2" (PyramidKV-style score
 * over the instruction window [n - alpha, n]; probabilities rebuilt as
 * exp(k.q - rowmax)/l from the prefill's outputs; key-major loop order;
 * only window query blocks visited).  For each sequence (length n, window
 * w = min(alpha, n) rows n-w .. n-1) and KV head h:
 *     S[h][i] = sum_{g in group(h)} sum_{q = n-w}^{n-1} [i <= q]
 *               exp(scale * q_g . k_i - m[g][q]) / l[g][q]
 *   q [T][h_q][d], k [T][h_kv][d] bf16; m, l [h_q][T] fp32 (only the window
 *   rows are read); scores [h_kv][T] fp32 (output; every token of every
 *   sequence is written).  alpha * G <= 256.
 * ---------------------------------------------------------------------- */
kvs_status kvs_window_scores(const kvs_bf16* q, const kvs_bf16* k, const float* m, const float* l,
                             float* scores, const int32_t* cu_seqlens, int32_t batch,
                             int32_t max_n, int32_t total_tokens, int32_t h_q, int32_t h_kv,
                             int32_t d, int32_t alpha, float scale, int32_t* status,
                             kvs_stream stream);

/* The same scores for n_layers consecutive layers in one launch.  Layer j's
 * tensors follow layer j-1's in the same buffers: q [n_layers][T][h_q][d],
 * k [n_layers][T][h_kv][d], m, l [n_layers][h_q][T], scores
 * [n_layers][h_kv][T] (one cu_seqlens for all layers).  A layer's scores
 * read only that layer's q, k, m and l, so they may be computed any time
 * after its prefill and before its selection: one launch over every
 * budgeted layer after the prefill loop replaces a launch per layer between
 * the prefills.  Results are bit-identical to kvs_window_scores per layer.
 * batch x n_layers <= 65535 and n_layers x T < 2^31; n_layers = 0 is a no-op.
 * (The batching over layers is this library's, not a step of the method.)
 */
kvs_status kvs_window_scores_layers(const kvs_bf16* q, const kvs_bf16* k, const float* m,
                                    const float* l, float* scores, const int32_t* cu_seqlens,
                                    int32_t batch, int32_t max_n, int32_t total_tokens,
                                    int32_t h_q, int32_t h_kv, int32_t d, int32_t alpha,
                                    float scale, int32_t n_layers, int32_t* status,
                                    kvs_stream stream);

/* ------------------------------------------------------------------------
 * 3. Top-k_l selection.
 * Source: Novita article, section "System model" (keep the higher-scoring and
 * nearer KV pairs), section "Key techniques 1" (first three layers full,
 * later layers evict the lowest scores), section "Key techniques 2" (per
 * layer l and head h keep the k_l highest-scoring tokens; the rest is
 * discarded for the whole generation).
 * One item = one (sequence, layer).  For each item and KV head h the row
 * scores[score_off + h * head_stride + i], i < n, is read and
 *   k >= n : kept = 0 .. n-1 (identity)
 *   else   : kept = {n-recent .. n-1} plus the (k - recent) highest scores of
 *            positions 0 .. n-recent-1, ties to the lower position,
 * written in ascending position order to
 *   kept_idx[idx_off + h * min(k, n) + j], j < min(k, n).
 * Scores are non-negative finite fp32 (compared as stored); recent <= k.
 * items: device array of n_items descriptors.
 * ---------------------------------------------------------------------- */
typedef struct {
  int64_t score_off; /* element offset of head 0's row in `scores` */
  int32_t n;         /* prompt length */
  int32_t k;         /* budget k_l (>= n means keep all) */
  int64_t idx_off;   /* element offset of head 0's output in `kept_idx` */
} kvs_select_item;

kvs_status kvs_select_topk(const float* scores, int64_t head_stride, const kvs_select_item* items,
                           int32_t n_items, int32_t h_kv, int32_t recent, int32_t* kept_idx,
                           int32_t* status, kvs_stream stream);

/* ------------------------------------------------------------------------
 * 4. Compaction into 16-token blocks.
 * Source: Ultralytics glossary "PagedAttention", section "How paging works"
 * (slot p % 16 of block table[p / 16]); Novita article, section "Key
 * techniques 1" (per-layer block-table strategies).
 * One item = one (sequence, layer).  For each item, head h and kept slot
 * j < k_eff, with p = kept_idx[idx_off + h * k_eff + j] and
 * b = block_tables[table_off + j / 16]:
 *     k_pool[b][h][j % 16][:] = k[src_tok + p][h][:]   (same for v)
 * a bit-exact copy (rows are items' (j) slots; all h_kv heads of a slot are
 * copied together).  row_off is the item's first row in the flattened
 * (item, j) enumeration: row_off(i) = sum of k_eff over items before i;
 * total_rows = sum of all k_eff.  items: device array.
 * A table entry of KVS_BLOCK_SKIP marks a block that already holds its rows
 * (a prefix block found by kvs_alloc_prefix_blocks): its slots are neither
 * read nor written.  Any other entry outside [0, num_blocks) skips the slot
 * and flags KVS_ERR_INVALID in `status`.
 * ---------------------------------------------------------------------- */
#define KVS_BLOCK_SKIP (-2)

typedef struct {
  int64_t src_tok;   /* first token of the item's K/V in `k` / `v` */
  int64_t idx_off;   /* element offset of head 0's kept indices */
  int64_t row_off;   /* prefix sum of k_eff over earlier items */
  int32_t n;         /* tokens of the item (kept indices must be < n) */
  int32_t k_eff;     /* kept tokens per head */
  int32_t table_off; /* element offset of the item's block table */
  int32_t reserved;  /* 0 */
} kvs_compact_item;

kvs_status kvs_compact_blocks(const kvs_bf16* k, const kvs_bf16* v, const kvs_compact_item* items,
                              int32_t n_items, int64_t total_rows, int32_t h_kv, int32_t d,
                              const int32_t* kept_idx, const int32_t* block_tables,
                              kvs_bf16* k_pool, kvs_bf16* v_pool, int32_t num_blocks,
                              int32_t* status, kvs_stream stream);

/* kvs_compact_blocks into an FP8 pool (d = 128 only).  Source: Ultralytics
 * glossary "PagedAttention", section "Related techniques" (FP8 cache
 * quantisation: keys and values at 8-bit precision, about half the memory of
 * 16-bit formats); format and scaling are this library's reading:
 *   - each cached row (slot r of block b, KV head h; d values) is stored as
 *     e4m3 codes with one fp32 scale s = amax / 448 (s = 1 for an all-zero
 *     row): code = e4m3 nearest to x / s, ties to even, saturating at 448;
 *     amax / 448 and x / s are IEEE fp32 divisions; the stored value is
 *     e4m3(code) * s;
 *   - k_pool [num_blocks][h_kv][16][128] uint8: row r of (b, h) at byte
 *     ((b * h_kv + h) * 16 + r) * 128, its 16-byte chunk c at chunk position
 *     c ^ (4 * (r & 1)) within the row;
 *   - v_pool [num_blocks][h_kv][128][16] uint8: transposed, element dd of
 *     slot r at byte ((b * h_kv + h) * 128 + dd) * 16 + r;
 *   - k_scale, v_scale [num_blocks][h_kv][16] fp32.
 * Slots past k_eff in an item's last block get zero codes and zero scales.
 * Other arguments as kvs_compact_blocks; n_items <= 4096; pool and scale
 * pointers 16-byte aligned. */
kvs_status kvs_compact_blocks_fp8(const kvs_bf16* k, const kvs_bf16* v,
                                  const kvs_compact_item* items, int32_t n_items,
                                  int64_t total_rows, int32_t h_kv, int32_t d,
                                  const int32_t* kept_idx, const int32_t* block_tables,
                                  uint8_t* k_pool, uint8_t* v_pool, float* k_scale,
                                  float* v_scale, int32_t num_blocks, int32_t* status,
                                  kvs_stream stream);

/* kvs_copy_blocks for FP8 pools (layout of kvs_compact_blocks_fp8; d = 128):
 * each pair copies the block's K and V codes of every head and their row
 * scales.  Two launches on `stream`. */
kvs_status kvs_copy_blocks_fp8(const int32_t* src, const int32_t* dst, int32_t count,
                               uint8_t* k_pool, uint8_t* v_pool, float* k_scale, float* v_scale,
                               int32_t num_blocks, int32_t h_kv, int32_t d, int32_t* status,
                               kvs_stream stream);

/* Copy whole blocks src[i] -> dst[i] in both pools (the copy of
 * copy-on-write; Ultralytics glossary "PagedAttention", section "Block
 * sharing between sequences").  src, dst: device int32 [count]. */
kvs_status kvs_copy_blocks(const int32_t* src, const int32_t* dst, int32_t count,
                           kvs_bf16* k_pool, kvs_bf16* v_pool, int32_t num_blocks, int32_t h_kv,
                           int32_t d, int32_t* status, kvs_stream stream);

/* ------------------------------------------------------------------------
 * 5. Paged decode attention (split-K over 16-token blocks).
 * Source: Ultralytics glossary "PagedAttention", section "How paging works"
 * (the kernel follows the block table and gathers K/V block by block);
 * Novita article, section "Key techniques 2" (PagedAttention on the decode
 * side).  One item = one (stream, layer) with `lens[i]` tokens already in
 * its table.  If k_new is not NULL the item's new k/v row is first written
 * at slot lens[i] (block table[lens[i] / 16], slot lens[i] % 16) and
 * attention runs over lens[i] + 1 tokens (the new token attends to itself);
 * otherwise over lens[i] tokens.  Per query head g (KV head g / G):
 *     out[i][g] = softmax_t(scale * q[i][g] . K_t) V
 *   q, out [batch][h_q][d]; k_new, v_new [batch][h_kv][d] (nullable)
 *   block_tables [batch][max_blocks] int32; lens [batch] int32 (batch <= 2048)
 *   table_patch  [batch] int32, nullable: entry >= 0 replaces
 *                block_tables[i][lens[i] / 16] before use and is written
 *                back there (the host allocator's new or copied-on-write
 *                last block); -1 = no change.
 *   lens_next    [batch] int32, nullable, must not alias lens: receives
 *                lens[i] + (k_new != NULL).
 *   workspace    scratch of kvs_paged_decode_workspace_size(batch, h_q, h_kv,
 *                d) bytes (split partials; the size covers the bf16 and the
 *                FP8 decode, whose launches differ in warps per CTA, so the
 *                bf16 decode alone accepts a little less); needs no
 *                initialisation.  Calls sharing a workspace must not overlap
 *                in time.
 *   q, out, the pools and the workspace must be 16-byte aligned
 *   (KVS_ERR_INVALID otherwise).
 * Two launches on `stream`: the split decode, then a merge of the splits (a
 * programmatic dependent launch that waits for the decode's partials).  A
 * batch whose per-item lengths and prefix would leave the kernel a single
 * shared-memory stage per warp (about 1250 bf16 items at G = 4) is decoded
 * in consecutive chunks of items, each chunk such a pair of launches, in
 * order on `stream` and reusing the workspace.
 * An item with zero tokens to attend (lens[i] == 0 and no append) gets no
 * output row.
 * ---------------------------------------------------------------------- */
size_t kvs_paged_decode_workspace_size(int32_t batch, int32_t h_q, int32_t h_kv, int32_t d);

/* Zero-fill a device buffer on `stream` (convenience for callers' scratch). */
kvs_status kvs_workspace_zero(void* workspace, size_t bytes, kvs_stream stream);

kvs_status kvs_paged_decode(const kvs_bf16* q, const kvs_bf16* k_new, const kvs_bf16* v_new,
                            kvs_bf16* k_pool, kvs_bf16* v_pool, int32_t num_blocks,
                            int32_t* block_tables, int32_t max_blocks, const int32_t* table_patch,
                            const int32_t* lens, int32_t* lens_next, int32_t batch, int32_t h_q,
                            int32_t h_kv, int32_t d, float scale, kvs_bf16* out, void* workspace,
                            size_t workspace_bytes, int32_t* status, kvs_stream stream);

/* Test hook for the bounded waits (no counterpart in the method: failure
 * detection of the library itself).  Same arguments and checks as
 * kvs_paged_decode without an append, but the decode's copy-issuing lane
 * arms each stage's barrier and starts none of the copies it announced, and
 * every barrier wait gives up after wait_ns (0 < wait_ns <= 1.5 s) instead
 * of the usual 1.5 s.  So every wait runs out: the kernel stores
 * KVS_ERR_DEVICE_TIMEOUT in `status` (nullable) and returns, nothing is left
 * in flight, and the context stays usable.  `out` rows are undefined
 * afterwards; the pools are not written.  Exists so that tests can drive the
 * timeout path without a fault; serving code has no reason to call it. */
kvs_status kvs_test_paged_decode_stalled(const kvs_bf16* q, kvs_bf16* k_pool, kvs_bf16* v_pool,
                                         int32_t num_blocks, int32_t* block_tables,
                                         int32_t max_blocks, const int32_t* lens, int32_t batch,
                                         int32_t h_q, int32_t h_kv, int32_t d, float scale,
                                         kvs_bf16* out, void* workspace, size_t workspace_bytes,
                                         uint32_t wait_ns, int32_t* status, kvs_stream stream);

/* ------------------------------------------------------------------------
 * Paged decode that allocates nothing (no counterpart in the method's
 * sources: this is a calling convention, not a step of the method).
 *
 * Some callers cannot hand the library a workspace: a serving process that
 * reserved all device memory for its paged pool up front and allows no
 * allocation on the decode path (an allocation there can fail under memory
 * pressure, fragment the reserved pool, or synchronise the device), or a
 * plain C host without a device allocator of its own.  This entry point takes
 * the same arguments and computes the same result as kvs_paged_decode, but
 * its split partials live in a device array built into the library, of
 * KVS_DECODE_STATIC_SCRATCH_BYTES; every GPU that loads the library holds
 * that array until the process exits.  It calls no cudaMalloc, cudaFree or
 * allocating library routine.
 *   - Sizes whose partials (the bf16 decode's share of
 *     kvs_paged_decode_workspace_size, which also covers the FP8 decode's
 *     larger launch) exceed the array are rejected with KVS_ERR_UNSUPPORTED
 *     before any launch.  With h_q = 32, h_kv = 8, d = 128 the array serves
 *     up to 624 items (one 32-layer sequence is 32 items and needs about
 *     7 MB); 625 are rejected.
 *   - The first call on a device looks up the array's device address on that
 *     device (the current one); make that first call before any stream
 *     capture.
 *   - The CUDA runtime creates the array when it first loads the library's
 *     decode code on a device (under lazy module loading, the default: the
 *     first decode call of any kind there, or the first call of this entry
 *     point).  A caller that means to reserve the rest of device memory for
 *     its pool should make one such call first, or that first call may find
 *     no room for the array and fail with KVS_ERR_CUDA.
 *   - All calls share the one array and it keeps the last call's contents;
 *     nothing in it needs to start at zero (each call writes its partials
 *     before reading them).  Calls that overlap on the GPU (on
 *     different streams, or from different threads) race on it.
 * ---------------------------------------------------------------------- */
#define KVS_DECODE_STATIC_SCRATCH_BYTES (16u << 20)

kvs_status kvs_paged_decode_static(const kvs_bf16* q, const kvs_bf16* k_new,
                                   const kvs_bf16* v_new, kvs_bf16* k_pool, kvs_bf16* v_pool,
                                   int32_t num_blocks, int32_t* block_tables, int32_t max_blocks,
                                   const int32_t* table_patch, const int32_t* lens,
                                   int32_t* lens_next, int32_t batch, int32_t h_q, int32_t h_kv,
                                   int32_t d, float scale, kvs_bf16* out, int32_t* status,
                                   kvs_stream stream);

/* ------------------------------------------------------------------------
 * Block allocator (host memory, single-threaded, not thread-safe).
 * Source: Ultralytics glossary "PagedAttention": sections "How paging
 * works" (a new block only when the last one is full, taken from wherever one
 * is free; the worked example pops the front of the free list) and "Block
 * sharing between sequences" (reference counts; copy before writing a block
 * others still use).  The free list is FIFO: allocation pops the head, a block
 * whose count reaches zero is appended to the tail.  All operations are O(1)
 * except creation.
 * ---------------------------------------------------------------------- */
typedef struct kvs_allocator kvs_allocator;

/* num_blocks physical blocks.  initial_free (host, nullable): the initial free
 * list order, n_initial distinct ids in [0, num_blocks); blocks not listed are
 * unmanaged (reference count 0, never handed out).  NULL = 0 .. num_blocks-1. */
kvs_status kvs_alloc_create(int32_t num_blocks, const int32_t* initial_free, int32_t n_initial,
                            kvs_allocator** out);
void kvs_alloc_destroy(kvs_allocator* a);
/* Pop the head of the free list; its count becomes 1.  KVS_ERR_OOM_BLOCKS if empty. */
kvs_status kvs_alloc_block(kvs_allocator* a, int32_t* out);
/* Pop `count` blocks into out (host); all or nothing. */
kvs_status kvs_alloc_blocks(kvs_allocator* a, int32_t count, int32_t* out);
kvs_status kvs_alloc_incref(kvs_allocator* a, int32_t block);
kvs_status kvs_alloc_decref(kvs_allocator* a, int32_t block);
/* If block is shared (count > 1): pop a new block, drop one reference to
 * `block`, *out = new block, *copied = 1 (the caller copies the contents).
 * Otherwise *out = block, *copied = 0. */
kvs_status kvs_alloc_cow(kvs_allocator* a, int32_t block, int32_t* out, int32_t* copied);
int32_t kvs_alloc_refcount(const kvs_allocator* a, int32_t block); /* -1 if out of range */
int32_t kvs_alloc_num_free(const kvs_allocator* a);
/* Copy up to cap free-list entries, head first, into buf (host); returns count. */
int32_t kvs_alloc_free_list(const kvs_allocator* a, int32_t* buf, int32_t cap);

/* Prefix blocks: prompt caching across requests by hashing whole blocks
 * (Ultralytics glossary "PagedAttention", section "Block sharing between
 * sequences", last paragraph).  For the n_tokens / 16 full blocks of a
 * prompt's token ids (host int32, n_tokens of them) in one layer that keeps
 * every token: block i is keyed by (layer, block i - 1 of this call or -1,
 * tokens[16 i .. 16 i + 15]).  A key held by the allocator (its block in use)
 * is a hit: that block gains a reference, hits[i] = 1.  Otherwise a block is
 * popped from the free list (count 1) and recorded under the key, hits[i] = 0.
 * A hit needs an equal key, not only an equal hash.  blocks, hits: host
 * int32 [n_tokens / 16]; *n_hits (nullable) = blocks found, which always form
 * a run from the first block.  A block's key is forgotten when its count
 * drops to zero.  KVS_ERR_OOM_BLOCKS (nothing changed) when the free list
 * cannot supply the blocks not found.  A caller that places a prompt this
 * way need not write the blocks found (their slots already hold the rows of
 * the same prefix): see KVS_BLOCK_SKIP. */
kvs_status kvs_alloc_prefix_blocks(kvs_allocator* a, int32_t layer, const int32_t* tokens,
                                   int32_t n_tokens, int32_t* blocks, int32_t* hits,
                                   int32_t* n_hits);
/* Number of blocks currently recorded as prefix blocks (-1 for NULL). */
int32_t kvs_alloc_prefix_entries(const kvs_allocator* a);

/* Host-side step preparation for a batch of decode items (one per (stream,
 * layer)), visited in order: for item i with length lens[i] (host) and table
 * row tables[i * max_blocks ..] (host):
 *   lens[i] % 16 == 0             -> pop a new block; patch[i] = it
 *   last block shared (count > 1) -> copy-on-write; patch[i] = new block and
 *                                    the pair (old, new) is appended to
 *                                    cow_src / cow_dst
 *   otherwise                     -> patch[i] = -1
 * The host table row is updated in place.  *n_cow receives the number of
 * copies (cow_src / cow_dst need room for n_items entries); *n_patch
 * (nullable) the number of entries of `patch` that are >= 0, so that a step
 * with none can pass table_patch = NULL to kvs_paged_decode.  If the pool runs
 * dry, returns KVS_ERR_OOM_BLOCKS with *n_done = items fully prepared. */
kvs_status kvs_decode_prepare(kvs_allocator* a, int32_t* tables, int32_t max_blocks,
                              const int32_t* lens, int32_t n_items, int32_t* patch,
                              int32_t* cow_src, int32_t* cow_dst, int32_t* n_cow,
                              int32_t* n_patch, int32_t* n_done);

/* ------------------------------------------------------------------------
 * One whole decode step in one native call: the host preparation above, the
 * uploads it needs and the paged decode (the per-step sequence of the
 * Ultralytics glossary "PagedAttention", section "How paging works", and of
 * the Novita article's serving loop; bundling it is this library's calling
 * convention, so that a serving loop spends microseconds of host time per
 * step).  In order, on `stream`:
 *   1. kvs_decode_prepare over the host mirrors tables_h [n_items][max_blocks]
 *      and lens_h [n_items] (lengths before this step's append);
 *   2. if blocks must be copied on write: the (old, new) pairs, staged in
 *      cow_h [2 n_items] host, are uploaded to cow_d [2 n_items] device and
 *      kvs_copy_blocks runs;
 *   3. if any table entry changed: patch_h [n_items] host is uploaded to
 *      patch_d [n_items] device and passed as table_patch;
 *   4. kvs_paged_decode with k_new / v_new appended (both required), lens ->
 *      lens_next on the device;
 *   5. lens_h[i] += 1 on the host.
 * patch_h and cow_h are read by copies queued on `stream`: use pinned memory
 * for an asynchronous upload, and do not write them again before those
 * copies have run (a ring of staging buffers guarded by events).  n_cow,
 * n_patch (nullable) receive this step's counts.  A preparation error
 * (KVS_ERR_OOM_BLOCKS, bad sizes) launches nothing; a launch error after the
 * preparation leaves the host mirrors prepared for the step.
 * ---------------------------------------------------------------------- */
kvs_status kvs_decode_step(kvs_allocator* a, int32_t* tables_h, int32_t* lens_h,
                           int32_t* patch_h, int32_t* cow_h, int32_t* patch_d, int32_t* cow_d,
                           const kvs_bf16* q, const kvs_bf16* k_new, const kvs_bf16* v_new,
                           kvs_bf16* k_pool, kvs_bf16* v_pool, int32_t num_blocks,
                           int32_t* block_tables, int32_t max_blocks, const int32_t* lens,
                           int32_t* lens_next, int32_t n_items, int32_t h_q, int32_t h_kv,
                           int32_t d, float scale, kvs_bf16* out, void* workspace,
                           size_t workspace_bytes, int32_t* status, int32_t* n_cow,
                           int32_t* n_patch, kvs_stream stream);

/* kvs_decode_step over FP8 pools (kvs_copy_blocks_fp8 for the copies,
 * kvs_paged_decode_fp8 for the decode; d = 128). */
kvs_status kvs_decode_step_fp8(kvs_allocator* a, int32_t* tables_h, int32_t* lens_h,
                               int32_t* patch_h, int32_t* cow_h, int32_t* patch_d,
                               int32_t* cow_d, const kvs_bf16* q, const kvs_bf16* k_new,
                               const kvs_bf16* v_new, uint8_t* k_pool, uint8_t* v_pool,
                               float* k_scale, float* v_scale, int32_t num_blocks,
                               int32_t* block_tables, int32_t max_blocks, const int32_t* lens,
                               int32_t* lens_next, int32_t n_items, int32_t h_q, int32_t h_kv,
                               int32_t d, float scale, kvs_bf16* out, void* workspace,
                               size_t workspace_bytes, int32_t* status, int32_t* n_cow,
                               int32_t* n_patch, kvs_stream stream);

/* ------------------------------------------------------------------------
 * 7. Decode-time scoring and fixed-budget replacement (budgeted layers).
 * Source: Novita article, section "Key techniques 1" (after the first three
 * layers a sliding-window strategy replaces the lowest-scoring KVs
 * automatically) and section "Key techniques 2" (the decode-side
 * PagedAttention works toward the same score S as the prefill).  Readings
 * (the pages give no formula): a budgeted item keeps exactly lens[i] = k_l
 * slots per KV head; a step's new token takes, per KV head, the slot of the
 * token with the lowest accumulated score among those at positions
 * <= new_pos[i] - recent (ties to the lower position); each step adds to
 * every cached token the attention probability the step's query heads give
 * it, summed over the KV head's query group.  A step is
 *   kvs_evict_place -> kvs_paged_decode (k_new = NULL, over lens[i] slots)
 *   -> kvs_decode_scores
 * on one stream (or, with the logits written by the decode itself,
 * kvs_evict_place -> kvs_paged_decode_logits -> kvs_decode_scores_from_logits).  State, device, per item i and KV head h, slot j < lens[i]:
 *   score [n_items][h_kv][max_slots] fp32: the accumulated score;
 *   pos   [n_items][h_kv][max_slots] int32: the token's position;
 *   new_pos [n_items] int32: the position of the step's new token.
 * Slot j lives at row j % 16 of block block_tables[i][j / 16] (as written by
 * kvs_compact_blocks).  Out-of-range table entries, lens[i] > max_slots, or
 * a head whose cached tokens are all recent store KVS_ERR_INVALID in status.
 * ---------------------------------------------------------------------- */

/* Choose each (item, KV head)'s slot for the step's token and write
 * k_new / v_new [n_items][h_kv][d] bf16 there; the slot's score becomes 0 and
 * its position new_pos[i].  One CTA per (item, KV head). */
kvs_status kvs_evict_place(const kvs_bf16* k_new, const kvs_bf16* v_new, kvs_bf16* k_pool,
                           kvs_bf16* v_pool, int32_t num_blocks, const int32_t* block_tables,
                           int32_t max_blocks, const int32_t* lens, const int32_t* new_pos,
                           float* score, int32_t* pos, int32_t max_slots, int32_t n_items,
                           int32_t h_kv, int32_t d, int32_t recent, int32_t* status,
                           kvs_stream stream);

/* kvs_evict_place over FP8 pools (layout and quantisation as
 * kvs_compact_blocks_fp8; d = 128 only).  The claimed slot, positions and
 * scores as kvs_evict_place; the new K and V rows are quantised the same way
 * as the compaction (per-row scale from the row's maximum magnitude, e4m3
 * codes) and written into the slot: K codes in the block's row layout, V
 * codes transposed, the two scales into k_scale / v_scale.  k_new / v_new
 * must be 8-byte aligned.  Errors as kvs_evict_place. */
kvs_status kvs_evict_place_fp8(const kvs_bf16* k_new, const kvs_bf16* v_new, uint8_t* k_pool,
                               uint8_t* v_pool, float* k_scale, float* v_scale,
                               int32_t num_blocks, const int32_t* block_tables,
                               int32_t max_blocks, const int32_t* lens, const int32_t* new_pos,
                               float* score, int32_t* pos, int32_t max_slots, int32_t n_items,
                               int32_t h_kv, int32_t d, int32_t recent, int32_t* status,
                               kvs_stream stream);

/* Add the step's attention probabilities to the scores: for each (item, KV
 * head), softmax over the lens[i] slots of scale * q_g . k_j for each query
 * head g of the group (q [n_items][h_q][d] bf16, K read from the pool), summed
 * over the group.  Then new_pos[i] += 1.  fp32 arithmetic; G <= 16.  Two
 * launches: the logits of every slot (a thread per slot, 256-slot chunks),
 * then per (item, KV head) the softmax and the score update.  workspace:
 * device scratch of kvs_decode_scores_workspace_size bytes (the logits and
 * each chunk's maxima; needs no initialisation). */
size_t kvs_decode_scores_workspace_size(int32_t n_items, int32_t h_q, int32_t h_kv,
                                        int32_t max_slots);

/* kvs_paged_decode over FP8 pools (layout and quantisation as
 * kvs_compact_blocks_fp8; d = 128 only).  The appended k_new / v_new rows
 * are quantised the same way into slot lens[i] (codes and scales).  The
 * result is the attention over the stored values e4m3(code) * s with q and
 * the probabilities (times each token's V scale and 2^10) rounded to fp16,
 * fp32 accumulation.  Input range: every q entry must satisfy |q| <= 65504
 * (a larger one turns into infinity in fp16 and the logits into NaN; entries
 * below about 6.1e-5 in magnitude keep only fp16-subnormal precision), and
 * |v| must stay below 28000.  Nothing checks these ranges.  Workspace, status
 * and every other argument as kvs_paged_decode. */
kvs_status kvs_paged_decode_fp8(const kvs_bf16* q, const kvs_bf16* k_new, const kvs_bf16* v_new,
                                uint8_t* k_pool, uint8_t* v_pool, float* k_scale, float* v_scale,
                                int32_t num_blocks, int32_t* block_tables, int32_t max_blocks,
                                const int32_t* table_patch, const int32_t* lens,
                                int32_t* lens_next, int32_t batch, int32_t h_q, int32_t h_kv,
                                int32_t d, float scale, kvs_bf16* out, void* workspace,
                                size_t workspace_bytes, int32_t* status, kvs_stream stream);

/* kvs_paged_decode that also writes every attended slot's logit, log2-scaled
 * (scale * log2(e) * q_g . k_j), to logits [batch][h_kv][G][logit_ld] fp32 at
 * [i][h][g][j] (slots j >= logit_ld are not written), and each query head's
 * log2 softmax denominator, log2(sum_j exp2(logit_j)), to lse [batch][h_q]
 * fp32 (items with no tokens leave theirs unwritten).  Both buffers are
 * caller-owned device memory and must be non-NULL.  With them a step's score
 * update reads the logits instead of K again and needs no reduction:
 *   kvs_evict_place -> kvs_paged_decode_logits -> kvs_decode_scores_from_logits */
kvs_status kvs_paged_decode_logits(const kvs_bf16* q, const kvs_bf16* k_new,
                                   const kvs_bf16* v_new, kvs_bf16* k_pool, kvs_bf16* v_pool,
                                   int32_t num_blocks, int32_t* block_tables, int32_t max_blocks,
                                   const int32_t* table_patch, const int32_t* lens,
                                   int32_t* lens_next, int32_t batch, int32_t h_q, int32_t h_kv,
                                   int32_t d, float scale, kvs_bf16* out, void* workspace,
                                   size_t workspace_bytes, float* logits, int32_t logit_ld,
                                   float* lse, int32_t* status, kvs_stream stream);

/* kvs_paged_decode_logits over FP8 pools: the decode of kvs_paged_decode_fp8
 * (same arguments, the same input range), which also writes every attended
 * slot's log2-scaled logit (the K row's scale included) and each query head's
 * log2 softmax denominator, in the layouts of kvs_paged_decode_logits.
 * Errors as kvs_paged_decode_fp8; a NULL logits or lse buffer, or logit_ld <=
 * 0, is KVS_ERR_INVALID with nothing launched.  Slots at or past logit_ld get
 * no logit. */
kvs_status kvs_paged_decode_logits_fp8(const kvs_bf16* q, const kvs_bf16* k_new,
                                       const kvs_bf16* v_new, uint8_t* k_pool, uint8_t* v_pool,
                                       float* k_scale, float* v_scale, int32_t num_blocks,
                                       int32_t* block_tables, int32_t max_blocks,
                                       const int32_t* table_patch, const int32_t* lens,
                                       int32_t* lens_next, int32_t batch, int32_t h_q,
                                       int32_t h_kv, int32_t d, float scale, kvs_bf16* out,
                                       void* workspace, size_t workspace_bytes, float* logits,
                                       int32_t logit_ld, float* lse, int32_t* status,
                                       kvs_stream stream);

/* The score update of kvs_decode_scores from those logits and denominators:
 * slot j of (item i, KV head h) gains sum_g exp2(logits[i][h][g][j] -
 * lse[i][h*G + g]) (the step's softmax over the lens[i] slots, summed over the
 * group); then new_pos[i] += 1.  One launch, a thread per slot; lens[i] <=
 * logit_ld and lens[i] <= max_slots, else KVS_ERR_INVALID in status. */
kvs_status kvs_decode_scores_from_logits(const float* logits, int32_t logit_ld, const float* lse,
                                         const int32_t* lens, float* score, int32_t* new_pos,
                                         int32_t max_slots, int32_t n_items, int32_t h_q,
                                         int32_t h_kv, int32_t* status, kvs_stream stream);

kvs_status kvs_decode_scores(const kvs_bf16* q, const kvs_bf16* k_pool, int32_t num_blocks,
                             const int32_t* block_tables, int32_t max_blocks, const int32_t* lens,
                             float* score, int32_t* new_pos, int32_t max_slots, int32_t n_items,
                             int32_t h_q, int32_t h_kv, int32_t d, float scale, void* workspace,
                             size_t workspace_bytes, int32_t* status, kvs_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* KVS_H_ */
