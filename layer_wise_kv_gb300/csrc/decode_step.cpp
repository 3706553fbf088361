// One decode step in one native call: the host allocator's preparation of
// every item, the uploads it calls for (copy-on-write pairs, the table
// patch) and the paged decode, queued on the caller's stream.
//
// Sources: Ultralytics glossary "PagedAttention", section "How paging works"
// (a new block when the last one is full; the kernel follows the table) and
// section "Block sharing between sequences" (copy-on-write of a shared last
// block); Novita article, section "Key techniques 2" (PagedAttention on the
// decode side of the serving loop).
#include <cuda_runtime.h>

#include <cstring>

#include "host_common.h"

namespace {

// The step for either pool type: bf16 pools (k_scale == nullptr) or FP8 pools.
kvs_status decode_step(const char* name, kvs_allocator* a, int32_t* tables_h, int32_t* lens_h,
                       int32_t* patch_h, int32_t* cow_h, int32_t* patch_d, int32_t* cow_d,
                       const kvs_bf16* q, const kvs_bf16* k_new, const kvs_bf16* v_new,
                       void* k_pool, void* v_pool, float* k_scale, float* v_scale, bool fp8,
                       int32_t num_blocks, int32_t* block_tables, int32_t max_blocks,
                       const int32_t* lens, int32_t* lens_next, int32_t n_items, int32_t h_q,
                       int32_t h_kv, int32_t d, float scale, kvs_bf16* out, void* workspace,
                       size_t workspace_bytes, int32_t* status, int32_t* n_cow, int32_t* n_patch,
                       kvs_stream stream) {
  KVS_REQUIRE(n_items >= 0, "%s: negative item count", name);
  if (n_cow) *n_cow = 0;
  if (n_patch) *n_patch = 0;
  if (n_items == 0) return KVS_OK;
  KVS_REQUIRE(a && tables_h && lens_h && patch_h && cow_h && patch_d && cow_d,
              "%s: NULL argument", name);
  KVS_REQUIRE(k_new && v_new, "%s: a step appends: k_new and v_new are required", name);
  KVS_REQUIRE(!fp8 || (k_scale && v_scale), "%s: FP8 pools need their scales", name);
  int32_t nc = 0, np = 0, done = 0;
  int32_t* cow_src = cow_h;
  int32_t* cow_dst = cow_h + n_items;
  kvs_status st = kvs_decode_prepare(a, tables_h, max_blocks, lens_h, n_items, patch_h, cow_src,
                                     cow_dst, &nc, &np, &done);
  if (st != KVS_OK) return st;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (nc > 0) {
    // pairs as [old x nc][new x nc], one upload
    std::memmove(cow_h + nc, cow_dst, static_cast<size_t>(nc) * sizeof(int32_t));
    KVS_CUDA(cudaMemcpyAsync(cow_d, cow_h, 2 * static_cast<size_t>(nc) * sizeof(int32_t),
                             cudaMemcpyHostToDevice, s),
             "kvs_decode_step: copy-on-write pair upload");
    st = fp8 ? kvs_copy_blocks_fp8(cow_d, cow_d + nc, nc, static_cast<uint8_t*>(k_pool),
                                   static_cast<uint8_t*>(v_pool), k_scale, v_scale, num_blocks,
                                   h_kv, d, status, stream)
             : kvs_copy_blocks(cow_d, cow_d + nc, nc, static_cast<kvs_bf16*>(k_pool),
                               static_cast<kvs_bf16*>(v_pool), num_blocks, h_kv, d, status,
                               stream);
    if (st != KVS_OK) return st;
  }
  if (np > 0) {
    KVS_CUDA(cudaMemcpyAsync(patch_d, patch_h, static_cast<size_t>(n_items) * sizeof(int32_t),
                             cudaMemcpyHostToDevice, s),
             "kvs_decode_step: table patch upload");
  }
  int32_t* patch = np > 0 ? patch_d : nullptr;
  st = fp8 ? kvs_paged_decode_fp8(q, k_new, v_new, static_cast<uint8_t*>(k_pool),
                                  static_cast<uint8_t*>(v_pool), k_scale, v_scale, num_blocks,
                                  block_tables, max_blocks, patch, lens, lens_next, n_items, h_q,
                                  h_kv, d, scale, out, workspace, workspace_bytes, status, stream)
           : kvs_paged_decode(q, k_new, v_new, static_cast<kvs_bf16*>(k_pool),
                              static_cast<kvs_bf16*>(v_pool), num_blocks, block_tables,
                              max_blocks, patch, lens, lens_next, n_items, h_q, h_kv, d, scale,
                              out, workspace, workspace_bytes, status, stream);
  if (st != KVS_OK) return st;
  for (int32_t i = 0; i < n_items; ++i) ++lens_h[i];
  if (n_cow) *n_cow = nc;
  if (n_patch) *n_patch = np;
  return KVS_OK;
}

}  // namespace

extern "C" kvs_status kvs_decode_step(kvs_allocator* a, int32_t* tables_h, int32_t* lens_h,
                                      int32_t* patch_h, int32_t* cow_h, int32_t* patch_d,
                                      int32_t* cow_d, const kvs_bf16* q, const kvs_bf16* k_new,
                                      const kvs_bf16* v_new, kvs_bf16* k_pool, kvs_bf16* v_pool,
                                      int32_t num_blocks, int32_t* block_tables,
                                      int32_t max_blocks, const int32_t* lens,
                                      int32_t* lens_next, int32_t n_items, int32_t h_q,
                                      int32_t h_kv, int32_t d, float scale, kvs_bf16* out,
                                      void* workspace, size_t workspace_bytes, int32_t* status,
                                      int32_t* n_cow, int32_t* n_patch, kvs_stream stream) {
  return decode_step("kvs_decode_step", a, tables_h, lens_h, patch_h, cow_h, patch_d, cow_d, q,
                     k_new, v_new, k_pool, v_pool, nullptr, nullptr, false, num_blocks,
                     block_tables, max_blocks, lens, lens_next, n_items, h_q, h_kv, d, scale,
                     out, workspace, workspace_bytes, status, n_cow, n_patch, stream);
}

extern "C" kvs_status kvs_decode_step_fp8(
    kvs_allocator* a, int32_t* tables_h, int32_t* lens_h, int32_t* patch_h, int32_t* cow_h,
    int32_t* patch_d, int32_t* cow_d, const kvs_bf16* q, const kvs_bf16* k_new,
    const kvs_bf16* v_new, uint8_t* k_pool, uint8_t* v_pool, float* k_scale, float* v_scale,
    int32_t num_blocks, int32_t* block_tables, int32_t max_blocks, const int32_t* lens,
    int32_t* lens_next, int32_t n_items, int32_t h_q, int32_t h_kv, int32_t d, float scale,
    kvs_bf16* out, void* workspace, size_t workspace_bytes, int32_t* status, int32_t* n_cow,
    int32_t* n_patch, kvs_stream stream) {
  return decode_step("kvs_decode_step_fp8", a, tables_h, lens_h, patch_h, cow_h, patch_d, cow_d,
                     q, k_new, v_new, k_pool, v_pool, k_scale, v_scale, true, num_blocks,
                     block_tables, max_blocks, lens, lens_next, n_items, h_q, h_kv, d, scale,
                     out, workspace, workspace_bytes, status, n_cow, n_patch, stream);
}
