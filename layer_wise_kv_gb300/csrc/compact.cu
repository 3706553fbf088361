// Compaction of kept K/V rows into 16-token blocks, and whole-block copies.
//
// Compaction: Ultralytics glossary "PagedAttention", section "How paging
// works" -- token slot j of a request lives at slot j % 16 of block
// table[j / 16]; Novita article, section "Key techniques 1" (after the
// sparsification step each layer keeps only its selected KV).  Block copies:
// same glossary, section "Block sharing between sequences" (copy-on-write).
//
// Both kernels are pure data movement, bound by HBM bandwidth: every byte is
// read once and written once with 16-byte vector accesses.  One warp moves one
// kept slot j of one item: for each KV head it reads the 2*d-byte K and V rows
// of the kept token (d=128: 256 B contiguous each) and writes them to the
// pool.  Algorithmic bytes per slot: 2 (K,V) * h_kv * d * 2 B read + the same
// written.
#include <cuda_runtime.h>

#include "fp8.cuh"
#include "host_common.h"
#include "ptx.cuh"

namespace kvs {
namespace {

constexpr int kWarpsPerCta = 8;

__device__ __forceinline__ int find_item(const kvs_compact_item* items, int n_items,
                                         int64_t row) {
  // last item with row_off <= row
  int lo = 0, hi = n_items - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (items[mid].row_off <= row) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__global__ void __launch_bounds__(kWarpsPerCta * 32)
compact_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
               const kvs_compact_item* __restrict__ items, int n_items, int64_t total_rows,
               int h_kv, int chunks_per_row /* d * 2 / 16 */,
               const int32_t* __restrict__ kept_idx, const int32_t* __restrict__ tables,
               uint4* __restrict__ k_pool, uint4* __restrict__ v_pool, int num_blocks,
               int32_t* status) {
  const int lane = threadIdx.x & 31;
  const int64_t warp_global = static_cast<int64_t>(blockIdx.x) * kWarpsPerCta + (threadIdx.x >> 5);
  const int64_t warp_stride = static_cast<int64_t>(gridDim.x) * kWarpsPerCta;
  const int per_head = chunks_per_row;            // 16-byte chunks per (token, head) row
  const int per_slot = 2 * h_kv * per_head;       // K and V, every head
  for (int64_t row = warp_global; row < total_rows; row += warp_stride) {
    const int it = find_item(items, n_items, row);
    const kvs_compact_item item = items[it];
    const int j = static_cast<int>(row - item.row_off);
    if (j >= item.k_eff) continue;                // a row past a short item (cannot happen
                                                  // with consistent row_off)
    const int block = tables[item.table_off + j / KVS_BLOCK_TOKENS];
    if (block == KVS_BLOCK_SKIP) continue;  // a prefix block already in place
    const bool block_ok = block >= 0 && block < num_blocks;
    if (!block_ok) {
      if (lane == 0) flag_status(status, KVS_ERR_INVALID);
      continue;
    }
    const int slot = j % KVS_BLOCK_TOKENS;
    // the kept token of every head for this slot, one lane per head
    const int p_lane = lane < h_kv ? kept_idx[item.idx_off + static_cast<int64_t>(lane) * item.k_eff + j] : 0;
    // all of the slot's loads in flight before its stores (8 x 16 B per lane
    // covers 2 x h_kv x d x 2 B up to h_kv * d = 1024)
    constexpr int kUnroll = 8;
    for (int c0 = 0; c0 < per_slot; c0 += 32 * kUnroll) {
      uint4 val[kUnroll];
      int64_t dst[kUnroll];
      bool is_v[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int c = c0 + u * 32 + lane;
        const bool in_range = c < per_slot;
        is_v[u] = in_range && c >= h_kv * per_head;
        const int cc = !in_range ? 0 : (is_v[u] ? c - h_kv * per_head : c);
        const int h = cc / per_head;
        const int part = cc - h * per_head;
        const int p = __shfl_sync(0xffffffffu, p_lane, h);  // every lane, every step
        dst[u] = -1;
        if (in_range) {
          if (p < 0 || p >= item.n) {
            flag_status(status, KVS_ERR_INVALID);
          } else {
            const int64_t src = ((item.src_tok + p) * h_kv + h) * per_head + part;
            val[u] = is_v[u] ? __ldg(v + src) : __ldg(k + src);
            dst[u] = ((static_cast<int64_t>(block) * h_kv + h) * KVS_BLOCK_TOKENS + slot) *
                         per_head + part;
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u)
        if (dst[u] >= 0) (is_v[u] ? v_pool : k_pool)[dst[u]] = val[u];
    }
  }
}

__global__ void copy_blocks_kernel(const int32_t* __restrict__ src, const int32_t* __restrict__ dst,
                                   int count, uint4* __restrict__ k_pool,
                                   uint4* __restrict__ v_pool, int num_blocks,
                                   int64_t chunks_per_block, int32_t* status) {
  const int64_t total = static_cast<int64_t>(count) * chunks_per_block * 2;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t per_pair = chunks_per_block * 2;
    const int pair = static_cast<int>(i / per_pair);
    int64_t off = i - pair * per_pair;
    uint4* pool = k_pool;
    if (off >= chunks_per_block) {
      pool = v_pool;
      off -= chunks_per_block;
    }
    const int s = src[pair], d = dst[pair];
    if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks) {
      flag_status(status, KVS_ERR_INVALID);
      continue;
    }
    pool[d * chunks_per_block + off] = pool[s * chunks_per_block + off];
  }
}

// Compaction into an FP8 pool (d = 128; layout and quantisation in fp8.cuh).
// One warp per (item, block of 16 kept slots, KV head): it loads the block's
// 16 kept K and V rows (every load in flight), quantises each row with the
// warp's max-reduction for the scale, writes the K rows as they come and
// gathers the V codes transposed in registers (lane l holds rows d = 4l ..
// 4l+3) for one 64-byte store per lane.  Slots past k_eff in an item's last
// block get zero codes and zero scales.  Blocks are enumerated through a
// per-CTA prefix of ceil(k_eff / 16) over the items.
constexpr int kF8MaxItems = 4096;

__global__ void __launch_bounds__(kWarpsPerCta * 32)
compact_fp8_kernel(const uint16_t* __restrict__ k, const uint16_t* __restrict__ v,
                   const kvs_compact_item* __restrict__ items, int n_items, int h_kv,
                   const int32_t* __restrict__ kept_idx, const int32_t* __restrict__ tables,
                   uint8_t* __restrict__ k_pool, uint8_t* __restrict__ v_pool,
                   float* __restrict__ k_scale, float* __restrict__ v_scale, int num_blocks,
                   int32_t* status) {
  __shared__ int pre[kF8MaxItems + 1];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 0) {
    const int per = (n_items + 31) / 32;
    const int b0 = lane * per, b1 = min(n_items, b0 + per);
    int sum = 0;
    for (int b = b0; b < b1; ++b) sum += (max(items[b].k_eff, 0) + KVS_BLOCK_TOKENS - 1) / KVS_BLOCK_TOKENS;
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    int run = incl - sum;
    for (int b = b0; b < b1; ++b) {
      pre[b] = run;
      run += (max(items[b].k_eff, 0) + KVS_BLOCK_TOKENS - 1) / KVS_BLOCK_TOKENS;
    }
    if (lane == 31) pre[n_items] = incl;
  }
  __syncthreads();
  const int64_t units = static_cast<int64_t>(pre[n_items]) * h_kv;
  for (int64_t u = static_cast<int64_t>(blockIdx.x) * kWarpsPerCta + warp; u < units;
       u += static_cast<int64_t>(gridDim.x) * kWarpsPerCta) {
    const int gb = static_cast<int>(u / h_kv);
    const int h = static_cast<int>(u - static_cast<int64_t>(gb) * h_kv);
    int lo = 0, hi = n_items - 1;  // last item with pre[item] <= gb
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pre[mid] <= gb) lo = mid; else hi = mid - 1;
    }
    const kvs_compact_item it = items[lo];
    const int jb = gb - pre[lo];
    const int b = tables[it.table_off + jb];
    if (b == KVS_BLOCK_SKIP) continue;  // a prefix block already in place
    if (b < 0 || b >= num_blocks) {
      if (lane == 0) flag_status(status, KVS_ERR_INVALID);
      continue;
    }
    const int valid = min(KVS_BLOCK_TOKENS, it.k_eff - jb * KVS_BLOCK_TOKENS);
    uint2 kr[KVS_BLOCK_TOKENS], vr[KVS_BLOCK_TOKENS];
#pragma unroll
    for (int r = 0; r < KVS_BLOCK_TOKENS; ++r) {
      kr[r] = vr[r] = make_uint2(0u, 0u);
      if (r < valid) {
        const int p = kept_idx[it.idx_off + static_cast<int64_t>(h) * it.k_eff +
                               jb * KVS_BLOCK_TOKENS + r];
        if (p < 0 || p >= it.n) {
          if (lane == 0) flag_status(status, KVS_ERR_INVALID);
        } else {
          const int64_t src = ((it.src_tok + p) * h_kv + h) * 128 + 4 * lane;
          kr[r] = __ldg(reinterpret_cast<const uint2*>(k + src));
          vr[r] = __ldg(reinterpret_cast<const uint2*>(v + src));
        }
      }
    }
    uint8_t* kt = k_pool + (static_cast<int64_t>(b) * h_kv + h) * KVS_BLOCK_TOKENS * 128;
    uint32_t vt[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) vt[i][0] = vt[i][1] = vt[i][2] = vt[i][3] = 0u;
    float ksc = 0.f, vsc = 0.f;
#pragma unroll
    for (int r = 0; r < KVS_BLOCK_TOKENS; ++r) {
      const float k0 = bf16_lo(kr[r].x), k1 = bf16_hi(kr[r].x), k2 = bf16_lo(kr[r].y),
                  k3 = bf16_hi(kr[r].y);
      const float v0 = bf16_lo(vr[r].x), v1 = bf16_hi(vr[r].x), v2 = bf16_lo(vr[r].y),
                  v3 = bf16_hi(vr[r].y);
      const float ka = warp_max(fmaxf(fmaxf(fabsf(k0), fabsf(k1)), fmaxf(fabsf(k2), fabsf(k3))));
      const float va = warp_max(fmaxf(fmaxf(fabsf(v0), fabsf(v1)), fmaxf(fabsf(v2), fabsf(v3))));
      const bool ok = r < valid;
      const float sk = f8_row_scale(ka), sv = f8_row_scale(va);
      const uint32_t kc = ok ? f8_quant4(k0, k1, k2, k3, sk) : 0u;
      const uint32_t vc = ok ? f8_quant4(v0, v1, v2, v3, sv) : 0u;
      *reinterpret_cast<uint32_t*>(kt + f8_k_off(r, 4 * lane)) = kc;
#pragma unroll
      for (int i = 0; i < 4; ++i) vt[i][r >> 2] |= ((vc >> (8 * i)) & 0xFFu) << (8 * (r & 3));
      if (lane == r) {
        ksc = ok ? sk : 0.f;
        vsc = ok ? sv : 0.f;
      }
    }
    uint8_t* vtile = v_pool + (static_cast<int64_t>(b) * h_kv + h) * 128 * KVS_BLOCK_TOKENS;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      *reinterpret_cast<uint4*>(vtile + (4 * lane + i) * KVS_BLOCK_TOKENS) =
          make_uint4(vt[i][0], vt[i][1], vt[i][2], vt[i][3]);
    if (lane < KVS_BLOCK_TOKENS) {
      const int64_t so = (static_cast<int64_t>(b) * h_kv + h) * KVS_BLOCK_TOKENS + lane;
      k_scale[so] = ksc;
      v_scale[so] = vsc;
    }
  }
}

int sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace kvs

extern "C" {

kvs_status kvs_compact_blocks(const kvs_bf16* k, const kvs_bf16* v, const kvs_compact_item* items,
                              int32_t n_items, int64_t total_rows, int32_t h_kv, int32_t d,
                              const int32_t* kept_idx, const int32_t* block_tables,
                              kvs_bf16* k_pool, kvs_bf16* v_pool, int32_t num_blocks,
                              int32_t* status, kvs_stream stream) {
  KVS_REQUIRE(n_items >= 0 && total_rows >= 0, "kvs_compact_blocks: negative sizes");
  if (n_items == 0 || total_rows == 0) return KVS_OK;
  KVS_REQUIRE(k && v && items && kept_idx && block_tables && k_pool && v_pool,
              "kvs_compact_blocks: NULL pointer");
  KVS_SUPPORTED(d == 64 || d == 128, "kvs_compact_blocks: d = %d (supported: 64, 128)", d);
  KVS_REQUIRE(h_kv > 0 && num_blocks > 0, "kvs_compact_blocks: h_kv / num_blocks must be > 0");
  KVS_SUPPORTED(h_kv <= 32, "kvs_compact_blocks: h_kv = %d (supported: up to 32)", h_kv);
  KVS_REQUIRE(kvs::aligned16(k) && kvs::aligned16(v) && kvs::aligned16(k_pool) &&
                  kvs::aligned16(v_pool),
              "kvs_compact_blocks: K/V and pool pointers must be 16-byte aligned");
  const int64_t warps = total_rows;
  int64_t grid = (warps + kvs::kWarpsPerCta - 1) / kvs::kWarpsPerCta;
  const int64_t cap = static_cast<int64_t>(kvs::sm_count()) * 8;
  if (grid > cap) grid = cap;
  kvs::compact_kernel<<<static_cast<unsigned>(grid), kvs::kWarpsPerCta * 32, 0,
                        static_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const uint4*>(k), reinterpret_cast<const uint4*>(v), items, n_items,
      total_rows, h_kv, d * 2 / 16, kept_idx, block_tables, reinterpret_cast<uint4*>(k_pool),
      reinterpret_cast<uint4*>(v_pool), num_blocks, status);
  KVS_CHECK_LAUNCH("kvs_compact_blocks");
  return KVS_OK;
}

kvs_status kvs_compact_blocks_fp8(const kvs_bf16* k, const kvs_bf16* v,
                                  const kvs_compact_item* items, int32_t n_items,
                                  int64_t total_rows, int32_t h_kv, int32_t d,
                                  const int32_t* kept_idx, const int32_t* block_tables,
                                  uint8_t* k_pool, uint8_t* v_pool, float* k_scale,
                                  float* v_scale, int32_t num_blocks, int32_t* status,
                                  kvs_stream stream) {
  KVS_REQUIRE(n_items >= 0 && total_rows >= 0, "kvs_compact_blocks_fp8: negative sizes");
  if (n_items == 0 || total_rows == 0) return KVS_OK;
  KVS_REQUIRE(k && v && items && kept_idx && block_tables && k_pool && v_pool && k_scale &&
                  v_scale,
              "kvs_compact_blocks_fp8: NULL pointer");
  KVS_SUPPORTED(d == 128, "kvs_compact_blocks_fp8: d = %d (supported: 128)", d);
  KVS_SUPPORTED(n_items <= kvs::kF8MaxItems, "kvs_compact_blocks_fp8: %d items > %d", n_items,
                kvs::kF8MaxItems);
  KVS_REQUIRE(h_kv > 0 && num_blocks > 0, "kvs_compact_blocks_fp8: h_kv / num_blocks must be > 0");
  KVS_REQUIRE(kvs::aligned16(k) && kvs::aligned16(v) && kvs::aligned16(k_pool) &&
                  kvs::aligned16(v_pool) && kvs::aligned16(k_scale) && kvs::aligned16(v_scale),
              "kvs_compact_blocks_fp8: K/V, pool and scale pointers must be 16-byte aligned");
  // units = sum over items of ceil(k_eff / 16) x h_kv <= (total_rows / 16 + n_items) x h_kv
  const int64_t units = (total_rows / KVS_BLOCK_TOKENS + n_items) * h_kv;
  int64_t grid = (units + kvs::kWarpsPerCta - 1) / kvs::kWarpsPerCta;
  const int64_t cap = static_cast<int64_t>(kvs::sm_count()) * 8;
  if (grid > cap) grid = cap;
  kvs::compact_fp8_kernel<<<static_cast<unsigned>(grid), kvs::kWarpsPerCta * 32, 0,
                            static_cast<cudaStream_t>(stream)>>>(
      k, v, items, n_items, h_kv, kept_idx, block_tables, k_pool, v_pool, k_scale, v_scale,
      num_blocks, status);
  KVS_CHECK_LAUNCH("kvs_compact_blocks_fp8");
  return KVS_OK;
}

kvs_status kvs_copy_blocks(const int32_t* src, const int32_t* dst, int32_t count,
                           kvs_bf16* k_pool, kvs_bf16* v_pool, int32_t num_blocks, int32_t h_kv,
                           int32_t d, int32_t* status, kvs_stream stream) {
  KVS_REQUIRE(count >= 0, "kvs_copy_blocks: negative count");
  if (count == 0) return KVS_OK;
  KVS_REQUIRE(src && dst && k_pool && v_pool, "kvs_copy_blocks: NULL pointer");
  KVS_SUPPORTED(d == 64 || d == 128, "kvs_copy_blocks: d = %d (supported: 64, 128)", d);
  KVS_REQUIRE(h_kv > 0 && num_blocks > 0, "kvs_copy_blocks: h_kv / num_blocks must be > 0");
  KVS_REQUIRE(kvs::aligned16(k_pool) && kvs::aligned16(v_pool),
              "kvs_copy_blocks: pool pointers must be 16-byte aligned");
  const int64_t chunks = static_cast<int64_t>(h_kv) * KVS_BLOCK_TOKENS * d * 2 / 16;
  const int64_t total = chunks * 2 * count;
  int64_t grid = (total + 255) / 256;
  const int64_t cap = static_cast<int64_t>(kvs::sm_count()) * 8;
  if (grid > cap) grid = cap;
  kvs::copy_blocks_kernel<<<static_cast<unsigned>(grid), 256, 0,
                            static_cast<cudaStream_t>(stream)>>>(
      src, dst, count, reinterpret_cast<uint4*>(k_pool), reinterpret_cast<uint4*>(v_pool),
      num_blocks, chunks, status);
  KVS_CHECK_LAUNCH("kvs_copy_blocks");
  return KVS_OK;
}

kvs_status kvs_copy_blocks_fp8(const int32_t* src, const int32_t* dst, int32_t count,
                               uint8_t* k_pool, uint8_t* v_pool, float* k_scale, float* v_scale,
                               int32_t num_blocks, int32_t h_kv, int32_t d, int32_t* status,
                               kvs_stream stream) {
  KVS_REQUIRE(count >= 0, "kvs_copy_blocks_fp8: negative count");
  if (count == 0) return KVS_OK;
  KVS_REQUIRE(src && dst && k_pool && v_pool && k_scale && v_scale,
              "kvs_copy_blocks_fp8: NULL pointer");
  KVS_SUPPORTED(d == 128, "kvs_copy_blocks_fp8: d = %d (supported: 128)", d);
  KVS_REQUIRE(h_kv > 0 && num_blocks > 0, "kvs_copy_blocks_fp8: h_kv / num_blocks must be > 0");
  KVS_REQUIRE(kvs::aligned16(k_pool) && kvs::aligned16(v_pool) && kvs::aligned16(k_scale) &&
                  kvs::aligned16(v_scale),
              "kvs_copy_blocks_fp8: pool and scale pointers must be 16-byte aligned");
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t cap = static_cast<int64_t>(kvs::sm_count()) * 8;
  // the codes (16 x d bytes per head and pool), then the row scales (16 floats)
  const int64_t chunk_counts[2] = {static_cast<int64_t>(h_kv) * KVS_BLOCK_TOKENS * d / 16,
                                   static_cast<int64_t>(h_kv) * KVS_BLOCK_TOKENS * 4 / 16};
  uint4* a_pools[2] = {reinterpret_cast<uint4*>(k_pool), reinterpret_cast<uint4*>(k_scale)};
  uint4* b_pools[2] = {reinterpret_cast<uint4*>(v_pool), reinterpret_cast<uint4*>(v_scale)};
  for (int i = 0; i < 2; ++i) {
    int64_t grid = (chunk_counts[i] * 2 * count + 255) / 256;
    if (grid > cap) grid = cap;
    kvs::copy_blocks_kernel<<<static_cast<unsigned>(grid), 256, 0, st>>>(
        src, dst, count, a_pools[i], b_pools[i], num_blocks, chunk_counts[i], status);
    KVS_CHECK_LAUNCH("kvs_copy_blocks_fp8");
  }
  return KVS_OK;
}

kvs_status kvs_workspace_zero(void* workspace, size_t bytes, kvs_stream stream) {
  if (bytes == 0) return KVS_OK;
  KVS_REQUIRE(workspace != nullptr, "kvs_workspace_zero: NULL workspace");
  KVS_CUDA(cudaMemsetAsync(workspace, 0, bytes, static_cast<cudaStream_t>(stream)),
           "kvs_workspace_zero");
  return KVS_OK;
}

}  // extern "C"
