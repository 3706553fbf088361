// Decode-time scoring and fixed-budget replacement in budgeted layers.
//
// Source: Novita article "How KV Sparsity achieves 1.5x acceleration for
// vLLM", section "Key techniques 1" (after the first three layers, a
// sliding-window strategy replaces the lowest-scoring KVs automatically) and
// section "Key techniques 2" (the decode-side PagedAttention works toward the
// same score S as the prefill).  The pages give no formula for the decode
// side; the readings: a budgeted item's cache keeps exactly k_l slots per KV
// head; each step's new token takes, per KV head, the slot of the token with
// the lowest accumulated score among those older than the recent window (ties
// to the lower position); every step adds to each cached token the attention
// probability the step's query heads give it, summed over the KV head's query
// group.
//
// A step is three launches on one stream: evict_place_kernel (choose the slot,
// write the new K/V row into it), kvs_paged_decode over the k_l slots (no
// append), decode_scores_kernel (the step's probabilities added to the
// scores).  Both kernels here run one CTA per (item, KV head).  The scores
// kernel recomputes the step's logits from q and the cached K rows (it reads
// K once more: k_l * d * 2 bytes per item and head) and keeps them in shared
// memory for the max, sum and probability passes.
#include <cuda_runtime.h>

#include <cmath>

#include "host_common.h"
#include "ptx.cuh"

namespace kvs {
namespace {

constexpr int kEvictThreads = 256;
constexpr float kLog2eE = 1.4426950408889634f;

// row of slot j (block table[j / 16], row j % 16) of KV head h, or -1 when the
// table entry is out of range
__device__ __forceinline__ int64_t slot_row(const int32_t* table, int max_blocks, int num_blocks,
                                            int h_kv, int h, int j) {
  const int lb = j / KVS_BLOCK_TOKENS;
  if (lb >= max_blocks) return -1;
  const int pb = table[lb];
  if (pb < 0 || pb >= num_blocks) return -1;
  return (static_cast<int64_t>(pb) * h_kv + h) * KVS_BLOCK_TOKENS + (j % KVS_BLOCK_TOKENS);
}

// (score, position) order: lower score first, ties to the lower position
__device__ __forceinline__ bool before(float s0, int p0, float s1, int p1) {
  return s0 < s1 || (s0 == s1 && p0 < p1);
}

__global__ void __launch_bounds__(kEvictThreads)
evict_place_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                   uint4* __restrict__ k_pool, uint4* __restrict__ v_pool, int num_blocks,
                   const int32_t* __restrict__ tables, int max_blocks,
                   const int32_t* __restrict__ lens, const int32_t* __restrict__ new_pos,
                   float* __restrict__ score, int32_t* __restrict__ pos, int max_slots, int h_kv,
                   int chunks /* d * 2 / 16 */, int recent, int32_t* status) {
  __shared__ float s_sc[kEvictThreads / 32];
  __shared__ int s_ps[kEvictThreads / 32], s_ix[kEvictThreads / 32];
  __shared__ int s_best;
  const int item = blockIdx.x, h = blockIdx.y;
  const int n = lens[item];
  const int np_ = new_pos[item];
  if (n <= 0 || n > max_slots) {
    if (threadIdx.x == 0 && n > max_slots) flag_status(status, KVS_ERR_INVALID);
    return;
  }
  const int64_t base = (static_cast<int64_t>(item) * h_kv + h) * max_slots;
  // lowest (score, position) among slots older than the recent window
  float bs = INFINITY;
  int bp = 0x7fffffff, bi = -1;
  for (int j = threadIdx.x; j < n; j += kEvictThreads) {
    const int pj = pos[base + j];
    if (pj > np_ - recent) continue;
    const float sj = score[base + j];
    if (bi < 0 || before(sj, pj, bs, bp)) {
      bs = sj;
      bp = pj;
      bi = j;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float os = __shfl_xor_sync(0xffffffffu, bs, o);
    const int op = __shfl_xor_sync(0xffffffffu, bp, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (oi >= 0 && (bi < 0 || before(os, op, bs, bp))) {
      bs = os;
      bp = op;
      bi = oi;
    }
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    s_sc[warp] = bs;
    s_ps[warp] = bp;
    s_ix[warp] = bi;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    bs = s_sc[0];
    bp = s_ps[0];
    bi = s_ix[0];
    for (int w = 1; w < kEvictThreads / 32; ++w)
      if (s_ix[w] >= 0 && (bi < 0 || before(s_sc[w], s_ps[w], bs, bp))) {
        bs = s_sc[w];
        bp = s_ps[w];
        bi = s_ix[w];
      }
    s_best = bi;
    if (bi < 0) {
      flag_status(status, KVS_ERR_INVALID);  // every cached token is recent
    } else {
      pos[base + bi] = np_;
      score[base + bi] = 0.f;
    }
  }
  __syncthreads();
  const int s = s_best;
  if (s < 0) return;
  const int64_t row =
      slot_row(tables + static_cast<int64_t>(item) * max_blocks, max_blocks, num_blocks, h_kv, h, s);
  if (row < 0) {
    if (threadIdx.x == 0) flag_status(status, KVS_ERR_INVALID);
    return;
  }
  const int64_t src = (static_cast<int64_t>(item) * h_kv + h) * chunks;
  for (int c = threadIdx.x; c < 2 * chunks; c += kEvictThreads) {
    if (c < chunks)
      k_pool[row * chunks + c] = k_new[src + c];
    else
      v_pool[row * chunks + (c - chunks)] = v_new[src + (c - chunks)];
  }
}

// One CTA per (item, KV head): logits of the G query heads against every
// slot, then per head the maximum and the sum of exponentials, then each
// slot's probability summed over the group, added to its score.  A thread
// owns whole slots: it issues every 16-byte load of a K row before it needs
// the first, and reads the group's query rows (fp32, shared memory) as
// broadcasts.  The item's block table is staged in shared memory.  The CTA of
// KV head 0 advances the item's next position once it is done.
constexpr int kScoreThreads = 256;
constexpr int kMaxTableSmem = 2048;  // table entries staged in shared memory

template <int D>
__global__ void __launch_bounds__(kScoreThreads, 2)
decode_scores_kernel(const uint16_t* __restrict__ q, const uint4* __restrict__ k_pool,
                     int num_blocks, const int32_t* __restrict__ tables, int max_blocks,
                     const int32_t* __restrict__ lens, float* __restrict__ score,
                     int32_t* __restrict__ new_pos, int max_slots, int h_q, int h_kv, int G,
                     float scale_log2, int32_t* status) {
  extern __shared__ __align__(16) float s_dyn[];  // logits [G][max_slots], then q [G][D]
  __shared__ int s_table[kMaxTableSmem];
  __shared__ float s_red[kScoreThreads / 32][16];
  __shared__ float s_m[16], s_il[16];
  constexpr int C = D / 8;  // 16-byte chunks per row
  float* s_logit = s_dyn;
  // q after the logits, padded to a multiple of four floats (16-byte reads)
  float* s_q = s_dyn + ((static_cast<size_t>(G) * max_slots + 3) & ~static_cast<size_t>(3));
  const int item = blockIdx.x, h = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = lens[item];
  if (n > 0 && n <= max_slots) {
    const int32_t* table = tables + static_cast<int64_t>(item) * max_blocks;
    const int nb = (n + KVS_BLOCK_TOKENS - 1) / KVS_BLOCK_TOKENS;
    const bool staged = nb <= kMaxTableSmem && nb <= max_blocks;
    if (staged)
      for (int b = threadIdx.x; b < nb; b += kScoreThreads) s_table[b] = table[b];
    for (int i = threadIdx.x; i < G * D; i += kScoreThreads)
      s_q[i] = bf16_lo(static_cast<uint32_t>(
          q[(static_cast<int64_t>(item) * h_q + h * G) * D + i]));
    __syncthreads();
    float mx[16];
#pragma unroll
    for (int g = 0; g < 16; ++g) mx[g] = -INFINITY;
    for (int j = threadIdx.x; j < n; j += kScoreThreads) {
      const int lb = j / KVS_BLOCK_TOKENS;
      const int pb = staged ? s_table[lb] : (lb < max_blocks ? table[lb] : -1);
      const bool ok = pb >= 0 && pb < num_blocks;
      if (!ok) flag_status(status, KVS_ERR_INVALID);
      const uint4* src = k_pool + ((static_cast<int64_t>(ok ? pb : 0) * h_kv + h) * KVS_BLOCK_TOKENS +
                                   (j % KVS_BLOCK_TOKENS)) * C;
      // the row in halves of H chunks: every load of a half in flight at once
      constexpr int H = C < 8 ? C : 8;
      float acc[16][2];
#pragma unroll
      for (int g = 0; g < 16; ++g) acc[g][0] = acc[g][1] = 0.f;
#pragma unroll
      for (int c0 = 0; c0 < C; c0 += H) {
        uint4 kr[H];
#pragma unroll
        for (int c = 0; c < H; ++c) kr[c] = ok ? __ldg(src + c0 + c) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int g = 0; g < 16; ++g) {
          if (g >= G) break;
          // the query elements of a chunk as two 16-byte shared-memory reads
          const float4* qg = reinterpret_cast<const float4*>(s_q + g * D + c0 * 8);
#pragma unroll
          for (int c = 0; c < H; ++c) {
            const float4 qa = qg[2 * c], qb = qg[2 * c + 1];
            acc[g][0] = fmaf(qa.x, bf16_lo(kr[c].x), acc[g][0]);
            acc[g][1] = fmaf(qa.y, bf16_hi(kr[c].x), acc[g][1]);
            acc[g][0] = fmaf(qa.z, bf16_lo(kr[c].y), acc[g][0]);
            acc[g][1] = fmaf(qa.w, bf16_hi(kr[c].y), acc[g][1]);
            acc[g][0] = fmaf(qb.x, bf16_lo(kr[c].z), acc[g][0]);
            acc[g][1] = fmaf(qb.y, bf16_hi(kr[c].z), acc[g][1]);
            acc[g][0] = fmaf(qb.z, bf16_lo(kr[c].w), acc[g][0]);
            acc[g][1] = fmaf(qb.w, bf16_hi(kr[c].w), acc[g][1]);
          }
        }
      }
#pragma unroll
      for (int g = 0; g < 16; ++g) {
        if (g >= G) break;
        const float a0 = acc[g][0], a1 = acc[g][1];
        const float lg = (a0 + a1) * scale_log2;
        s_logit[g * max_slots + j] = lg;
        mx[g] = fmaxf(mx[g], lg);
      }
    }
    // per head: maximum over the slots
#pragma unroll
    for (int g = 0; g < 16; ++g) {
      if (g >= G) break;
      float v = mx[g];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
      if (lane == 0) s_red[warp][g] = v;
    }
    __syncthreads();
    if (threadIdx.x < G) {
      float m = -INFINITY;
      for (int w = 0; w < kScoreThreads / 32; ++w) m = fmaxf(m, s_red[w][threadIdx.x]);
      s_m[threadIdx.x] = m;
    }
    __syncthreads();
    // per head: sum of exp2(logit - max)
    float sm[16];
#pragma unroll
    for (int g = 0; g < 16; ++g) sm[g] = 0.f;
    for (int j = threadIdx.x; j < n; j += kScoreThreads)
#pragma unroll
      for (int g = 0; g < 16; ++g)
        if (g < G) sm[g] += ex2(s_logit[g * max_slots + j] - s_m[g]);
#pragma unroll
    for (int g = 0; g < 16; ++g) {
      if (g >= G) break;
      float v = sm[g];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) s_red[warp][g] = v;
    }
    __syncthreads();
    if (threadIdx.x < G) {
      float l = 0.f;
      for (int w = 0; w < kScoreThreads / 32; ++w) l += s_red[w][threadIdx.x];
      s_il[threadIdx.x] = 1.0f / l;
    }
    __syncthreads();
    // each slot's probability, summed over the group, added to its score
    float* sc = score + (static_cast<int64_t>(item) * h_kv + h) * max_slots;
    for (int j = threadIdx.x; j < n; j += kScoreThreads) {
      float p = 0.f;
#pragma unroll
      for (int g = 0; g < 16; ++g)
        if (g < G) p += ex2(s_logit[g * max_slots + j] - s_m[g]) * s_il[g];
      sc[j] += p;
    }
  } else if (n > max_slots && threadIdx.x == 0) {
    flag_status(status, KVS_ERR_INVALID);
  }
  if (h == 0 && threadIdx.x == 0) new_pos[item] += 1;
}

}  // namespace
}  // namespace kvs

extern "C" kvs_status kvs_evict_place(const kvs_bf16* k_new, const kvs_bf16* v_new,
                                      kvs_bf16* k_pool, kvs_bf16* v_pool, int32_t num_blocks,
                                      const int32_t* block_tables, int32_t max_blocks,
                                      const int32_t* lens, const int32_t* new_pos, float* score,
                                      int32_t* pos, int32_t max_slots, int32_t n_items,
                                      int32_t h_kv, int32_t d, int32_t recent, int32_t* status,
                                      kvs_stream stream) {
  KVS_REQUIRE(n_items >= 0, "kvs_evict_place: negative item count");
  if (n_items == 0) return KVS_OK;
  KVS_REQUIRE(k_new && v_new && k_pool && v_pool && block_tables && lens && new_pos && score &&
                  pos,
              "kvs_evict_place: NULL pointer");
  KVS_SUPPORTED(d == 64 || d == 128, "kvs_evict_place: d = %d (supported: 64, 128)", d);
  KVS_REQUIRE(h_kv > 0 && num_blocks > 0 && max_blocks > 0 && max_slots > 0 && recent >= 1 &&
                  n_items <= 65535 && h_kv <= 65535,
              "kvs_evict_place: bad sizes");
  KVS_REQUIRE(((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new) |
                reinterpret_cast<uintptr_t>(k_pool) | reinterpret_cast<uintptr_t>(v_pool)) & 15) == 0,
              "kvs_evict_place: k_new, v_new and the pools must be 16-byte aligned");
  kvs::evict_place_kernel<<<dim3(n_items, h_kv), kvs::kEvictThreads, 0,
                            static_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const uint4*>(k_new), reinterpret_cast<const uint4*>(v_new),
      reinterpret_cast<uint4*>(k_pool), reinterpret_cast<uint4*>(v_pool), num_blocks, block_tables,
      max_blocks, lens, new_pos, score, pos, max_slots, h_kv, d * 2 / 16, recent, status);
  KVS_CHECK_LAUNCH("kvs_evict_place");
  return KVS_OK;
}

extern "C" kvs_status kvs_decode_scores(const kvs_bf16* q, const kvs_bf16* k_pool,
                                        int32_t num_blocks, const int32_t* block_tables,
                                        int32_t max_blocks, const int32_t* lens, float* score,
                                        int32_t* new_pos, int32_t max_slots, int32_t n_items,
                                        int32_t h_q, int32_t h_kv, int32_t d, float scale,
                                        int32_t* status, kvs_stream stream) {
  KVS_REQUIRE(n_items >= 0, "kvs_decode_scores: negative item count");
  if (n_items == 0) return KVS_OK;
  KVS_REQUIRE(q && k_pool && block_tables && lens && score && new_pos,
              "kvs_decode_scores: NULL pointer");
  KVS_SUPPORTED(d == 64 || d == 128, "kvs_decode_scores: d = %d (supported: 64, 128)", d);
  KVS_REQUIRE(h_kv > 0 && h_q > 0 && h_q % h_kv == 0 && num_blocks > 0 && max_blocks > 0 &&
                  max_slots > 0 && n_items <= 65535 && h_kv <= 65535,
              "kvs_decode_scores: bad sizes");
  const int G = h_q / h_kv;
  KVS_SUPPORTED(G <= 16, "kvs_decode_scores: group size %d > 16", G);
  const size_t smem =
      (((static_cast<size_t>(G) * max_slots + 3) & ~static_cast<size_t>(3)) +
       static_cast<size_t>(G) * d) * sizeof(float);
  KVS_SUPPORTED(smem <= 200 * 1024, "kvs_decode_scores: %d slots x %d heads exceed shared memory",
                max_slots, G);
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const float sl2 = scale * kvs::kLog2eE;
  const dim3 grid(n_items, h_kv);
  static bool configured = false;  // the shared-memory limit, once per process
  if (!configured) {
    KVS_CUDA(cudaFuncSetAttribute(kvs::decode_scores_kernel<128>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024),
             "kvs_decode_scores: shared-memory limit");
    KVS_CUDA(cudaFuncSetAttribute(kvs::decode_scores_kernel<64>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024),
             "kvs_decode_scores: shared-memory limit");
    configured = true;
  }
  if (d == 128) {
    kvs::decode_scores_kernel<128><<<grid, kvs::kScoreThreads, smem, st>>>(
        reinterpret_cast<const uint16_t*>(q), reinterpret_cast<const uint4*>(k_pool), num_blocks,
        block_tables, max_blocks, lens, score, new_pos, max_slots, h_q, h_kv, G, sl2, status);
  } else {
    kvs::decode_scores_kernel<64><<<grid, kvs::kScoreThreads, smem, st>>>(
        reinterpret_cast<const uint16_t*>(q), reinterpret_cast<const uint4*>(k_pool), num_blocks,
        block_tables, max_blocks, lens, score, new_pos, max_slots, h_q, h_kv, G, sl2, status);
  }
  KVS_CHECK_LAUNCH("kvs_decode_scores");
  return KVS_OK;
}
