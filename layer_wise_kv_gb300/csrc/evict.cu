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

#include "fp8.cuh"
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

// The slot (item, KV head h) gives its new token: the lowest (score,
// position) among slots older than the recent window; its position becomes
// new_pos[item] and its score 0.  Every thread of the CTA returns the slot,
// -1 when there is none (empty or oversized length, every token recent: the
// latter two flag KVS_ERR_INVALID).
__device__ int claim_slot(int item, int h, const int32_t* __restrict__ lens,
                          const int32_t* __restrict__ new_pos, float* __restrict__ score,
                          int32_t* __restrict__ pos, int max_slots, int h_kv, int recent,
                          int32_t* status) {
  __shared__ float s_sc[kEvictThreads / 32];
  __shared__ int s_ps[kEvictThreads / 32], s_ix[kEvictThreads / 32];
  __shared__ int s_best;
  const int n = lens[item];
  const int np_ = new_pos[item];
  if (n <= 0 || n > max_slots) {
    if (threadIdx.x == 0 && n > max_slots) flag_status(status, KVS_ERR_INVALID);
    return -1;
  }
  const int64_t base = (static_cast<int64_t>(item) * h_kv + h) * max_slots;
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
  return s_best;
}

__global__ void __launch_bounds__(kEvictThreads)
evict_place_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                   uint4* __restrict__ k_pool, uint4* __restrict__ v_pool, int num_blocks,
                   const int32_t* __restrict__ tables, int max_blocks,
                   const int32_t* __restrict__ lens, const int32_t* __restrict__ new_pos,
                   float* __restrict__ score, int32_t* __restrict__ pos, int max_slots, int h_kv,
                   int chunks /* d * 2 / 16 */, int recent, int32_t* status) {
  const int item = blockIdx.x, h = blockIdx.y;
  const int s = claim_slot(item, h, lens, new_pos, score, pos, max_slots, h_kv, recent, status);
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

// The same over FP8 pools (d = 128; layout of kvs_compact_blocks_fp8): the
// new K and V rows are quantised as the compaction does (per-row scale from
// the row's maximum magnitude, e4m3 codes) and written into the claimed
// slot, K codes in the block's row layout, V codes transposed, and the scales.
// One warp writes: lane l holds dimensions 4l .. 4l+3.
__global__ void __launch_bounds__(kEvictThreads)
evict_place_fp8_kernel(const uint2* __restrict__ k_new, const uint2* __restrict__ v_new,
                       uint8_t* __restrict__ k_pool, uint8_t* __restrict__ v_pool,
                       float* __restrict__ k_scale, float* __restrict__ v_scale, int num_blocks,
                       const int32_t* __restrict__ tables, int max_blocks,
                       const int32_t* __restrict__ lens, const int32_t* __restrict__ new_pos,
                       float* __restrict__ score, int32_t* __restrict__ pos, int max_slots, int h_kv,
                       int recent, int32_t* status) {
  constexpr int D = 128;
  const int item = blockIdx.x, h = blockIdx.y;
  const int s = claim_slot(item, h, lens, new_pos, score, pos, max_slots, h_kv, recent, status);
  if (s < 0) return;
  const int64_t row =
      slot_row(tables + static_cast<int64_t>(item) * max_blocks, max_blocks, num_blocks, h_kv, h, s);
  if (row < 0) {
    if (threadIdx.x == 0) flag_status(status, KVS_ERR_INVALID);
    return;
  }
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  const int slot = s % KVS_BLOCK_TOKENS;
  const int64_t block_row = row - slot;  // the block's first row of this head
  const int64_t src = (static_cast<int64_t>(item) * h_kv + h) * (D / 4) + lane;
  const uint2 kw = __ldg(k_new + src);
  const uint2 vw = __ldg(v_new + src);
  const float k0 = bf16_lo(kw.x), k1 = bf16_hi(kw.x), k2 = bf16_lo(kw.y), k3 = bf16_hi(kw.y);
  const float v0 = bf16_lo(vw.x), v1 = bf16_hi(vw.x), v2 = bf16_lo(vw.y), v3 = bf16_hi(vw.y);
  const float sk =
      f8_row_scale(warp_max(fmaxf(fmaxf(fabsf(k0), fabsf(k1)), fmaxf(fabsf(k2), fabsf(k3)))));
  const float sv =
      f8_row_scale(warp_max(fmaxf(fmaxf(fabsf(v0), fabsf(v1)), fmaxf(fabsf(v2), fabsf(v3)))));
  const uint32_t kc = f8_quant4(k0, k1, k2, k3, sk);
  const uint32_t vc = f8_quant4(v0, v1, v2, v3, sv);
  uint8_t* kp = k_pool + block_row * D;
  uint8_t* vp = v_pool + block_row * D;
  *reinterpret_cast<uint32_t*>(kp + f8_k_off(slot, 4 * lane)) = kc;
#pragma unroll
  for (int i = 0; i < 4; ++i)
    vp[(4 * lane + i) * KVS_BLOCK_TOKENS + slot] = static_cast<uint8_t>(vc >> (8 * i));
  if (lane == 0) {
    k_scale[row] = sk;
    v_scale[row] = sv;
  }
}

// The scores in two launches.  decode_logits_kernel: one CTA per (256-slot
// chunk, item, KV head), a thread per slot; the thread issues every 16-byte
// load of its K row (in halves) before it needs one, takes the group's query
// rows (fp32, shared memory) as 16-byte broadcasts, and writes the G logits
// (log2 units) of its slot; the CTA writes each head's maximum over its
// chunk.  decode_scores_update_kernel: one CTA per (item, KV head): each
// head's maximum over the chunks, its sum of exponentials, then every slot's
// probability summed over the group, added to the slot's score; the CTA of KV
// head 0 advances the item's next position.
constexpr int kScoreThreads = 256;  // also the slots of one chunk

// workspace: logits [n_items][h_kv][G][ld], then chunk maxima
// [n_items][h_kv][n_chunks][G]; ld = max_slots rounded up to four floats
__host__ __device__ inline int64_t logit_ld(int max_slots) { return (max_slots + 3) & ~3; }

template <int D>
__global__ void __launch_bounds__(kScoreThreads, 2)
decode_logits_kernel(const uint16_t* __restrict__ q, const uint4* __restrict__ k_pool,
                     int num_blocks, const int32_t* __restrict__ tables, int max_blocks,
                     const int32_t* __restrict__ lens, float* __restrict__ logits,
                     float* __restrict__ chunk_max, int max_slots, int n_chunks, int h_q, int h_kv,
                     int G, float scale_log2, int32_t* status) {
  __shared__ __align__(16) float s_q[16 * D];
  __shared__ float s_red[kScoreThreads / 32][16];
  constexpr int C = D / 8;  // 16-byte chunks per row
  const int chunk = blockIdx.x, item = blockIdx.y, h = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = lens[item];
  const int j0 = chunk * kScoreThreads;
  if (n <= 0 || n > max_slots) {
    if (chunk == 0 && h == 0 && threadIdx.x == 0 && n > max_slots)
      flag_status(status, KVS_ERR_INVALID);
    return;
  }
  if (j0 >= n) return;
  for (int i = threadIdx.x; i < G * D; i += kScoreThreads)
    s_q[i] = bf16_lo(static_cast<uint32_t>(q[(static_cast<int64_t>(item) * h_q + h * G) * D + i]));
  __syncthreads();
  const int j = j0 + threadIdx.x;
  float lg[16];
#pragma unroll
  for (int g = 0; g < 16; ++g) lg[g] = -INFINITY;
  if (j < n) {
    const int lb = j / KVS_BLOCK_TOKENS;
    const int pb = lb < max_blocks ? tables[static_cast<int64_t>(item) * max_blocks + lb] : -1;
    const bool ok = pb >= 0 && pb < num_blocks;
    if (!ok) flag_status(status, KVS_ERR_INVALID);
    const uint4* src = k_pool + ((static_cast<int64_t>(ok ? pb : 0) * h_kv + h) * KVS_BLOCK_TOKENS +
                                 (j % KVS_BLOCK_TOKENS)) * C;
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
    float* out = logits + (static_cast<int64_t>(item) * h_kv + h) * G * logit_ld(max_slots);
#pragma unroll
    for (int g = 0; g < 16; ++g) {
      if (g >= G) break;
      lg[g] = (acc[g][0] + acc[g][1]) * scale_log2;
      out[g * logit_ld(max_slots) + j] = lg[g];
    }
  }
#pragma unroll
  for (int g = 0; g < 16; ++g) {
    if (g >= G) break;
    float v = lg[g];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (lane == 0) s_red[warp][g] = v;
  }
  __syncthreads();
  if (threadIdx.x < G) {
    float m = -INFINITY;
    for (int w = 0; w < kScoreThreads / 32; ++w) m = fmaxf(m, s_red[w][threadIdx.x]);
    chunk_max[((static_cast<int64_t>(item) * h_kv + h) * n_chunks + chunk) * G + threadIdx.x] = m;
  }
}

__global__ void __launch_bounds__(kScoreThreads)
decode_scores_update_kernel(const float* __restrict__ logits, const float* __restrict__ chunk_max,
                            const int32_t* __restrict__ lens, float* __restrict__ score,
                            int32_t* __restrict__ new_pos, int max_slots, int n_chunks, int h_kv,
                            int G) {
  __shared__ float s_red[kScoreThreads / 32][16];
  __shared__ float s_m[16], s_il[16];
  const int item = blockIdx.x, h = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = lens[item];
  if (n > 0 && n <= max_slots) {
    const int64_t ld = logit_ld(max_slots);
    const float* lgt = logits + (static_cast<int64_t>(item) * h_kv + h) * G * ld;
    const int nc = (n + kScoreThreads - 1) / kScoreThreads;
    if (threadIdx.x < G) {
      float m = -INFINITY;
      for (int c = 0; c < nc; ++c)
        m = fmaxf(m, chunk_max[((static_cast<int64_t>(item) * h_kv + h) * n_chunks + c) * G +
                               threadIdx.x]);
      s_m[threadIdx.x] = m;
    }
    __syncthreads();
    float sm[16];
#pragma unroll
    for (int g = 0; g < 16; ++g) sm[g] = 0.f;
    for (int j = threadIdx.x; j < n; j += kScoreThreads)
#pragma unroll
      for (int g = 0; g < 16; ++g)
        if (g < G) sm[g] += ex2(lgt[g * ld + j] - s_m[g]);
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
    float* sc = score + (static_cast<int64_t>(item) * h_kv + h) * max_slots;
    for (int j = threadIdx.x; j < n; j += kScoreThreads) {
      float p = 0.f;
#pragma unroll
      for (int g = 0; g < 16; ++g)
        if (g < G) p += ex2(lgt[g * ld + j] - s_m[g]) * s_il[g];
      sc[j] += p;
    }
  }
  if (h == 0 && threadIdx.x == 0) new_pos[item] += 1;
}

// The score update from what the decode kernel wrote (kvs_paged_decode_logits):
// each slot's log2-scaled logit per query head and each head's log2 softmax
// denominator, so a slot's probability is exp2(logit - lse) with no reduction
// left to do.  A thread per slot, kScoreThreads-slot chunks; grid (chunks,
// h_kv, items).  The first CTA of KV head 0 advances the item's next position.
__global__ void __launch_bounds__(kScoreThreads)
scores_from_logits_kernel(const float* __restrict__ logits, int ld, const float* __restrict__ lse,
                          const int32_t* __restrict__ lens, float* __restrict__ score,
                          int32_t* __restrict__ new_pos, int max_slots, int h_kv, int G,
                          int32_t* status) {
  const int item = blockIdx.z, h = blockIdx.y;
  const int j = blockIdx.x * kScoreThreads + threadIdx.x;
  const int n = lens[item];
  const bool lead = blockIdx.x == 0 && h == 0 && threadIdx.x == 0;
  if (n > max_slots || n > ld) {
    if (lead) flag_status(status, KVS_ERR_INVALID);
  } else if (j < n) {
    const int64_t ih = static_cast<int64_t>(item) * h_kv + h;
    const float* lg = logits + ih * G * ld + j;
    const float* ls = lse + ih * G;
    float p = 0.f;
#pragma unroll
    for (int g = 0; g < 16; ++g)
      if (g < G) p += ex2(lg[static_cast<int64_t>(g) * ld] - ls[g]);
    score[ih * max_slots + j] += p;
  }
  if (lead) new_pos[item] += 1;
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

extern "C" kvs_status kvs_evict_place_fp8(const kvs_bf16* k_new, const kvs_bf16* v_new,
                                          uint8_t* k_pool, uint8_t* v_pool, float* k_scale,
                                          float* v_scale, int32_t num_blocks,
                                          const int32_t* block_tables, int32_t max_blocks,
                                          const int32_t* lens, const int32_t* new_pos,
                                          float* score, int32_t* pos, int32_t max_slots,
                                          int32_t n_items, int32_t h_kv, int32_t d,
                                          int32_t recent, int32_t* status, kvs_stream stream) {
  KVS_REQUIRE(n_items >= 0, "kvs_evict_place_fp8: negative item count");
  if (n_items == 0) return KVS_OK;
  KVS_REQUIRE(k_new && v_new && k_pool && v_pool && k_scale && v_scale && block_tables && lens &&
                  new_pos && score && pos,
              "kvs_evict_place_fp8: NULL pointer");
  KVS_SUPPORTED(d == 128, "kvs_evict_place_fp8: d = %d (supported: 128)", d);
  KVS_REQUIRE(h_kv > 0 && num_blocks > 0 && max_blocks > 0 && max_slots > 0 && recent >= 1 &&
                  n_items <= 65535 && h_kv <= 65535,
              "kvs_evict_place_fp8: bad sizes");
  KVS_REQUIRE(((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) & 7) == 0 &&
                  ((reinterpret_cast<uintptr_t>(k_pool) | reinterpret_cast<uintptr_t>(v_pool)) & 3) == 0,
              "kvs_evict_place_fp8: k_new / v_new must be 8-byte and the pools 4-byte aligned");
  kvs::evict_place_fp8_kernel<<<dim3(n_items, h_kv), kvs::kEvictThreads, 0,
                                static_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const uint2*>(k_new), reinterpret_cast<const uint2*>(v_new), k_pool, v_pool,
      k_scale, v_scale, num_blocks, block_tables, max_blocks, lens, new_pos, score, pos, max_slots,
      h_kv, recent, status);
  KVS_CHECK_LAUNCH("kvs_evict_place_fp8");
  return KVS_OK;
}

extern "C" size_t kvs_decode_scores_workspace_size(int32_t n_items, int32_t h_q, int32_t h_kv,
                                                   int32_t max_slots) {
  if (n_items <= 0 || h_q <= 0 || h_kv <= 0 || max_slots <= 0 || h_q % h_kv != 0) return 0;
  const int64_t G = h_q / h_kv;
  const int64_t n_chunks = (max_slots + kvs::kScoreThreads - 1) / kvs::kScoreThreads;
  return static_cast<size_t>(static_cast<int64_t>(n_items) * h_kv * G *
                             (kvs::logit_ld(max_slots) + n_chunks) * sizeof(float));
}

extern "C" kvs_status kvs_decode_scores(const kvs_bf16* q, const kvs_bf16* k_pool,
                                        int32_t num_blocks, const int32_t* block_tables,
                                        int32_t max_blocks, const int32_t* lens, float* score,
                                        int32_t* new_pos, int32_t max_slots, int32_t n_items,
                                        int32_t h_q, int32_t h_kv, int32_t d, float scale,
                                        void* workspace, size_t workspace_bytes, int32_t* status,
                                        kvs_stream stream) {
  KVS_REQUIRE(n_items >= 0, "kvs_decode_scores: negative item count");
  if (n_items == 0) return KVS_OK;
  KVS_REQUIRE(q && k_pool && block_tables && lens && score && new_pos && workspace,
              "kvs_decode_scores: NULL pointer");
  KVS_SUPPORTED(d == 64 || d == 128, "kvs_decode_scores: d = %d (supported: 64, 128)", d);
  KVS_REQUIRE(h_kv > 0 && h_q > 0 && h_q % h_kv == 0 && num_blocks > 0 && max_blocks > 0 &&
                  max_slots > 0 && n_items <= 65535 && h_kv <= 65535,
              "kvs_decode_scores: bad sizes");
  const int G = h_q / h_kv;
  KVS_SUPPORTED(G <= 16, "kvs_decode_scores: group size %d > 16", G);
  const size_t need = kvs_decode_scores_workspace_size(n_items, h_q, h_kv, max_slots);
  KVS_REQUIRE(workspace_bytes >= need, "kvs_decode_scores: workspace %zu bytes < %zu needed",
              workspace_bytes, need);
  KVS_REQUIRE((reinterpret_cast<uintptr_t>(k_pool) & 15) == 0,
              "kvs_decode_scores: the K pool must be 16-byte aligned");
  const int n_chunks = (max_slots + kvs::kScoreThreads - 1) / kvs::kScoreThreads;
  KVS_SUPPORTED(n_chunks <= 65535, "kvs_decode_scores: %d slots per item is too many", max_slots);
  float* logits = static_cast<float*>(workspace);
  float* chunk_max = logits + static_cast<int64_t>(n_items) * h_kv * G * kvs::logit_ld(max_slots);
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const float sl2 = scale * kvs::kLog2eE;
  const dim3 grid_l(n_chunks, n_items, h_kv);
  if (d == 128)
    kvs::decode_logits_kernel<128><<<grid_l, kvs::kScoreThreads, 0, st>>>(
        reinterpret_cast<const uint16_t*>(q), reinterpret_cast<const uint4*>(k_pool), num_blocks,
        block_tables, max_blocks, lens, logits, chunk_max, max_slots, n_chunks, h_q, h_kv, G, sl2,
        status);
  else
    kvs::decode_logits_kernel<64><<<grid_l, kvs::kScoreThreads, 0, st>>>(
        reinterpret_cast<const uint16_t*>(q), reinterpret_cast<const uint4*>(k_pool), num_blocks,
        block_tables, max_blocks, lens, logits, chunk_max, max_slots, n_chunks, h_q, h_kv, G, sl2,
        status);
  KVS_CHECK_LAUNCH("kvs_decode_scores (logits)");
  kvs::decode_scores_update_kernel<<<dim3(n_items, h_kv), kvs::kScoreThreads, 0, st>>>(
      logits, chunk_max, lens, score, new_pos, max_slots, n_chunks, h_kv, G);
  KVS_CHECK_LAUNCH("kvs_decode_scores (update)");
  return KVS_OK;
}

extern "C" kvs_status kvs_decode_scores_from_logits(const float* logits, int32_t logit_ld,
                                                    const float* lse, const int32_t* lens,
                                                    float* score,
                                                    int32_t* new_pos, int32_t max_slots,
                                                    int32_t n_items, int32_t h_q, int32_t h_kv,
                                                    int32_t* status, kvs_stream stream) {
  KVS_REQUIRE(n_items >= 0, "kvs_decode_scores_from_logits: negative item count");
  if (n_items == 0) return KVS_OK;
  KVS_REQUIRE(logits && lse && lens && score && new_pos,
              "kvs_decode_scores_from_logits: NULL pointer");
  KVS_REQUIRE(h_kv > 0 && h_q > 0 && h_q % h_kv == 0 && max_slots > 0 && logit_ld > 0 &&
                  n_items <= 65535 && h_kv <= 65535,
              "kvs_decode_scores_from_logits: bad sizes");
  KVS_SUPPORTED(h_q / h_kv <= 16, "kvs_decode_scores_from_logits: group size %d > 16",
                h_q / h_kv);
  const unsigned chunks = static_cast<unsigned>((max_slots + kvs::kScoreThreads - 1) /
                                                kvs::kScoreThreads);
  kvs::scores_from_logits_kernel<<<dim3(chunks, h_kv, n_items), kvs::kScoreThreads, 0,
                                   static_cast<cudaStream_t>(stream)>>>(
      logits, logit_ld, lse, lens, score, new_pos, max_slots, h_kv, h_q / h_kv, status);
  KVS_CHECK_LAUNCH("kvs_decode_scores_from_logits");
  return KVS_OK;
}
