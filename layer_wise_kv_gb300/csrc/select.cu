// Per-(layer, KV head) top-k_l selection with a forced recent window.
//
// Source: Novita article "How KV Sparsity achieves 1.5x acceleration for
// vLLM" -- section "System model" (prune low-score KV pairs, keep the
// higher-scoring and nearer ones), section "Key techniques 1" (first three
// layers full cache, later layers evict the lowest scores), section "Key
// techniques 2" (per layer l and head h keep the top-k_l tokens by score;
// the rest is discarded for the whole generation).
//
// One CTA per (item, KV head) row.  The row's fp32 scores are mapped to
// order-preserving 32-bit keys and a 4-pass MSB-first radix select (8 bits per
// pass, per-warp shared-memory histograms) finds the key T of the
// (k - recent)-th largest candidate and how many candidates equal to T must be
// kept.  A final ordered pass keeps every candidate with key > T and the
// lowest-position ones with key == T (ties to the lower position), writing
// indices in ascending position with block-wide prefix sums; the recent
// window follows.  The decisions are exact integer comparisons on the stored
// fp32 values.
#include <cuda_runtime.h>

#include "host_common.h"
#include "ptx.cuh"

namespace kvs {
namespace {

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kPerThread = 8;  // consecutive positions per thread in the output pass

__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t b = __float_as_uint(f);
  if (b == 0x80000000u) b = 0u;  // -0.0 compares equal to +0.0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Exclusive block-wide prefix sum of one int per thread; also returns the total.
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_sums, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kSelWarps ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kSelWarps) warp_sums[lane] = w;  // inclusive warp prefix
  }
  __syncthreads();
  total = warp_sums[kSelWarps - 1];
  const int before = warp == 0 ? 0 : warp_sums[warp - 1];
  __syncthreads();  // warp_sums is reused by the next call
  return before + x - v;
}

__global__ void __launch_bounds__(kSelThreads)
select_kernel(const float* __restrict__ scores, int64_t head_stride,
              const kvs_select_item* __restrict__ items, int h_kv, int recent,
              int32_t* __restrict__ kept_idx, int32_t* status) {
  __shared__ uint32_t hist[kSelWarps][256];
  __shared__ int warp_sums[kSelWarps];
  __shared__ uint32_t s_digit;
  __shared__ int s_remaining;

  const int it = blockIdx.x / h_kv;
  const int h = blockIdx.x - it * h_kv;
  const kvs_select_item item = items[it];
  const int n = item.n;
  const int k = item.k;
  const int tid = threadIdx.x;
  if (n <= 0) return;
  const int k_eff = k < n ? k : n;
  int32_t* out = kept_idx + item.idx_off + static_cast<int64_t>(h) * k_eff;
  const float* s = scores + item.score_off + static_cast<int64_t>(h) * head_stride;

  if (k >= n) {  // full cache: identity
    for (int i = tid; i < n; i += kSelThreads) out[i] = i;
    return;
  }
  if (recent > k || k < 0) {
    if (tid == 0) flag_status(status, KVS_ERR_INVALID);
    return;
  }
  const int nc = n - recent;    // candidates: positions 0 .. nc-1
  const int want = k - recent;  // candidates kept
  for (int i = nc + tid; i < n; i += kSelThreads) out[want + (i - nc)] = i;
  if (want == 0) return;

  // ---- radix select of the want-th largest candidate key ----
  const int warp = tid >> 5;
  uint32_t prefix = 0, mask = 0;
  int remaining = want;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int b = tid; b < kSelWarps * 256; b += kSelThreads) (&hist[0][0])[b] = 0;
    __syncthreads();
    for (int i = tid; i < nc; i += kSelThreads) {
      const uint32_t key = order_key(__ldg(s + i));
      if ((key & mask) == prefix) atomicAdd(&hist[warp][(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    // thread t < 256 owns digit (255 - t): inclusive scan from the top digit
    int cnt = 0;
    if (tid < 256) {
      const int dgt = 255 - tid;
#pragma unroll
      for (int w = 0; w < kSelWarps; ++w) cnt += static_cast<int>(hist[w][dgt]);
    }
    int total;
    const int above = block_exclusive_scan(tid < 256 ? cnt : 0, warp_sums, total);
    if (tid < 256 && above < remaining && above + cnt >= remaining) {
      s_digit = static_cast<uint32_t>(255 - tid);
      s_remaining = remaining - above;
    }
    __syncthreads();
    prefix |= s_digit << shift;
    mask |= 255u << shift;
    remaining = s_remaining;
    __syncthreads();
  }
  const uint32_t T = prefix;     // key of the want-th largest candidate
  const int need_eq = remaining; // candidates equal to T to keep (lowest positions)

  // ---- ordered output pass ----
  int eq_run = 0, out_run = 0;
  for (int base = 0; base < nc; base += kSelThreads * kPerThread) {
    const int p0 = base + tid * kPerThread;
    uint32_t keys[kPerThread];
    int n_eq = 0;
#pragma unroll
    for (int e = 0; e < kPerThread; ++e) {
      const int p = p0 + e;
      keys[e] = p < nc ? order_key(__ldg(s + p)) : 0u;
      n_eq += (p < nc && keys[e] == T) ? 1 : 0;
    }
    int tot_eq;
    int eq_rank = eq_run + block_exclusive_scan(n_eq, warp_sums, tot_eq);
    int n_keep = 0;
    uint32_t keep_bits = 0;
#pragma unroll
    for (int e = 0; e < kPerThread; ++e) {
      const int p = p0 + e;
      bool keep = false;
      if (p < nc) {
        if (keys[e] > T) keep = true;
        else if (keys[e] == T) { keep = eq_rank < need_eq; ++eq_rank; }
      }
      if (keep) { keep_bits |= 1u << e; ++n_keep; }
    }
    int tot_keep;
    int pos = out_run + block_exclusive_scan(n_keep, warp_sums, tot_keep);
#pragma unroll
    for (int e = 0; e < kPerThread; ++e)
      if (keep_bits & (1u << e)) out[pos++] = p0 + e;
    eq_run += tot_eq;
    out_run += tot_keep;
  }
  if (tid == 0 && out_run != want) flag_status(status, KVS_ERR_INVALID);  // NaN scores
}

}  // namespace
}  // namespace kvs

extern "C" kvs_status kvs_select_topk(const float* scores, int64_t head_stride,
                                      const kvs_select_item* items, int32_t n_items,
                                      int32_t h_kv, int32_t recent, int32_t* kept_idx,
                                      int32_t* status, kvs_stream stream) {
  KVS_REQUIRE(n_items >= 0 && h_kv > 0 && recent >= 0, "kvs_select_topk: bad sizes");
  if (n_items == 0) return KVS_OK;
  KVS_REQUIRE(scores && items && kept_idx, "kvs_select_topk: NULL pointer");
  KVS_REQUIRE(static_cast<int64_t>(n_items) * h_kv < (1ll << 31), "kvs_select_topk: too many rows");
  kvs::select_kernel<<<static_cast<unsigned>(n_items * h_kv), kvs::kSelThreads, 0,
                       static_cast<cudaStream_t>(stream)>>>(scores, head_stride, items, h_kv,
                                                            recent, kept_idx, status);
  KVS_CHECK_LAUNCH("kvs_select_topk");
  return KVS_OK;
}
