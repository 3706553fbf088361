// Window scores S on the 5th-generation tensor cores.
//
// Source: Novita article "How KV Sparsity achieves 1.5x acceleration for
// vLLM", section "Key techniques 2: attention modification": the score of a
// key is the sum of the softmax probabilities the last alpha (instruction)
// queries give it; each probability is rebuilt as exp(k.q - rowmax)/l from
// the prefill's stored row maximum and normaliser; the loop order is turned
// from q.k to k.q so the column sum over queries becomes a per-key row sum
// kept in registers; only the window's query block is visited (the
// article's example: 5000 x 256 instead of 5000 x 5000 pairs).
//
// One CTA per (layer, sequence, KV head, tile of 128 keys); a launch covers
// one or several consecutive layers of stacked buffers.  TMA brings the key tile
// (128 x d) and the window block of the head's G query heads (alpha x G rows
// x d, ordered [query][head]) into 128-byte-swizzled shared memory; one
// thread issues tcgen05.mma with M = 128 keys, N = alpha*G (rounded up to 16)
// window rows, K = d, accumulating S^T = K Q_w^T in TMEM.  Each of the 128
// threads then owns one key row: it reads its N logits from TMEM
// (tcgen05.ld 32x32b), and sums exp2(s*scale*log2e - m*log2e) / l over the
// causally visible window columns.  No atomics, no cross-thread reduction.
#include <cuda_runtime.h>

#include "host_common.h"
#include "ptx.cuh"
#include "tma_host.h"

namespace kvs {
namespace {

constexpr int kScoreThreads = 128;
constexpr int kKeyTile = 128;
constexpr float kLog2eS = 1.4426950408889634f;

struct ScoreParams {
  const float* m;
  const float* l;
  float* scores;
  const int32_t* cu_seqlens;
  int32_t* status;
  int total, h_q, h_kv, group, alpha, n_cols, n_pad, batch;
  float scale_log2;
};

template <int D>
struct ScoreSmem {
  static constexpr int kKBytes = kKeyTile * D * 2;  // D/64 chunks of 128 rows x 128 B
  __host__ __device__ static int q_chunk_bytes(int n_pad) { return n_pad * 128; }
  static size_t bytes(int n_pad) {
    return 1024 + kKBytes + static_cast<size_t>(D / 64) * q_chunk_bytes(n_pad) +
           3 * 256 * 4 /* mcol, ilcol, qcol */ + 64;
  }
};

template <int D>
__global__ void __launch_bounds__(kScoreThreads)
window_scores_kernel(const __grid_constant__ CUtensorMap k_map,
                     const __grid_constant__ CUtensorMap q_map, const ScoreParams p) {
  using L = ScoreSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* k_s = smem;
  uint8_t* q_s = smem + L::kKBytes;
  const int q_chunk = L::q_chunk_bytes(p.n_pad);
  float* mcol = reinterpret_cast<float*>(q_s + (D / 64) * q_chunk);
  float* ilcol = mcol + 256;
  int* qcol = reinterpret_cast<int*>(ilcol + 256);
  uint64_t* bars = reinterpret_cast<uint64_t*>(qcol + 256);  // [0] tma, [1] mma
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  // launched as a programmatic dependent: wait for the previous grid on the
  // stream (its m and l) before touching global memory
  griddep_launch_dependents();
  griddep_wait();
  // blockIdx.z = layer * batch + sequence; a layer's Q and K rows follow the
  // previous layer's in the tensor maps (row = layer * total + token), its
  // m, l and scores sit one [heads][total] plane further on
  const int li = blockIdx.z / p.batch;
  const int b = blockIdx.z - li * p.batch;
  const int h = blockIdx.y;
  const int row0 = li * p.total;
  const float* m_l = p.m + static_cast<int64_t>(li) * p.h_q * p.total;
  const float* l_l = p.l + static_cast<int64_t>(li) * p.h_q * p.total;
  float* scores_l = p.scores + static_cast<int64_t>(li) * p.h_kv * p.total;
  const int seq0 = p.cu_seqlens[b];
  const int n = p.cu_seqlens[b + 1] - seq0;
  const int key0 = blockIdx.x * kKeyTile;
  if (key0 >= n) return;
  const int w = n < p.alpha ? n : p.alpha;  // window rows of this sequence
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t ncols = p.n_pad <= 32 ? 32 : (p.n_pad <= 64 ? 64 : (p.n_pad <= 128 ? 128 : 256));

  if (warp == 0) {
    tmem_alloc(tmem_slot, ncols);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int win_start = seq0 + n - p.alpha;  // may precede the sequence: masked below
  if (tid == 0) {
    mbar_arrive_expect_tx(&bars[0], L::kKBytes + (D / 64) * p.n_cols * 128);
#pragma unroll
    for (int c = 0; c < D / 64; ++c) {
      tma_load_3d(k_s + c * (kKeyTile * 128), &k_map, &bars[0], c * 64, h, row0 + seq0 + key0);
      tma_load_3d(q_s + c * q_chunk, &q_map, &bars[0], c * 64, h * p.group, row0 + win_start);
    }
  }
  // per window column: m * log2(e), 1 / l and the query position (-1 for a
  // column outside this sequence's window, which no key can see)
  for (int c = tid; c < p.n_pad; c += kScoreThreads) {
    float mc = 0.f, il = 0.f;
    int qc = -1;
    if (c < p.n_cols) {
      const int t = c / p.group;             // window query index 0 .. alpha-1
      const int g = h * p.group + (c - t * p.group);
      if (t >= p.alpha - w) {
        const int64_t at = static_cast<int64_t>(g) * p.total + win_start + t;
        mc = m_l[at] * kLog2eS;
        il = 1.0f / l_l[at];
        qc = n - p.alpha + t;
      }
    }
    mcol[c] = mc;
    ilcol[c] = il;
    qcol[c] = qc;
  }
  if (tid == 0) {
    if (!mbar_wait(&bars[0], 0)) {
      flag_status(p.status, KVS_ERR_DEVICE_TIMEOUT);
      *abort_flag = 1;
    } else {
      tc_fence_after();
      const uint32_t idesc = idesc_bf16_f32(128, p.n_pad, 0);
      const uint32_t ka = smem_u32(k_s), qa = smem_u32(q_s);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t adesc = smem_desc_sw128(ka + c * (kKeyTile * 128) + kk * 32, 16, 1024);
          const uint64_t bdesc = smem_desc_sw128(qa + c * q_chunk + kk * 32, 16, 1024);
          mma_ss(tmem, adesc, bdesc, idesc, (c | kk) != 0 ? 1u : 0u);
        }
      }
      mma_commit(&bars[1]);
    }
  }
  __syncthreads();
  bool ok = !*abort_flag;
  if (ok && !mbar_wait(&bars[1], 0)) {
    flag_status(p.status, KVS_ERR_DEVICE_TIMEOUT);
    ok = false;
  }
  ok = __all_sync(0xffffffffu, ok);  // tcgen05.ld below is warp-collective
  tc_fence_after();

  const int key = key0 + warp * 32 + lane;  // this thread's key (row of the tile)
  float acc = 0.f;
  if (ok) {
    const uint32_t row_addr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    for (int c0 = 0; c0 < p.n_pad; c0 += 32) {
      uint32_t r[32];
      tmem_ld32(row_addr + c0, r);
      tmem_wait_ld();
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const int c = c0 + e;
        if (c < p.n_cols) {
          const float x = ex2(fmaf(__uint_as_float(r[e]), p.scale_log2, -mcol[c])) * ilcol[c];
          acc += key <= qcol[c] ? x : 0.f;
        }
      }
    }
  }
  if (key < n) scores_l[static_cast<int64_t>(h) * p.total + seq0 + key] = acc;

  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, ncols);
}

struct QKMaps {
  const void* q = nullptr;
  const void* k = nullptr;
  int total = 0, h_q = 0, h_kv = 0, d = 0, box_rows = 0, box_heads = 0;
  CUtensorMap qm, km;
};

// 3-D map over a [T][H][d] bf16 tensor with a box of (64, heads, rows).
bool map_thd(CUtensorMap* m, const void* base, int total, int heads, int d, int box_heads,
             int box_rows) {
  const uint64_t dims[3] = {static_cast<uint64_t>(d), static_cast<uint64_t>(heads),
                            static_cast<uint64_t>(total)};
  const uint64_t strides[2] = {static_cast<uint64_t>(d) * 2,
                               static_cast<uint64_t>(d) * 2 * heads};
  const uint32_t box[3] = {64, static_cast<uint32_t>(box_heads), static_cast<uint32_t>(box_rows)};
  return make_bf16_map(m, base, 3, dims, strides, box);
}

template <int D>
kvs_status launch_scores(const CUtensorMap& km, const CUtensorMap& qm, const ScoreParams& prm,
                         int max_n, int batch, int n_layers, cudaStream_t st) {
  const size_t smem = ScoreSmem<D>::bytes(prm.n_pad);
  static bool configured = false;
  if (!configured) {
    KVS_CUDA(cudaFuncSetAttribute(window_scores_kernel<D>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, 232448),
             "kvs_window_scores: raising the shared-memory limit");
    configured = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((max_n + kKeyTile - 1) / kKeyTile, prm.h_kv, batch * n_layers);
  cfg.blockDim = dim3(kScoreThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  KVS_CUDA(cudaLaunchKernelEx(&cfg, window_scores_kernel<D>, km, qm, prm),
           "kvs_window_scores (launch)");
  return KVS_OK;
}

}  // namespace
}  // namespace kvs

namespace kvs {
namespace {

kvs_status window_scores(const char* fn, const kvs_bf16* q, const kvs_bf16* k, const float* m,
                         const float* l, float* scores, const int32_t* cu_seqlens, int32_t batch,
                         int32_t max_n, int32_t total_tokens, int32_t h_q, int32_t h_kv, int32_t d,
                         int32_t alpha, float scale, int32_t n_layers, int32_t* status,
                         kvs_stream stream) {
  KVS_REQUIRE(batch >= 0 && n_layers >= 0, "%s: negative batch or layer count", fn);
  if (batch == 0 || total_tokens == 0 || n_layers == 0) return KVS_OK;
  KVS_REQUIRE(q && k && m && l && scores && cu_seqlens, "%s: NULL pointer", fn);
  KVS_SUPPORTED(d == 64 || d == 128, "%s: d = %d (supported: 64, 128)", fn, d);
  KVS_REQUIRE(h_kv > 0 && h_q > 0 && h_q % h_kv == 0, "%s: bad head counts", fn);
  KVS_REQUIRE(alpha >= 1 && max_n >= 1 && total_tokens >= 1, "%s: bad sizes", fn);
  KVS_SUPPORTED(static_cast<int64_t>(batch) * n_layers <= 65535,
                "%s: batch x layers = %lld > 65535", fn,
                static_cast<long long>(batch) * n_layers);
  KVS_REQUIRE(static_cast<int64_t>(total_tokens) * n_layers < (1ll << 31),
              "%s: layers x tokens exceed 32-bit TMA row coordinates", fn);
  const int G = h_q / h_kv;
  KVS_SUPPORTED(alpha * G <= 256, "%s: alpha * G = %d > 256", fn, alpha * G);
  KVS_REQUIRE((reinterpret_cast<uintptr_t>(q) & 15) == 0 && (reinterpret_cast<uintptr_t>(k) & 15) == 0,
              "%s: q and k must be 16-byte aligned", fn);
  ScoreParams prm;
  prm.m = m;
  prm.l = l;
  prm.scores = scores;
  prm.cu_seqlens = cu_seqlens;
  prm.status = status;
  prm.total = total_tokens;
  prm.h_q = h_q;
  prm.h_kv = h_kv;
  prm.group = G;
  prm.alpha = alpha;
  prm.n_cols = alpha * G;
  prm.n_pad = (alpha * G + 15) / 16 * 16;
  prm.batch = batch;
  prm.scale_log2 = scale * kLog2eS;

  // the maps cover every layer of the call: rows = layers x tokens
  const int rows = total_tokens * n_layers;
  static thread_local QKMaps cache;
  if (cache.q != q || cache.k != k || cache.total != rows || cache.h_q != h_q ||
      cache.h_kv != h_kv || cache.d != d || cache.box_rows != alpha || cache.box_heads != G) {
    if (!map_thd(&cache.km, k, rows, h_kv, d, 1, kKeyTile) ||
        !map_thd(&cache.qm, q, rows, h_q, d, G, alpha)) {
      cache.q = nullptr;
      return KVS_ERR_CUDA;
    }
    cache.q = q;
    cache.k = k;
    cache.total = rows;
    cache.h_q = h_q;
    cache.h_kv = h_kv;
    cache.d = d;
    cache.box_rows = alpha;
    cache.box_heads = G;
  }
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (d == 128) return launch_scores<128>(cache.km, cache.qm, prm, max_n, batch, n_layers, st);
  return launch_scores<64>(cache.km, cache.qm, prm, max_n, batch, n_layers, st);
}

}  // namespace
}  // namespace kvs

extern "C" kvs_status kvs_window_scores(const kvs_bf16* q, const kvs_bf16* k, const float* m,
                                        const float* l, float* scores, const int32_t* cu_seqlens,
                                        int32_t batch, int32_t max_n, int32_t total_tokens,
                                        int32_t h_q, int32_t h_kv, int32_t d, int32_t alpha,
                                        float scale, int32_t* status, kvs_stream stream) {
  return kvs::window_scores("kvs_window_scores", q, k, m, l, scores, cu_seqlens, batch, max_n,
                            total_tokens, h_q, h_kv, d, alpha, scale, 1, status, stream);
}

extern "C" kvs_status kvs_window_scores_layers(const kvs_bf16* q, const kvs_bf16* k,
                                               const float* m, const float* l, float* scores,
                                               const int32_t* cu_seqlens, int32_t batch,
                                               int32_t max_n, int32_t total_tokens, int32_t h_q,
                                               int32_t h_kv, int32_t d, int32_t alpha, float scale,
                                               int32_t n_layers, int32_t* status,
                                               kvs_stream stream) {
  return kvs::window_scores("kvs_window_scores_layers", q, k, m, l, scores, cu_seqlens, batch,
                            max_n, total_tokens, h_q, h_kv, d, alpha, scale, n_layers, status,
                            stream);
}
