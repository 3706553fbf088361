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
// Persistent form (batches of up to kPMaxBatch sequences): one CTA per SM
// takes a contiguous run of the launch's key tiles, numbered (layer,
// sequence, KV head, tile).  Warp 8 copies: each K tile (128 x d) into a
// ring of up to kPMaxStages stages, and the window block of each (layer,
// sequence, head) group into one of two buffers, the next group's a few
// tiles into the current one.  Warp 9 issues, per tile, S^T = K Q_w^T into
// one of four TMEM buffers (two for windows wider than 128 columns), all of
// a tile's MMAs from one elected thread.  Warps 0-7 sum, in two sets of four
// that take alternate tiles, so that the two summing warps of a scheduler
// are never at the same step: a thread owns one key row (TMEM lane) of its
// set's tiles, reads its logits a few 16-column chunks at a time (the next
// chunks loading while it sums the current ones) and sums
// exp2(s*scale*log2e - c) over the window columns, with c = m*log2e +
// log2(l) per column (so 1/l is in the exponent, and a column outside the
// window gets a c that makes its term 0), two columns at a time on the
// packed fp32 path; only the tile holding the window's own keys applies the
// causal mask.  The common window widths (32, 64, 128, 256 columns) have
// compile-time chunk counts.  Each group's m and l columns are loaded a
// group ahead.  Otherwise (very large batches):
// one CTA per (layer, sequence, KV head, tile of 128 keys); a launch covers
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
constexpr int kPMaxStages = 4;
constexpr int kPThreads = 320;
constexpr int kPMaxBatch = 2048;

struct ScoreParams {
  const float* m;
  const float* l;
  float* scores;
  const int32_t* cu_seqlens;
  int32_t* status;
  int total, h_q, h_kv, group, alpha, n_cols, n_pad, batch, n_layers;
  float scale_log2;
  // persistent form: shared-memory offsets
  int n_stages, q_off, col_off, pre_off, bar_off, misc_off;
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

// Persistent form.  Shared memory: K ring [n_stages][D/64][128 x 128 B],
// window buffers [2][D/64][n_pad x 128 B], column values [2][2][256] (-c and
// the query position), the tile prefix over sequences [batch + 1] and the
// sequence starts [batch + 1], barriers, TMEM address, abort flag.
struct PTile {
  int layer, b, head, tile, tiles_b, seq0, n;
};

// pre: tiles per sequence as a prefix [batch + 1]; cu: the sequences' first
// tokens [batch + 1] (both in shared memory)
__device__ __forceinline__ PTile ptile_at(int64_t t, const int* pre, const int* cu,
                                          const ScoreParams& p) {
  PTile x;
  const int64_t per_layer = static_cast<int64_t>(pre[p.batch]) * p.h_kv;
  x.layer = static_cast<int>(t / per_layer);
  const int r = static_cast<int>(t - x.layer * per_layer);
  int lo = 0, hi = p.batch - 1;  // last sequence with pre[b] * h_kv <= r
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pre[mid] * p.h_kv <= r) lo = mid; else hi = mid - 1;
  }
  x.b = lo;
  x.tiles_b = pre[lo + 1] - pre[lo];
  const int r2 = r - pre[lo] * p.h_kv;
  x.head = r2 / x.tiles_b;
  x.tile = r2 - x.head * x.tiles_b;
  x.seq0 = cu[lo];
  x.n = cu[lo + 1] - x.seq0;
  return x;
}

// The tile after x in the numbering (layer, sequence, head, tile), without a
// division: the next tile of the head, else the next head, else the next
// sequence with tiles, else the next layer.
__device__ __forceinline__ void ptile_next(PTile& x, const int* pre, const int* cu,
                                           const ScoreParams& p) {
  if (++x.tile < x.tiles_b) return;
  x.tile = 0;
  if (++x.head < p.h_kv) return;
  x.head = 0;
  do {
    if (++x.b == p.batch) {
      x.b = 0;
      ++x.layer;
    }
  } while (pre[x.b + 1] == pre[x.b]);
  x.tiles_b = pre[x.b + 1] - pre[x.b];
  x.seq0 = cu[x.b];
  x.n = cu[x.b + 1] - x.seq0;
}

// Sum over the NCH 16-column chunks of one key row held in TMEM, no column
// masked: exp2(s * scale_log2 + (-c)) per column, two columns at a time on the
// packed fp32 path.  Chunks come from TMEM a few at a time, the next ones
// loading while the current ones are summed.
template <int NCH>
__device__ __forceinline__ float sum_row_visible(uint32_t row_addr, const float* cg,
                                                 uint64_t sc2) {
  // chunks per round trip: four (two when there are sixteen, to stay within
  // the 168 registers a thread of a 320-thread CTA may hold)
  constexpr int RT = NCH < 4 ? NCH : (NCH >= 16 ? 2 : 4);
  constexpr int NT = NCH / RT;
  uint32_t r[2][RT][16];
  uint64_t acc2[4] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f), f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
#pragma unroll
  for (int u = 0; u < RT; ++u) tmem_ld16(row_addr + u * 16, r[0][u]);
  tmem_wait_ld();
#pragma unroll
  for (int tr = 0; tr < NT; ++tr) {
    if (tr + 1 < NT) {
#pragma unroll
      for (int u = 0; u < RT; ++u) tmem_ld16(row_addr + ((tr + 1) * RT + u) * 16, r[(tr + 1) & 1][u]);
    }
#pragma unroll
    for (int u = 0; u < RT; ++u) {
      const ulonglong2* cv = reinterpret_cast<const ulonglong2*>(cg + (tr * RT + u) * 16);
#pragma unroll
      for (int e4 = 0; e4 < 4; ++e4) {
        const ulonglong2 c4 = cv[e4];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int e = 4 * e4 + 2 * h;
          float t0, t1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(r[tr & 1][u][e]),
                                   __uint_as_float(r[tr & 1][u][e + 1])),
                           sc2, h ? c4.y : c4.x),
                    t0, t1);
          acc2[(e4 & 1) * 2 + h] = f2_add(acc2[(e4 & 1) * 2 + h], f2_pack(ex2(t0), ex2(t1)));
        }
      }
    }
    if (tr + 1 < NT) tmem_wait_ld();
  }
  float a[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) f2_unpack(acc2[i], a[2 * i], a[2 * i + 1]);
  return ((a[0] + a[1]) + (a[2] + a[3])) + ((a[4] + a[5]) + (a[6] + a[7]));
}

// Any chunk count, masked or not: one chunk at a time, column by column,
// counting a column only where the key is at or before its query.
__device__ __forceinline__ float sum_row_masked(uint32_t row_addr, const float* cg, const int* qc,
                                                int n_chunks, int key, float scale_log2) {
  float acc = 0.f;
  for (int k0 = 0; k0 < n_chunks; ++k0) {
    uint32_t r[16];
    tmem_ld16(row_addr + k0 * 16, r);
    tmem_wait_ld();
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const float xv = ex2(fmaf(__uint_as_float(r[e]), scale_log2, cg[k0 * 16 + e]));
      acc += key <= qc[k0 * 16 + e] ? xv : 0.f;
    }
  }
  return acc;
}

// NCH > 0: the window block is NCH 16-column chunks (compile time); 0: any.
template <int D, int NCH>
__global__ void __launch_bounds__(kPThreads, 1)
window_scores_persistent(const __grid_constant__ CUtensorMap k_map,
                         const __grid_constant__ CUtensorMap q_map, const ScoreParams p) {
  constexpr int kK = kKeyTile * D * 2;  // one K tile
  const int NS = p.n_stages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int q_chunk = p.n_pad * 128;
  const int q_buf = (D / 64) * q_chunk;
  float* cols = reinterpret_cast<float*>(smem + p.col_off);  // [2][2][256]: -c, query position
  int* pre = reinterpret_cast<int*>(smem + p.pre_off);
  int* cu = pre + (p.batch + 1);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.bar_off);
  uint64_t* k_full = bars;
  uint64_t* k_empty = k_full + NS;
  uint64_t* q_full = k_empty + NS;
  uint64_t* q_empty = q_full + 2;
  uint64_t* s_full = q_empty + 2;
  uint64_t* s_empty = s_full + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + p.misc_off);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + p.misc_off + 4);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t ncols = p.n_pad <= 32 ? 32 : (p.n_pad <= 64 ? 64 : (p.n_pad <= 128 ? 128 : 256));
  // TMEM buffers of S^T: four when they fit in the 512 columns (the launch
  // asks for enough shared memory that no other CTA shares the SM), else two;
  // even tiles go to buffers 0 and 2, odd ones to 1 and 3
  const int nb_log = ncols <= 128 ? 2 : 1;
  const int nbuf = 1 << nb_log;

  // launched as a programmatic dependent: wait for the previous grid on the
  // stream (its m and l) before touching global memory
  griddep_launch_dependents();
  griddep_wait();
  if (warp == 9) {
    tmem_alloc(tmem_slot, nbuf * ncols);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], 4);  // one arrival per warp of the set that reads it
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  for (int b = tid; b <= p.batch; b += kPThreads) cu[b] = p.cu_seqlens[b];
  // tiles per sequence, as a prefix (one warp)
  if (warp == 0) {
    const int per = (p.batch + 31) / 32;
    const int b0 = lane * per, b1 = min(p.batch, b0 + per);
    int sum = 0;
    for (int b = b0; b < b1; ++b)
      sum += (p.cu_seqlens[b + 1] - p.cu_seqlens[b] + kKeyTile - 1) / kKeyTile;
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    int run = incl - sum;
    for (int b = b0; b < b1; ++b) {
      pre[b] = run;
      run += (p.cu_seqlens[b + 1] - p.cu_seqlens[b] + kKeyTile - 1) / kKeyTile;
    }
    if (lane == 31) pre[p.batch] = incl;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int64_t total = static_cast<int64_t>(pre[p.batch]) * p.h_kv * p.n_layers;
  const int64_t lo = total * blockIdx.x / gridDim.x;
  const int64_t hi = total * (blockIdx.x + 1) / gridDim.x;
  auto fail = [&]() {
    flag_status(p.status, KVS_ERR_DEVICE_TIMEOUT);
    *abort_flag = 1;
  };

  if (warp == 8) {
    // ------------------------------------------------------------ copies
    if (lane == 0) {
      int qi = 0, ki = 0;
      PTile x = ptile_at(lo, pre, cu, p);
      // Q windows are loaded in group order into two buffers; qn counts the
      // loads issued, qi the groups reached.  The next group's window is
      // loaded NS tiles into the current group (or at its last tile): by then
      // the MMA warp has finished the group before, whose buffer it reuses.
      int qn = 0;
      auto load_q = [&](const PTile& g) -> bool {
        const int qb = qn & 1;
        if (qn >= 2 && !mbar_wait(&q_empty[qb], ((qn >> 1) & 1) ^ 1)) return false;
        mbar_arrive_expect_tx(&q_full[qb], (D / 64) * p.n_cols * 128);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(smem + p.q_off + qb * q_buf + c * q_chunk, &q_map, &q_full[qb], c * 64,
                      g.head * p.group, g.layer * p.total + g.seq0 + g.n - p.alpha);
        ++qn;
        return true;
      };
      int g_first = 0;  // tile index, within its head, of the group's first tile in range
      for (int64_t t = lo; t < hi && !*abort_flag; ++t, ptile_next(x, pre, cu, p)) {
        const int row0 = x.layer * p.total;
        if (t == lo || x.tile == 0) {
          if (qn == qi && !load_q(x)) {
            fail();
            break;
          }
          ++qi;
          g_first = x.tile;
        }
        const int s = ki % NS;
        if (ki >= NS && !mbar_wait(&k_empty[s], ((ki / NS) & 1) ^ 1)) {
          fail();
          break;
        }
        mbar_arrive_expect_tx(&k_full[s], kK);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(smem + s * kK + c * (kKeyTile * 128), &k_map, &k_full[s], c * 64, x.head,
                      row0 + x.seq0 + x.tile * kKeyTile);
        ++ki;
        if (qn == qi && (x.tile - g_first >= NS || x.tile == x.tiles_b - 1) &&
            t + (x.tiles_b - x.tile) < hi) {
          PTile y = x;  // the first tile of the next group
          y.tile = y.tiles_b - 1;
          ptile_next(y, pre, cu, p);
          if (!load_q(y)) {
            fail();
            break;
          }
        }
      }
      // every copy issued has landed before the CTA may end
      for (int i = ki > NS ? ki - NS : 0; i < ki; ++i)
        if (!mbar_wait(&k_full[i % NS], (i / NS) & 1)) break;
      for (int i = qn > 2 ? qn - 2 : 0; i < qn; ++i)
        if (!mbar_wait(&q_full[i & 1], (i >> 1) & 1)) break;
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMAs
    const uint32_t idesc = idesc_bf16_f32(128, p.n_pad, 0);
    bool ok = true;
    auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
      ok = ok && __all_sync(0xffffffffu, mbar_wait(bar, parity));
      if (ok) tc_fence_after();
      return ok;
    };
    int qi = 0, ki = 0, qb = 0;
    PTile x = ptile_at(lo, pre, cu, p);
    for (int64_t t = lo; t < hi && ok; ++t, ptile_next(x, pre, cu, p)) {
      if (t == lo || x.tile == 0) {
        qb = qi & 1;
        if (!wait(&q_full[qb], (qi >> 1) & 1)) break;
        ++qi;
      }
      const int s = ki % NS, tb = ki & (nbuf - 1);
      if (!wait(&k_full[s], (ki / NS) & 1)) break;
      if (ki >= nbuf && !wait(&s_empty[tb], ((ki >> nb_log) & 1) ^ 1)) break;
      // one elected thread issues the tile's MMAs and commits; the operand
      // descriptors step through K by adding to their start-address field
      // (shared addresses are below 256 KB, so the 14-bit field never carries)
      const uint64_t a0 = smem_desc_sw128(smem_u32(smem + s * kK), 16, 1024);
      const uint64_t b0 = smem_desc_sw128(smem_u32(smem + p.q_off + qb * q_buf), 16, 1024);
      if (elect_one()) {
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ss(tmem + tb * ncols, a0 + static_cast<uint64_t>((c * (kKeyTile * 128) + kk * 32) >> 4),
                   b0 + static_cast<uint64_t>((c * q_chunk + kk * 32) >> 4), idesc,
                   (c | kk) != 0 ? 1u : 0u);
        }
        mma_commit(&s_full[tb]);
        mma_commit(&k_empty[s]);
        if (x.tile == x.tiles_b - 1 || t == hi - 1) mma_commit(&q_empty[qb]);
      }
      __syncwarp();
      ++ki;
    }
    if (!ok && lane == 0) fail();
  } else {
    // ------------------------------------------------------------ sums
    // Two sets of four warps take alternate tiles (set = tile parity), so
    // that the two warps of a scheduler are never at the same step; a thread
    // owns one key row of its set's tiles and sums over all columns.  Column
    // tid of each group (256 summing threads cover n_pad <= 256) is computed
    // at the group's start, from m and l loaded while the previous group ran.
    const int set = warp >> 2;
    float pm = 0.f, pl = 1.f;
    auto load_cols = [&](const PTile& x) {
      const float* m_l = p.m + static_cast<int64_t>(x.layer) * p.h_q * p.total;
      const float* l_l = p.l + static_cast<int64_t>(x.layer) * p.h_q * p.total;
      const int w = x.n < p.alpha ? x.n : p.alpha;
      const int c = tid;
      const int t_ = c / p.group;
      if (c < p.n_cols && t_ >= p.alpha - w) {
        const int64_t at = static_cast<int64_t>(x.head * p.group + (c - t_ * p.group)) * p.total +
                           x.seq0 + x.n - p.alpha + t_;
        pm = m_l[at];
        pl = l_l[at];
      }
    };
    int gi = 0, ki = 0;
    // after a wait runs out the warp stops reading TMEM but still passes the
    // group barriers, so that the other set never waits on it there
    bool ok = true;
    PTile x = ptile_at(lo, pre, cu, p);
    if (lo < hi) load_cols(x);
    const int n_chunks = p.n_pad / 16;
    const uint64_t sc2 = f2_pack(p.scale_log2, p.scale_log2);
    const int kr = (warp & 3) * 32 + lane;  // key row of the tile
    for (int64_t t = lo; t < hi; ++t, ptile_next(x, pre, cu, p), ++ki) {
      if (t == lo || x.tile == 0) {
        // this group's columns: -c = -(m log2e + log2 l), kept negated so
        // that a pair of them is an operand of the packed FMA as read, and
        // the query position
        float* cg = cols + (gi & 1) * 2 * 256;
        const int w = x.n < p.alpha ? x.n : p.alpha;
        const int c = tid;
        if (c < p.n_pad) {
          const int t_ = c / p.group;
          const bool vis = c < p.n_cols && t_ >= p.alpha - w;
          cg[c] = vis ? -fmaf(pm, kLog2eS, __log2f(pl)) : -3.0e38f;
          reinterpret_cast<int*>(cg)[256 + c] = vis ? x.n - p.alpha + t_ : -1;
        }
        asm volatile("bar.sync 1, 256;" ::: "memory");  // the summing warps only
        ++gi;
        const int64_t tn = t + (x.tiles_b - x.tile);
        if (tn < hi) {
          // the first tile of the next group: this head's tiles end here
          PTile y = x;
          y.tile = y.tiles_b - 1;
          ptile_next(y, pre, cu, p);
          load_cols(y);
        }
      }
      if ((ki & 1) != set || !ok) continue;
      const float* cg = cols + ((gi - 1) & 1) * 2 * 256;
      const int* qc = reinterpret_cast<const int*>(cg) + 256;
      const int tb = ki & (nbuf - 1);
      ok = __all_sync(0xffffffffu,
                      !*abort_flag && mbar_wait(&s_full[tb], (ki >> nb_log) & 1));
      if (!ok) continue;
      tc_fence_after();
      const int key = x.tile * kKeyTile + kr;
      const bool masked = x.tile * kKeyTile + kKeyTile > x.n - p.alpha;  // holds window keys
      const uint32_t row_addr = tmem + tb * ncols + (static_cast<uint32_t>((warp & 3) * 32) << 16);
      float sum;
      if (NCH > 0 && !masked)
        sum = sum_row_visible<NCH == 0 ? 1 : NCH>(row_addr, cg, sc2);
      else
        sum = sum_row_masked(row_addr, cg, qc, n_chunks, masked ? key : -1, p.scale_log2);
      // every logit of the buffer this warp reads is in registers: free it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_empty[tb]);
      if (key < x.n) {
        float* scores_l = p.scores + static_cast<int64_t>(x.layer) * p.h_kv * p.total;
        scores_l[static_cast<int64_t>(x.head) * p.total + x.seq0 + key] = sum;
      }
    }
    if (!ok) fail();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 9) tmem_dealloc(tmem, nbuf * ncols);
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

// Shared-memory plan of the persistent form; 0 if it does not fit.
template <int D>
size_t plan_persistent(ScoreParams& prm) {
  const size_t kK = static_cast<size_t>(kKeyTile) * D * 2;
  const size_t q_buf = static_cast<size_t>(D / 64) * prm.n_pad * 128;
  for (int ns = kPMaxStages; ns >= 2; --ns) {
    size_t off = ns * kK;
    const size_t q_off = off;
    off += 2 * q_buf;
    const size_t col_off = off;
    off += 2 * 2 * 256 * 4;
    const size_t pre_off = off;
    off += static_cast<size_t>(2 * (prm.batch + 1)) * 4;
    off = (off + 7) & ~static_cast<size_t>(7);
    const size_t bar_off = off;
    off += static_cast<size_t>(2 * ns + 12) * 8;
    const size_t misc_off = off;
    off += 16;
    if (off + 1024 <= 232448) {
      prm.n_stages = ns;
      prm.q_off = static_cast<int>(q_off);
      prm.col_off = static_cast<int>(col_off);
      prm.pre_off = static_cast<int>(pre_off);
      prm.bar_off = static_cast<int>(bar_off);
      prm.misc_off = static_cast<int>(misc_off);
      return off + 1024;
    }
  }
  return 0;
}

int sm_count_scores() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

template <int D, int NCH>
kvs_status launch_persistent(const CUtensorMap& km, const CUtensorMap& qm, const ScoreParams& prm,
                             const cudaLaunchConfig_t& cfg) {
  static bool configured = false;
  if (!configured) {
    KVS_CUDA(cudaFuncSetAttribute(window_scores_persistent<D, NCH>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, 232448),
             "kvs_window_scores: raising the shared-memory limit");
    configured = true;
  }
  KVS_CUDA(cudaLaunchKernelEx(&cfg, window_scores_persistent<D, NCH>, km, qm, prm),
           "kvs_window_scores (launch)");
  return KVS_OK;
}

template <int D>
kvs_status launch_scores(const CUtensorMap& km, const CUtensorMap& qm, ScoreParams prm,
                         int max_n, int batch, int n_layers, cudaStream_t st) {
  const size_t psmem = batch <= kPMaxBatch ? plan_persistent<D>(prm) : 0;
  if (psmem != 0) {
    // at most one CTA per key tile; the tile count is only known on the device,
    // max_n bounds it from above
    const int64_t tiles_max = static_cast<int64_t>((max_n + kKeyTile - 1) / kKeyTile) * batch *
                              prm.h_kv * n_layers;
    const int grid = static_cast<int>(tiles_max < sm_count_scores() ? tiles_max : sm_count_scores());
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kPThreads);
    // four TMEM buffers take all 512 columns: ask for more than half of the
    // SM's shared memory so that no second CTA lands on the SM and waits for
    // them
    const bool four_buf = prm.n_pad <= 128;
    cfg.dynamicSmemBytes = four_buf && psmem < (116u << 10) ? (116u << 10) : psmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // the usual window widths (alpha x G of 32, 64, 128 or 256 columns) get
    // the compile-time row sum
    switch (prm.n_pad / 16) {
      case 2: return launch_persistent<D, 2>(km, qm, prm, cfg);
      case 4: return launch_persistent<D, 4>(km, qm, prm, cfg);
      case 8: return launch_persistent<D, 8>(km, qm, prm, cfg);
      case 16: return launch_persistent<D, 16>(km, qm, prm, cfg);
      default: return launch_persistent<D, 0>(km, qm, prm, cfg);
    }
  }
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
  prm.n_layers = n_layers;
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
