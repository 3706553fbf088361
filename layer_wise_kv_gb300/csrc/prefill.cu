// Causal prefill attention that also returns each row's max logit m and
// normaliser l, on the 5th-generation tensor cores.
//
// Source: Novita article "How KV Sparsity achieves 1.5x acceleration for
// vLLM", section "Key techniques 2: attention modification": FlashAttention-2
// (Figure 7) walks Q in chunks over K/V blocks, keeps a running row maximum and
// l, and divides O by l at the end; the modification also returns the row
// maximum and l (small outputs, slight cost) so the scoring pass can rebuild
// softmax probabilities without a second attention pass.
//
// Kernel layout (one CTA per (query head, 128-query tile, sequence)):
//   warp 4      TMA producer: Q tile once, then K_j / V_j tiles (128 keys x d,
//               128-byte swizzle) into a 2-stage ring each.
//   warp 5      MMA issuer (one thread): S_j = Q K_j^T into TMEM buffer j%2
//               (M=128, N=128, K=d), and O += P_{j-1} V_{j-1} with P read from
//               TMEM (the A operand) and V from shared memory (MN-major B).
//   warps 0-3   softmax warpgroup, one thread per query row: load S_j from
//               TMEM, causal mask on the diagonal tile, online max in the log2
//               domain with lazy rescaling (O and l are rescaled only when the
//               row maximum grows by more than 8, i.e. a factor of 256), P as
//               bf16 written back over S_j in TMEM; finally O / l, m and l.
// TMEM: S buffers at columns [0,128) and [128,256), O at [256, 256+d).
// Every wait on an mbarrier is bounded; on a timeout the kernel records
// KVS_ERR_DEVICE_TIMEOUT, drains its own copies and MMAs, frees TMEM and ends.
#include <cuda_runtime.h>

#include "host_common.h"
#include "ptx.cuh"
#include "tma_host.h"

namespace kvs {
namespace {

constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kStagesKV = 2;
constexpr int kPrefillThreads = 192;
constexpr float kLog2eP = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

struct PrefillParams {
  uint16_t* o;
  float* m;
  float* l;
  const int32_t* cu_seqlens;
  int32_t* status;
  int total, h_q, h_kv, group, n_qtiles_max;
  float scale_log2;
};

template <int D>
struct PrefillSmem {
  static constexpr int kTile = kBN * D * 2;  // one 128 x D bf16 tile = D/64 chunks of 16 KB
  static constexpr int kChunk = 128 * 128;
  // V ring first (see the note on descriptor reach), then K ring, then Q.
  static constexpr int kV = 0;
  static constexpr int kK = kV + kStagesKV * kTile;
  static constexpr int kQ = kK + kStagesKV * kTile;
  static constexpr int kBar = kQ + kTile;
  // barriers: q_full, k_full[2], k_empty[2], v_full[2], v_empty[2], s_full[2],
  // p_full[2], o_done, drain
  static constexpr int kNumBars = 1 + 2 * kStagesKV * 2 + 2 + 2 + 2;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr size_t kBytes = 1024 + kMisc + 16;
};

template <int D>
__global__ void __launch_bounds__(kPrefillThreads, 1)
prefill_attn_kernel(const __grid_constant__ CUtensorMap q_map,
                    const __grid_constant__ CUtensorMap k_map,
                    const __grid_constant__ CUtensorMap v_map, const PrefillParams p) {
  using L = PrefillSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = k_full + kStagesKV;
  uint64_t* v_full = k_empty + kStagesKV;
  uint64_t* v_empty = v_full + kStagesKV;
  uint64_t* s_full = v_empty + kStagesKV;
  uint64_t* p_full = s_full + 2;
  uint64_t* o_done = p_full + 2;
  uint64_t* drain = o_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);

  const int g = blockIdx.x;   // query head
  const int b = blockIdx.z;   // sequence
  const int seq0 = p.cu_seqlens[b];
  const int n = p.cu_seqlens[b + 1] - seq0;
  const int ntiles = (n + kBM - 1) / kBM;
  const int qt = ntiles - 1 - static_cast<int>(blockIdx.y);  // longest tiles first
  if (qt < 0) return;
  const int q0 = qt * kBM;       // first query of the tile (within the sequence)
  const int nkv = qt + 1;        // causal: key tiles 0 .. qt
  const int hk = g / p.group;    // KV head
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (warp == 0) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < kStagesKV; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&p_full[s], kBM);
    }
    mbar_init(o_done, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tmem_o = tmem + 256;

  auto fail_timeout = [&]() {
    flag_status(p.status, KVS_ERR_DEVICE_TIMEOUT);
    *abort_flag = 1;
  };

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int issued_k = 0, issued_v = 0;
      mbar_arrive_expect_tx(q_full, L::kTile);
#pragma unroll
      for (int c = 0; c < D / 64; ++c)
        tma_load_3d(smem + L::kQ + c * L::kChunk, &q_map, q_full, c * 64, g, seq0 + q0);
      for (int j = 0; j < nkv && !*abort_flag; ++j) {
        const int s = j % kStagesKV;
        const uint32_t ph = (j / kStagesKV) & 1;
        const int tok = seq0 + j * kBN;
        if (!mbar_wait(&k_empty[s], ph ^ 1)) { fail_timeout(); break; }
        mbar_arrive_expect_tx(&k_full[s], L::kTile);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(smem + L::kK + s * L::kTile + c * L::kChunk, &k_map, &k_full[s], c * 64, hk,
                      tok);
        ++issued_k;
        if (!mbar_wait(&v_empty[s], ph ^ 1)) { fail_timeout(); break; }
        mbar_arrive_expect_tx(&v_full[s], L::kTile);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(smem + L::kV + s * L::kTile + c * L::kChunk, &v_map, &v_full[s], c * 64, hk,
                      tok);
        ++issued_v;
      }
      // drain: every load we issued has landed before the CTA may exit
      mbar_wait(q_full, 0);
      for (int j = issued_k > kStagesKV ? issued_k - kStagesKV : 0; j < issued_k; ++j)
        if (!mbar_wait(&k_full[j % kStagesKV], (j / kStagesKV) & 1)) break;
      for (int j = issued_v > kStagesKV ? issued_v - kStagesKV : 0; j < issued_v; ++j)
        if (!mbar_wait(&v_full[j % kStagesKV], (j / kStagesKV) & 1)) break;
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_s = idesc_bf16_f32(kBM, kBN, 0);
      const uint32_t idesc_o = idesc_bf16_f32(kBM, D, 1);
      const uint32_t qa = smem_u32(smem + L::kQ);
      bool ok = mbar_wait(q_full, 0);
      if (!ok) fail_timeout();
      auto issue_pv = [&](int jj) -> bool {
        const int pb = jj & 1;
        if (!mbar_wait(&p_full[pb], (jj >> 1) & 1)) return false;
        const int sv = jj % kStagesKV;
        if (!mbar_wait(&v_full[sv], (jj / kStagesKV) & 1)) return false;
        tc_fence_after();
        const uint32_t vb = smem_u32(smem + L::kV + sv * L::kTile);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          // B = V_j: MN-major, 64-column atoms kChunk bytes apart (LBO), 8-key
          // groups 1024 bytes apart (SBO); 16 keys per step = 2048 bytes
          const uint64_t bdesc = smem_desc_sw128(vb + kk * 2048, L::kChunk, 1024);
          mma_ts(tmem_o, tmem + pb * 128 + kk * 8, bdesc, idesc_o, (jj > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&v_empty[sv]);
        mma_commit(o_done);
        return true;
      };
      for (int j = 0; j < nkv && ok && !*abort_flag; ++j) {
        const int sk = j % kStagesKV;
        if (!mbar_wait(&k_full[sk], (j / kStagesKV) & 1)) { ok = false; break; }
        tc_fence_after();
        const uint32_t kb = smem_u32(smem + L::kK + sk * L::kTile);
        const uint32_t s_tmem = tmem + (j & 1) * 128;
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t adesc = smem_desc_sw128(qa + c * L::kChunk + kk * 32, 16, 1024);
            const uint64_t bdesc = smem_desc_sw128(kb + c * L::kChunk + kk * 32, 16, 1024);
            mma_ss(s_tmem, adesc, bdesc, idesc_s, (c | kk) != 0 ? 1u : 0u);
          }
        }
        mma_commit(&s_full[j & 1]);
        mma_commit(&k_empty[sk]);
        if (j >= 1 && !issue_pv(j - 1)) { ok = false; break; }
      }
      if (ok && !*abort_flag && !issue_pv(nkv - 1)) ok = false;
      if (!ok) fail_timeout();
      // drain: all MMAs we issued are complete before TMEM may be freed
      mma_commit(drain);
      mbar_wait(drain, 0);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int r = tid;                    // row of the tile (TMEM lane)
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    float m_ref = -INFINITY;              // exponent reference (lazy)
    float m_max = -INFINITY;              // true running maximum
    float l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < nkv; ++j) {
      const int sb = j & 1;
      if (*abort_flag) { ok = false; break; }
      if (!__all_sync(0xffffffffu, mbar_wait(&s_full[sb], (j >> 1) & 1))) {
        fail_timeout();
        ok = false;
        break;
      }
      tc_fence_after();
      float s[kBN];
#pragma unroll
      for (int c = 0; c < kBN / 32; ++c) {
        uint32_t rr[32];
        tmem_ld32(tmem + lane_base + sb * 128 + c * 32, rr);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) s[c * 32 + e] = __uint_as_float(rr[e]) * p.scale_log2;
      }
      if (j == qt) {  // diagonal tile: key column c visible iff c <= r
#pragma unroll
        for (int c = 0; c < kBN; ++c) s[c] = c <= r ? s[c] : -INFINITY;
      }
      float mt = -INFINITY;
#pragma unroll
      for (int c = 0; c < kBN; ++c) mt = fmaxf(mt, s[c]);
      m_max = fmaxf(m_max, mt);
      const bool need = m_max > m_ref + kRescaleThreshold;
      const float m_new = need ? m_max : m_ref;
      const float factor = ex2(m_ref - m_new);  // 1 when unchanged, 0 on the first tile
      if (__any_sync(0xffffffffu, need) && j > 0) {
        // O holds PV of tiles < j; wait until PV_{j-1} has landed, then rescale
        if (!__all_sync(0xffffffffu, mbar_wait(o_done, (j - 1) & 1))) {
          fail_timeout();
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t rr[32];
          tmem_ld32(tmem_o + lane_base + c * 32, rr);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) rr[e] = __float_as_uint(__uint_as_float(rr[e]) * factor);
          tmem_st32(tmem_o + lane_base + c * 32, rr);
        }
        tmem_wait_st();
      }
      l_run *= factor;
      m_ref = m_new;
      float rs = 0.f;
#pragma unroll
      for (int c = 0; c < kBN / 32; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float p0 = ex2(s[c * 32 + 2 * e] - m_ref);
          const float p1 = ex2(s[c * 32 + 2 * e + 1] - m_ref);
          rs += p0 + p1;
          pk[e] = pack_bf16x2(p0, p1);
        }
        tmem_st16(tmem + lane_base + sb * 128 + c * 16, pk);
      }
      l_run += rs;
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&p_full[sb]);
    }
    // epilogue: O / l, m, l (tcgen05.ld is warp-collective: decide per warp)
    ok = __all_sync(0xffffffffu, ok && !*abort_flag);
    const bool o_ready = ok && __all_sync(0xffffffffu, mbar_wait(o_done, (nkv - 1) & 1));
    if (o_ready) {
      tc_fence_after();
      const int qi = q0 + r;
      const bool row_ok = qi < n;
      const float inv_l = 1.0f / l_run;
      uint16_t* orow = p.o + (static_cast<int64_t>(seq0 + qi) * p.h_q + g) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t rr[32];
        tmem_ld32(tmem_o + lane_base + c * 32, rr);
        tmem_wait_ld();
        if (row_ok) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(rr[8 * v + 0]) * inv_l, __uint_as_float(rr[8 * v + 1]) * inv_l);
            w.y = pack_bf16x2(__uint_as_float(rr[8 * v + 2]) * inv_l, __uint_as_float(rr[8 * v + 3]) * inv_l);
            w.z = pack_bf16x2(__uint_as_float(rr[8 * v + 4]) * inv_l, __uint_as_float(rr[8 * v + 5]) * inv_l);
            w.w = pack_bf16x2(__uint_as_float(rr[8 * v + 6]) * inv_l, __uint_as_float(rr[8 * v + 7]) * inv_l);
            dst[v] = w;
          }
        }
      }
      if (row_ok) {
        const int64_t at = static_cast<int64_t>(g) * p.total + seq0 + qi;
        p.m[at] = m_max * kLn2;
        p.l[at] = l_run * ex2(m_ref - m_max);
      }
    } else if (ok) {
      fail_timeout();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

struct PrefillMaps {
  const void* q = nullptr;
  const void* k = nullptr;
  const void* v = nullptr;
  int total = 0, h_q = 0, h_kv = 0, d = 0;
  CUtensorMap qm, km, vm;
};

bool map_rows(CUtensorMap* m, const void* base, int total, int heads, int d) {
  const uint64_t dims[3] = {static_cast<uint64_t>(d), static_cast<uint64_t>(heads),
                            static_cast<uint64_t>(total)};
  const uint64_t strides[2] = {static_cast<uint64_t>(d) * 2,
                               static_cast<uint64_t>(d) * 2 * heads};
  const uint32_t box[3] = {64, 1, 128};
  return make_bf16_map(m, base, 3, dims, strides, box);
}

template <int D>
kvs_status launch_prefill(const PrefillMaps& mp, const PrefillParams& prm, int batch,
                          cudaStream_t st) {
  static bool configured = false;
  if (!configured) {
    KVS_CUDA(cudaFuncSetAttribute(prefill_attn_kernel<D>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(PrefillSmem<D>::kBytes)),
             "kvs_prefill_attn_lse: raising the shared-memory limit");
    configured = true;
  }
  dim3 grid(prm.h_q, prm.n_qtiles_max, batch);
  prefill_attn_kernel<D><<<grid, kPrefillThreads, PrefillSmem<D>::kBytes, st>>>(mp.qm, mp.km,
                                                                               mp.vm, prm);
  KVS_CHECK_LAUNCH("kvs_prefill_attn_lse");
  return KVS_OK;
}

}  // namespace
}  // namespace kvs

extern "C" kvs_status kvs_prefill_attn_lse(const kvs_bf16* q, const kvs_bf16* k,
                                           const kvs_bf16* v, kvs_bf16* o, float* m, float* l,
                                           const int32_t* cu_seqlens, int32_t batch,
                                           int32_t max_n, int32_t total_tokens, int32_t h_q,
                                           int32_t h_kv, int32_t d, float scale,
                                           int32_t* status, kvs_stream stream) {
  KVS_REQUIRE(batch >= 0, "kvs_prefill_attn_lse: negative batch");
  if (batch == 0 || total_tokens == 0) return KVS_OK;
  KVS_REQUIRE(q && k && v && o && m && l && cu_seqlens, "kvs_prefill_attn_lse: NULL pointer");
  KVS_SUPPORTED(d == 64 || d == 128, "kvs_prefill_attn_lse: d = %d (supported: 64, 128)", d);
  KVS_REQUIRE(h_kv > 0 && h_q > 0 && h_q % h_kv == 0, "kvs_prefill_attn_lse: bad head counts");
  KVS_REQUIRE(max_n >= 1 && total_tokens >= 1 && batch <= 65535,
              "kvs_prefill_attn_lse: bad sizes");
  KVS_REQUIRE(((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o)) & 15) == 0,
              "kvs_prefill_attn_lse: q, k, v, o must be 16-byte aligned");
  kvs::PrefillParams prm;
  prm.o = o;
  prm.m = m;
  prm.l = l;
  prm.cu_seqlens = cu_seqlens;
  prm.status = status;
  prm.total = total_tokens;
  prm.h_q = h_q;
  prm.h_kv = h_kv;
  prm.group = h_q / h_kv;
  prm.n_qtiles_max = (max_n + kvs::kBM - 1) / kvs::kBM;
  prm.scale_log2 = scale * kvs::kLog2eP;
  KVS_REQUIRE(prm.n_qtiles_max <= 65535, "kvs_prefill_attn_lse: max_n too large");

  static thread_local kvs::PrefillMaps cache;
  if (cache.q != q || cache.k != k || cache.v != v || cache.total != total_tokens ||
      cache.h_q != h_q || cache.h_kv != h_kv || cache.d != d) {
    if (!kvs::map_rows(&cache.qm, q, total_tokens, h_q, d) ||
        !kvs::map_rows(&cache.km, k, total_tokens, h_kv, d) ||
        !kvs::map_rows(&cache.vm, v, total_tokens, h_kv, d)) {
      cache.q = nullptr;
      return KVS_ERR_CUDA;
    }
    cache.q = q;
    cache.k = k;
    cache.v = v;
    cache.total = total_tokens;
    cache.h_q = h_q;
    cache.h_kv = h_kv;
    cache.d = d;
  }
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (d == 128) return kvs::launch_prefill<128>(cache, prm, batch, st);
  return kvs::launch_prefill<64>(cache, prm, batch, st);
}
