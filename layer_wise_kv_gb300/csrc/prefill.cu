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
// Work items are (query head, pair of 128-row query tiles, sequence); the
// lower tile A and the upper tile B of a pair share every K/V tile.  The CTAs
// are persistent (one per SM) and walk the items in a snake order over a
// numbering that runs from the longest pairs down, keeping TMEM, barriers and
// the K/V ring across items: the next item's Q load and first QK^T overlap the
// current item's last tiles and epilogue, and only the first item of a CTA
// pays the start-up.
// Kernel layout:
//   warp 8      TMA producer: per item Q_A, K_0, Q_B, V_0, then K_j / V_j tiles
//               (128 keys x d, 128-byte swizzle) into 2-stage rings; an L2
//               prefetch of the next item's Q.
//   warp 9      MMA issuer (the whole warp, one elected lane per instruction):
//               S_t = Q_t K_j^T into TMEM (M=N=128,
//               K=d) and O_t += P_t V_j with P_t read from TMEM as the A operand
//               and V_j as an MN-major shared-memory B operand.  Issue order
//               PV_A(j), S_A(j+1), PV_B(j), S_B(j+1): the tensor core works on
//               one tile while the other tile's softmax runs.
//   warps 0-3   softmax warpgroup of tile A, warps 4-7 of tile B; one thread
//               per query row holds its whole 128-key S row in registers: causal
//               mask on the diagonal tile, online maximum in the log2 domain
//               (the TMEM loads return each 32-key maximum) with lazy rescaling (O and l are rescaled only when the row
//               maximum grows by more than 8, a factor of 256), P as bf16
//               written back over S in TMEM; finally O / l, m and l.
// TMEM (512 columns): S_A [0,128), S_B [128,256), O_A [256,384), O_B [384,512).
//
// While the tensor core reads both operands of Q K^T from shared memory it
// takes nearly all of the shared-memory bandwidth, and every shared-memory
// access of another thread (an mbarrier test, a flag load) then waits on the
// order of a hundred cycles.  The MMA queue holds only a few instructions, so
// the issuing warp keeps shared-memory accesses off the boundaries between
// MMA groups: it tests the K/V "full" barriers where it waits for the softmax
// anyway (the loads land long before they are needed), it reads no abort flag
// in the loop, and it commits only what a consumer waits on.  The commit that signals S_t(j)
// also covers PV_t(j-1), issued before it, so the softmax may rescale O_t as
// soon as S_t(j) is visible; O_t's own barrier is committed once, after the last
// PV_t.
// Every wait on an mbarrier is bounded; on a timeout the kernel records
// KVS_ERR_DEVICE_TIMEOUT, drains its own copies and MMAs, frees TMEM and ends.
#include <cuda_runtime.h>

#include "host_common.h"
#include "ptx.cuh"
#include "tma_host.h"

namespace kvs {
namespace {

constexpr int kBM = 128;            // rows per query tile
constexpr int kBN = 128;            // keys per K/V tile
constexpr int kStagesKV = 2;
constexpr int kPrefillThreads = 320;
constexpr float kLog2eP = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

struct PrefillParams {
  uint16_t* o;
  float* m;
  float* l;
  const int32_t* cu_seqlens;
  int32_t* status;
  int total, h_q, h_kv, group, n_pairs_max, batch, n_layers;
  int n_items;  // h_q x batch x n_layers x n_pairs_max work items (some empty)
  float scale_log2;
};

template <int D>
struct PrefillSmem {
  static constexpr int kTile = kBN * D * 2;  // one 128 x D bf16 tile = D/64 chunks of 16 KB
  static constexpr int kChunk = 128 * 128;
  // V ring first (an MN-major descriptor reaches furthest), then K ring, Q_A, Q_B.
  static constexpr int kV = 0;
  static constexpr int kK = kV + kStagesKV * kTile;
  static constexpr int kQ = kK + kStagesKV * kTile;
  static constexpr int kBar = kQ + 2 * kTile;
  // barriers: q_full[2], q_empty[2], k_full[2], k_empty[2], v_full[2],
  // v_empty[2], s_full[2], p_half[2], p_full[2], o_done[2], drain
  static constexpr int kNumBars = 4 + 4 * kStagesKV + 2 + 2 + 2 + 2 + 1;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr size_t kBytes = 1024 + kMisc + 16;
};

// A work item: one query head g of one pair of 128-row query tiles (A: rows
// q0 .. q0+127, B: q0+128 .. q0+255, q0 = 256 pr) of sequence b of one layer.
// Items are numbered layer slowest, then pair rank from the top of the
// sequence (y), then sequence, then head: within a layer the numbering runs
// from the longest pairs down (an item whose sequence has fewer than y + 1
// pairs is empty), and the layers follow one another, so a layer's K and V
// stay in L2 while its items run and only the last layer's short items make
// the launch's tail.  Layers are stacked: layer j's rows follow layer j-1's in
// the Q/K/V maps and in O (row = j * total + token), its m and l sit one
// [h_q][total] plane further on.
struct PItem {
  bool valid;
  int g, pr, seq0, n;  // seq0: the sequence's first row in the stacked rows
  // causal: tile A sees key tiles 0 .. 2pr, tile B 0 .. 2pr+1
  __device__ __forceinline__ int nkv_a() const { return 2 * pr + 1; }
  __device__ __forceinline__ int nkv_b() const { return 2 * pr + 2; }
};

__device__ __forceinline__ PItem item_at(int idx, const PrefillParams& p) {
  PItem it;
  it.g = idx % p.h_q;
  const int rest = idx / p.h_q;
  const int b = rest % p.batch;
  const int rest2 = rest / p.batch;
  const int y = rest2 % p.n_pairs_max;
  const int layer = rest2 / p.n_pairs_max;
  const int tok0 = p.cu_seqlens[b];
  it.n = p.cu_seqlens[b + 1] - tok0;
  it.seq0 = layer * p.total + tok0;
  const int npairs = (it.n + 2 * kBM - 1) / (2 * kBM);
  it.pr = npairs - 1 - y;
  it.valid = it.pr >= 0;
  return it;
}

// The k-th item of CTA c out of G persistent CTAs: a snake over the item
// numbering (c, 2G-1-c, 2G+c, ...), which evens out the descending sizes.
__device__ __forceinline__ int item_pos(int k, int c, int G) {
  return k * G + ((k & 1) ? (G - 1 - c) : c);
}

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
  uint64_t* q_full = bars;                 // [tile]
  uint64_t* q_empty = bars + 2;            // [tile]: the item's S_t MMAs are done with Q_t
  uint64_t* k_full = bars + 4;
  uint64_t* k_empty = k_full + kStagesKV;
  uint64_t* v_full = k_empty + kStagesKV;
  uint64_t* v_empty = v_full + kStagesKV;
  uint64_t* s_full = v_empty + kStagesKV;  // [tile]
  uint64_t* p_half = s_full + 2;           // [tile]: P of keys 0..63 written
  uint64_t* p_full = p_half + 2;           // [tile]: all of P written
  uint64_t* o_done = p_full + 2;           // [tile]: one phase per item, after its last PV
  uint64_t* drain = o_done + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);

  const int cta = blockIdx.x, n_cta = gridDim.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (warp == 0) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(&q_full[t], 1);
      mbar_init(&q_empty[t], 1);
    }
    for (int s = 0; s < kStagesKV; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&p_half[t], kBM / 32);  // one arrival per softmax warp
      mbar_init(&p_full[t], kBM / 32);
      mbar_init(&o_done[t], 1);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // launched as a programmatic dependent: the set-up above overlaps the
  // previous kernel's tail; nothing in global memory is touched before it ends
  griddep_launch_dependents();
  griddep_wait();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  auto fail_timeout = [&]() {
    flag_status(p.status, KVS_ERR_DEVICE_TIMEOUT);
    *abort_flag = 1;
  };

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    // Per item: Q_A (once the previous item's last S_A is done with the
    // buffer), K_0, Q_B (once its last S_B is done), V_0, then K_j / V_j.
    // K_0 and Q_A come first because the MMA warp starts the item's S_A(0)
    // inside the previous item's last iteration.
    if (lane == 0) {
      int n_qt[2] = {0, 0}, n_k = 0, n_v = 0;  // Q_t, K and V tiles issued so far
      bool ok = true;
      auto load_q = [&](int t, const PItem& it) -> bool {
        if (n_qt[t] > 0 && !mbar_wait(&q_empty[t], (n_qt[t] - 1) & 1)) return false;
        mbar_arrive_expect_tx(&q_full[t], L::kTile);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(smem + L::kQ + t * L::kTile + c * L::kChunk, &q_map, &q_full[t], c * 64,
                      it.g, it.seq0 + it.pr * 2 * kBM + t * kBM);
        ++n_qt[t];
        return true;
      };
      auto load_k = [&](const PItem& it, int hk, int j) -> bool {
        const int s = n_k % kStagesKV;
        if (!mbar_wait(&k_empty[s], ((n_k / kStagesKV) & 1) ^ 1)) return false;
        mbar_arrive_expect_tx(&k_full[s], L::kTile);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(smem + L::kK + s * L::kTile + c * L::kChunk, &k_map, &k_full[s], c * 64, hk,
                      it.seq0 + j * kBN);
        ++n_k;
        return true;
      };
      auto load_v = [&](const PItem& it, int hk, int j) -> bool {
        const int s = n_v % kStagesKV;
        if (!mbar_wait(&v_empty[s], ((n_v / kStagesKV) & 1) ^ 1)) return false;
        mbar_arrive_expect_tx(&v_full[s], L::kTile);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(smem + L::kV + s * L::kTile + c * L::kChunk, &v_map, &v_full[s], c * 64, hk,
                      it.seq0 + j * kBN);
        ++n_v;
        return true;
      };
      for (int k = 0; ok && !*abort_flag; ++k) {
        const int pos = item_pos(k, cta, n_cta);
        if (pos >= p.n_items) break;
        const PItem it = item_at(pos, p);
        if (!it.valid) continue;
        const int hk = it.g / p.group;
        ok = load_q(0, it) && load_k(it, hk, 0) && load_q(1, it) && load_v(it, hk, 0);
        if (!ok) break;
        // the next item's Q is read once, from HBM: start it towards L2 now
        for (int k2 = k + 1;; ++k2) {
          const int pos2 = item_pos(k2, cta, n_cta);
          if (pos2 >= p.n_items) break;
          const PItem nx = item_at(pos2, p);
          if (!nx.valid) continue;
#pragma unroll
          for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int c = 0; c < D / 64; ++c)
              tma_prefetch_3d(&q_map, c * 64, nx.g, nx.seq0 + nx.pr * 2 * kBM + t * kBM);
          break;
        }
        for (int j = 1; j < it.nkv_b() && ok; ++j) ok = load_k(it, hk, j) && load_v(it, hk, j);
      }
      if (!ok) fail_timeout();
      // drain: every load we issued has landed before the CTA may exit
      for (int t = 0; t < 2; ++t)
        if (n_qt[t] > 0) mbar_wait(&q_full[t], (n_qt[t] - 1) & 1);
      for (int j = n_k > kStagesKV ? n_k - kStagesKV : 0; j < n_k; ++j)
        if (!mbar_wait(&k_full[j % kStagesKV], (j / kStagesKV) & 1)) break;
      for (int j = n_v > kStagesKV ? n_v - kStagesKV : 0; j < n_v; ++j)
        if (!mbar_wait(&v_full[j % kStagesKV], (j / kStagesKV) & 1)) break;
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the issue loop in lockstep and one elected lane
    // issues each tcgen05 instruction: with uniform control flow the
    // descriptor arithmetic stays on the uniform datapath, and the issue does
    // not starve behind the softmax warps that share this SM sub-partition (a
    // single lane in a divergent branch needs several times the issue slots).
    const uint32_t idesc_s = idesc_bf16_f32(kBM, kBN, 0);
    const uint32_t idesc_o = idesc_bf16_f32(kBM, D, 1);
    // Base descriptors, built once.  The start-address field holds address
    // >> 4 in its low 14 bits; every operand lies inside shared memory, so
    // adding (byte offset >> 4) to the descriptor moves the start address
    // without touching the other fields.
    const uint64_t dq = smem_desc_sw128(smem_u32(smem + L::kQ), 16, 1024);
    const uint64_t dk = smem_desc_sw128(smem_u32(smem + L::kK), 16, 1024);
    // V: MN-major, 64-column atoms kChunk bytes apart (LBO), 8-key groups
    // 1024 bytes apart (SBO); 16 keys per K-step = 2048 bytes
    const uint64_t dv = smem_desc_sw128(smem_u32(smem + L::kV), L::kChunk, 1024);
    bool ok = true;
    // a bounded wait, uniform over the warp; on success orders the following
    // MMAs after it
    auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
      ok = ok && __all_sync(0xffffffffu, mbar_wait(bar, parity));
      if (ok) tc_fence_after();
      return ok;
    };
    auto commit = [&](uint64_t* bar) {
      if (elect_one()) mma_commit(bar);
    };
    // S_t = Q_t K^T with K in ring stage s
    auto issue_s = [&](int t, int s) {
      const uint64_t qa = dq + static_cast<uint64_t>((t * L::kTile) >> 4);
      const uint64_t kb = dk + static_cast<uint64_t>((s * L::kTile) >> 4);
      const uint32_t d_tmem = tmem + t * 128;
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t off = static_cast<uint64_t>(((c * L::kChunk) >> 4) + kk * 2);
          if (elect_one()) mma_ss(d_tmem, qa + off, kb + off, idesc_s, (c | kk) != 0 ? 1u : 0u);
        }
      }
      commit(&s_full[t]);
    };
    // K-steps [k0, k1) of O_t += P_t V with V in ring stage s; the item's
    // first key tile (first) overwrites O_t
    auto issue_pv = [&](int t, int s, bool first, int k0, int k1) {
      const uint64_t vb = dv + static_cast<uint64_t>((s * L::kTile) >> 4);
      const uint32_t o_tmem = tmem + 256 + t * 128;
      const uint32_t p_tmem = tmem + t * 128;
#pragma unroll
      for (int kk = k0; kk < k1; ++kk)
        if (elect_one())
          mma_ts(o_tmem, p_tmem + kk * 8, vb + static_cast<uint64_t>(kk * (2048 >> 4)), idesc_o,
                 (!first || kk > 0) ? 1u : 0u);
    };
    // K_{j+1} and V_j are waited for at the top of iteration j, where the warp
    // would otherwise wait for the softmax: both loads were issued about an
    // iteration earlier and have landed, so no wait sits between MMA groups.
    // Item boundaries are pipelined: the next item's S_A(0) is issued right
    // after this item's last PV_A (its Q_A and K_0 are loaded by then) and its
    // S_B(0) right after the last PV_B, so each softmax warpgroup finds its
    // next tile ready when it leaves its epilogue.  The softmax's first P of
    // an item is written after it has read the previous item's O, so the
    // p_half wait also orders the item's first PV (which overwrites O) after
    // that read.
    int k_next = 0;
    auto next_item = [&]() -> PItem {
      for (;; ++k_next) {
        const int pos = item_pos(k_next, cta, n_cta);
        if (pos >= p.n_items) {
          PItem none;
          none.valid = false;
          return none;
        }
        const PItem it = item_at(pos, p);
        if (it.valid) {
          ++k_next;
          return it;
        }
      }
    };
    int n_q = 0, ring = 0, n_pa = 0, n_pb = 0;  // items, ring tiles, P tiles of A / B
    PItem cur = next_item();
    // the first item's S_A(0), S_B(0)
    if (cur.valid && wait(&q_full[0], 0) && wait(&k_full[0], 0)) {
      issue_s(0, 0);
      if (cur.nkv_a() == 1) commit(&q_empty[0]);
      if (wait(&q_full[1], 0)) {
        issue_s(1, 0);
        commit(&k_empty[0]);
      }
    }
    while (cur.valid && ok) {
      const PItem nxt = next_item();
      const int ring_n = ring + cur.nkv_b();  // ring position of the next item's K_0 / V_0
      const uint32_t qph = (n_q + 1) & 1;   // the next item's Q phase
      for (int j = 0; j < cur.nkv_b(); ++j) {
        const int r = ring + j;  // ring position of key tile j
        const bool more = j + 1 < cur.nkv_b();
        const int s = r % kStagesKV, s1 = (r + 1) % kStagesKV;
        if (!wait(&v_full[s], (r / kStagesKV) & 1)) break;
        if (more && !wait(&k_full[s1], ((r + 1) / kStagesKV) & 1)) break;
        if (j < cur.nkv_a()) {
          if (!wait(&p_half[0], n_pa & 1)) break;
          issue_pv(0, s, j == 0, 0, kBN / 32);
          if (!wait(&p_full[0], n_pa & 1)) break;
          issue_pv(0, s, j == 0, kBN / 32, kBN / 16);
          ++n_pa;
          if (j + 1 < cur.nkv_a()) {
            issue_s(0, s1);
            if (j + 2 == cur.nkv_a()) commit(&q_empty[0]);  // the item's last S_A
          } else {
            commit(&o_done[0]);
            if (nxt.valid) {                                // the next item's S_A(0)
              if (!wait(&q_full[0], qph) ||
                  !wait(&k_full[ring_n % kStagesKV], (ring_n / kStagesKV) & 1))
                break;
              issue_s(0, ring_n % kStagesKV);
              if (nxt.nkv_a() == 1) commit(&q_empty[0]);
            }
          }
        }
        if (!wait(&p_half[1], n_pb & 1)) break;
        issue_pv(1, s, j == 0, 0, kBN / 32);
        if (!wait(&p_full[1], n_pb & 1)) break;
        issue_pv(1, s, j == 0, kBN / 32, kBN / 16);
        ++n_pb;
        commit(&v_empty[s]);
        if (more) {
          issue_s(1, s1);
          commit(&k_empty[s1]);
          if (j + 2 == cur.nkv_b()) commit(&q_empty[1]);     // the item's last S_B
        } else {
          commit(&o_done[1]);
          if (nxt.valid) {                                  // the next item's S_B(0)
            if (!wait(&q_full[1], qph)) break;
            issue_s(1, ring_n % kStagesKV);
            commit(&k_empty[ring_n % kStagesKV]);
          }
        }
      }
      ++n_q;
      ring = ring_n;
      cur = nxt;
    }
    if (!ok && lane == 0) fail_timeout();
    // drain: all MMAs we issued are complete before TMEM may be freed
    commit(drain);
    __all_sync(0xffffffffu, mbar_wait(drain, 0));
  } else {
    // ------------------------------------------------------------ softmax
    const int t = warp >> 2;              // 0: tile A, 1: tile B
    const int r = tid & 127;              // row of the tile (TMEM lane)
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t s_tm = tmem + lane_base + t * 128;
    const uint32_t o_tm = tmem + lane_base + 256 + t * 128;
    const float sl2 = p.scale_log2;
    bool ok = true;
    int n_s = 0, n_it = 0;                // S tiles and items of this tile slot so far
    int k_next = 0;
    // the next non-empty item of this CTA (looked up an item ahead, so its
    // loads of the sequence bounds stay off the path between items)
    auto next_item = [&]() -> PItem {
      for (;; ++k_next) {
        const int pos = item_pos(k_next, cta, n_cta);
        if (pos >= p.n_items) {
          PItem none;
          none.valid = false;
          return none;
        }
        const PItem x = item_at(pos, p);
        if (x.valid) {
          ++k_next;
          return x;
        }
      }
    };
    PItem it_next = next_item();
    while (ok && it_next.valid) {
    const PItem it = it_next;
    it_next = next_item();
    const int nkv = t == 0 ? it.nkv_a() : it.nkv_b();
    float m_ref = -INFINITY;              // exponent reference (lazy)
    float m_max = -INFINITY;              // true running maximum (log2 units)
    float l_run = 0.f;
    for (int j = 0; j < nkv; ++j, ++n_s) {
      if (!__all_sync(0xffffffffu, mbar_wait(&s_full[t], n_s & 1))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const bool diag = j == nkv - 1;     // key column c visible iff c <= r
      uint32_t sr[kBN];
      float mx4[kBN / 32];
#pragma unroll
      for (int c = 0; c < kBN / 32; ++c)
        mx4[c] = tmem_ld32_max(s_tm + c * 32, *reinterpret_cast<uint32_t(*)[32]>(sr + c * 32));
      tmem_wait_ld();
      // the row maximum: off the diagonal it comes with the loads; on the
      // diagonal tile only keys c <= r count
      float mt = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
      if (diag) {
        float mx8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx8[i] = -INFINITY;
#pragma unroll
        for (int c = 0; c < kBN; ++c)
          mx8[c & 7] = c > r ? mx8[c & 7] : fmaxf(mx8[c & 7], __uint_as_float(sr[c]));
        mt = fmaxf(fmax3(mx8[0], mx8[1], mx8[2]),
                   fmaxf(fmax3(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
      }
      m_max = fmaxf(m_max, mt * sl2);
      const bool need = m_max > m_ref + kRescaleThreshold;
      const float m_new = need ? m_max : m_ref;
      const float factor = ex2(m_ref - m_new);  // 1 when unchanged, 0 on the first tile
      if (__any_sync(0xffffffffu, need) && j > 0) {
        // O holds PV of tiles < j, complete: S_t(j), visible above, was
        // committed after PV_t(j-1).  Rescale it before the first half of P
        // lets PV_t(j) start.
        // (16 columns at a time: the S row is still held in registers)
#pragma unroll 1
        for (int c = 0; c < D / 16; ++c) {
          uint32_t rr[16];
          tmem_ld16(o_tm + c * 16, rr);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) rr[e] = __float_as_uint(__uint_as_float(rr[e]) * factor);
          tmem_st16(o_tm + c * 16, rr);
        }
      }
      // P = exp2(s * scale_log2 - m_new) as bf16 over the first half of the S
      // columns, 64 keys -> 32 packed columns at a time; each half is
      // announced as soon as it is in TMEM (one arrival per warp), so PV_t(j)
      // on keys 0..63 overlaps the exponentials of keys 64..127.  The scaling
      // and the row sum run on fp32 pairs.
      const uint64_t sc2 = f2_pack(sl2, sl2);
      const uint64_t nm2 = f2_pack(-m_new, -m_new);
      uint64_t acc2[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) acc2[i] = f2_pack(0.f, 0.f);
#pragma unroll
      for (int c = 0; c < kBN / 64; ++c) {
        uint32_t pk[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int k0 = c * 64 + 2 * e;
          float t0, t1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[k0]), __uint_as_float(sr[k0 + 1])), sc2, nm2),
                    t0, t1);
          float p0 = ex2(t0);
          float p1 = ex2(t1);
          if (diag) {
            p0 = k0 <= r ? p0 : 0.f;
            p1 = k0 + 1 <= r ? p1 : 0.f;
          }
          acc2[e & 3] = f2_add(acc2[e & 3], f2_pack(p0, p1));
          pk[e] = pack_bf16x2(p0, p1);
        }
        tmem_st32(s_tm + c * 32, pk);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(c == 0 ? &p_half[t] : &p_full[t]);
      }
      float rs0, rs1;
      f2_unpack(f2_add(f2_add(acc2[0], acc2[1]), f2_add(acc2[2], acc2[3])), rs0, rs1);
      l_run = l_run * factor + (rs0 + rs1);
      m_ref = m_new;
    }
    if (!ok) break;
    // epilogue of the item: O / l, m, l (tcgen05.ld is warp-collective:
    // decide per warp).  The O reads complete (wait::ld) before this warp
    // writes the next item's first P, which is what lets that item's first PV
    // overwrite O.
    const bool o_ready = __all_sync(0xffffffffu, !*abort_flag && mbar_wait(&o_done[t], n_it & 1));
    ++n_it;
    if (!o_ready) {
      ok = false;
      break;
    }
    tc_fence_after();
    {
      const int qi = it.pr * 2 * kBM + t * kBM + r;
      const bool row_ok = qi < it.n;
      const float inv_l = 1.0f / l_run;
      uint32_t rr[D];
#pragma unroll
      for (int c = 0; c < D / 32; ++c)
        tmem_ld32(o_tm + c * 32, *reinterpret_cast<uint32_t(*)[32]>(rr + c * 32));
      tmem_wait_ld();
      if (row_ok) {
        uint4* dst = reinterpret_cast<uint4*>(
            p.o + (static_cast<int64_t>(it.seq0 + qi) * p.h_q + it.g) * D);
#pragma unroll
        for (int v = 0; v < D / 8; ++v) {
          uint4 w;
          w.x = pack_bf16x2(__uint_as_float(rr[8 * v + 0]) * inv_l, __uint_as_float(rr[8 * v + 1]) * inv_l);
          w.y = pack_bf16x2(__uint_as_float(rr[8 * v + 2]) * inv_l, __uint_as_float(rr[8 * v + 3]) * inv_l);
          w.z = pack_bf16x2(__uint_as_float(rr[8 * v + 4]) * inv_l, __uint_as_float(rr[8 * v + 5]) * inv_l);
          w.w = pack_bf16x2(__uint_as_float(rr[8 * v + 6]) * inv_l, __uint_as_float(rr[8 * v + 7]) * inv_l);
          dst[v] = w;
        }
        // m, l [layer][h_q][total]; seq0 = layer * total + first token
        const int layer = it.seq0 / p.total;
        const int64_t at = (static_cast<int64_t>(layer) * p.h_q + it.g) * p.total +
                           (it.seq0 - layer * p.total) + qi;
        p.m[at] = m_max * kLn2;
        p.l[at] = l_run * ex2(m_ref - m_max);
      }
    }
    }  // items
    if (!ok) fail_timeout();
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
  // persistent: one CTA per SM (fewer if there are fewer items)
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (sms <= 0) sms = 1;
  const int grid = prm.n_items < sms ? prm.n_items : sms;
  // a programmatic dependent launch: the kernel waits for the previous grid on
  // the stream before it reads or writes global memory
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kPrefillThreads);
  cfg.dynamicSmemBytes = PrefillSmem<D>::kBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  KVS_CUDA(cudaLaunchKernelEx(&cfg, prefill_attn_kernel<D>, mp.qm, mp.km, mp.vm, prm),
           "kvs_prefill_attn_lse (launch)");
  return KVS_OK;
}

}  // namespace
}  // namespace kvs

namespace kvs {
namespace {

kvs_status prefill_attn(const char* fn, const kvs_bf16* q, const kvs_bf16* k, const kvs_bf16* v,
                        kvs_bf16* o, float* m, float* l, const int32_t* cu_seqlens, int32_t batch,
                        int32_t max_n, int32_t total_tokens, int32_t h_q, int32_t h_kv, int32_t d,
                        float scale, int32_t n_layers, int32_t* status, kvs_stream stream) {
  KVS_REQUIRE(batch >= 0 && n_layers >= 0, "%s: negative batch or layer count", fn);
  if (batch == 0 || total_tokens == 0 || n_layers == 0) return KVS_OK;
  KVS_REQUIRE(q && k && v && o && m && l && cu_seqlens, "%s: NULL pointer", fn);
  KVS_SUPPORTED(d == 64 || d == 128, "%s: d = %d (supported: 64, 128)", fn, d);
  KVS_REQUIRE(h_kv > 0 && h_q > 0 && h_q % h_kv == 0, "%s: bad head counts", fn);
  KVS_REQUIRE(max_n >= 1 && total_tokens >= 1 && batch <= 65535, "%s: bad sizes", fn);
  KVS_REQUIRE(static_cast<int64_t>(total_tokens) * n_layers < (1ll << 31),
              "%s: layers x tokens exceed 32-bit TMA row coordinates", fn);
  KVS_REQUIRE(((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o)) & 15) == 0,
              "%s: q, k, v, o must be 16-byte aligned", fn);
  PrefillParams prm;
  prm.o = o;
  prm.m = m;
  prm.l = l;
  prm.cu_seqlens = cu_seqlens;
  prm.status = status;
  prm.total = total_tokens;
  prm.h_q = h_q;
  prm.h_kv = h_kv;
  prm.group = h_q / h_kv;
  prm.n_pairs_max = (max_n + 2 * kBM - 1) / (2 * kBM);
  prm.batch = batch;
  prm.n_layers = n_layers;
  prm.scale_log2 = scale * kLog2eP;
  KVS_REQUIRE(static_cast<int64_t>(prm.n_pairs_max) * batch * h_q * n_layers < (1ll << 31),
              "%s: too many work items", fn);
  prm.n_items = prm.n_pairs_max * batch * h_q * n_layers;

  // the maps cover every layer of the call: rows = layers x tokens
  const int rows = total_tokens * n_layers;
  static thread_local PrefillMaps cache;
  if (cache.q != q || cache.k != k || cache.v != v || cache.total != rows ||
      cache.h_q != h_q || cache.h_kv != h_kv || cache.d != d) {
    if (!map_rows(&cache.qm, q, rows, h_q, d) || !map_rows(&cache.km, k, rows, h_kv, d) ||
        !map_rows(&cache.vm, v, rows, h_kv, d)) {
      cache.q = nullptr;
      return KVS_ERR_CUDA;
    }
    cache.q = q;
    cache.k = k;
    cache.v = v;
    cache.total = rows;
    cache.h_q = h_q;
    cache.h_kv = h_kv;
    cache.d = d;
  }
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (d == 128) return launch_prefill<128>(cache, prm, batch, st);
  return launch_prefill<64>(cache, prm, batch, st);
}

}  // namespace
}  // namespace kvs

extern "C" kvs_status kvs_prefill_attn_lse(const kvs_bf16* q, const kvs_bf16* k,
                                           const kvs_bf16* v, kvs_bf16* o, float* m, float* l,
                                           const int32_t* cu_seqlens, int32_t batch,
                                           int32_t max_n, int32_t total_tokens, int32_t h_q,
                                           int32_t h_kv, int32_t d, float scale,
                                           int32_t* status, kvs_stream stream) {
  return kvs::prefill_attn("kvs_prefill_attn_lse", q, k, v, o, m, l, cu_seqlens, batch, max_n,
                           total_tokens, h_q, h_kv, d, scale, 1, status, stream);
}

extern "C" kvs_status kvs_prefill_attn_lse_layers(const kvs_bf16* q, const kvs_bf16* k,
                                                  const kvs_bf16* v, kvs_bf16* o, float* m,
                                                  float* l, const int32_t* cu_seqlens,
                                                  int32_t batch, int32_t max_n,
                                                  int32_t total_tokens, int32_t h_q, int32_t h_kv,
                                                  int32_t d, float scale, int32_t n_layers,
                                                  int32_t* status, kvs_stream stream) {
  return kvs::prefill_attn("kvs_prefill_attn_lse_layers", q, k, v, o, m, l, cu_seqlens, batch,
                           max_n, total_tokens, h_q, h_kv, d, scale, n_layers, status, stream);
}
