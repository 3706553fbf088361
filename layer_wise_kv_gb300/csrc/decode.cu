// Paged decode attention, split-K over 16-token blocks, with the step's k/v
// appended in the same pass.
//
// Source: Ultralytics glossary "PagedAttention", section "How paging works"
// (the attention kernel follows the request's block table and gathers keys
// and values block by block; storage need not be contiguous); Novita article
// "How KV Sparsity achieves 1.5x acceleration for vLLM", section "Key
// techniques 2" (PagedAttention serves the decode side of the sparsified
// cache).
//
// Design (HBM-bound: ~4 flop per byte of K/V):
// * A unit is (item, KV head, split of 256 tokens = 16 blocks).  Persistent
//   CTAs walk units round-robin; each CTA has one producer warp and eight
//   consumer warps.  Per-CTA unit lists come from a prefix sum over the
//   items' split counts, computed from `lens` in shared memory, so the launch
//   needs no host knowledge of the lengths.
// * The producer streams each block's K and V rows for the head (16 x d bf16
//   each, contiguous in the pool) into a 16-stage shared-memory ring with 2-D
//   TMA loads (128-byte swizzle), mbarrier-tracked.
// * Consumer warp w takes blocks w, w+8 of the unit.  The G query rows of the
//   KV head form the M=16 side of mma.sync m16n8k16 (bf16 in, fp32 out): S =
//   q K^T (K fragments by ldmatrix), online softmax in registers (log2
//   domain), O += P V (V fragments by ldmatrix.trans).  The tensor pipe only
//   takes the instruction count off the issue slots; the bound is HBM.
// * Warps merge through shared memory at the end of a unit; an item with one
//   split writes `out` directly, otherwise the unit writes an unnormalised
//   partial (m, l, o) to the workspace and the last unit of (item, head) to
//   finish (an atomic counter, no waiting) merges all partials and resets the
//   counter.
#include <cuda_runtime.h>

#include "host_common.h"
#include "ptx.cuh"
#include "tma_host.h"

namespace kvs {
namespace {

constexpr int kConsumers = 8;
constexpr int kDecThreads = (kConsumers + 1) * 32;
constexpr int kStages = 16;
constexpr int kSplitBlocks = 16;
constexpr int kSplitTokens = kSplitBlocks * KVS_BLOCK_TOKENS;
constexpr int kMaxG = 16;
constexpr float kLog2e = 1.4426950408889634f;

struct DecodeParams {
  const uint16_t* q;
  const uint16_t* k_new;
  const uint16_t* v_new;
  uint16_t* k_pool;
  uint16_t* v_pool;
  int32_t* tables;
  const int32_t* patch;
  const int32_t* lens;
  int32_t* lens_next;
  uint16_t* out;
  float* ws_part;
  int32_t* ws_count;
  int32_t* status;
  int batch, max_blocks, num_blocks, h_q, h_kv, group, s_max, append;
  float scale_log2;
};

template <int D>
struct DecodeSmem {
  static constexpr int kBoxBytes = KVS_BLOCK_TOKENS * 128;         // 16 rows x 64 bf16
  static constexpr int kBlockBytes = KVS_BLOCK_TOKENS * D * 2;     // one head's K (or V) block
  static constexpr int kStageBytes = 2 * kBlockBytes;
  static constexpr int kRing = kStages * kStageBytes;
  static constexpr int kScratchFloats = kConsumers * kMaxG * (D + 2);
  // ring | full[kStages] | empty[kStages] | scratch | flags | prefix[batch+1]
  static constexpr int kBarOff = kRing;
  static constexpr int kScratchOff = kBarOff + 2 * kStages * 8;
  static constexpr int kFlagOff = kScratchOff + kScratchFloats * 4;
  static constexpr int kPrefixOff = kFlagOff + 16;
  static size_t bytes(int batch) { return 1024 + kPrefixOff + 4 * (batch + 1); }
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// byte offset of 16-byte chunk `c` (0 .. D/8-1) of row `r` in a block stored
// as D/64 boxes of 16 rows x 128 B with the 128-byte swizzle
__device__ __forceinline__ uint32_t sw_off(int r, int c) {
  return static_cast<uint32_t>((c >> 3) * (KVS_BLOCK_TOKENS * 128) + r * 128 +
                               (((c & 7) ^ (r & 7)) << 4));
}

struct Unit {
  int item, h, split, ns, nblk, len, lens0;
};

__device__ __forceinline__ Unit decode_unit(int u, const int* prefix, int batch, int h_kv,
                                            int append) {
  int lo = 0, hi = batch - 1;  // last item with prefix[item] <= u
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= u) lo = mid; else hi = mid - 1;
  }
  Unit x;
  x.item = lo;
  const int units = prefix[lo + 1] - prefix[lo];
  x.ns = units / h_kv;
  const int local = u - prefix[lo];
  x.h = local / x.ns;
  x.split = local - x.h * x.ns;
  return x;
}

template <int D>
__global__ void __launch_bounds__(kDecThreads, 1)
paged_decode_kernel(const __grid_constant__ CUtensorMap k_map,
                    const __grid_constant__ CUtensorMap v_map, const DecodeParams p) {
  using L = DecodeSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* empty = full + kStages;
  float* scratch = reinterpret_cast<float*>(smem + L::kScratchOff);
  volatile int* flags = reinterpret_cast<volatile int*>(smem + L::kFlagOff);  // [0] abort, [1] last
  int* prefix = reinterpret_cast<int*>(smem + L::kPrefixOff);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.group;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    flags[0] = 0;
    flags[1] = 0;
    fence_mbar_init();
  }
  // prefix over items of (splits x heads); one warp, each lane a contiguous range
  if (warp == 0) {
    const int per = (p.batch + 31) / 32;
    const int b0 = lane * per;
    const int b1 = min(p.batch, b0 + per);
    int sum = 0;
    for (int b = b0; b < b1; ++b) {
      const int len = p.lens[b] + p.append;
      const int ns = len > 0 ? (len + kSplitTokens - 1) / kSplitTokens : 0;
      sum += ns * p.h_kv;
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    int run = incl - sum;
    for (int b = b0; b < b1; ++b) {
      prefix[b] = run;
      const int len = p.lens[b] + p.append;
      const int ns = len > 0 ? (len + kSplitTokens - 1) / kSplitTokens : 0;
      run += ns * p.h_kv;
    }
    if (lane == 31) prefix[p.batch] = incl;
  }
  __syncthreads();
  const int total_units = prefix[p.batch];

  if (warp == kConsumers) {
    // ------------------------------------------------------------ producer
    int g = 0;
    for (int u = blockIdx.x; u < total_units; u += gridDim.x) {
      if (flags[0]) break;
      Unit x = decode_unit(u, prefix, p.batch, p.h_kv, p.append);
      const int lens0 = p.lens[x.item];
      const int len = lens0 + p.append;
      const int tok0 = x.split * kSplitTokens;
      const int nblk = min(kSplitBlocks, (len - tok0 + KVS_BLOCK_TOKENS - 1) / KVS_BLOCK_TOKENS);
      // every lane fetches one table entry of the unit
      int phys = 0;
      if (lane < nblk) {
        const int lb = x.split * kSplitBlocks + lane;
        int patch = -1;
        if (p.append && p.patch != nullptr && lb == lens0 / KVS_BLOCK_TOKENS) patch = p.patch[x.item];
        phys = patch >= 0 ? patch : p.tables[static_cast<int64_t>(x.item) * p.max_blocks + lb];
        if (phys < 0 || phys >= p.num_blocks || lb >= p.max_blocks) {
          flag_status(p.status, KVS_ERR_INVALID);
          phys = 0;
        }
      }
      for (int j = 0; j < nblk; ++j) {
        const int pb = __shfl_sync(0xffffffffu, phys, j);
        const int s = g % kStages;
        const uint32_t ph = (g / kStages) & 1;
        bool ok = true;
        if (lane == 0) {
          ok = mbar_wait(&empty[s], ph ^ 1);
          if (!ok) {
            flag_status(p.status, KVS_ERR_DEVICE_TIMEOUT);
            flags[0] = 1;
          } else {
            mbar_arrive_expect_tx(&full[s], L::kStageBytes);
            uint8_t* st = smem + s * L::kStageBytes;
            const int row = (pb * p.h_kv + x.h) * KVS_BLOCK_TOKENS;
#pragma unroll
            for (int b = 0; b < D / 64; ++b) {
              tma_load_2d(st + b * L::kBoxBytes, &k_map, &full[s], b * 64, row);
              tma_load_2d(st + L::kBlockBytes + b * L::kBoxBytes, &v_map, &full[s], b * 64, row);
            }
          }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        ++g;
      }
    }
    // make sure no load of ours is still landing in shared memory when we leave
    if (lane == 0) {
      const int first = g > kStages ? g - kStages : 0;
      for (int gg = first; gg < g; ++gg)
        if (!mbar_wait(&full[gg % kStages], (gg / kStages) & 1)) break;
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int ra = lane >> 2;   // rows (query heads of the group) ra and ra + 8
  const int rb = ra + 8;
  const int cq = (lane & 3) * 2;
  const uint32_t ring = smem_u32(smem);
  int g_base = 0;
  for (int u = blockIdx.x; u < total_units; u += gridDim.x) {
    Unit x = decode_unit(u, prefix, p.batch, p.h_kv, p.append);
    const int lens0 = p.lens[x.item];
    const int len = lens0 + p.append;
    const int tok_split = x.split * kSplitTokens;
    const int nblk = min(kSplitBlocks, (len - tok_split + KVS_BLOCK_TOKENS - 1) / KVS_BLOCK_TOKENS);

    // q fragments of the group's query rows (rows >= G are zero)
    uint32_t qa[D / 16][4];
    {
      const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
          p.q + (static_cast<int64_t>(x.item) * p.h_q + x.h * G) * D);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const int c0 = (ks * 16 + cq) >> 1;
        qa[ks][0] = ra < G ? __ldg(qrow + ra * (D / 2) + c0) : 0u;
        qa[ks][1] = rb < G ? __ldg(qrow + rb * (D / 2) + c0) : 0u;
        qa[ks][2] = ra < G ? __ldg(qrow + ra * (D / 2) + c0 + 4) : 0u;
        qa[ks][3] = rb < G ? __ldg(qrow + rb * (D / 2) + c0 + 4) : 0u;
      }
    }
    float o[D / 8][4];
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
    float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;

    for (int j = warp; j < nblk; j += kConsumers) {
      const int g = g_base + j;
      const int s = g % kStages;
      const uint32_t ph = (g / kStages) & 1;
      if (!flags[0]) {
        bool ok = true;
        if (lane == 0) {
          ok = mbar_wait(&full[s], ph);
          if (!ok) {
            flag_status(p.status, KVS_ERR_DEVICE_TIMEOUT);
            flags[0] = 1;
          }
        }
        __syncwarp();
      }
      const bool aborted = flags[0] != 0;
      const uint32_t kst = ring + s * L::kStageBytes;
      const uint32_t vst = kst + L::kBlockBytes;
      const int tok0 = tok_split + j * KVS_BLOCK_TOKENS;

      // the block holding the appended token: put the new row into the stage
      // and into the pool
      if (p.append && !aborted && lens0 >= tok0 && lens0 < tok0 + KVS_BLOCK_TOKENS) {
        const int slot = lens0 - tok0;
        const int lb = lens0 / KVS_BLOCK_TOKENS;
        int pb = (p.patch != nullptr && p.patch[x.item] >= 0)
                     ? p.patch[x.item]
                     : p.tables[static_cast<int64_t>(x.item) * p.max_blocks + lb];
        const bool pb_ok = pb >= 0 && pb < p.num_blocks;
        const int per = D / 8;  // 16-byte chunks per row
        if (lane < 2 * per) {
          const bool is_v = lane >= per;
          const int c = is_v ? lane - per : lane;
          const uint4* src = reinterpret_cast<const uint4*>(
              (is_v ? p.v_new : p.k_new) + (static_cast<int64_t>(x.item) * p.h_kv + x.h) * D);
          const uint4 val = __ldg(src + c);
          uint8_t* st = smem + s * L::kStageBytes + (is_v ? L::kBlockBytes : 0);
          *reinterpret_cast<uint4*>(st + sw_off(slot, c)) = val;
          if (pb_ok) {
            uint4* dst = reinterpret_cast<uint4*>(
                (is_v ? p.v_pool : p.k_pool) +
                ((static_cast<int64_t>(pb) * p.h_kv + x.h) * KVS_BLOCK_TOKENS + slot) * D);
            dst[c] = val;
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
      }

      // S = q K^T for the 16 tokens of the block
      float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      {
        const int mi = lane >> 3, rr = lane & 7;
        const int tok = (mi >> 1) * 8 + rr;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kst + sw_off(tok, ks * 2 + (mi & 1)), b0, b1, b2, b3);
          mma16816(sc[0], qa[ks], b0, b1);
          mma16816(sc[1], qa[ks], b2, b3);
        }
      }
      // online softmax (log2 domain); rows ra, rb; columns cq, cq+1, 8+cq, 9+cq
      float mx_a = -INFINITY, mx_b = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int t = tok0 + nt * 8 + cq + e;
          const bool valid = t < len;
          sc[nt][e] = valid ? sc[nt][e] * p.scale_log2 : -INFINITY;
          sc[nt][2 + e] = valid ? sc[nt][2 + e] * p.scale_log2 : -INFINITY;
          mx_a = fmaxf(mx_a, sc[nt][e]);
          mx_b = fmaxf(mx_b, sc[nt][2 + e]);
        }
      }
      mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 1));
      mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 2));
      mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 1));
      mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 2));
      const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
      const float al_a = ex2(m_a - mn_a), al_b = ex2(m_b - mn_b);
      m_a = mn_a;
      m_b = mn_b;
      float ps_a = 0.f, ps_b = 0.f;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          sc[nt][e] = ex2(sc[nt][e] - mn_a);
          sc[nt][2 + e] = ex2(sc[nt][2 + e] - mn_b);
          ps_a += sc[nt][e];
          ps_b += sc[nt][2 + e];
        }
      }
      l_a = l_a * al_a + ps_a;
      l_b = l_b * al_b + ps_b;
#pragma unroll
      for (int nt = 0; nt < D / 8; ++nt) {
        o[nt][0] *= al_a;
        o[nt][1] *= al_a;
        o[nt][2] *= al_b;
        o[nt][3] *= al_b;
      }
      uint32_t pa[4];
      pa[0] = pack_bf16x2(sc[0][0], sc[0][1]);
      pa[1] = pack_bf16x2(sc[0][2], sc[0][3]);
      pa[2] = pack_bf16x2(sc[1][0], sc[1][1]);
      pa[3] = pack_bf16x2(sc[1][2], sc[1][3]);
      // O += P V
      {
        const int mi = lane >> 3, rr = lane & 7;
        const int tok = (mi & 1) * 8 + rr;
#pragma unroll
        for (int np = 0; np < D / 16; ++np) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vst + sw_off(tok, np * 2 + (mi >> 1)), b0, b1, b2, b3);
          mma16816(o[2 * np], pa, b0, b1);
          mma16816(o[2 * np + 1], pa, b2, b3);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    g_base += nblk;

    // ---- merge the consumer warps of this unit ----
    l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
    l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
    float* wsc = scratch + warp * kMaxG * (D + 2);
    if (ra < G) {
#pragma unroll
      for (int nt = 0; nt < D / 8; ++nt) {
        wsc[ra * (D + 2) + nt * 8 + cq] = o[nt][0];
        wsc[ra * (D + 2) + nt * 8 + cq + 1] = o[nt][1];
      }
      if ((lane & 3) == 0) {
        wsc[ra * (D + 2) + D] = m_a;
        wsc[ra * (D + 2) + D + 1] = l_a;
      }
    }
    if (rb < G) {
#pragma unroll
      for (int nt = 0; nt < D / 8; ++nt) {
        wsc[rb * (D + 2) + nt * 8 + cq] = o[nt][2];
        wsc[rb * (D + 2) + nt * 8 + cq + 1] = o[nt][3];
      }
      if ((lane & 3) == 0) {
        wsc[rb * (D + 2) + D] = m_b;
        wsc[rb * (D + 2) + D + 1] = l_b;
      }
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumers * 32) : "memory");

    const int out_row0 = x.item * p.h_q + x.h * G;
    const int64_t part_slot = (static_cast<int64_t>(x.item) * p.h_kv + x.h) * p.s_max + x.split;
    float* part = p.ws_part + part_slot * G * (D + 2);
    for (int e = threadIdx.x; e < G * D; e += kConsumers * 32) {
      const int r = e / D, c = e - r * D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kConsumers; ++w)
        M = fmaxf(M, scratch[w * kMaxG * (D + 2) + r * (D + 2) + D]);
      float Lsum = 0.f, O = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumers; ++w) {
        const float* ws = scratch + w * kMaxG * (D + 2) + r * (D + 2);
        const float f = ex2(ws[D] - M);
        Lsum += ws[D + 1] * f;
        O += ws[c] * f;
      }
      if (x.ns == 1) {
        const float val = O / Lsum;
        const uint32_t b = pack_bf16x2(val, 0.f);
        p.out[static_cast<int64_t>(out_row0 + r) * D + c] = static_cast<uint16_t>(b & 0xFFFFu);
      } else {
        part[r * D + c] = O;
        if (c == 0) {
          part[G * D + r] = M;
          part[G * D + G + r] = Lsum;
        }
      }
    }
    if (x.ns > 1) {
      __threadfence();
      asm volatile("bar.sync 1, %0;" ::"n"(kConsumers * 32) : "memory");
      if (threadIdx.x == 0) {
        const int old = atomicAdd(p.ws_count + x.item * p.h_kv + x.h, 1);
        flags[1] = (old == x.ns - 1) ? 1 : 0;
      }
      asm volatile("bar.sync 1, %0;" ::"n"(kConsumers * 32) : "memory");
      if (flags[1]) {
        __threadfence();
        const float* base = p.ws_part + (static_cast<int64_t>(x.item) * p.h_kv + x.h) * p.s_max *
                                            G * (D + 2);
        for (int e = threadIdx.x; e < G * D; e += kConsumers * 32) {
          const int r = e / D, c = e - r * D;
          float M = -INFINITY;
          for (int sp = 0; sp < x.ns; ++sp)
            M = fmaxf(M, __ldcg(base + static_cast<int64_t>(sp) * G * (D + 2) + G * D + r));
          float Lsum = 0.f, O = 0.f;
          for (int sp = 0; sp < x.ns; ++sp) {
            const float* pr = base + static_cast<int64_t>(sp) * G * (D + 2);
            const float f = ex2(__ldcg(pr + G * D + r) - M);
            Lsum += __ldcg(pr + G * D + G + r) * f;
            O += __ldcg(pr + r * D + c) * f;
          }
          const uint32_t b = pack_bf16x2(O / Lsum, 0.f);
          p.out[static_cast<int64_t>(out_row0 + r) * D + c] = static_cast<uint16_t>(b & 0xFFFFu);
        }
        if (threadIdx.x == 0) p.ws_count[x.item * p.h_kv + x.h] = 0;
      }
    }
    // table patch and length bookkeeping, once per item
    if (threadIdx.x == 0 && x.split == 0 && x.h == 0) {
      if (p.append && p.patch != nullptr && p.patch[x.item] >= 0)
        p.tables[static_cast<int64_t>(x.item) * p.max_blocks + lens0 / KVS_BLOCK_TOKENS] =
            p.patch[x.item];
      if (p.lens_next != nullptr) p.lens_next[x.item] = len;
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumers * 32) : "memory");
  }
}

struct MapCache {
  const void* base = nullptr;
  int num_blocks = 0, h_kv = 0, d = 0;
  CUtensorMap map;
};

bool pool_map(MapCache& c, const void* pool, int num_blocks, int h_kv, int d) {
  if (c.base == pool && c.num_blocks == num_blocks && c.h_kv == h_kv && c.d == d) return true;
  const uint64_t dims[2] = {static_cast<uint64_t>(d),
                            static_cast<uint64_t>(num_blocks) * h_kv * KVS_BLOCK_TOKENS};
  const uint64_t strides[1] = {static_cast<uint64_t>(d) * 2};
  const uint32_t box[2] = {64, KVS_BLOCK_TOKENS};
  if (!make_bf16_map(&c.map, pool, 2, dims, strides, box)) {
    c.base = nullptr;
    return false;
  }
  c.base = pool;
  c.num_blocks = num_blocks;
  c.h_kv = h_kv;
  c.d = d;
  return true;
}

int s_max_for(int max_len) { return (max_len + kSplitTokens - 1) / kSplitTokens; }

int sm_count_dec() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

template <int D>
kvs_status launch_decode(const DecodeParams& prm, const CUtensorMap& km, const CUtensorMap& vm,
                         int grid, cudaStream_t stream) {
  const size_t smem = DecodeSmem<D>::bytes(prm.batch);
  static bool configured = false;
  if (!configured) {
    KVS_CUDA(cudaFuncSetAttribute(paged_decode_kernel<D>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, 232448),
             "kvs_paged_decode: raising the shared-memory limit");
    configured = true;
  }
  paged_decode_kernel<D><<<grid, kDecThreads, smem, stream>>>(km, vm, prm);
  KVS_CHECK_LAUNCH("kvs_paged_decode");
  return KVS_OK;
}

}  // namespace
}  // namespace kvs

extern "C" {

size_t kvs_paged_decode_workspace_size(int32_t batch, int32_t h_q, int32_t h_kv, int32_t d,
                                       int32_t max_len) {
  if (batch <= 0 || h_kv <= 0 || h_q <= 0 || d <= 0 || max_len <= 0) return 0;
  const int64_t G = h_q / h_kv;
  const int64_t counters = static_cast<int64_t>(batch) * h_kv;
  const int64_t counter_bytes = (counters * 4 + 255) / 256 * 256;
  const int64_t parts = counters * kvs::s_max_for(max_len) * G * (d + 2);
  return static_cast<size_t>(counter_bytes + parts * 4);
}

kvs_status kvs_paged_decode(const kvs_bf16* q, const kvs_bf16* k_new, const kvs_bf16* v_new,
                            kvs_bf16* k_pool, kvs_bf16* v_pool, int32_t num_blocks,
                            int32_t* block_tables, int32_t max_blocks, const int32_t* table_patch,
                            const int32_t* lens, int32_t* lens_next, int32_t batch,
                            int32_t max_len, int32_t h_q, int32_t h_kv, int32_t d, float scale,
                            kvs_bf16* out, void* workspace, size_t workspace_bytes,
                            int32_t* status, kvs_stream stream) {
  KVS_REQUIRE(batch >= 0, "kvs_paged_decode: negative batch");
  if (batch == 0) return KVS_OK;
  KVS_REQUIRE(q && k_pool && v_pool && block_tables && lens && out && workspace,
              "kvs_paged_decode: NULL pointer");
  KVS_REQUIRE((k_new == nullptr) == (v_new == nullptr),
              "kvs_paged_decode: k_new and v_new must both be given or both be NULL");
  KVS_SUPPORTED(d == 64 || d == 128, "kvs_paged_decode: d = %d (supported: 64, 128)", d);
  KVS_REQUIRE(h_kv > 0 && h_q > 0 && h_q % h_kv == 0, "kvs_paged_decode: bad head counts");
  KVS_SUPPORTED(h_q / h_kv <= kvs::kMaxG, "kvs_paged_decode: group size %d > %d", h_q / h_kv,
                kvs::kMaxG);
  KVS_REQUIRE(num_blocks > 0 && max_blocks > 0 && max_len > 0, "kvs_paged_decode: bad sizes");
  KVS_REQUIRE(static_cast<int64_t>(num_blocks) * h_kv * KVS_BLOCK_TOKENS < (1ll << 31),
              "kvs_paged_decode: pool too large for 32-bit TMA row coordinates");
  KVS_REQUIRE(static_cast<int64_t>(max_blocks) * KVS_BLOCK_TOKENS >= max_len,
              "kvs_paged_decode: max_len %d exceeds the table capacity", max_len);
  KVS_REQUIRE((reinterpret_cast<uintptr_t>(k_pool) & 15) == 0 &&
                  (reinterpret_cast<uintptr_t>(v_pool) & 15) == 0 &&
                  (reinterpret_cast<uintptr_t>(q) & 15) == 0,
              "kvs_paged_decode: q and pools must be 16-byte aligned");
  KVS_REQUIRE(batch <= 8192, "kvs_paged_decode: batch %d > 8192", batch);
  const size_t need = kvs_paged_decode_workspace_size(batch, h_q, h_kv, d, max_len);
  KVS_REQUIRE(workspace_bytes >= need, "kvs_paged_decode: workspace %zu bytes < %zu needed",
              workspace_bytes, need);
  static thread_local kvs::MapCache kc, vc;
  if (!kvs::pool_map(kc, k_pool, num_blocks, h_kv, d) ||
      !kvs::pool_map(vc, v_pool, num_blocks, h_kv, d))
    return KVS_ERR_CUDA;

  kvs::DecodeParams prm;
  prm.q = q;
  prm.k_new = k_new;
  prm.v_new = v_new;
  prm.k_pool = k_pool;
  prm.v_pool = v_pool;
  prm.tables = block_tables;
  prm.patch = table_patch;
  prm.lens = lens;
  prm.lens_next = lens_next;
  prm.out = out;
  const int64_t counters = static_cast<int64_t>(batch) * h_kv;
  const int64_t counter_bytes = (counters * 4 + 255) / 256 * 256;
  prm.ws_count = static_cast<int32_t*>(workspace);
  prm.ws_part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + counter_bytes);
  prm.status = status;
  prm.batch = batch;
  prm.max_blocks = max_blocks;
  prm.num_blocks = num_blocks;
  prm.h_q = h_q;
  prm.h_kv = h_kv;
  prm.group = h_q / h_kv;
  prm.s_max = kvs::s_max_for(max_len);
  prm.append = k_new != nullptr ? 1 : 0;
  prm.scale_log2 = scale * kvs::kLog2e;
  // persistent grid: one CTA per SM, never more CTAs than units
  const int64_t units_ub = counters * prm.s_max;
  const int grid = static_cast<int>(units_ub < kvs::sm_count_dec() ? units_ub : kvs::sm_count_dec());
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (d == 128) return kvs::launch_decode<128>(prm, kc.map, vc.map, grid, st);
  return kvs::launch_decode<64>(prm, kc.map, vc.map, grid, st);
}

}  // extern "C"
