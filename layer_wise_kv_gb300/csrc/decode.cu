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
// * The work is the sequence of (item, KV head) segments, each a run of
//   16-token blocks.  Persistent CTAs (one per SM; twelve warps, sixteen
//   over FP8 pools) split the concatenated block sequence into equal
//   contiguous ranges, one per warp (stream-K): every warp streams the same number of bytes, whatever the mix
//   of lengths, and a segment is cut into at most a few pieces.  Segment
//   offsets come from a prefix sum over `lens` in shared memory, so the launch
//   needs no host knowledge of the lengths.
// * A warp runs its range with no CTA-wide barrier: its own 2- or 3-stage
//   shared-memory ring (as shared memory allows), refilled by its lane 0 with 2-D TMA loads (128-byte
//   swizzle) of each block's K and V rows for the head (16 x d bf16 each,
//   contiguous in the pool) plus, with a piece's first block, a linear bulk
//   copy of the group's q rows.  Block-table entries are fetched 32 at a time,
//   one chunk ahead.
// * Per 16-token block the products run transposed on mma.sync m16n8k16
//   (bf16 in, fp32 out), with the block's tokens as the M=16 side and the G
//   query heads of the KV head as the N side (8 per n-tile): S^T = K q^T (K
//   fragments by ldmatrix), online softmax per head in registers (log2
//   domain), P^T turned into a B fragment with movmatrix, O^T += V^T P^T (V
//   fragments by ldmatrix.trans).  The tensor pipe only takes the instruction
//   count off the issue slots; the bound is HBM.
// * A segment covered by one piece writes `out` directly; otherwise each piece
//   writes an unnormalised partial (m, l, o) to its workspace slot (warp index
//   + segment index, unique).  A second, small kernel (one CTA per segment,
//   every partial load in flight at once) merges them; it is a programmatic
//   dependent launch that recomputes the split from the lengths while decode
//   drains and only then waits for decode's partials.  The decode kernel itself needs no fence,
//   atomic or wait between warps.
#include <cuda_runtime.h>

#include <mutex>

#include "fp8.cuh"
#include "host_common.h"
#include "ptx.cuh"
#include "tma_host.h"

// Built-in scratch of kvs_paged_decode_static: the split index and partials
// for callers that cannot provide a workspace.  Host code never uses the name
// as an address; it looks the device address up per device (below).
static __device__ __align__(256) unsigned char g_decode_static_scratch[KVS_DECODE_STATIC_SCRATCH_BYTES];

namespace kvs {
namespace {

#ifndef KVS_DECODE_WARPS
#define KVS_DECODE_WARPS 12
#endif
constexpr int kWarps = KVS_DECODE_WARPS;
// FP8 pools: a block is half the bytes, so 16 warps fit two stages each, and
// the kernel is latency-bound per warp (more warps, more chains in flight)
constexpr int kWarpsF8 = 16;
constexpr int kMaxWarps = kWarps > kWarpsF8 ? kWarps : kWarpsF8;
__host__ __device__ constexpr int dec_warps(bool f8) { return f8 ? kWarpsF8 : kWarps; }
constexpr int kMaxGrid = 256;
constexpr int kMaxG = 16;
constexpr int kMaxBatch = 2048;
constexpr int kMaxStages = 8;
constexpr float kLog2e = 1.4426950408889634f;
// FP8 pools: P is multiplied by each token's V scale times kPvScale before the
// f16 P.V product (keeping P' in f16's normal range down to p * |v| ~ 3e-5
// and below its overflow for |v| < 28000), and the result by 1 / kPvScale.
constexpr float kPvScale = 1024.0f;

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
  float* logits;   // optional: [batch][h_kv][G][logit_ld] fp32, log2-scaled logits
  int logit_ld;
  float* lse;      // with logits: [batch][h_q] fp32, log2 of each head's softmax denominator
  float* k_scale;  // FP8 pools: per-row scales [num_blocks][h_kv][16]
  float* v_scale;
  int32_t* status;
  uint64_t wait_ns;  // limit of every mbarrier wait
  int stall;         // test hook: issue no copies, so that every wait runs out
  int batch, max_blocks, num_blocks, h_q, h_kv, group, append, n_stages;
  int q_bytes, q_stride, q_off, bar_off, pb_off, idx_off;
  float scale_log2;
};

// A stage: one head's K block then its V block (bf16: 16 x d each, as D/64
// TMA boxes; FP8: 16 x d codes and the transposed V codes, then the 16 K and
// 16 V row scales).
template <int D, bool kF8 = false>
struct DecodeLayout {
  static constexpr int kBoxBytes = KVS_BLOCK_TOKENS * 128;       // 16 rows x 64 bf16
  static constexpr int kBlockBytes = KVS_BLOCK_TOKENS * D * (kF8 ? 1 : 2);
  static constexpr int kScaleOff = 2 * kBlockBytes;
  static constexpr int kStageBytes = 2 * kBlockBytes + (kF8 ? 2 * KVS_BLOCK_TOKENS * 4 : 0);
  static_assert(kStageBytes % 16 == 0 && kScaleOff % 16 == 0 && kBoxBytes % 1024 == 0,
                "stages, scale rows and TMA boxes keep their alignment");
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

__device__ __forceinline__ void mma16816_f16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                             uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

// byte offset of 16-byte chunk `c` (0 .. D/8-1) of row `r` in a block stored
// as D/64 boxes of 16 rows x 128 B with the 128-byte swizzle
__device__ __forceinline__ uint32_t sw_off(int r, int c) {
  return static_cast<uint32_t>((c >> 3) * (KVS_BLOCK_TOKENS * 128) + r * 128 +
                               (((c & 7) ^ (r & 7)) << 4));
}

// floats in one partial record: G rows of D accumulators, then the G maxima and
// the G sums, padded to whole float4s so that every record starts 16-byte
// aligned (the merge reads records as float4; G*(D+2) floats alone are not a
// multiple of four when G is odd)
__host__ __device__ constexpr int part_floats(int G, int D) { return (G * (D + 2) + 3) & ~3; }

// An item's length as the decode uses it: lens[i] clamped to [0, max_blocks *
// 16 - append], so that its blocks (appended token included) stay inside its
// table row and the block counts stay small enough for 32-bit prefix sums.
// Returns whether the given length was already in range.
__device__ __forceinline__ bool clamp_len(int v, int max_blocks, int append, int& out) {
  const int64_t hi = static_cast<int64_t>(max_blocks) * KVS_BLOCK_TOKENS - append;
  out = v < 0 ? 0 : (static_cast<int64_t>(v) > hi ? static_cast<int>(hi) : v);
  return out == v;
}

// owner warp of global block b when T blocks are split evenly over W warps
// (warp w owns [w*T/W, (w+1)*T/W))
__device__ __forceinline__ int owner_of(int64_t b, int64_t T, int W) {
  const int64_t w = ((b + 1) * W - 1) / T;
  return static_cast<int>(w < W - 1 ? w : W - 1);
}

struct Piece {
  bool valid;
  int item, h, seg, blk0, nblk, lens0, len, first_slot, npieces;
  int patch;    // the item's table patch (-1: none); loaded here, first used when issuing
  int64_t end;  // global block index just past the piece
};

// The piece of warp-range [pos, range_end) that starts at pos.
__device__ __forceinline__ Piece piece_at(int64_t pos, int64_t range_end, int64_t T, int W,
                                          const int* prefix, const int* lens_s,
                                          const DecodeParams& p) {
  Piece x;
  x.valid = pos < range_end;
  if (!x.valid) {
    x.item = x.h = x.seg = x.blk0 = x.nblk = x.lens0 = x.len = x.first_slot = x.npieces = 0;
    x.patch = -1;
    x.end = pos;
    return x;
  }
  int lo = 0, hi = p.batch - 1;  // last item with prefix[item] <= pos
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= pos) lo = mid; else hi = mid - 1;
  }
  x.item = lo;
  x.lens0 = lens_s[lo];
  x.len = x.lens0 + p.append;
  const int nb = (x.len + KVS_BLOCK_TOKENS - 1) / KVS_BLOCK_TOKENS;  // blocks per head
  const int local = static_cast<int>(pos - prefix[lo]);
  x.h = local / nb;
  x.blk0 = local - x.h * nb;
  x.seg = lo * p.h_kv + x.h;
  const int64_t seg_lo = prefix[lo] + static_cast<int64_t>(x.h) * nb;
  const int64_t seg_hi = seg_lo + nb;
  x.end = seg_hi < range_end ? seg_hi : range_end;
  x.nblk = static_cast<int>(x.end - pos);
  const int w_lo = owner_of(seg_lo, T, W);
  x.npieces = owner_of(seg_hi - 1, T, W) - w_lo + 1;
  x.first_slot = w_lo + x.seg;
  x.patch = (p.append && p.patch != nullptr) ? p.patch[x.item] : -1;
  return x;
}

// Table entry of block (base + lane) of the piece, as stored (-1 past its end).
// Nothing here reads the loaded value, so the load stays in flight until the
// entry is issued (a chunk or a piece later); resolve_block checks it then.
__device__ __forceinline__ int fetch_chunk(const Piece& x, int base, int lane,
                                           const DecodeParams& p) {
  const int j = base + lane;
  const int lb = x.blk0 + j;
  if (!x.valid || j >= x.nblk || lb >= p.max_blocks) return -1;
  return p.tables[static_cast<int64_t>(x.item) * p.max_blocks + lb];
}

// Physical block of block j of the piece from its table entry: the item's
// patch replaces the entry of the block that receives the appended token.
// Returns -1 (and flags the status) for an entry outside the pool.
__device__ __forceinline__ int resolve_block(const Piece& x, int j, int entry,
                                             const DecodeParams& p) {
  int pb = entry;
  if (p.append && x.patch >= 0 && x.blk0 + j == x.lens0 / KVS_BLOCK_TOKENS) pb = x.patch;
  if (pb < 0 || pb >= p.num_blocks) {
    flag_status(p.status, KVS_ERR_INVALID);
    return -1;
  }
  return pb;
}

// kF8: the pools hold FP8 codes and row scales (layout in fp8.cuh; d = 128).
// Each block's K and V codes and scales arrive by linear bulk copies; K and V
// fragments are 4-byte shared-memory loads turned into f16 pairs (exact), the
// products run on the f16 form of the same MMA, the K scales multiply the
// logits and the V scales (times kPvScale) the probabilities that enter P.V
// (the denominators use the unscaled ones).  So that K and V need
// no byte transposes, the MMA's token order inside a block is permuted: row
// rho of S^T (and k-slot rho of P^T V) is token tau(rho) = 4 (rho/2 % 4) +
// rho % 2 + 2 (rho / 8), and q's d order follows the order of the K bytes a
// thread holds.
template <int D, int NT, bool kLogits, bool kF8 = false>
__global__ void __launch_bounds__(dec_warps(kF8) * 32, 1)
paged_decode_kernel(const __grid_constant__ CUtensorMap k_map,
                    const __grid_constant__ CUtensorMap v_map, const DecodeParams p) {
  static_assert(!kF8 || D == 128, "FP8 pools: d = 128");
  using L = DecodeLayout<D, kF8>;
  constexpr int kWarps = dec_warps(kF8);
  constexpr int kDecThreads = kWarps * 32;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int NS = p.n_stages;
  const int G = p.group;
  uint8_t* my_stages = smem + warp * NS * L::kStageBytes;
  uint8_t* my_q = smem + p.q_off + warp * 2 * p.q_stride;
  uint64_t* my_full = reinterpret_cast<uint64_t*>(smem + p.bar_off) + warp * NS;
  // per stage: the physical block its copy reads (written by lane 0 when it
  // issues the copy, read by the warp after the stage's barrier completes)
  int* my_pb = reinterpret_cast<int*>(smem + p.pb_off) + warp * NS;
  int* prefix = reinterpret_cast<int*>(smem + p.idx_off);  // [batch + 1], in blocks
  int* lens_s = prefix + (p.batch + 1);

  // the merge launched after this grid may be set up now; it waits for this
  // grid's completion (and the visibility of its writes) before reading
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) {
    if constexpr (!kF8) {
      tma_prefetch_desc(&k_map);
      tma_prefetch_desc(&v_map);
    }
    for (int i = 0; i < kWarps * NS; ++i) mbar_init(reinterpret_cast<uint64_t*>(smem + p.bar_off) + i, 1);
    fence_mbar_init();
  }
  // The block tables are read right after the length prefix: start them
  // towards L2 now, one 128-byte line per thread over the grid, so that the
  // first table reads wait on L2 rather than on a second DRAM round trip.
  {
    const int64_t tbytes = static_cast<int64_t>(p.batch) * p.max_blocks * 4;
    for (int64_t off = (static_cast<int64_t>(blockIdx.x) * kDecThreads + threadIdx.x) * 128;
         off < tbytes; off += static_cast<int64_t>(gridDim.x) * kDecThreads * 128)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char*>(p.tables) + off));
  }
  for (int b = threadIdx.x; b < p.batch; b += kDecThreads)
    if (!clamp_len(p.lens[b], p.max_blocks, p.append, lens_s[b]))
      flag_status(p.status, KVS_ERR_INVALID);
  __syncthreads();
  // prefix over items of (blocks x heads); one warp, each lane a contiguous range
  if (warp == 0) {
    const int per = (p.batch + 31) / 32;
    const int b0 = lane * per;
    const int b1 = min(p.batch, b0 + per);
    int sum = 0;
    for (int b = b0; b < b1; ++b)
      sum += (lens_s[b] + p.append + KVS_BLOCK_TOKENS - 1) / KVS_BLOCK_TOKENS * p.h_kv;
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    int run = incl - sum;
    for (int b = b0; b < b1; ++b) {
      prefix[b] = run;
      run += (lens_s[b] + p.append + KVS_BLOCK_TOKENS - 1) / KVS_BLOCK_TOKENS * p.h_kv;
    }
    if (lane == 31) prefix[p.batch] = incl;
  }
  __syncthreads();
  const int64_t T = prefix[p.batch];
  // W warps take part, never more than there are blocks, so that every range
  // holds at least one block (the piece counts below rely on it)
  const int W = static_cast<int>(T < gridDim.x * kWarps ? T : gridDim.x * kWarps);
  const int w = blockIdx.x * kWarps + warp;
  if (w >= W) return;
  const int64_t r_lo = T * w / W;
  const int64_t r_hi = T * (w + 1) / W;

  Piece cur = piece_at(r_lo, r_hi, T, W, prefix, lens_s, p);
  Piece nxt = piece_at(cur.end, r_hi, T, W, prefix, lens_s, p);
  // issue-side table chunks: tb (current chunk of the issuing piece), tb_n
  // (its next chunk), tb_q (first chunk of the piece after cur)
  int tb = fetch_chunk(cur, 0, lane, p);
  int tb_n = fetch_chunk(cur, 32, lane, p);
  int tb_q = fetch_chunk(nxt, 0, lane, p);
  int tb_base = 0;

  const uint32_t stages_u32 = smem_u32(my_stages);
  int g_iss = 0, g_cons = 0;
  bool iss_next = false;  // issue pointer in nxt (else in cur)
  int iss_j = 0;          // next block of the issuing piece
  int k = 0;              // index of cur among this warp's pieces (q buffer parity)
  bool aborted = false;

  auto issue = [&](const Piece& x, int j, int entry, int qpar) {
    if (lane == 0) {
      const int s = g_iss % NS;
      // the physical block (-1: corrupt entry; the copy then reads block 0 and
      // the consumer writes nothing into the pool for it)
      const int pbr = resolve_block(x, j, entry, p);
      my_pb[s] = pbr;
      const int pb = pbr < 0 ? 0 : pbr;
      uint8_t* st = my_stages + s * L::kStageBytes;
      mbar_arrive_expect_tx(&my_full[s], L::kStageBytes + (j == 0 ? p.q_bytes : 0));
      if (p.stall) {  // test hook: the copies this stage expects never start
        ++g_iss;
        return;
      }
      const int row = (pb * p.h_kv + x.h) * KVS_BLOCK_TOKENS;
      if constexpr (kF8) {
        const int64_t off = static_cast<int64_t>(row) * D;
        bulk_load(st, reinterpret_cast<const uint8_t*>(p.k_pool) + off, L::kBlockBytes,
                  &my_full[s]);
        bulk_load(st + L::kBlockBytes, reinterpret_cast<const uint8_t*>(p.v_pool) + off,
                  L::kBlockBytes, &my_full[s]);
        bulk_load(st + L::kScaleOff, p.k_scale + row, KVS_BLOCK_TOKENS * 4, &my_full[s]);
        bulk_load(st + L::kScaleOff + KVS_BLOCK_TOKENS * 4, p.v_scale + row,
                  KVS_BLOCK_TOKENS * 4, &my_full[s]);
      } else {
#pragma unroll
        for (int b = 0; b < D / 64; ++b) {
          tma_load_2d(st + b * L::kBoxBytes, &k_map, &my_full[s], b * 64, row);
          tma_load_2d(st + L::kBlockBytes + b * L::kBoxBytes, &v_map, &my_full[s], b * 64, row);
        }
      }
      if (j == 0)
        bulk_load(my_q + qpar * p.q_stride,
                  p.q + (static_cast<int64_t>(x.item) * p.h_q + x.h * G) * D, p.q_bytes,
                  &my_full[s]);
    }
    ++g_iss;
  };
  auto top_up = [&]() {
    while (g_iss < g_cons + NS) {
      const Piece& x = iss_next ? nxt : cur;
      if (iss_j >= x.nblk) {
        if (iss_next || !nxt.valid) break;
        iss_next = true;  // move the issue pointer into the next piece
        iss_j = 0;
        tb = tb_q;
        tb_n = fetch_chunk(nxt, 32, lane, p);
        tb_base = 0;
        continue;
      }
      if (iss_j - tb_base >= 32) {
        tb = tb_n;
        tb_base += 32;
        tb_n = fetch_chunk(x, tb_base + 32, lane, p);
      }
      const int entry = __shfl_sync(0xffffffffu, tb, iss_j - tb_base);
      issue(x, iss_j, entry, (k + (iss_next ? 1 : 0)) & 1);
      ++iss_j;
    }
  };

  while (cur.valid && !aborted) {
    top_up();
    // NT n-tiles of 8 query heads; per thread: heads hc = nt*8 + 2*(lane%4) + {0,1}
    uint32_t qb[D / 16][NT][2];  // B fragments of q^T (k = d, n = head)
    float o[D / 16][NT][4];      // O^T accumulators (m = d, n = head)
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) o[mt][nt][0] = o[mt][nt][1] = o[mt][nt][2] = o[mt][nt][3] = 0.f;
    float m_h[NT][2], l_h[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      m_h[nt][0] = m_h[nt][1] = -INFINITY;
      l_h[nt][0] = l_h[nt][1] = 0.f;
    }

    for (int j = 0; j < cur.nblk; ++j) {
      const int s = g_cons % NS;
      if (!__all_sync(0xffffffffu, mbar_wait(&my_full[s], (g_cons / NS) & 1, p.wait_ns))) {
        flag_status(p.status, KVS_ERR_DEVICE_TIMEOUT);
        aborted = true;
        break;
      }
      if (j == 0) {  // the group's q rows arrived with the piece's first block
        const uint8_t* qs = my_q + (k & 1) * p.q_stride;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const int hd = nt * 8 + (lane >> 2);
            if constexpr (kF8) {
              // k-slots 2t, 2t+1 / 2t+8, 2t+9 of step ks are d = base + 0, 1 / 2, 3
              const int t = lane & 3;
              const int base = ks < 4 ? 16 * t + 4 * ks : 64 + 16 * t + 4 * (ks - 4);
              const int off = (hd * D + base) * 2;
              qb[ks][nt][0] =
                  hd < G ? bf16x2_to_f16x2(*reinterpret_cast<const uint32_t*>(qs + off)) : 0u;
              qb[ks][nt][1] =
                  hd < G ? bf16x2_to_f16x2(*reinterpret_cast<const uint32_t*>(qs + off + 4)) : 0u;
            } else {
              const int off = hd * D * 2 + (ks * 16 + (lane & 3) * 2) * 2;
              qb[ks][nt][0] = hd < G ? *reinterpret_cast<const uint32_t*>(qs + off) : 0u;
              qb[ks][nt][1] = hd < G ? *reinterpret_cast<const uint32_t*>(qs + off + 16) : 0u;
            }
          }
      }
      const uint32_t kst = stages_u32 + s * L::kStageBytes;
      const uint32_t vst = kst + L::kBlockBytes;
      const int tok0 = (cur.blk0 + j) * KVS_BLOCK_TOKENS;

      // the block holding the appended token: put the new row into the stage
      // and into the pool
      if (p.append && cur.lens0 >= tok0 && cur.lens0 < tok0 + KVS_BLOCK_TOKENS) {
        const int slot = cur.lens0 - tok0;
        const int pb = my_pb[s];  // resolved when the stage was issued
        if constexpr (kF8) {
          // quantise the new rows (lane l holds d = 4l .. 4l+3) into the stage and the pool
          const int64_t nrow = (static_cast<int64_t>(cur.item) * p.h_kv + cur.h) * D + 4 * lane;
          const uint2 kw = __ldg(reinterpret_cast<const uint2*>(p.k_new + nrow));
          const uint2 vw = __ldg(reinterpret_cast<const uint2*>(p.v_new + nrow));
          const float k0 = bf16_lo(kw.x), k1 = bf16_hi(kw.x), k2 = bf16_lo(kw.y), k3 = bf16_hi(kw.y);
          const float v0 = bf16_lo(vw.x), v1 = bf16_hi(vw.x), v2 = bf16_lo(vw.y), v3 = bf16_hi(vw.y);
          const float sk = f8_row_scale(
              warp_max(fmaxf(fmaxf(fabsf(k0), fabsf(k1)), fmaxf(fabsf(k2), fabsf(k3)))));
          const float sv = f8_row_scale(
              warp_max(fmaxf(fmaxf(fabsf(v0), fabsf(v1)), fmaxf(fabsf(v2), fabsf(v3)))));
          const uint32_t kc = f8_quant4(k0, k1, k2, k3, sk);
          const uint32_t vc = f8_quant4(v0, v1, v2, v3, sv);
          uint8_t* st = my_stages + s * L::kStageBytes;
          const int ko = f8_k_off(slot, 4 * lane);
          *reinterpret_cast<uint32_t*>(st + ko) = kc;
#pragma unroll
          for (int i = 0; i < 4; ++i)
            st[L::kBlockBytes + (4 * lane + i) * KVS_BLOCK_TOKENS + slot] =
                static_cast<uint8_t>(vc >> (8 * i));
          if (lane == 0) {
            reinterpret_cast<float*>(st + L::kScaleOff)[slot] = sk;
            reinterpret_cast<float*>(st + L::kScaleOff)[KVS_BLOCK_TOKENS + slot] = sv;
          }
          if (pb >= 0 && pb < p.num_blocks) {
            const int64_t row = (static_cast<int64_t>(pb) * p.h_kv + cur.h) * KVS_BLOCK_TOKENS;
            uint8_t* kp = reinterpret_cast<uint8_t*>(p.k_pool) + row * D;
            uint8_t* vp = reinterpret_cast<uint8_t*>(p.v_pool) + row * D;
            *reinterpret_cast<uint32_t*>(kp + ko) = kc;
#pragma unroll
            for (int i = 0; i < 4; ++i)
              vp[(4 * lane + i) * KVS_BLOCK_TOKENS + slot] = static_cast<uint8_t>(vc >> (8 * i));
            if (lane == 0) {
              p.k_scale[row + slot] = sk;
              p.v_scale[row + slot] = sv;
            }
          }
          fence_proxy_async_smem();  // before a later bulk refill of this stage
        }
        const int per = D / 8;  // 16-byte chunks per row
        if (!kF8 && lane < 2 * per) {
          const bool is_v = lane >= per;
          const int c = is_v ? lane - per : lane;
          const uint4* src = reinterpret_cast<const uint4*>(
              (is_v ? p.v_new : p.k_new) + (static_cast<int64_t>(cur.item) * p.h_kv + cur.h) * D);
          const uint4 val = __ldg(src + c);
          uint8_t* st = my_stages + s * L::kStageBytes + (is_v ? L::kBlockBytes : 0);
          *reinterpret_cast<uint4*>(st + sw_off(slot, c)) = val;
          if (pb >= 0 && pb < p.num_blocks) {
            uint4* dst = reinterpret_cast<uint4*>(
                (is_v ? p.v_pool : p.k_pool) +
                ((static_cast<int64_t>(pb) * p.h_kv + cur.h) * KVS_BLOCK_TOKENS + slot) * D);
            dst[c] = val;
          }
          fence_proxy_async_smem();  // before a later TMA refill of this stage
        }
        __syncwarp();
      }
      // the last block: slots past the length hold undefined bytes (possibly
      // NaN patterns); P is 0 there, but 0 * NaN is NaN, so zero those V rows
      if (tok0 + KVS_BLOCK_TOKENS > cur.len) {
        const int valid = cur.len - tok0;
        const int per = D / 8;
        uint8_t* vs = my_stages + s * L::kStageBytes + L::kBlockBytes;
        if constexpr (kF8) {
          // transposed V: keep the first `valid` bytes of each of the d rows
          uint32_t m[4];
#pragma unroll
          for (int w4 = 0; w4 < 4; ++w4) {
            const int nb = min(4, max(0, valid - 4 * w4));
            m[w4] = nb >= 4 ? 0xFFFFFFFFu : ((1u << (8 * nb)) - 1u);
          }
#pragma unroll
          for (int i = 0; i < D / 32; ++i) {
            uint4* r = reinterpret_cast<uint4*>(vs + ((D / 32) * lane + i) * KVS_BLOCK_TOKENS);
            uint4 x = *r;
            x.x &= m[0];
            x.y &= m[1];
            x.z &= m[2];
            x.w &= m[3];
            *r = x;
          }
        } else {
          for (int idx = lane; idx < (KVS_BLOCK_TOKENS - valid) * per; idx += 32) {
            const int r = valid + idx / per;
            *reinterpret_cast<uint4*>(vs + sw_off(r, idx % per)) = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        fence_proxy_async_smem();  // before a later TMA refill of this stage
        __syncwarp();
      }

      // S^T = K q^T: rows = tokens (lane/4, lane/4 + 8), columns = heads.
      // Two accumulator chains (even / odd k-steps) halve the dependent MMA chain.
      float sa[NT][4], sb[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) sa[nt][e] = sb[nt][e] = 0.f;
      // the block tokens of this thread's S^T rows (g = lane / 4 and g + 8)
      const int tr0 = kF8 ? (((lane >> 3) << 2) | ((lane >> 2) & 1)) : (lane >> 2);
      const int tr1 = kF8 ? tr0 + 2 : tr0 + 8;
      if constexpr (kF8) {
        // K rows tr0, tr1: this thread's 16-byte chunks t and t + 4 of each
        const int t = lane & 3, sw = (tr0 & 1) << 2;
        const uint8_t* kt = my_stages + s * L::kStageBytes;
        const uint4 c00 = *reinterpret_cast<const uint4*>(kt + tr0 * D + ((t ^ sw) << 4));
        const uint4 c01 = *reinterpret_cast<const uint4*>(kt + tr0 * D + (((t + 4) ^ sw) << 4));
        const uint4 c10 = *reinterpret_cast<const uint4*>(kt + tr1 * D + ((t ^ sw) << 4));
        const uint4 c11 = *reinterpret_cast<const uint4*>(kt + tr1 * D + (((t + 4) ^ sw) << 4));
        const uint32_t w0[8] = {c00.x, c00.y, c00.z, c00.w, c01.x, c01.y, c01.z, c01.w};
        const uint32_t w1[8] = {c10.x, c10.y, c10.z, c10.w, c11.x, c11.y, c11.z, c11.w};
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          uint32_t a[4];
          e4m3x4_to_f16x2(w0[ks], a[0], a[2]);
          e4m3x4_to_f16x2(w1[ks], a[1], a[3]);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            if (ks & 1) mma16816_f16(sb[nt], a, qb[ks][nt][0], qb[ks][nt][1]);
            else mma16816_f16(sa[nt], a, qb[ks][nt][0], qb[ks][nt][1]);
          }
        }
      } else {
        const int mi = lane >> 3, rr = lane & 7;
        const int tok = (mi & 1) * 8 + rr;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          uint32_t a[4];
          ldsm_x4(kst + sw_off(tok, ks * 2 + (mi >> 1)), a[0], a[1], a[2], a[3]);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            if (ks & 1) mma16816(sb[nt], a, qb[ks][nt][0], qb[ks][nt][1]);
            else mma16816(sa[nt], a, qb[ks][nt][0], qb[ks][nt][1]);
          }
        }
      }
      // online softmax per head (log2 domain): a head's 16 scores sit in the 8
      // lanes with the same lane % 4 (rows lane/4 and lane/4 + 8)
      const bool v0 = tok0 + tr0 < cur.len;
      const bool v1 = tok0 + tr1 < cur.len;
      float sc0 = p.scale_log2, sc1 = p.scale_log2;
      float pv0 = 1.f, pv1 = 1.f;  // FP8: the V scale of each row's token, times kPvScale
      if constexpr (kF8) {
        const float* sks = reinterpret_cast<const float*>(my_stages + s * L::kStageBytes +
                                                          L::kScaleOff);
        sc0 *= sks[tr0];
        sc1 *= sks[tr1];
        pv0 = v0 ? sks[KVS_BLOCK_TOKENS + tr0] * kPvScale : 0.f;
        pv1 = v1 ? sks[KVS_BLOCK_TOKENS + tr1] * kPvScale : 0.f;
      }
      uint32_t pb0[NT], pb1[NT];
      bool rescale = false;
      float al[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        float s0[2], s1[2], mx[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          s0[e] = v0 ? (sa[nt][e] + sb[nt][e]) * sc0 : -INFINITY;
          s1[e] = v1 ? (sa[nt][2 + e] + sb[nt][2 + e]) * sc1 : -INFINITY;
          if constexpr (kLogits) {
            // every slot's logit for the score update (head hd, slots tok0 + lane/4, +8)
            const int hd = nt * 8 + (lane & 3) * 2 + e;
            if (hd < G) {
              float* lg = p.logits +
                          ((static_cast<int64_t>(cur.item) * p.h_kv + cur.h) * G + hd) * p.logit_ld;
              const int t0 = tok0 + tr0, t1 = tok0 + tr1;
              if (v0 && t0 < p.logit_ld) lg[t0] = s0[e];
              if (v1 && t1 < p.logit_ld) lg[t1] = s1[e];
            }
          }
          mx[e] = fmaxf(s0[e], s1[e]);
          mx[e] = fmaxf(mx[e], __shfl_xor_sync(0xffffffffu, mx[e], 4));
          mx[e] = fmaxf(mx[e], __shfl_xor_sync(0xffffffffu, mx[e], 8));
          mx[e] = fmaxf(mx[e], __shfl_xor_sync(0xffffffffu, mx[e], 16));
          const float mn = fmaxf(m_h[nt][e], mx[e]);
          al[nt][e] = ex2(m_h[nt][e] - mn);
          rescale |= mn != m_h[nt][e];
          m_h[nt][e] = mn;
          s0[e] = ex2(s0[e] - mn);
          s1[e] = ex2(s1[e] - mn);
          l_h[nt][e] = l_h[nt][e] * al[nt][e] + (s0[e] + s1[e]);
        }
        // P^T (tokens x heads) -> B fragments (k = tokens, n = heads)
        if constexpr (kF8) {
          pb0[nt] = movmatrix_t(pack_f16x2(s0[0] * pv0, s0[1] * pv0));
          pb1[nt] = movmatrix_t(pack_f16x2(s1[0] * pv1, s1[1] * pv1));
        } else {
          pb0[nt] = movmatrix_t(pack_bf16x2(s0[0], s0[1]));
          pb1[nt] = movmatrix_t(pack_bf16x2(s1[0], s1[1]));
        }
      }
      if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            o[mt][nt][0] *= al[nt][0];
            o[mt][nt][1] *= al[nt][1];
            o[mt][nt][2] *= al[nt][0];
            o[mt][nt][3] *= al[nt][1];
          }
      }
      // O^T += V^T P^T: A = V^T (m = d, k = tokens) by ldmatrix.trans
      if constexpr (kF8) {
        // transposed V codes: row d, bytes 4t .. 4t+3 = tokens of k-slots 2t, 2t+1, 2t+8, 2t+9
        const int gq = lane >> 2, t = lane & 3;
        const uint8_t* vt = my_stages + s * L::kStageBytes + L::kBlockBytes;
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
          const uint32_t x0 =
              *reinterpret_cast<const uint32_t*>(vt + (mt * 16 + gq) * KVS_BLOCK_TOKENS + 4 * t);
          const uint32_t x1 = *reinterpret_cast<const uint32_t*>(
              vt + (mt * 16 + gq + 8) * KVS_BLOCK_TOKENS + 4 * t);
          uint32_t a[4];
          e4m3x4_to_f16x2(x0, a[0], a[2]);
          e4m3x4_to_f16x2(x1, a[1], a[3]);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma16816_f16(o[mt][nt], a, pb0[nt], pb1[nt]);
        }
      } else {
        const int mi = lane >> 3, rr = lane & 7;
        const int tok = (mi >> 1) * 8 + rr;
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
          uint32_t a[4];
          ldsm_x4_t(vst + sw_off(tok, mt * 2 + (mi & 1)), a[0], a[1], a[2], a[3]);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma16816(o[mt][nt], a, pb0[nt], pb1[nt]);
        }
      }
      __syncwarp();
      ++g_cons;
      top_up();
    }
    if (aborted) break;

    // ---- the piece's result ----
    // per head: l summed over the 8 lanes sharing lane % 4
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        l_h[nt][e] += __shfl_xor_sync(0xffffffffu, l_h[nt][e], 4);
        l_h[nt][e] += __shfl_xor_sync(0xffffffffu, l_h[nt][e], 8);
        l_h[nt][e] += __shfl_xor_sync(0xffffffffu, l_h[nt][e], 16);
      }
    const int64_t out_row0 = static_cast<int64_t>(cur.item) * p.h_q + cur.h * G;
    const int dr = lane >> 2;  // d offset inside an m-tile (and + 8)
    if (cur.npieces == 1) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int hd = nt * 8 + (lane & 3) * 2 + e;
          if (hd < G) {
            const float il = (kF8 ? 1.0f / kPvScale : 1.0f) / l_h[nt][e];
            if constexpr (kLogits)
              if (lane < 4) p.lse[out_row0 + hd] = m_h[nt][e] + log2f(l_h[nt][e]);
            uint16_t* orow = p.out + (out_row0 + hd) * D;
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
              orow[mt * 16 + dr] =
                  static_cast<uint16_t>(pack_bf16x2(o[mt][nt][e] * il, 0.f) & 0xFFFFu);
              orow[mt * 16 + dr + 8] =
                  static_cast<uint16_t>(pack_bf16x2(o[mt][nt][2 + e] * il, 0.f) & 0xFFFFu);
            }
          }
        }
    } else {
      const int rec = part_floats(G, D);
      float* part = p.ws_part + static_cast<int64_t>(w + cur.seg) * rec;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int hd = nt * 8 + (lane & 3) * 2 + e;
          if (hd < G) {
            const float os = kF8 ? 1.0f / kPvScale : 1.0f;
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
              part[hd * D + mt * 16 + dr] = o[mt][nt][e] * os;
              part[hd * D + mt * 16 + dr + 8] = o[mt][nt][2 + e] * os;
            }
            if (lane < 4) {
              part[G * D + hd] = m_h[nt][e];
              part[G * D + G + hd] = l_h[nt][e];
            }
          }
        }
    }
    // table patch and length bookkeeping, once per item (its head-0 segment start)
    if (lane == 0 && cur.blk0 == 0 && cur.h == 0) {
      if (p.append && cur.patch >= 0)
        p.tables[static_cast<int64_t>(cur.item) * p.max_blocks + cur.lens0 / KVS_BLOCK_TOKENS] =
            cur.patch;
      if (p.lens_next != nullptr) p.lens_next[cur.item] = cur.len;
    }

    // ---- next piece ----
    ++k;
    cur = nxt;
    if (!iss_next) {  // nothing of the new cur was issued yet (cannot happen
      iss_j = 0;      // while it is valid, kept for safety)
      tb = tb_q;
      tb_n = fetch_chunk(cur, 32, lane, p);
      tb_base = 0;
    }
    iss_next = false;
    nxt = piece_at(cur.end, r_hi, T, W, prefix, lens_s, p);
    tb_q = fetch_chunk(nxt, 0, lane, p);
  }
  // leave no load of ours landing in shared memory after we return
  if (lane == 0)
    for (int g = g_cons; g < g_iss; ++g)
      if (!mbar_wait(&my_full[g % NS], (g / NS) & 1, p.wait_ns)) break;
  __syncwarp();
}

// Merge of the pieces of every split segment: one CTA per (item, KV head).
// Pieces are combined as softmax partials: with M the largest piece maximum,
// out = sum_p exp2(m_p - M) o_p / sum_p exp2(m_p - M) l_p.  The CTA's
// kMergeGroups thread groups take every kMergeGroups-th piece; a thread owns
// four output values of one head and folds its pieces in batches of up to
// kMergeBatch, all loads of a batch in flight together, with a running maximum;
// the groups' results are then combined the same way through shared memory.
// With lse given, each head's log2(sum_p exp2(m_p - M) l_p) + M is written too.
// Launched as a programmatic dependent of the decode kernel: the grid is set
// up while decode drains and waits here until decode's writes are visible.
constexpr int kMergeGroups = 4;
constexpr int kMergeGroupThreads = 128;
constexpr int kMergeThreads = kMergeGroups * kMergeGroupThreads;
constexpr int kMergeBatch = 6;

template <int D>
__global__ void __launch_bounds__(kMergeThreads, 2)
decode_merge_kernel(const float* __restrict__ ws_part, const int32_t* __restrict__ lens, int batch,
                    int max_blocks, int append, int h_q, int h_kv, int G, int n_warps,
                    uint16_t* __restrict__ out, float* __restrict__ lse) {
  __shared__ float4 s_acc[kMergeGroups][kMergeGroupThreads];
  __shared__ float2 s_ml[kMergeGroups][kMergeGroupThreads];
  __shared__ int s_total, s_before;
  const int seg = blockIdx.x;
  const int item = seg / h_kv, h = seg - item * h_kv;
  // The decode kernel's split, recomputed from the lengths (an input of the
  // decode, read before waiting for it): T blocks over W = min(T, n_warps)
  // equal warp ranges; this segment's pieces are the ranges w_lo .. w_hi.
  {
    const int per = (batch + kMergeThreads - 1) / kMergeThreads;
    const int b0 = threadIdx.x * per, b1 = min(batch, b0 + per);
    int sum = 0, before = 0;
    for (int b = b0; b < b1; ++b) {
      int lb;
      clamp_len(lens[b], max_blocks, append, lb);  // as the decode kernel clamps it
      const int nbk = (lb + append + KVS_BLOCK_TOKENS - 1) / KVS_BLOCK_TOKENS * h_kv;
      if (b < item) before += nbk;
      sum += nbk;
    }
    if (threadIdx.x == 0) s_total = s_before = 0;
    __syncthreads();
    atomicAdd(&s_total, sum);
    atomicAdd(&s_before, before);
    __syncthreads();
  }
  const int64_t T = s_total;
  int len_item;
  clamp_len(lens[item], max_blocks, append, len_item);
  const int nb = (len_item + append + KVS_BLOCK_TOKENS - 1) / KVS_BLOCK_TOKENS;
  if (nb == 0) return;  // no tokens: no output row
  const int64_t seg_lo = s_before + static_cast<int64_t>(h) * nb;
  const int W = static_cast<int>(T < n_warps ? T : n_warps);
  const int w_lo = owner_of(seg_lo, T, W);
  const int np = owner_of(seg_lo + nb - 1, T, W) - w_lo + 1;
  if (np <= 1) return;  // written directly by its only piece
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int rec = part_floats(G, D);
  const float* base = ws_part + static_cast<int64_t>(w_lo + seg) * rec;
  const int64_t out_row0 = static_cast<int64_t>(item) * h_q + h * G;
  const int grp = threadIdx.x / kMergeGroupThreads;
  const int t = threadIdx.x % kMergeGroupThreads;
  for (int e0 = 0; e0 < G * D / 4; e0 += kMergeGroupThreads) {
    const int e4 = e0 + t;
    const bool act = e4 < G * D / 4;
    const int r = act ? (e4 * 4) / D : 0;
    const int c = e4 * 4 - r * D;
    float M = -INFINITY, lsum = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (act) {
      // pieces in batches of kMergeBatch per thread: every load of a batch is
      // issued before any is used (a guarded body, not a loop remainder, so
      // short folds do not serialise their L2 round trips)
      for (int sp0 = grp; sp0 < np; sp0 += kMergeGroups * kMergeBatch) {
        float mm[kMergeBatch], ll[kMergeBatch];
        float4 vv[kMergeBatch];
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u) {
          const int sp = sp0 + u * kMergeGroups;
          mm[u] = -INFINITY;
          ll[u] = 0.f;
          vv[u] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (sp < np) {
            const float* pr = base + static_cast<int64_t>(sp) * rec;
            mm[u] = __ldcg(pr + G * D + r);
            ll[u] = __ldcg(pr + G * D + G + r);
            vv[u] = __ldcg(reinterpret_cast<const float4*>(pr + r * D + c));
          }
        }
        float mn = M;
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u) mn = fmaxf(mn, mm[u]);
        const float sc = ex2(M - mn);  // 0 on the first batch (M = -inf, mn finite)
        acc.x *= sc;
        acc.y *= sc;
        acc.z *= sc;
        acc.w *= sc;
        lsum *= sc;
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u) {
          if (sp0 + u * kMergeGroups < np) {
            const float wgt = ex2(mm[u] - mn);
            acc.x += wgt * vv[u].x;
            acc.y += wgt * vv[u].y;
            acc.z += wgt * vv[u].z;
            acc.w += wgt * vv[u].w;
            lsum += wgt * ll[u];
          }
        }
        M = mn;
      }
    }
    s_acc[grp][t] = acc;
    s_ml[grp][t] = make_float2(M, lsum);
    __syncthreads();
    if (grp == 0 && act) {
      float Mt = -INFINITY;
#pragma unroll
      for (int g2 = 0; g2 < kMergeGroups; ++g2) Mt = fmaxf(Mt, s_ml[g2][t].x);
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
      float ls = 0.f;
#pragma unroll
      for (int g2 = 0; g2 < kMergeGroups; ++g2) {
        const float2 ml = s_ml[g2][t];
        if (ml.x == -INFINITY) continue;  // a group without pieces
        const float wgt = ex2(ml.x - Mt);
        const float4 v4 = s_acc[g2][t];
        a.x += wgt * v4.x;
        a.y += wgt * v4.y;
        a.z += wgt * v4.z;
        a.w += wgt * v4.w;
        ls += wgt * ml.y;
      }
      const float il = 1.0f / ls;
      if (lse != nullptr && c == 0) lse[out_row0 + r] = Mt + log2f(ls);
      uint2 w2;
      w2.x = pack_bf16x2(a.x * il, a.y * il);
      w2.y = pack_bf16x2(a.z * il, a.w * il);
      *reinterpret_cast<uint2*>(out + (out_row0 + r) * D + c) = w2;
    }
    __syncthreads();
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


// Partial slots one launch may touch: one per (warp, segment it touches),
// slot = warp + segment, for `warps` warps per CTA.
size_t workspace_need(int32_t batch, int32_t h_q, int32_t h_kv, int32_t d, int warps) {
  if (batch <= 0 || h_kv <= 0 || h_q <= 0 || d <= 0) return 0;
  const int64_t G = h_q / h_kv;
  const int64_t slots = static_cast<int64_t>(kMaxGrid) * warps +
                        static_cast<int64_t>(batch) * h_kv;
  return static_cast<size_t>(slots * part_floats(static_cast<int>(G), d) * 4);
}

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

constexpr int kSmemLimit = 232448;

// Shared-memory plan for a launch; returns the bytes, 0 if it cannot fit.
template <int D, bool kF8>
size_t plan_smem(DecodeParams& prm) {
  using L = DecodeLayout<D, kF8>;
  constexpr int kWarps = dec_warps(kF8);
  prm.q_bytes = prm.group * D * 2;
  prm.q_stride = (prm.q_bytes + 127) / 128 * 128;
  for (int ns = kMaxStages; ns >= 1; --ns) {
    size_t off = static_cast<size_t>(kWarps) * ns * L::kStageBytes;
    const size_t q_off = off;
    off += static_cast<size_t>(kWarps) * 2 * prm.q_stride;
    const size_t bar_off = off;
    off += static_cast<size_t>(kWarps) * ns * 8;
    const size_t pb_off = off;
    off += static_cast<size_t>(kWarps) * ns * 4;
    const size_t idx_off = off;
    off += static_cast<size_t>(2 * prm.batch + 1) * 4;
    const size_t total = off + 1024;
    if (total <= kSmemLimit) {
      prm.n_stages = ns;
      prm.q_off = static_cast<int>(q_off);
      prm.bar_off = static_cast<int>(bar_off);
      prm.pb_off = static_cast<int>(pb_off);
      prm.idx_off = static_cast<int>(idx_off);
      return total;
    }
  }
  return 0;
}

template <int D, int NT, bool kF8 = false>
kvs_status launch_decode(DecodeParams& prm, const CUtensorMap& km, const CUtensorMap& vm,
                         cudaStream_t stream) {
  const size_t smem = plan_smem<D, kF8>(prm);
  if (smem == 0) return fail(KVS_ERR_UNSUPPORTED, "kvs_paged_decode: shared-memory plan does not fit");
  static bool configured = false;
  if (!configured) {
    if constexpr (kF8) {
      KVS_CUDA(cudaFuncSetAttribute(paged_decode_kernel<D, NT, false, true>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit),
               "kvs_paged_decode: raising the shared-memory limit");
      KVS_CUDA(cudaFuncSetAttribute(paged_decode_kernel<D, NT, true, true>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit),
               "kvs_paged_decode: raising the shared-memory limit");
    } else {
      KVS_CUDA(cudaFuncSetAttribute(paged_decode_kernel<D, NT, false>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit),
               "kvs_paged_decode: raising the shared-memory limit");
      KVS_CUDA(cudaFuncSetAttribute(paged_decode_kernel<D, NT, true>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit),
               "kvs_paged_decode: raising the shared-memory limit");
    }
    configured = true;
  }
  const int grid = sm_count_dec() < kMaxGrid ? sm_count_dec() : kMaxGrid;
  constexpr int kWarps = dec_warps(kF8);
  constexpr int kDecThreads = kWarps * 32;
  if constexpr (kF8) {
    if (prm.logits != nullptr)
      paged_decode_kernel<D, NT, true, true><<<grid, kDecThreads, smem, stream>>>(km, vm, prm);
    else
      paged_decode_kernel<D, NT, false, true><<<grid, kDecThreads, smem, stream>>>(km, vm, prm);
  } else if (prm.logits != nullptr)
    paged_decode_kernel<D, NT, true><<<grid, kDecThreads, smem, stream>>>(km, vm, prm);
  else
    paged_decode_kernel<D, NT, false><<<grid, kDecThreads, smem, stream>>>(km, vm, prm);
  KVS_CHECK_LAUNCH("kvs_paged_decode");
  // the merge as a programmatic dependent launch (it waits for decode inside)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(prm.batch * prm.h_kv));
  cfg.blockDim = dim3(kMergeThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  KVS_CUDA(cudaLaunchKernelEx(&cfg, decode_merge_kernel<D>, static_cast<const float*>(prm.ws_part),
                              prm.lens, prm.batch, prm.max_blocks, prm.append, prm.h_q, prm.h_kv,
                              prm.group,
                              grid * kWarps, prm.out, prm.logits != nullptr ? prm.lse : nullptr),
           "kvs_paged_decode (merge launch)");
  return KVS_OK;
}

}  // namespace
}  // namespace kvs

extern "C" {

size_t kvs_paged_decode_workspace_size(int32_t batch, int32_t h_q, int32_t h_kv, int32_t d) {
  // enough for either pool type's decode
  return kvs::workspace_need(batch, h_q, h_kv, d, kvs::kMaxWarps);
}

}  // extern "C"

namespace {

kvs_status paged_decode_impl(const kvs_bf16* q, const kvs_bf16* k_new, const kvs_bf16* v_new,
                             kvs_bf16* k_pool, kvs_bf16* v_pool, int32_t num_blocks,
                             int32_t* block_tables, int32_t max_blocks, const int32_t* table_patch,
                             const int32_t* lens, int32_t* lens_next, int32_t batch, int32_t h_q,
                             int32_t h_kv, int32_t d, float scale, kvs_bf16* out, void* workspace,
                             size_t workspace_bytes, int32_t* status, kvs_stream stream,
                             float* logits, int32_t logit_ld, float* lse,
                             float* k_scale = nullptr, float* v_scale = nullptr,
                             bool fp8 = false, uint64_t wait_ns = kvs::kWaitLimitNs,
                             bool stall = false) {
  KVS_REQUIRE(batch >= 0, "kvs_paged_decode: negative batch");
  if (batch == 0) return KVS_OK;
  KVS_REQUIRE(q && k_pool && v_pool && block_tables && lens && out && workspace,
              "kvs_paged_decode: NULL pointer");
  KVS_REQUIRE((k_new == nullptr) == (v_new == nullptr),
              "kvs_paged_decode: k_new and v_new must both be given or both be NULL");
  KVS_REQUIRE(lens_next == nullptr || lens_next != lens,
              "kvs_paged_decode: lens_next must not alias lens");
  KVS_SUPPORTED(d == 64 || d == 128, "kvs_paged_decode: d = %d (supported: 64, 128)", d);
  KVS_REQUIRE(h_kv > 0 && h_q > 0 && h_q % h_kv == 0, "kvs_paged_decode: bad head counts");
  KVS_SUPPORTED(h_q / h_kv <= kvs::kMaxG, "kvs_paged_decode: group size %d > %d", h_q / h_kv,
                kvs::kMaxG);
  KVS_SUPPORTED(batch <= kvs::kMaxBatch, "kvs_paged_decode: batch %d > %d", batch,
                kvs::kMaxBatch);
  KVS_REQUIRE(num_blocks > 0 && max_blocks > 0, "kvs_paged_decode: bad sizes");
  // the kernels' block counts (lengths clamped to each table row) are 32-bit sums
  KVS_REQUIRE(static_cast<int64_t>(batch) * max_blocks * h_kv < (1ll << 31),
              "kvs_paged_decode: batch x max_blocks x h_kv must stay below 2^31");
  KVS_REQUIRE(static_cast<int64_t>(num_blocks) * h_kv * KVS_BLOCK_TOKENS < (1ll << 31),
              "kvs_paged_decode: pool too large for 32-bit TMA row coordinates");
  KVS_REQUIRE((reinterpret_cast<uintptr_t>(k_pool) & 15) == 0 &&
                  (reinterpret_cast<uintptr_t>(v_pool) & 15) == 0 &&
                  (reinterpret_cast<uintptr_t>(q) & 15) == 0 &&
                  (reinterpret_cast<uintptr_t>(out) & 15) == 0 &&
                  (reinterpret_cast<uintptr_t>(workspace) & 15) == 0,
              "kvs_paged_decode: q, out, pools and workspace must be 16-byte aligned");
  const int64_t G = h_q / h_kv;
  const size_t need = kvs::workspace_need(batch, h_q, h_kv, d, kvs::dec_warps(fp8));
  KVS_REQUIRE(workspace_bytes >= need, "kvs_paged_decode: workspace %zu bytes < %zu needed",
              workspace_bytes, need);
  static thread_local kvs::MapCache kc, vc;
  if (fp8) {
    KVS_SUPPORTED(d == 128, "kvs_paged_decode_fp8: d = %d (supported: 128)", d);
    KVS_REQUIRE(k_scale && v_scale && (reinterpret_cast<uintptr_t>(k_scale) & 15) == 0 &&
                    (reinterpret_cast<uintptr_t>(v_scale) & 15) == 0,
                "kvs_paged_decode_fp8: scales must be non-NULL and 16-byte aligned");
  } else if (!kvs::pool_map(kc, k_pool, num_blocks, h_kv, d) ||
             !kvs::pool_map(vc, v_pool, num_blocks, h_kv, d)) {
    return KVS_ERR_CUDA;
  }

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
  prm.ws_part = static_cast<float*>(workspace);
  prm.logits = logits;
  prm.logit_ld = logit_ld;
  prm.lse = lse;
  prm.k_scale = k_scale;
  prm.v_scale = v_scale;
  prm.status = status;
  prm.wait_ns = wait_ns;
  prm.stall = stall ? 1 : 0;
  prm.batch = batch;
  prm.max_blocks = max_blocks;
  prm.num_blocks = num_blocks;
  prm.h_q = h_q;
  prm.h_kv = h_kv;
  prm.group = static_cast<int>(G);
  prm.append = k_new != nullptr ? 1 : 0;
  prm.scale_log2 = scale * kvs::kLog2e;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  auto launch = [&](kvs::DecodeParams& pr) -> kvs_status {
    if (fp8) {
      static const CUtensorMap unused = {};  // FP8 blocks arrive by linear bulk copies
      if (G <= 8) return kvs::launch_decode<128, 1, true>(pr, unused, unused, st);
      return kvs::launch_decode<128, 2, true>(pr, unused, unused, st);
    }
    if (G <= 8) {
      if (d == 128) return kvs::launch_decode<128, 1>(pr, kc.map, vc.map, st);
      return kvs::launch_decode<64, 1>(pr, kc.map, vc.map, st);
    }
    if (d == 128) return kvs::launch_decode<128, 2>(pr, kc.map, vc.map, st);
    return kvs::launch_decode<64, 2>(pr, kc.map, vc.map, st);
  };
  // stages per warp that the shared-memory plan leaves for nb items (their
  // lengths and prefix take shared memory too); 0: it does not fit
  auto stages = [&](int nb) -> int {
    kvs::DecodeParams pr = prm;
    pr.batch = nb;
    const size_t sm = fp8 ? kvs::plan_smem<128, true>(pr)
                          : (d == 128 ? kvs::plan_smem<128, false>(pr) : kvs::plan_smem<64, false>(pr));
    return sm == 0 ? 0 : pr.n_stages;
  };
  // A batch whose per-item arrays would leave a single stage per warp (no
  // load in flight while a block is computed) is decoded in consecutive
  // chunks of items that keep two: each chunk a decode launch and its merge,
  // in order on the stream, reusing the workspace (a chunk's decode is an
  // ordinary launch, so it starts once the previous chunk's merge is done).
  int chunk = batch;
  while (chunk > 1 && stages(chunk) < 2) chunk = (chunk + 1) / 2;
  if (chunk == batch) return launch(prm);
  for (int b0 = 0; b0 < batch; b0 += chunk) {
    const int nb = batch - b0 < chunk ? batch - b0 : chunk;
    kvs::DecodeParams pc = prm;
    pc.batch = nb;
    pc.q = q + static_cast<int64_t>(b0) * h_q * d;
    pc.k_new = k_new ? k_new + static_cast<int64_t>(b0) * h_kv * d : nullptr;
    pc.v_new = v_new ? v_new + static_cast<int64_t>(b0) * h_kv * d : nullptr;
    pc.tables = block_tables + static_cast<int64_t>(b0) * max_blocks;
    pc.patch = table_patch ? table_patch + b0 : nullptr;
    pc.lens = lens + b0;
    pc.lens_next = lens_next ? lens_next + b0 : nullptr;
    pc.out = out + static_cast<int64_t>(b0) * h_q * d;
    pc.logits = logits ? logits + static_cast<int64_t>(b0) * h_kv * G * logit_ld : nullptr;
    pc.lse = lse ? lse + static_cast<int64_t>(b0) * h_q : nullptr;
    const kvs_status rc = launch(pc);
    if (rc != KVS_OK) return rc;
  }
  return KVS_OK;
}

}  // namespace

extern "C" {

kvs_status kvs_paged_decode(const kvs_bf16* q, const kvs_bf16* k_new, const kvs_bf16* v_new,
                            kvs_bf16* k_pool, kvs_bf16* v_pool, int32_t num_blocks,
                            int32_t* block_tables, int32_t max_blocks, const int32_t* table_patch,
                            const int32_t* lens, int32_t* lens_next, int32_t batch, int32_t h_q,
                            int32_t h_kv, int32_t d, float scale, kvs_bf16* out, void* workspace,
                            size_t workspace_bytes, int32_t* status, kvs_stream stream) {
  return paged_decode_impl(q, k_new, v_new, k_pool, v_pool, num_blocks, block_tables, max_blocks,
                           table_patch, lens, lens_next, batch, h_q, h_kv, d, scale, out,
                           workspace, workspace_bytes, status, stream, nullptr, 0, nullptr);
}

kvs_status kvs_paged_decode_fp8(const kvs_bf16* q, const kvs_bf16* k_new, const kvs_bf16* v_new,
                                uint8_t* k_pool, uint8_t* v_pool, float* k_scale, float* v_scale,
                                int32_t num_blocks, int32_t* block_tables, int32_t max_blocks,
                                const int32_t* table_patch, const int32_t* lens,
                                int32_t* lens_next, int32_t batch, int32_t h_q, int32_t h_kv,
                                int32_t d, float scale, kvs_bf16* out, void* workspace,
                                size_t workspace_bytes, int32_t* status, kvs_stream stream) {
  return paged_decode_impl(q, k_new, v_new, reinterpret_cast<kvs_bf16*>(k_pool),
                           reinterpret_cast<kvs_bf16*>(v_pool), num_blocks, block_tables,
                           max_blocks, table_patch, lens, lens_next, batch, h_q, h_kv, d, scale,
                           out, workspace, workspace_bytes, status, stream, nullptr, 0, nullptr,
                           k_scale, v_scale, true);
}

kvs_status kvs_paged_decode_logits(const kvs_bf16* q, const kvs_bf16* k_new,
                                   const kvs_bf16* v_new, kvs_bf16* k_pool, kvs_bf16* v_pool,
                                   int32_t num_blocks, int32_t* block_tables, int32_t max_blocks,
                                   const int32_t* table_patch, const int32_t* lens,
                                   int32_t* lens_next, int32_t batch, int32_t h_q, int32_t h_kv,
                                   int32_t d, float scale, kvs_bf16* out, void* workspace,
                                   size_t workspace_bytes, float* logits, int32_t logit_ld,
                                   float* lse, int32_t* status, kvs_stream stream) {
  KVS_REQUIRE(logits != nullptr && logit_ld > 0 && lse != nullptr,
              "kvs_paged_decode_logits: no logits or lse buffer");
  return paged_decode_impl(q, k_new, v_new, k_pool, v_pool, num_blocks, block_tables, max_blocks,
                           table_patch, lens, lens_next, batch, h_q, h_kv, d, scale, out,
                           workspace, workspace_bytes, status, stream, logits, logit_ld, lse);
}

kvs_status kvs_paged_decode_logits_fp8(const kvs_bf16* q, const kvs_bf16* k_new,
                                       const kvs_bf16* v_new, uint8_t* k_pool, uint8_t* v_pool,
                                       float* k_scale, float* v_scale, int32_t num_blocks,
                                       int32_t* block_tables, int32_t max_blocks,
                                       const int32_t* table_patch, const int32_t* lens,
                                       int32_t* lens_next, int32_t batch, int32_t h_q,
                                       int32_t h_kv, int32_t d, float scale, kvs_bf16* out,
                                       void* workspace, size_t workspace_bytes, float* logits,
                                       int32_t logit_ld, float* lse, int32_t* status,
                                       kvs_stream stream) {
  KVS_REQUIRE(logits != nullptr && logit_ld > 0 && lse != nullptr,
              "kvs_paged_decode_logits_fp8: no logits or lse buffer");
  return paged_decode_impl(q, k_new, v_new, reinterpret_cast<kvs_bf16*>(k_pool),
                           reinterpret_cast<kvs_bf16*>(v_pool), num_blocks, block_tables,
                           max_blocks, table_patch, lens, lens_next, batch, h_q, h_kv, d, scale,
                           out, workspace, workspace_bytes, status, stream, logits, logit_ld, lse,
                           k_scale, v_scale, true);
}

kvs_status kvs_test_paged_decode_stalled(const kvs_bf16* q, kvs_bf16* k_pool, kvs_bf16* v_pool,
                                         int32_t num_blocks, int32_t* block_tables,
                                         int32_t max_blocks, const int32_t* lens, int32_t batch,
                                         int32_t h_q, int32_t h_kv, int32_t d, float scale,
                                         kvs_bf16* out, void* workspace, size_t workspace_bytes,
                                         uint32_t wait_ns, int32_t* status, kvs_stream stream) {
  KVS_REQUIRE(wait_ns > 0 && wait_ns <= kvs::kWaitLimitNs,
              "kvs_test_paged_decode_stalled: wait_ns must be in (0, %llu]",
              static_cast<unsigned long long>(kvs::kWaitLimitNs));
  return paged_decode_impl(q, nullptr, nullptr, k_pool, v_pool, num_blocks, block_tables,
                           max_blocks, nullptr, lens, nullptr, batch, h_q, h_kv, d, scale, out,
                           workspace, workspace_bytes, status, stream, nullptr, 0, nullptr,
                           nullptr, nullptr, false, wait_ns, true);
}

}  // extern "C"

namespace {

// Device address of the built-in scratch on the current device, looked up
// once per device.  Returns nullptr (and records the error) on failure.
void* static_scratch_address() {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    kvs::set_error("kvs_paged_decode_static: no usable current device");
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_decode_static_scratch);
    if (e != cudaSuccess) {
      kvs::set_error("kvs_paged_decode_static: cudaGetSymbolAddress failed: %s",
                     cudaGetErrorString(e));
      return nullptr;
    }
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace

extern "C" kvs_status kvs_paged_decode_static(const kvs_bf16* q, const kvs_bf16* k_new,
                                              const kvs_bf16* v_new, kvs_bf16* k_pool,
                                              kvs_bf16* v_pool, int32_t num_blocks,
                                              int32_t* block_tables, int32_t max_blocks,
                                              const int32_t* table_patch, const int32_t* lens,
                                              int32_t* lens_next, int32_t batch, int32_t h_q,
                                              int32_t h_kv, int32_t d, float scale,
                                              kvs_bf16* out, int32_t* status, kvs_stream stream) {
  KVS_REQUIRE(batch >= 0, "kvs_paged_decode_static: negative batch");
  if (batch == 0) return KVS_OK;
  KVS_REQUIRE(h_kv > 0 && h_q > 0 && h_q % h_kv == 0, "kvs_paged_decode_static: bad head counts");
  const size_t need = kvs::workspace_need(batch, h_q, h_kv, d, kvs::dec_warps(false));
  if (need > KVS_DECODE_STATIC_SCRATCH_BYTES)
    return kvs::fail(KVS_ERR_UNSUPPORTED,
                     "kvs_paged_decode_static: this batch needs %zu bytes of scratch; the "
                     "built-in array holds %u (use kvs_paged_decode with a workspace)",
                     need, static_cast<unsigned>(KVS_DECODE_STATIC_SCRATCH_BYTES));
  void* scratch = static_scratch_address();
  if (scratch == nullptr) return KVS_ERR_CUDA;
  return kvs_paged_decode(q, k_new, v_new, k_pool, v_pool, num_blocks, block_tables, max_blocks,
                          table_patch, lens, lens_next, batch, h_q, h_kv, d, scale, out, scratch,
                          KVS_DECODE_STATIC_SCRATCH_BYTES, status, stream);
}
