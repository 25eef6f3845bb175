// Paged K/V cache: one-token decode attention over a paged cache with grouped
// heads, and the append of the new token's K/V.  Page "CUDA KV Cache：分页存储与长上下
// 文 Decode 极致优化" (chengzipai.xyz): cache[P][2][T][Hkv][D] with token t of
// request b on physical page block_table[b, t / T] at offset t % T (section 2);
// query head h reads key/value head h / (Hq / Hkv) (section 3.3); the append
// writes the newest token's K and V at that address with 16-byte stores (section
// 4); the decode keeps FP32 running max m, sum l and output o across pages
// (section 5), serves a group of query heads from one copy of each K/V page
// (section 6.3), looks a page id up once per page (section 6.1) and splits long
// contexts into segments merged with the online-softmax law (section 6.4).
//
// GB300 mapping: one CTA per (request, K/V head, chunk of HC <= 8 query heads of
// the group, key segment); five warps.  A producer warp issues the TMA copies:
// each page of one K/V head as (T tokens x 64 dims) boxes with the 128-byte
// swizzle, into a 2-stage ring of 64-token tiles, with the page ids in a rolling
// window in shared memory and the tile's valid-row mask beside it.  Four compute
// warps each take 16 tokens of every tile and run their own online softmax over
// them (section 5's recurrence, per warp), merged once at the end with the
// section 6.4 law.  The HC query heads are the rows of mma.sync m16n8k16
// products padded to 16 (the decode is HBM-bound at a few FLOP per byte, so the
// padding costs nothing; tcgen05 would need M >= 64):
//   S^T-free scores: S (heads x 8 tokens) = Q (heads x 16 dims) K^T, K^T fragments
//                    read with ldmatrix straight from the swizzled boxes, fp32
//                    accumulation, Q fragments held in registers;
//   softmax: the S accumulator layout is the A-operand layout of the next
//            product, so p goes to 16 bits in registers with no shared memory;
//   O += P V: V fragments read with ldmatrix.trans, fp32 accumulators per warp.
// No K/V element is converted to fp32 and no block barrier is taken per tile.
// Page and row offsets use shifts (page sizes are powers of two).
// Page ids outside [0, P) and lengths outside [0, max_pages * T] are not read:
// the kernel records ATTN_ERR_BAD_INDEX in the status word and treats them as
// empty.
#pragma once
#include <cuda.h>
#include <cstdint>

#include "ptx.cuh"

namespace eca {

constexpr int kDecTile = 64;     // tokens per tile
constexpr int kDecStages = 2;
constexpr int kDecWarps = 4;     // compute warps: 16 tokens of every tile each
constexpr int kDecThreads = 32 * (kDecWarps + 1);  // and one producer warp
constexpr int kDecIdRing = 64;  // page ids staged in shared memory, a rolling window of the segment

struct DecodeParams {
  const void* q;            // [B, Hq, D] 16-bit
  const int* block_table;   // [B, max_pages]
  const int* lengths;       // [B]
  void* out;                // [B, Hq, D] 16-bit (no split)
  float* lse;               // [B, Hq] or null (no split)
  float* part_o;            // split: [splits, B, Hq, D] fp32
  float* part_lse;          // split: [splits, B, Hq] fp32
  int* status;
  int B, Hq, Hkv, page_size, max_pages, num_pages;
  int head_chunks;          // chunks of HC query heads per K/V head
  int splits, seg_pages;    // key segments of seg_pages logical pages
  float scale_log2e;
  unsigned long long wait_limit_ns;
  int timeout_code, bad_index_code;
  // Split only: one counter per (request, K/V head, head chunk), zero on entry and
  // left zero; the last segment to finish merges the group's partial results.
  // Null: a separate merge kernel does it.
  unsigned* counters;
};

template <int D>
struct DecodeSmem {
  static constexpr int kKindBytes = kDecTile * D * 2;  // one kind (K or V) of a tile
  static constexpr int kStageBytes = 2 * kKindBytes;
  static constexpr int kRingOff = 0;
  static constexpr int kRedOff = kRingOff;  // fp32 [warps][8][D] partial outputs at the end, over the idle ring
  static constexpr int kRowsOff = kDecStages * kStageBytes;         // uint64 [stages]: valid rows of the staged tile
  static constexpr int kIdsOff = kRowsOff + 8 * kDecStages;         // int32 page-id window
  static constexpr int kQFragOff = kIdsOff + kDecIdRing * 4;        // uint32 [D/16][32 lanes][2] query fragments
  static constexpr int kStatOff = kQFragOff + (D / 16) * 32 * 8;     // fp32 [warps][8] m, then [warps][8] l
  static constexpr int kBarOff = kStatOff + 2 * kDecWarps * 8 * 4;  // full[stages], then empty[stages]
  static constexpr int kMiscOff = kBarOff + 2 * kDecStages * 8;     // abort flag, last-segment flag
  static constexpr int kBytes = kMiscOff + 16;
  static constexpr int kDynamicBytes = kBytes + 1024;
  static_assert(kDecWarps * 8 * D * 4 <= kDecStages * kStageBytes, "reduction buffer fits over the ring");
  static_assert(kBarOff % 8 == 0, "mbarriers are 8-byte aligned");
};

template <bool BF16>
__device__ __forceinline__ float to_f32(uint16_t h) {
  if constexpr (BF16) {
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
  } else {
    float f;
    asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"(h));
    return f;
  }
}

template <bool BF16>
__device__ __forceinline__ float2 to_f32x2(uint32_t w) {
  return make_float2(to_f32<BF16>(static_cast<uint16_t>(w & 0xffffu)), to_f32<BF16>(static_cast<uint16_t>(w >> 16)));
}

// Byte offset, inside one kind of a tile, of the 16-byte chunk c (0 .. D/8 - 1) of
// token row r.  Rows are staged as swizzled (T x 64) boxes: box (page, half) holds
// T rows of 128 B, and chunk index c % 8 is stored at position (c % 8) ^ (row % 8).
template <int D>
__device__ __forceinline__ int dec_chunk_offset(int r, int c, int log2T) {
  const int T = 1 << log2T;
  const int page = r >> log2T, rr = r & (T - 1);
  const int box = page * (D / 64) + (c >> 3);
  return ((box * T + rr) << 7) + (((c & 7) ^ (rr & 7)) << 4);
}

// Four 8x8 16-bit matrices from shared memory; lane l gives the address of row
// l % 8 of matrix l / 8 (16 contiguous bytes), and receives row l / 4, elements
// 2 (l % 4) and 2 (l % 4) + 1 of each matrix (transposed with .trans).
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// D (16 x 8, fp32) += A (16 x 16, row) B (16 x 8, col), 16-bit inputs; d0, d1 hold
// row l / 4 of the accumulator, d2, d3 row l / 4 + 8.
template <bool BF16>
__device__ __forceinline__ void mma_16816(float& d0, float& d1, float& d2, float& d3, uint32_t a0, uint32_t a1,
                                          uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1) {
  if constexpr (BF16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d0), "+f"(d1), "+f"(d2), "+f"(d3)
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d0), "+f"(d1), "+f"(d2), "+f"(d3)
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

template <int D, bool BF16, int HC>
__global__ void __maxnreg__(128) paged_decode_kernel(const __grid_constant__ CUtensorMap tm_cache,
                                                                   const DecodeParams p) {
  static_assert(HC >= 1 && HC <= 8, "query heads per CTA are rows 0-7 of the padded products");
  using L = DecodeSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t sbase = (raw_base + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw_base);
  float* red_s = reinterpret_cast<float*>(smem + L::kRedOff);
  volatile unsigned long long* rows_s = reinterpret_cast<volatile unsigned long long*>(smem + L::kRowsOff);
  int* ids_s = reinterpret_cast<int*>(smem + L::kIdsOff);
  uint2* qfrag_s = reinterpret_cast<uint2*>(smem + L::kQFragOff);
  float* wm_s = reinterpret_cast<float*>(smem + L::kStatOff);  // [warp][8] running max
  float* wl_s = wm_s + kDecWarps * 8;                            // [warp][8] running sum
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff);
  auto full = [&](int s) -> uint32_t { return sbase + L::kBarOff + 8u * static_cast<uint32_t>(s); };
  auto empty = [&](int s) -> uint32_t { return sbase + L::kBarOff + 8u * static_cast<uint32_t>(kDecStages + s); };

  // Launched with programmatic serialisation: the next launch may be scheduled at
  // once, and no global memory is read before the grid ahead of this one finished.
  grid_launch_dependents();
  // The cache's tensor map comes from the launch's own parameters: its descriptor
  // fetch starts before the wait and overlaps the page-id and length reads.
  if (threadIdx.x == kDecWarps * 32) tma_prefetch_map(&tm_cache);
  grid_dependency_wait();
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  // unit: (b, kv head, head chunk, segment), segment fastest
  int u = blockIdx.x;
  const int seg = u % p.splits;
  u /= p.splits;
  const int chunk = u % p.head_chunks;
  u /= p.head_chunks;
  const int kvh = u % p.Hkv;
  const int b = u / p.Hkv;
  const int group = p.Hq / p.Hkv;
  const int qh0 = kvh * group + chunk * HC;  // first query head of this CTA
  const int T = p.page_size;
  const int log2T = 31 - __clz(T);
  const int pages_per_tile = kDecTile >> log2T;

  // The segment's first page ids are read together with the length rather than
  // after it (the table row holds max_pages entries, so the read stays inside it);
  // ids past the request's last page are read but never followed.
  const int* table_row = p.block_table + static_cast<size_t>(b) * p.max_pages;
  const int pg_begin = seg * p.seg_pages;
  int id_first = -1;
  if (tid < kDecIdRing && pg_begin + tid < min(p.max_pages, pg_begin + p.seg_pages)) {
    id_first = table_row[pg_begin + tid];
  }
  int len = p.lengths[b];
  if (len < 0 || len > p.max_pages * T) {
    if (tid == 0) atomicExch(p.status, p.bad_index_code);
    len = len < 0 ? 0 : p.max_pages * T;
  }
  const int n_pages = (len + T - 1) >> log2T;
  const int pg_end = min(n_pages, pg_begin + p.seg_pages);
  const int n_tiles = pg_end > pg_begin ? (pg_end - pg_begin + pages_per_tile - 1) / pages_per_tile : 0;

  if (tid == 0) {
    for (int s = 0; s < kDecStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), kDecWarps);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  // Page ids of the segment in a rolling window of kDecIdRing slots (slot = page % ring),
  // read from global memory once each and range-checked when used (rejected ids
  // are recorded and their pages skipped).
  auto checked_id = [&](int id) {
    if (id < 0 || id >= p.num_pages) {
      atomicExch(p.status, p.bad_index_code);
      return -1;
    }
    return id;
  };
  if (tid < kDecIdRing && pg_begin + tid < pg_end) ids_s[tid] = id_first;
  // Q of the chunk as A fragments of the score products (rows = heads, padded with
  // zeros to 16), the same for every compute warp: entry [k][l] holds, for lane l,
  // dims 16 k + 2 (l % 4) .. + 1 and the same + 8 of head l / 4.
  for (int e = tid; e < (D / 16) * 32; e += kDecThreads) {
    const int k = e / 32, l = e % 32, h = l >> 2;
    uint2 v = make_uint2(0u, 0u);
    if (h < HC) {
      const uint32_t* qg = reinterpret_cast<const uint32_t*>(static_cast<const uint16_t*>(p.q) +
                                                             (static_cast<size_t>(b) * p.Hq + qh0 + h) * D);
      v = make_uint2(qg[8 * k + (l & 3)], qg[8 * k + 4 + (l & 3)]);
    }
    qfrag_s[e] = v;
  }
  __syncthreads();
  const Watchdog wd{abort_flag, p.status, p.wait_limit_ns, p.timeout_code};
  const int head = lane >> 2;  // query head (row of the products) of this lane's accumulators
  float m_run = -INFINITY;     // compute warps: running max of head `head`, base-2 domain
  float l_run = 0.f;           // this lane's part of the running sum
  float o[D / 8][2];           // O (+)= P V, row `head`, 8 columns per block
#pragma unroll
  for (int d = 0; d < D / 8; ++d) o[d][0] = o[d][1] = 0.f;
  // Rows 8-15 of the padded products (P rows of no head, always 0) land in shared
  // sink registers, four pairs so the products stay in independent chains.
  float sink[4][2] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
  bool ok = true;

  if (warp == kDecWarps) {
    // ----------------------------------------------------------------- producer
    if (lane == 0) {
      // Each decode step reads its K/V once: evict-first.
      const uint64_t pol = policy_evict_first();
      // The window is refilled with cp.async: after tile i is issued, its slots
      // receive the page ids kDecIdRing pages further on, which are first needed at
      // least kDecIdRing / 8 = 8 tiles later; waiting until at most 7 refill groups
      // are in flight before reading the window keeps the copies off the path.
      int issued = 0;
      for (int i = 0; i < n_tiles; ++i) {
        const int slot = i % kDecStages;
        if (i >= kDecStages && !wd.wait(empty(slot), static_cast<uint32_t>((i / kDecStages) - 1) & 1u)) {
          ok = false;
          break;
        }
        asm volatile("cp.async.wait_group 7;" ::: "memory");
        const int first = i * pages_per_tile;  // within the segment
        const int np = min(pages_per_tile, pg_end - pg_begin - first);
        const int first_page = pg_begin + first;
        const int tok0 = first_page << log2T;  // logical token of tile row 0
        // Rows that hold a token of this segment on an accepted page; the rest (past
        // the length, past the segment, or on a rejected page) are empty.
        unsigned long long rows_ok = 0;
        int good = 0;
        int ids[8];  // the tile's page ids, range-checked (-1: rejected, not read)
#pragma unroll
        for (int pp = 0; pp < 8; ++pp) ids[pp] = pp < np ? checked_id(ids_s[(first + pp) % kDecIdRing]) : -1;
#pragma unroll
        for (int pp = 0; pp < 8; ++pp) {
          if (ids[pp] < 0) continue;
          ++good;
          const int lo = pp << log2T, hi = min((pp + 1) << log2T, len - tok0);
          if (hi > lo) rows_ok |= (hi - lo == 64 ? ~0ull : ((1ull << (hi - lo)) - 1)) << lo;
        }
        rows_s[slot] = rows_ok;
        mbar_arrive_expect_tx(full(slot), static_cast<uint32_t>(good * 2 * (D / 64) * T * 128));
        const uint32_t stage = sbase + L::kRingOff + slot * L::kStageBytes;
#pragma unroll
        for (int pp = 0; pp < 8; ++pp) {
          const int id = ids[pp];
          if (id < 0) continue;
          for (int kind = 0; kind < 2; ++kind) {
            for (int h = 0; h < D / 64; ++h) {
              const uint32_t dst = stage + kind * L::kKindBytes + (pp * (D / 64) + h) * T * 128;
              tma_load_3d(dst, &tm_cache, full(slot), 64 * h, kvh, (id * 2 + kind) * T, pol);
            }
          }
        }
        ++issued;
        // This tile's window slots now take the pages kDecIdRing further on.
        for (int pp = 0; pp < np; ++pp) {
          const int page = pg_begin + first + pp + kDecIdRing;
          if (page < pg_end) {
            asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(ids_s + (first + pp) % kDecIdRing)),
                         "l"(table_row + page)
                         : "memory");
          }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
      }
      asm volatile("cp.async.wait_all;" ::: "memory");
      // let every copy issued here land before the block exits
      for (int i = (issued > kDecStages ? issued - kDecStages : 0); i < issued; ++i) {
        wd.drain(full(i % kDecStages), static_cast<uint32_t>(i / kDecStages) & 1u);
      }
    }
  } else {
    // ------------------------------------------------------------ compute warps
    const float c = p.scale_log2e;
    const int tok_w = 16 * warp;  // this warp's rows of every tile
    for (int i = 0; i < n_tiles; ++i) {
      const int slot = i % kDecStages;
      if (!__all_sync(0xffffffffu, wd.wait(full(slot), static_cast<uint32_t>(i / kDecStages) & 1u))) {
        ok = false;
        break;
      }
      const unsigned long long rows_ok = rows_s[slot];
      const uint32_t kt = sbase + L::kRingOff + slot * L::kStageBytes;
      const uint32_t vt = kt + L::kKindBytes;
      // S = Q K^T for this warp's two 8-token blocks; ldmatrix row address of lane l:
      // token block + l % 8, 16-byte chunk (8 dims) 4 kk + l / 8 (two k-steps per load).
      float sacc[2][4];
#pragma unroll
      for (int nb = 0; nb < 2; ++nb) {
        sacc[nb][0] = sacc[nb][1] = sacc[nb][2] = sacc[nb][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < D / 32; ++kk) {
          uint32_t kb[4];
          ldsm_x4(kt + dec_chunk_offset<D>(tok_w + 8 * nb + (lane & 7), 4 * kk + (lane >> 3), log2T), kb);
          const uint2 qa0 = qfrag_s[(2 * kk) * 32 + lane], qa1 = qfrag_s[(2 * kk + 1) * 32 + lane];
          mma_16816<BF16>(sacc[nb][0], sacc[nb][1], sacc[nb][2], sacc[nb][3], qa0.x, 0u, qa0.y, 0u, kb[0], kb[1]);
          mma_16816<BF16>(sacc[nb][0], sacc[nb][1], sacc[nb][2], sacc[nb][3], qa1.x, 0u, qa1.y, 0u, kb[2], kb[3]);
        }
      }
      // This lane holds head `head` at tokens tok_w + 8 nb + 2 (lane % 4) + e.
      float x[4];
#pragma unroll
      for (int nb = 0; nb < 2; ++nb) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int r = tok_w + 8 * nb + 2 * (lane & 3) + e;
          x[2 * nb + e] = ((rows_ok >> r) & 1ull) ? sacc[nb][e] * c : -INFINITY;
        }
      }
      // online softmax over this warp's tokens: m' = max(m, max s), p = 2^(s - m'),
      // l' = l 2^(m - m') + sum p (the four lanes of a head share m)
      float mt = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
      mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
      mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
      const float m_new = fmaxf(m_run, mt);
      const float alpha = m_run == -INFINITY ? 0.f : ex2(m_run - m_new);
      float pe[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) pe[e] = m_new == -INFINITY ? 0.f : ex2(x[e] - m_new);
      l_run = l_run * alpha + ((pe[0] + pe[1]) + (pe[2] + pe[3]));
      m_run = m_new;
#pragma unroll
      for (int d = 0; d < D / 8; ++d) {
        o[d][0] *= alpha;
        o[d][1] *= alpha;
      }
      // P as the A fragment of O += P V (rows = heads, k = the warp's 16 tokens)
      const uint32_t pa0 = pack2<BF16>(pe[0], pe[1]);
      const uint32_t pa2 = pack2<BF16>(pe[2], pe[3]);
      // V fragments with ldmatrix.trans; lane l: token tok_w + l % 8 + 8 ((l / 8) % 2),
      // 16-byte chunk (8 dims) 2 dp + l / 16: dims blocks 2 dp and 2 dp + 1.
      // Empty rows have p = 0; their V may not be a number, so p 0 x NaN would
      // poison the sum: skip the tile's products when any of the warp's rows is empty
      // and zero their V through the mask below instead.
      const unsigned long long mine = (rows_ok >> tok_w) & 0xffffull;
      if (mine == 0xffffull) {
#pragma unroll
        for (int dp = 0; dp < D / 16; ++dp) {
          uint32_t vb[4];
          ldsm_x4_trans(vt + dec_chunk_offset<D>(tok_w + (lane & 7) + 8 * ((lane >> 3) & 1), 2 * dp + (lane >> 4), log2T),
                        vb);
          mma_16816<BF16>(o[2 * dp][0], o[2 * dp][1], sink[dp % 4][0], sink[dp % 4][1], pa0, 0u, pa2, 0u, vb[0],
                          vb[1]);
          mma_16816<BF16>(o[2 * dp + 1][0], o[2 * dp + 1][1], sink[(dp + 2) % 4][0], sink[(dp + 2) % 4][1], pa0, 0u,
                          pa2, 0u, vb[2], vb[3]);
        }
      } else if (mine != 0) {
        // Partly empty: the V fragment entries of empty rows are replaced by zero.
        // Lane l holds, in each fragment register, rows (tokens) 2 (l % 4) and + 1
        // (b0b1) and the same + 8 (b2b3).
        const int r0 = 2 * (lane & 3);
        const uint32_t keep01 = (((mine >> r0) & 1ull) ? 0x0000ffffu : 0u) | (((mine >> (r0 + 1)) & 1ull) ? 0xffff0000u : 0u);
        const uint32_t keep89 =
            (((mine >> (r0 + 8)) & 1ull) ? 0x0000ffffu : 0u) | (((mine >> (r0 + 9)) & 1ull) ? 0xffff0000u : 0u);
#pragma unroll
        for (int dp = 0; dp < D / 16; ++dp) {
          uint32_t vb[4];
          ldsm_x4_trans(vt + dec_chunk_offset<D>(tok_w + (lane & 7) + 8 * ((lane >> 3) & 1), 2 * dp + (lane >> 4), log2T),
                        vb);
          mma_16816<BF16>(o[2 * dp][0], o[2 * dp][1], sink[dp % 4][0], sink[dp % 4][1], pa0, 0u, pa2, 0u,
                          vb[0] & keep01, vb[1] & keep89);
          mma_16816<BF16>(o[2 * dp + 1][0], o[2 * dp + 1][1], sink[(dp + 2) % 4][0], sink[(dp + 2) % 4][1], pa0,
                          0u, pa2, 0u, vb[2] & keep01, vb[3] & keep89);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty(slot));
    }
    // this warp's state for the merge: the four lanes of a head add their sums
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
    if ((lane & 3) == 0) {
      wm_s[warp * 8 + head] = m_run;
      wl_s[warp * 8 + head] = l_run;
    }
  }
  __syncthreads();  // every copy has landed (the producer drained), every warp's state is in
  // Merge of the warps (section 6.4): M = max m_w, L = sum l_w 2^(m_w - M),
  // O = sum o_w 2^(m_w - M) / L; each compute warp scales its partial output.
  if (warp < kDecWarps) {
    float mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) mx = fmaxf(mx, wm_s[w * 8 + head]);
    const float sc = m_run == -INFINITY ? 0.f : ex2(m_run - mx);
    if (head < HC) {
#pragma unroll
      for (int d = 0; d < D / 8; ++d) {
        *reinterpret_cast<float2*>(red_s + (warp * 8 + head) * D + 8 * d + 2 * (lane & 3)) =
            make_float2(o[d][0] * sc, o[d][1] * sc);
      }
    }
  }
  __syncthreads();
  if (ok && !wd.aborted()) {
    // O = o / L and lse = (M + log2 L) ln 2; an empty context gives O = 0 and lse = -inf
    for (int idx = tid; idx < HC * (D / 2); idx += kDecThreads) {
      const int k = idx / (D / 2), cp = idx % (D / 2);
      float mx = -INFINITY;
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) mx = fmaxf(mx, wm_s[w * 8 + k]);
      float l = 0.f;
      float2 acc = make_float2(0.f, 0.f);
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) {
        const float mw = wm_s[w * 8 + k];
        l += mw == -INFINITY ? 0.f : wl_s[w * 8 + k] * ex2(mw - mx);
        const float2 part = *reinterpret_cast<const float2*>(red_s + (w * 8 + k) * D + 2 * cp);
        acc.x += part.x;
        acc.y += part.y;
      }
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const size_t row = static_cast<size_t>(b) * p.Hq + qh0 + k;
      if (p.part_o != nullptr) {
        *reinterpret_cast<float2*>(p.part_o + (static_cast<size_t>(seg) * p.B * p.Hq + row) * D + 2 * cp) =
            make_float2(acc.x * inv, acc.y * inv);
      } else {
        *reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(p.out) + row * D + 2 * cp) =
            pack2<BF16>(acc.x * inv, acc.y * inv);
      }
      if (cp == 0) {
        const float lse = l > 0.f ? (mx + log2f(l)) * 0.69314718055994530942f : -INFINITY;
        if (p.part_o != nullptr) {
          p.part_lse[static_cast<size_t>(seg) * p.B * p.Hq + row] = lse;
        } else if (p.lse != nullptr) {
          p.lse[row] = lse;
        }
      }
    }
  }
  if (p.part_o == nullptr || p.counters == nullptr) return;
  // Merge of the segments (section 6.4, log-sum-exp form) by the group's last
  // segment to finish: lse = ln sum_s e^(lse_s), O = sum_s e^(lse_s - lse) O_s.
  const int valid = min(p.splits, (n_pages + p.seg_pages - 1) / p.seg_pages);  // segments with pages
  volatile int* last_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
  const size_t stride = static_cast<size_t>(p.B) * p.Hq;
  if (seg < valid) {
    __syncthreads();  // this segment's partial results are written
    if (tid == 0) {
      __threadfence();
      unsigned* counter = p.counters + static_cast<size_t>(blockIdx.x / p.splits);
      const bool last = atomicAdd(counter, 1u) == static_cast<unsigned>(valid - 1);
      if (last) {
        *counter = 0u;  // back to zero for the next launch
        __threadfence();
      }
      *last_flag = last ? 1 : 0;
    }
    __syncthreads();
    if (*last_flag == 0) return;
  } else if (!(valid == 0 && seg == 0)) {
    return;  // an empty segment; an empty request is finished by its segment 0
  }
  // Every thread takes one (head, four columns) share and reads, six segments at a
  // time, their log-sum-exps and partial outputs in one round trip, folding each
  // group in with the online law (running max m, sums rescaled by e^(m_old - m)).
  for (int idx = tid; idx < HC * (D / 4); idx += kDecThreads) {
    const int k = idx / (D / 4), c4 = idx % (D / 4);
    const size_t row = static_cast<size_t>(b) * p.Hq + qh0 + k;
    float m = -INFINITY;
    float wsum = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < valid; s0 += 6) {
      float ls[6];
      float4 os[6];
#pragma unroll
      for (int i = 0; i < 6; ++i) {
        ls[i] = -INFINITY;
        os[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (s0 + i < valid) {
          const size_t r_s = static_cast<size_t>(s0 + i) * stride + row;
          ls[i] = __ldcg(p.part_lse + r_s);
          os[i] = __ldcg(reinterpret_cast<const float4*>(p.part_o + r_s * D + 4 * c4));
        }
      }
      float mc = m;
#pragma unroll
      for (int i = 0; i < 6; ++i) mc = fmaxf(mc, ls[i]);
      if (mc == -INFINITY) continue;
      const float sc = m == -INFINITY ? 0.f : expf(m - mc);
      wsum *= sc;
      acc.x *= sc;
      acc.y *= sc;
      acc.z *= sc;
      acc.w *= sc;
#pragma unroll
      for (int i = 0; i < 6; ++i) {
        const float wgt = ls[i] == -INFINITY ? 0.f : expf(ls[i] - mc);
        if (wgt == 0.f) continue;  // (an unwritten partial is never read into the sums)
        wsum += wgt;
        acc.x += wgt * os[i].x;
        acc.y += wgt * os[i].y;
        acc.z += wgt * os[i].z;
        acc.w += wgt * os[i].w;
      }
      m = mc;
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    uint2 packed = make_uint2(pack2<BF16>(acc.x * inv, acc.y * inv), pack2<BF16>(acc.z * inv, acc.w * inv));
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(p.out) + row * D + 4 * c4) = packed;
    if (c4 == 0 && p.lse != nullptr) p.lse[row] = wsum > 0.f ? m + logf(wsum) : -INFINITY;
  }
}

// Merge of the decode segments (section 6.4 of the page, in log-sum-exp form as in
// the prefill merge): rows are (b, query head); segment s is non-empty when its
// first logical page is below the request's page count.
template <int D, bool BF16>
__global__ void __launch_bounds__(256) paged_decode_combine(const DecodeParams p) {
  grid_dependency_wait();  // the partials come from the decode grid just ahead
  const int lane = threadIdx.x % 32;
  const long long rows = static_cast<long long>(p.B) * p.Hq;
  for (long long r = static_cast<long long>(blockIdx.x) * 8 + threadIdx.x / 32; r < rows; r += gridDim.x * 8LL) {
    const int b = static_cast<int>(r / p.Hq);
    int len = p.lengths[b];
    len = len < 0 ? 0 : (len > p.max_pages * p.page_size ? p.max_pages * p.page_size : len);
    const int n_pages = (len + p.page_size - 1) / p.page_size;
    const int valid = min(p.splits, (n_pages + p.seg_pages - 1) / p.seg_pages);
    const size_t stride = static_cast<size_t>(p.B) * p.Hq;
    float m = -INFINITY;
    for (int s = 0; s < valid; ++s) m = fmaxf(m, p.part_lse[s * stride + r]);
    float wsum = 0.f;
    float acc[D / 32];
#pragma unroll
    for (int i = 0; i < D / 32; ++i) acc[i] = 0.f;
    if (m != -INFINITY) {
      for (int s = 0; s < valid; ++s) {
        const float lse_s = p.part_lse[s * stride + r];
        if (lse_s == -INFINITY) continue;
        const float wgt = expf(lse_s - m);
        wsum += wgt;
#pragma unroll
        for (int i = 0; i < D / 32; ++i) acc[i] += wgt * p.part_o[(s * stride + r) * D + lane + 32 * i];
      }
    }
    uint16_t* dst = static_cast<uint16_t*>(p.out) + static_cast<size_t>(r) * D;
#pragma unroll
    for (int i = 0; i < D / 32; ++i) {
      const float val = wsum > 0.f ? acc[i] / wsum : 0.f;
      dst[lane + 32 * i] = static_cast<uint16_t>(pack2<BF16>(val, 0.f) & 0xffffu);
    }
    if (p.lse != nullptr && lane == 0) p.lse[r] = wsum > 0.f ? m + logf(wsum) : -INFINITY;
  }
}

// Append of the newest token (position lengths[b] - 1) of every request: row
// (b, kind, head) of new_kv [B, 2, Hkv, D] goes to cache[page][kind][offset][head],
// 16-byte stores, one warp per row.
struct AppendParams {
  const void* new_kv;
  void* cache;
  const int* block_table;
  const int* lengths;
  int* status;
  int B, Hkv, D, page_size, max_pages, num_pages, bad_index_code;
};

__global__ void __launch_bounds__(256) paged_append_kernel(const AppendParams p) {
  grid_launch_dependents();
  grid_dependency_wait();
  const long long rows = static_cast<long long>(p.B) * 2 * p.Hkv;
  const int lane = threadIdx.x % 32;
  const int vecs = p.D / 8;  // 16-byte vectors per row
  for (long long r = static_cast<long long>(blockIdx.x) * 8 + threadIdx.x / 32; r < rows; r += gridDim.x * 8LL) {
    const int b = static_cast<int>(r / (2 * p.Hkv));
    const int kind = static_cast<int>((r / p.Hkv) % 2);
    const int head = static_cast<int>(r % p.Hkv);
    const int token = p.lengths[b] - 1;
    if (token < 0 || token >= p.max_pages * p.page_size) {
      if (lane == 0) atomicExch(p.status, p.bad_index_code);
      continue;
    }
    const int page = p.block_table[static_cast<size_t>(b) * p.max_pages + token / p.page_size];
    if (page < 0 || page >= p.num_pages) {
      if (lane == 0) atomicExch(p.status, p.bad_index_code);
      continue;
    }
    const size_t src = static_cast<size_t>(r) * p.D;
    const size_t dst =
        (((static_cast<size_t>(page) * 2 + kind) * p.page_size + token % p.page_size) * p.Hkv + head) * p.D;
    const uint4* s = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.new_kv) + src);
    uint4* d = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.cache) + dst);
    for (int v = lane; v < vecs; v += 32) d[v] = s[v];
  }
}

}  // namespace eca
