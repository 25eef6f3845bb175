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
// GB300 mapping: one CTA per (request, K/V head, chunk of HC query heads of the
// group, key segment); 128 threads.  TMA brings each page of one K/V head as a
// (T tokens x 64 dims) box with the 128-byte swizzle into a 3-stage ring of
// 64-token tiles; thread 0 issues the copies.  With M = HC <= 8 query rows the
// arithmetic is far below the tensor-core shapes and the kernel is HBM-bound
// (about 4 FLOP per byte), so scores and P V run on the FP32 pipes:
//   scores: two threads per token row, each converting half of the K row to fp32
//           once and using it for every head of the chunk (one shuffle joins
//           the halves);
//   softmax: one warp per head, lanes over the tile's tokens (shuffle reductions);
//   P V: one thread per column pair and run of tokens, HC packed accumulators,
//        p stored token-major so one vector load serves four heads; the runs'
//        partial sums meet once per unit, in the ring's memory once every copy
//        has been consumed.
// About 73 KB of shared memory, so three CTAs share an SM.
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
constexpr int kDecThreads = 128;
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
};

template <int D>
struct DecodeSmem {
  static constexpr int kKindBytes = kDecTile * D * 2;  // one kind (K or V) of a tile
  static constexpr int kStageBytes = 2 * kKindBytes;
  static constexpr int kRingOff = 0;
  static constexpr int kQOff = kDecStages * kStageBytes;           // fp32 [8][D], pre-scaled query
  static constexpr int kSOff = kQOff + 8 * D * 4;                  // fp32 [8][64] scores
  static constexpr int kPOff = kSOff + 8 * kDecTile * 4;           // fp32 [64][8] p, token-major
  static constexpr int kRedOff = kRingOff;  // fp32 partial outputs (8 KB), over the ring once it is idle
  static constexpr int kIdsOff = kPOff + kDecTile * 8 * 4;         // int32 page-id window
  static constexpr int kStatOff = kIdsOff + kDecIdRing * 4;      // fp32 [8] alpha, [8] m, [8] l
  static constexpr int kBarOff = kStatOff + 3 * 8 * 4;
  static constexpr int kMiscOff = kBarOff + kDecStages * 8;        // abort flag
  static constexpr int kBytes = kMiscOff + 16;
  static constexpr int kDynamicBytes = kBytes + 1024;
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

template <int D, bool BF16, int HC>
__global__ void __launch_bounds__(kDecThreads) paged_decode_kernel(const __grid_constant__ CUtensorMap tm_cache,
                                                                   const DecodeParams p) {
  using L = DecodeSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t sbase = (raw_base + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw_base);
  float* q_s = reinterpret_cast<float*>(smem + L::kQOff);
  float* s_s = reinterpret_cast<float*>(smem + L::kSOff);
  float* p_s = reinterpret_cast<float*>(smem + L::kPOff);
  float* red_s = reinterpret_cast<float*>(smem + L::kRedOff);
  int* ids_s = reinterpret_cast<int*>(smem + L::kIdsOff);
  float* alpha_s = reinterpret_cast<float*>(smem + L::kStatOff);
  float* m_s = alpha_s + 8;
  float* l_s = alpha_s + 16;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff);
  auto bar = [&](int i) -> uint32_t { return sbase + L::kBarOff + 8u * static_cast<uint32_t>(i); };

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

  int len = p.lengths[b];
  if (len < 0 || len > p.max_pages * T) {
    if (tid == 0) atomicExch(p.status, p.bad_index_code);
    len = len < 0 ? 0 : p.max_pages * T;
  }
  const int n_pages = (len + T - 1) >> log2T;
  const int pg_begin = seg * p.seg_pages;
  const int pg_end = min(n_pages, pg_begin + p.seg_pages);
  const int n_tiles = pg_end > pg_begin ? (pg_end - pg_begin + pages_per_tile - 1) / pages_per_tile : 0;

  if (tid == 0) {
    for (int s = 0; s < kDecStages; ++s) mbar_init(bar(s), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  // Page ids of the segment in a rolling window of kDecIdRing slots (slot = page % ring),
  // read from global memory once each; rejected ids become -1.
  auto checked_id = [&](int id) {
    if (id < 0 || id >= p.num_pages) {
      atomicExch(p.status, p.bad_index_code);
      return -1;
    }
    return id;
  };
  const int* table_row = p.block_table + static_cast<size_t>(b) * p.max_pages;
  if (tid < kDecIdRing && pg_begin + tid < pg_end) ids_s[tid] = checked_id(table_row[pg_begin + tid]);
  // query rows of this chunk, scaled by scale * log2(e), in fp32
  const uint16_t* qg = static_cast<const uint16_t*>(p.q) + (static_cast<size_t>(b) * p.Hq + qh0) * D;
  for (int i = tid; i < HC * D; i += kDecThreads) q_s[i] = to_f32<BF16>(qg[i]) * p.scale_log2e;
  if (tid < HC) {
    m_s[tid] = -INFINITY;
    l_s[tid] = 0.f;
  }
  __syncthreads();
  const Watchdog wd{abort_flag, p.status, p.wait_limit_ns, p.timeout_code};

  // Copies of tile i: both kinds of its pages; a page id out of range is not read.
  // Each decode step reads its K/V once: evict-first.
  const uint64_t pol = policy_evict_first();
  auto issue_tile = [&](int i) {
    const int slot = i % kDecStages;
    const uint32_t stage = sbase + L::kRingOff + slot * L::kStageBytes;
    const int first = i * pages_per_tile;  // within the segment
    const int np = min(pages_per_tile, pg_end - pg_begin - first);
    int good = 0;
    for (int pp = 0; pp < np; ++pp) good += ids_s[(first + pp) % kDecIdRing] >= 0 ? 1 : 0;
    mbar_arrive_expect_tx(bar(slot), static_cast<uint32_t>(good * 2 * (D / 64) * T * 128));
    for (int pp = 0; pp < np; ++pp) {
      const int id = ids_s[(first + pp) % kDecIdRing];
      if (id < 0) continue;
      for (int kind = 0; kind < 2; ++kind) {
        for (int h = 0; h < D / 64; ++h) {
          const uint32_t dst = stage + kind * L::kKindBytes + (pp * (D / 64) + h) * T * 128;
          tma_load_3d(dst, &tm_cache, bar(slot), 64 * h, kvh, (id * 2 + kind) * T, pol);
        }
      }
    }
  };

  // Score mapping: two threads per token row, each owning half of the D columns.
  const int s_row = tid >> 1, s_half = tid & 1;
  // P V mapping: one thread per column pair, the tile's 64 tokens split into kTokSplit runs.
  constexpr int kPairs = D / 2;
  constexpr int kTokSplit = kDecThreads / kPairs;  // 2 (D = 128) or 4 (D = 64)
  constexpr int kRun = kDecTile / kTokSplit;
  const int cp = tid % kPairs, run = tid / kPairs;
  float2 acc[HC];
#pragma unroll
  for (int k = 0; k < HC; ++k) acc[k] = make_float2(0.f, 0.f);

  int issued = 0;  // tiles whose copies thread 0 has started
  if (tid == 0) {
    tma_prefetch_map(&tm_cache);
    for (int i = 0; i < kDecStages - 1 && i < n_tiles; ++i) issue_tile(issued++);
  }
  bool ok = true;
  for (int i = 0; i < n_tiles && ok; ++i) {
    // The pages of this tile leave the id window after it; their slots take the pages
    // kDecIdRing further on.  The load starts now and is stored at the end of the tile.
    const int refill = i * pages_per_tile + kDecIdRing + tid;  // within the segment
    const bool refills = tid < pages_per_tile && pg_begin + refill < pg_end;
    const int refill_id = refills ? table_row[pg_begin + refill] : -1;
    if (tid == 0 && i + kDecStages - 1 < n_tiles) issue_tile(issued++);
    const int slot = i % kDecStages;
    const bool got = wd.wait(bar(slot), static_cast<uint32_t>(i / kDecStages) & 1u);
    if (!__syncthreads_and(got)) {
      ok = false;
      break;
    }
    const uint8_t* kt = smem + L::kRingOff + slot * L::kStageBytes;
    const uint8_t* vt = kt + L::kKindBytes;
    const int first_page = pg_begin + i * pages_per_tile;
    const int tok0 = first_page << log2T;  // logical token of tile row 0
    // Rows that hold a token of this segment on an accepted page; the rest (past the
    // length, past the segment, or on a rejected page) are empty.
    uint64_t rows_ok = 0;
    for (int pp = 0; pp < pages_per_tile && first_page + pp < pg_end; ++pp) {
      if (ids_s[(first_page - pg_begin + pp) % kDecIdRing] < 0) continue;
      const int lo = pp << log2T, hi = min((pp + 1) << log2T, len - tok0);
      if (hi > lo) rows_ok |= (hi - lo == 64 ? ~0ull : ((1ull << (hi - lo)) - 1)) << lo;
    }

    // scores s = q . k in the base-2 domain: this thread's half row of K, converted once,
    // against every head of the chunk; the two halves meet through one shuffle.
    {
      const bool live = (rows_ok >> s_row) & 1ull;
      float kf[D / 2];
      if (live) {
#pragma unroll
        for (int c = 0; c < D / 16; ++c) {
          const uint4 w = *reinterpret_cast<const uint4*>(kt + dec_chunk_offset<D>(s_row, s_half * (D / 16) + c, log2T));
          const float2 a = to_f32x2<BF16>(w.x), bb = to_f32x2<BF16>(w.y), cc = to_f32x2<BF16>(w.z),
                       dd = to_f32x2<BF16>(w.w);
          kf[8 * c + 0] = a.x;
          kf[8 * c + 1] = a.y;
          kf[8 * c + 2] = bb.x;
          kf[8 * c + 3] = bb.y;
          kf[8 * c + 4] = cc.x;
          kf[8 * c + 5] = cc.y;
          kf[8 * c + 6] = dd.x;
          kf[8 * c + 7] = dd.y;
        }
      } else {
#pragma unroll
        for (int e = 0; e < D / 2; ++e) kf[e] = 0.f;
      }
#pragma unroll
      for (int k = 0; k < HC; ++k) {
        const float4* qq = reinterpret_cast<const float4*>(q_s + k * D + s_half * (D / 2));
        float2 a2 = make_float2(0.f, 0.f), b2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int e = 0; e < D / 8; ++e) {
          const float4 qv = qq[e];
          a2 = __ffma2_rn(make_float2(qv.x, qv.y), make_float2(kf[4 * e], kf[4 * e + 1]), a2);
          b2 = __ffma2_rn(make_float2(qv.z, qv.w), make_float2(kf[4 * e + 2], kf[4 * e + 3]), b2);
        }
        float dot = (a2.x + a2.y) + (b2.x + b2.y);
        dot += __shfl_xor_sync(0xffffffffu, dot, 1);
        if (s_half == 0) s_s[k * kDecTile + s_row] = live ? dot : -INFINITY;
      }
    }
    __syncthreads();

    // online softmax, one warp per head: m' = max(m, max s), p = 2^(s - m'), l' = l 2^(m - m') + sum p
    for (int qh = warp; qh < HC; qh += kDecThreads / 32) {
      const float s0 = s_s[qh * kDecTile + lane], s1 = s_s[qh * kDecTile + lane + 32];
      float mx = fmaxf(s0, s1);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float m_old = m_s[qh];
      const float m_new = fmaxf(m_old, mx);
      const float p0 = m_new == -INFINITY ? 0.f : ex2(s0 - m_new);
      const float p1 = m_new == -INFINITY ? 0.f : ex2(s1 - m_new);
      float sum = p0 + p1;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
      const float alpha = m_old == -INFINITY ? 0.f : ex2(m_old - m_new);
      p_s[lane * 8 + qh] = p0;
      p_s[(lane + 32) * 8 + qh] = p1;
      __syncwarp();
      if (lane == 0) {
        alpha_s[qh] = alpha;
        m_s[qh] = m_new;
        l_s[qh] = l_s[qh] * alpha + sum;
      }
    }
    __syncthreads();

    // o = alpha o + sum_r p_r v_r: this thread's column pair over its run of rows.
    // Empty rows are skipped (their V is never read: its data may not be a number).
#pragma unroll
    for (int k = 0; k < HC; ++k) {
      const float al = alpha_s[k];
      acc[k] = __fmul2_rn(acc[k], make_float2(al, al));
    }
    const int c = (2 * cp) >> 3, within = ((2 * cp) & 7) * 2;  // 16-byte chunk and byte inside it
    const uint64_t run_mask = (rows_ok >> (run * kRun)) & ((kRun == 64 ? ~0ull : (1ull << kRun) - 1));
    if (run_mask == (kRun == 64 ? ~0ull : (1ull << kRun) - 1)) {
#pragma unroll 4
      for (int j = 0; j < kRun; ++j) {
        const int r = run * kRun + j;
        const float2 v = to_f32x2<BF16>(*reinterpret_cast<const uint32_t*>(vt + dec_chunk_offset<D>(r, c, log2T) + within));
        const float4* pp = reinterpret_cast<const float4*>(p_s + r * 8);
        const float4 pa = pp[0];
        const float pr[8] = {pa.x, pa.y, pa.z, pa.w, 0.f, 0.f, 0.f, 0.f};
        float4 pb = make_float4(0.f, 0.f, 0.f, 0.f);
        if (HC > 4) pb = pp[1];
#pragma unroll
        for (int k = 0; k < HC; ++k) {
          const float pk = k < 4 ? pr[k] : (k == 4 ? pb.x : (k == 5 ? pb.y : (k == 6 ? pb.z : pb.w)));
          acc[k] = __ffma2_rn(make_float2(pk, pk), v, acc[k]);
        }
      }
    } else {
      for (int j = 0; j < kRun; ++j) {
        if (!((run_mask >> j) & 1ull)) continue;
        const int r = run * kRun + j;
        const float2 v = to_f32x2<BF16>(*reinterpret_cast<const uint32_t*>(vt + dec_chunk_offset<D>(r, c, log2T) + within));
#pragma unroll
        for (int k = 0; k < HC; ++k) {
          const float pk = p_s[r * 8 + k];
          acc[k] = __ffma2_rn(make_float2(pk, pk), v, acc[k]);
        }
      }
    }
    if (refills) ids_s[refill % kDecIdRing] = checked_id(refill_id);
    __syncthreads();  // the stage, the scores and p may be overwritten now
  }

  if (ok) {
    // the runs' partial outputs meet in shared memory, then O = o / l and
    // lse = (m + log2 l) ln 2; an empty context gives O = 0 and lse = -inf
    if (run > 0) {
#pragma unroll
      for (int k = 0; k < HC; ++k)
        *reinterpret_cast<float2*>(red_s + ((run - 1) * 8 + k) * D + 2 * cp) = acc[k];
    }
    __syncthreads();
    if (run == 0) {
#pragma unroll
      for (int k = 0; k < HC; ++k) {
        float2 o = acc[k];
        for (int rr = 1; rr < kTokSplit; ++rr) {
          const float2 part = *reinterpret_cast<const float2*>(red_s + ((rr - 1) * 8 + k) * D + 2 * cp);
          o.x += part.x;
          o.y += part.y;
        }
        const float l = l_s[k];
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const size_t row = static_cast<size_t>(b) * p.Hq + qh0 + k;
        if (p.part_o != nullptr) {
          *reinterpret_cast<float2*>(p.part_o + (static_cast<size_t>(seg) * p.B * p.Hq + row) * D + 2 * cp) =
              make_float2(o.x * inv, o.y * inv);
        } else {
          *reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(p.out) + row * D + 2 * cp) = pack2<BF16>(o.x * inv, o.y * inv);
        }
        if (cp == 0) {
          const float lse = l > 0.f ? (m_s[k] + log2f(l)) * 0.69314718055994530942f : -INFINITY;
          if (p.part_o != nullptr) {
            p.part_lse[static_cast<size_t>(seg) * p.B * p.Hq + row] = lse;
          } else if (p.lse != nullptr) {
            p.lse[row] = lse;
          }
        }
      }
    }
  }
  // let every copy thread 0 issued land before the block exits
  if (tid == 0) {
    for (int i = (issued > kDecStages ? issued - kDecStages : 0); i < issued; ++i) {
      wd.drain(bar(i % kDecStages), static_cast<uint32_t>(i / kDecStages) & 1u);
    }
  }
  __syncthreads();
}

// Merge of the decode segments (section 6.4 of the page, in log-sum-exp form as in
// the prefill merge): rows are (b, query head); segment s is non-empty when its
// first logical page is below the request's page count.
template <int D, bool BF16>
__global__ void __launch_bounds__(256) paged_decode_combine(const DecodeParams p) {
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
