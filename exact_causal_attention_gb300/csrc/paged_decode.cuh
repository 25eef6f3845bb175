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
//   scores: one thread per (head, token) dot product, reading the swizzled K row;
//   softmax: one warp per head, lanes over the tile's tokens (shuffle reductions);
//   P V: one thread per output column, HC accumulators in registers.
// Page ids outside [0, P) and lengths outside [0, max_pages * T] are not read:
// the kernel records ATTN_ERR_BAD_INDEX in the status word and treats them as
// empty.
#pragma once
#include <cuda.h>
#include <cstdint>

#include "ptx.cuh"

namespace eca {

constexpr int kDecTile = 64;     // tokens per tile
constexpr int kDecStages = 3;
constexpr int kDecThreads = 128;

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
  static constexpr int kSOff = kQOff + 8 * D * 4;                  // fp32 [8][64] scores, then p
  static constexpr int kStatOff = kSOff + 8 * kDecTile * 4;        // fp32 [8] alpha, [8] m, [8] l
  static constexpr int kBarOff = kStatOff + 3 * 8 * 4;
  static constexpr int kMiscOff = kBarOff + kDecStages * 8;        // abort flag
  static constexpr int kBytes = kMiscOff + 16;
  static constexpr int kDynamicBytes = kBytes + 1024;
};

// Element d of token row r of a tile kind (K or V) staged as swizzled T x 64 boxes.
template <int D>
__device__ __forceinline__ int dec_elem_offset(int r, int d, int T) {
  const int page = r / T, rr = r % T, half = d / 64, c = (d % 64) / 8;
  const int box = page * (D / 64) + half;
  return box * T * 128 + rr * 128 + ((c ^ (rr % 8)) * 16) + (d % 8) * 2;  // bytes
}

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
  const int pages_per_tile = kDecTile / T;

  int len = p.lengths[b];
  if (len < 0 || len > p.max_pages * T) {
    if (tid == 0) atomicExch(p.status, p.bad_index_code);
    len = len < 0 ? 0 : p.max_pages * T;
  }
  const int n_pages = (len + T - 1) / T;
  const int pg_begin = seg * p.seg_pages;
  const int pg_end = min(n_pages, pg_begin + p.seg_pages);
  const int n_tiles = pg_end > pg_begin ? (pg_end - pg_begin + pages_per_tile - 1) / pages_per_tile : 0;

  if (tid == 0) {
    for (int s = 0; s < kDecStages; ++s) mbar_init(bar(s), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
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
    const int first = pg_begin + i * pages_per_tile;
    const int np = min(pages_per_tile, pg_end - first);
    int good = 0;
    int ids[kDecTile / 8];
    for (int pp = 0; pp < np; ++pp) {
      const int id = p.block_table[static_cast<size_t>(b) * p.max_pages + first + pp];
      if (id < 0 || id >= p.num_pages) {
        atomicExch(p.status, p.bad_index_code);
        ids[pp] = -1;
      } else {
        ids[pp] = id;
        ++good;
      }
    }
    mbar_arrive_expect_tx(bar(slot), static_cast<uint32_t>(good * 2 * (D / 64) * T * 128));
    for (int pp = 0; pp < np; ++pp) {
      if (ids[pp] < 0) continue;
      for (int kind = 0; kind < 2; ++kind) {
        for (int h = 0; h < D / 64; ++h) {
          const uint32_t dst = stage + kind * L::kKindBytes + (pp * (D / 64) + h) * T * 128;
          tma_load_3d(dst, &tm_cache, bar(slot), 64 * h, kvh, (ids[pp] * 2 + kind) * T, pol);
        }
      }
    }
  };

  float o[HC];
#pragma unroll
  for (int k = 0; k < HC; ++k) o[k] = 0.f;
  constexpr int kColsPerPass = D;                      // one output column per thread per head set
  constexpr int kHeadSets = kDecThreads / kColsPerPass;  // 1 (D = 128) or 2 (D = 64)
  const int col = tid % D;
  const int hset = tid / D;

  int issued = 0;  // tiles whose copies thread 0 has started
  if (tid == 0) {
    tma_prefetch_map(&tm_cache);
    for (int i = 0; i < kDecStages - 1 && i < n_tiles; ++i) issue_tile(issued++);
  }
  bool ok = true;
  for (int i = 0; i < n_tiles && ok; ++i) {
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
    const int tok0 = first_page * T;  // logical token of tile row 0
    // Rows that hold a token of this segment on an accepted page; the rest (past the
    // length, past the segment, or on a rejected page) are empty.
    uint64_t rows_ok = 0;
    for (int pp = 0; pp < pages_per_tile && first_page + pp < pg_end; ++pp) {
      const int id = p.block_table[static_cast<size_t>(b) * p.max_pages + first_page + pp];
      if (id < 0 || id >= p.num_pages) continue;
      const int lo = pp * T, hi = min((pp + 1) * T, len - tok0);
      for (int r = lo; r < hi; ++r) rows_ok |= 1ull << r;
    }
    auto row_ok = [&](int r) { return ((rows_ok >> r) & 1ull) != 0; };

    // scores: s = q . k (already in the base-2 domain)
    for (int w = tid; w < HC * kDecTile; w += kDecThreads) {
      const int qh = w / kDecTile, r = w % kDecTile;
      float acc = 0.f;
      if (row_ok(r)) {
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
          const uint4 kv = *reinterpret_cast<const uint4*>(kt + dec_elem_offset<D>(r, c * 8, T));
          const float* qq = q_s + qh * D + c * 8;
          const float2 k0 = to_f32x2<BF16>(kv.x), k1 = to_f32x2<BF16>(kv.y);
          const float2 k2 = to_f32x2<BF16>(kv.z), k3 = to_f32x2<BF16>(kv.w);
          acc = fmaf(qq[0], k0.x, acc);
          acc = fmaf(qq[1], k0.y, acc);
          acc = fmaf(qq[2], k1.x, acc);
          acc = fmaf(qq[3], k1.y, acc);
          acc = fmaf(qq[4], k2.x, acc);
          acc = fmaf(qq[5], k2.y, acc);
          acc = fmaf(qq[6], k3.x, acc);
          acc = fmaf(qq[7], k3.y, acc);
        }
      } else {
        acc = -INFINITY;
      }
      s_s[qh * kDecTile + r] = acc;
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
      s_s[qh * kDecTile + lane] = p0;
      s_s[qh * kDecTile + lane + 32] = p1;
      __syncwarp();
      if (lane == 0) {
        alpha_s[qh] = alpha;
        m_s[qh] = m_new;
        l_s[qh] = l_s[qh] * alpha + sum;
      }
    }
    __syncthreads();

    // o = alpha o + sum_r p_r v_r for this thread's column; rows with p = 0 are skipped
    // (an empty row's V is never read: its data may not be a number).
#pragma unroll
    for (int k = 0; k < HC; ++k) {
      if (k % kHeadSets == hset) o[k] *= alpha_s[k];
    }
    for (int r = 0; r < kDecTile; ++r) {
      if (!row_ok(r)) continue;
      const float v = to_f32<BF16>(*reinterpret_cast<const uint16_t*>(vt + dec_elem_offset<D>(r, col, T)));
#pragma unroll
      for (int k = 0; k < HC; ++k) {
        if (k % kHeadSets == hset) o[k] = fmaf(s_s[k * kDecTile + r], v, o[k]);
      }
    }
    __syncthreads();  // the stage and the scores may be overwritten now
  }

  if (ok) {
    // epilogue: O = o / l, lse = (m + log2 l) ln 2; an empty context gives O = 0, lse = -inf
#pragma unroll
    for (int k = 0; k < HC; ++k) {
      if (k % kHeadSets != hset) continue;
      const float l = l_s[k];
      const float val = l > 0.f ? o[k] / l : 0.f;
      const size_t row = static_cast<size_t>(b) * p.Hq + qh0 + k;
      if (p.part_o != nullptr) {
        p.part_o[(static_cast<size_t>(seg) * p.B * p.Hq + row) * D + col] = val;
      } else {
        uint16_t* dst = static_cast<uint16_t*>(p.out) + row * D + col;
        const uint32_t packed = pack2<BF16>(val, 0.f);
        *dst = static_cast<uint16_t>(packed & 0xffffu);
      }
      if (col == 0) {
        const float lse = l > 0.f ? (m_s[k] + log2f(l)) * 0.69314718055994530942f : -INFINITY;
        if (p.part_o != nullptr) {
          p.part_lse[static_cast<size_t>(seg) * p.B * p.Hq + row] = lse;
        } else if (p.lse != nullptr) {
          p.lse[row] = lse;
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
