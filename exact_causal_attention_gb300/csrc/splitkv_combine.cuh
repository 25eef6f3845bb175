// Merge of key-split partial results ("CUDA KV Cache：分页存储与长上下文 Decode
// 极致优化", chengzipai.xyz, section 6.4): segment s of a row holds its
// normalised output O_s = o_s / l_s and lse_s = m_s + ln l_s.  The page's merge
//     m = max_s m_s,  l = sum_s l_s e^(m_s - m),  o = sum_s o_s e^(m_s - m),  O = o / l
// is, in these terms, lse = ln sum_s e^(lse_s) and O = sum_s e^(lse_s - lse) O_s
// (l_s e^(m_s - m) / l = e^(lse_s - lse)).  HBM-bound: one warp per query row,
// each lane holding D/32 consecutive columns.
#pragma once
#include <cstdint>

#include "ptx.cuh"

namespace eca {

struct CombineParams {
  const float* part_o;    // [splits, BH, N, D]
  const float* part_lse;  // [splits, BH, N]
  void* o;                // [BH, N, D] 16-bit
  float* lse;             // [BH, N] or null
  int BH;
  int N;
  int n_tiles;    // key tiles of the sequence
  int seg_tiles;  // key tiles per segment
  int splits;
  int causal;
};

template <int D, bool BF16>
__global__ void __launch_bounds__(256) splitkv_combine_kernel(const CombineParams p) {
  constexpr int kPer = D / 32;  // columns per lane: 4 (D = 128) or 2 (D = 64)
  // Launched with programmatic serialisation right behind the attention kernel
  // that writes the partials: read none before that grid has finished.
  grid_dependency_wait();
  const int lane = threadIdx.x % 32;
  const long long rows = static_cast<long long>(p.BH) * p.N;
  const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x / 32);
  for (long long r = static_cast<long long>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32; r < rows;
       r += warps) {
    const int row = static_cast<int>(r % p.N);
    // Segments holding at least one key this row's 128-row query tile looks at.
    const int need = p.causal ? row / 128 + 1 : p.n_tiles;
    const int valid = (need + p.seg_tiles - 1) / p.seg_tiles < p.splits ? (need + p.seg_tiles - 1) / p.seg_tiles
                                                                         : p.splits;
    const size_t stride = static_cast<size_t>(p.BH) * p.N;  // between segments, in rows
    float m = -INFINITY;
    for (int s = 0; s < valid; ++s) m = fmaxf(m, p.part_lse[s * stride + r]);
    float acc[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) acc[i] = 0.f;
    float wsum = 0.f;
    for (int s = 0; s < valid; ++s) {
      const float wgt = expf(p.part_lse[s * stride + r] - m);
      wsum += wgt;
      const float* src = p.part_o + (s * stride + r) * D + lane * kPer;
      if constexpr (kPer == 4) {
        const float4 v = *reinterpret_cast<const float4*>(src);
        acc[0] += wgt * v.x;
        acc[1] += wgt * v.y;
        acc[2] += wgt * v.z;
        acc[3] += wgt * v.w;
      } else {
        const float2 v = *reinterpret_cast<const float2*>(src);
        acc[0] += wgt * v.x;
        acc[1] += wgt * v.y;
      }
    }
    const float inv = 1.f / wsum;
    uint16_t* dst = static_cast<uint16_t*>(p.o) + static_cast<size_t>(r) * D + lane * kPer;
    if constexpr (kPer == 4) {
      *reinterpret_cast<uint2*>(dst) = make_uint2(pack2<BF16>(acc[0] * inv, acc[1] * inv),
                                                  pack2<BF16>(acc[2] * inv, acc[3] * inv));
    } else {
      *reinterpret_cast<uint32_t*>(dst) = pack2<BF16>(acc[0] * inv, acc[1] * inv);
    }
    if (p.lse != nullptr && lane == 0) p.lse[r] = m + logf(wsum);
  }
}

}  // namespace eca
