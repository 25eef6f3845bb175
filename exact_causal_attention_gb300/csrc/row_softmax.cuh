// Row softmax of an fp32 M x N matrix, y = exp(x - max) / sum exp(x - max) per
// row, in one pass over HBM when the row fits on chip.  The method is the online
// softmax of the page "Softmax kernels V1-V9" (lpnh.cn/news/2830604): each thread
// keeps a running (m, d) over its elements with one exponential per element
// (section 4.5: e = exp(-|x - m|) serves both branches), states are merged with
// m = max(m1, m2), d = d1 e^(m1 - m) + d2 e^(m2 - m), an empty state (-inf, 0)
// being skipped (section 4.6), across a warp by shuffles and across warps
// through shared memory; then every element is written as exp(x - m) / d.
//
// Schedules (rows contiguous, N elements each):
//   * warp per row (section 4.9's layout), row held in registers: N <= 2048;
//   * 128 threads per row, two rows per block, row held in registers: N <= 4096
//     (a short matrix then still fits in one wave of blocks);
//   * 256-thread block per row, row held in registers: N <= 16384;
//   * 256-thread block per row, two passes over the row: larger N.
// Loads and stores are 16-byte vectors when N is a multiple of 4 (rows then
// start 16-byte aligned), scalar otherwise (the page's N = 257 case).
// Launched with programmatic stream serialisation: each kernel lets the next grid
// launch at once and waits for the grid ahead of it before touching memory.
#pragma once
#include <cstdint>

#include "ptx.cuh"

namespace eca {

struct OnlineMD {
  float m;  // running max
  float d;  // running sum of exp(x - m)
};

// One element into the state (section 4.5's shared exponential).  -inf adds nothing.
__device__ __forceinline__ void md_push(OnlineMD& s, float x) {
  if (x == -INFINITY) return;
  const float e = __expf(-fabsf(x - s.m));  // s.m = -inf gives e = 0
  if (x > s.m) {
    s.d = s.d * e + 1.f;
    s.m = x;
  } else {
    s.d += e;
  }
}

// Merge law of section 4.6 with the empty-state guard.
__device__ __forceinline__ OnlineMD md_merge(OnlineMD a, OnlineMD b) {
  if (b.d == 0.f) return a;
  if (a.d == 0.f) return b;
  const float m = fmaxf(a.m, b.m);
  return OnlineMD{m, a.d * __expf(a.m - m) + b.d * __expf(b.m - m)};
}

__device__ __forceinline__ OnlineMD md_warp_reduce(OnlineMD s) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    OnlineMD o;
    o.m = __shfl_xor_sync(0xffffffffu, s.m, off);
    o.d = __shfl_xor_sync(0xffffffffu, s.d, off);
    s = md_merge(s, o);
  }
  return s;
}

// Merge over each group of WPR consecutive warps of a 256-thread block (one row
// per group), result broadcast to every thread of the group.
template <int WPR>
__device__ __forceinline__ OnlineMD md_block_reduce(OnlineMD s, OnlineMD* smem) {
  s = md_warp_reduce(s);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  __syncthreads();  // smem may still be read from a previous reduction
  if (lane == 0) smem[warp] = s;
  __syncthreads();
  OnlineMD t = lane < WPR ? smem[warp / WPR * WPR + lane] : OnlineMD{-INFINITY, 0.f};
  t = md_warp_reduce(t);
  return t;
}

// Register-cached row softmax: TPR threads per row (32, 128 or 256), ITEMS elements per
// thread, VEC = float4 accesses.  Element e of a thread sits at position
// (k * TPR + tid) * 4 + c for vectors (k = e / 4, c = e % 4), else k * TPR + tid.
template <int TPR, int ITEMS, bool VEC>
__global__ void __launch_bounds__(256) row_softmax_cached(const float* x, float* y, long long M, int N) {
  __shared__ OnlineMD red[8];
  grid_launch_dependents();
  grid_dependency_wait();
  const int tid = threadIdx.x % TPR;
  const int rows_per_block = 256 / TPR;
  const long long row = static_cast<long long>(blockIdx.x) * rows_per_block + threadIdx.x / TPR;
  const bool active = row < M;  // a whole warp shares one row, so this is warp-uniform
  const float* xr = x + (active ? row : 0) * static_cast<long long>(N);
  float* yr = y + (active ? row : 0) * static_cast<long long>(N);
  float v[ITEMS];
  OnlineMD s{-INFINITY, 0.f};
  if (VEC) {
#pragma unroll
    for (int k = 0; k < ITEMS / 4; ++k) {
      const int pos = (k * TPR + tid) * 4;
      float4 f = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      if (active && pos < N) f = *reinterpret_cast<const float4*>(xr + pos);
      v[4 * k] = f.x;
      v[4 * k + 1] = f.y;
      v[4 * k + 2] = f.z;
      v[4 * k + 3] = f.w;
    }
  } else {
#pragma unroll
    for (int k = 0; k < ITEMS; ++k) {
      const int pos = k * TPR + tid;
      v[k] = (active && pos < N) ? xr[pos] : -INFINITY;
    }
  }
#pragma unroll
  for (int e = 0; e < ITEMS; ++e) md_push(s, v[e]);
  s = TPR == 32 ? md_warp_reduce(s) : md_block_reduce<TPR / 32>(s, red);
  if (s.d == 0.f) s.m = 0.f;  // a row of -inf only: written as zeros
  const float inv = s.d > 0.f ? 1.f / s.d : 0.f;
  if (!active) return;
  if (VEC) {
#pragma unroll
    for (int k = 0; k < ITEMS / 4; ++k) {
      const int pos = (k * TPR + tid) * 4;
      if (pos < N) {
        *reinterpret_cast<float4*>(yr + pos) =
            make_float4(__expf(v[4 * k] - s.m) * inv, __expf(v[4 * k + 1] - s.m) * inv,
                        __expf(v[4 * k + 2] - s.m) * inv, __expf(v[4 * k + 3] - s.m) * inv);
      }
    }
  } else {
#pragma unroll
    for (int k = 0; k < ITEMS; ++k) {
      const int pos = k * TPR + tid;
      if (pos < N) yr[pos] = __expf(v[k] - s.m) * inv;
    }
  }
}

// Rows too long for registers: one block per row, a pass for (m, d), a pass to write.
template <bool VEC>
__global__ void __launch_bounds__(256) row_softmax_stream(const float* x, float* y, long long M, int N) {
  __shared__ OnlineMD red[8];
  grid_launch_dependents();
  grid_dependency_wait();
  const long long row = blockIdx.x;
  if (row >= M) return;
  const float* xr = x + row * static_cast<long long>(N);
  float* yr = y + row * static_cast<long long>(N);
  OnlineMD s{-INFINITY, 0.f};
  if (VEC) {
    for (int pos = threadIdx.x * 4; pos < N; pos += 256 * 4) {
      const float4 f = *reinterpret_cast<const float4*>(xr + pos);
      md_push(s, f.x);
      md_push(s, f.y);
      md_push(s, f.z);
      md_push(s, f.w);
    }
  } else {
    for (int pos = threadIdx.x; pos < N; pos += 256) md_push(s, xr[pos]);
  }
  s = md_block_reduce<8>(s, red);
  if (s.d == 0.f) s.m = 0.f;  // a row of -inf only: written as zeros
  const float inv = s.d > 0.f ? 1.f / s.d : 0.f;
  if (VEC) {
    for (int pos = threadIdx.x * 4; pos < N; pos += 256 * 4) {
      const float4 f = *reinterpret_cast<const float4*>(xr + pos);
      *reinterpret_cast<float4*>(yr + pos) = make_float4(__expf(f.x - s.m) * inv, __expf(f.y - s.m) * inv,
                                                         __expf(f.z - s.m) * inv, __expf(f.w - s.m) * inv);
    }
  } else {
    for (int pos = threadIdx.x; pos < N; pos += 256) yr[pos] = __expf(xr[pos] - s.m) * inv;
  }
}

}  // namespace eca
