// Shared-memory ingress probe (a measurement tool, not part of the library): C CTAs,
// one per SM, each stream bytes into a shared-memory ring of 16 KB slots with bulk
// copies (one producer lane issues `cp.async.bulk` into a slot once a consumer warp,
// which does nothing else, has released it).  Two sources: each CTA's own 2 MB of
// HBM with the L2 flushed before every timed launch, and each CTA's own 512 KB read 8
// times over (L2-resident after the first pass).  A second kernel runs the same ring in
// clusters of two CTAs where each CTA fetches half of every slot with a multicast copy
// that lands in both CTAs' shared memory, so each SM receives every byte but issues
// half the requests and the pair reads each byte from L2 once.  Both forms are also run
// with tiled tensor copies (`cp.async.bulk.tensor`, 128-B swizzle, boxes of 64 fp16 columns
// as the attention kernel loads its K and V tiles): 128-row boxes for a CTA alone, 64-row
// boxes multicast to the pair, whose consumers release each slot to the peer with a
// release-ordered remote arrive (as a consumer that read the slot must) or, to time the
// copies alone, a relaxed one.  Every wait is bounded.  Prints one JSON object of GB/s
// received, in all and per SM.  Built and run by `python bench.py --ingress`.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>

namespace {

constexpr int kChunk = 16384;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;
__device__ int g_wait_expired;

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void bar_init(uint32_t b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(b), "r"(count) : "memory");
}

__device__ __forceinline__ bool bar_wait(uint32_t b, uint32_t parity) {
  const unsigned long long t0 = global_ns();
  while (true) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(b), "r"(parity)
        : "memory");
    if (done) return true;
    if (global_ns() - t0 > kWaitLimitNs) {
      atomicExch(&g_wait_expired, 1);
      return false;
    }
  }
}

// Streams `passes` times over this CTA's `bytes_per_cta` of `src`, S slots in flight.
template <int S>
__global__ void __launch_bounds__(64, 1) stream_kernel(const uint8_t* src, size_t bytes_per_cta, int passes) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) unsigned long long bars[2 * S];  // full[S], then empty[S]
  const uint32_t ring = (static_cast<uint32_t>(__cvta_generic_to_shared(smem_raw)) + 1023u) & ~1023u;
  const uint32_t bar0 = static_cast<uint32_t>(__cvta_generic_to_shared(bars));
  if (threadIdx.x == 0) {
    for (int s = 0; s < 2 * S; ++s) bar_init(bar0 + 8u * s, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const int chunks = static_cast<int>(bytes_per_cta / kChunk);
  const int n = chunks * passes;
  const uint8_t* mine = src + static_cast<size_t>(blockIdx.x) * bytes_per_cta;
  if (threadIdx.x == 0) {
    for (int i = 0; i < n; ++i) {
      const int s = i % S;
      const uint32_t full = bar0 + 8u * s, empty = bar0 + 8u * (S + s);
      if (i >= S && !bar_wait(empty, static_cast<uint32_t>((i / S) - 1) & 1u)) break;
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(full), "r"(kChunk) : "memory");
      asm volatile(
          "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
              ring + static_cast<uint32_t>(s * kChunk)),
          "l"(mine + static_cast<size_t>(i % chunks) * kChunk), "r"(kChunk), "r"(full)
          : "memory");
    }
  } else if (threadIdx.x == 32) {
    // Every copy lands before the block can exit: the consumer waits for each one.
    for (int i = 0; i < n; ++i) {
      const int s = i % S;
      if (!bar_wait(bar0 + 8u * s, static_cast<uint32_t>(i / S) & 1u)) break;
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar0 + 8u * (S + s)) : "memory");
    }
  }
  __syncthreads();
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release;\n barrier.cluster.wait.acquire;" ::: "memory");
}

// Clusters of two CTAs stream `passes` times over the pair's `bytes_per_pair` of `src`.  Slot s
// of both CTAs is filled by two multicast copies of kChunk / 2 bytes, one issued by each CTA,
// each completing on the slot's full barrier in both CTAs (which expects kChunk bytes).  A slot
// is refilled only after both CTAs' consumers released it: the empty barriers count two
// arrivals, the CTA's own and the peer's (a remote arrive).
template <int S>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(64, 1)
    multicast_kernel(const uint8_t* src, size_t bytes_per_pair, int passes) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) unsigned long long bars[2 * S];  // full[S], then empty[S]
  constexpr int kHalf = kChunk / 2;
  const uint32_t ring = (static_cast<uint32_t>(__cvta_generic_to_shared(smem_raw)) + 1023u) & ~1023u;
  const uint32_t bar0 = static_cast<uint32_t>(__cvta_generic_to_shared(bars));
  const uint32_t rank = cluster_rank();
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) bar_init(bar0 + 8u * s, 1);
    for (int s = 0; s < S; ++s) bar_init(bar0 + 8u * (S + s), 2);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  cluster_sync();  // the peer's barriers are initialised before any copy or arrive targets them
  const int chunks = static_cast<int>(bytes_per_pair / kChunk);
  const int n = chunks * passes;
  const uint8_t* mine = src + static_cast<size_t>(blockIdx.x / 2) * bytes_per_pair;
  if (threadIdx.x == 0) {
    for (int i = 0; i < n; ++i) {
      const int s = i % S;
      const uint32_t full = bar0 + 8u * s, empty = bar0 + 8u * (S + s);
      if (i >= S && !bar_wait(empty, static_cast<uint32_t>((i / S) - 1) & 1u)) break;
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(full), "r"(kChunk) : "memory");
      const uint16_t both = 0x3;
      asm volatile(
          "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster"
          " [%0], [%1], %2, [%3], %4;" ::"r"(ring + static_cast<uint32_t>(s * kChunk) + rank * kHalf),
          "l"(mine + static_cast<size_t>(i % chunks) * kChunk + rank * kHalf), "r"(kHalf), "r"(full), "h"(both)
          : "memory");
    }
  } else if (threadIdx.x == 32) {
    for (int i = 0; i < n; ++i) {
      const int s = i % S;
      if (!bar_wait(bar0 + 8u * s, static_cast<uint32_t>(i / S) & 1u)) break;
      const uint32_t empty = bar0 + 8u * (S + s);
      uint32_t remote;
      asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(empty), "r"(rank ^ 1u));
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(empty) : "memory");
      asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote) : "memory");
    }
  }
  // On the normal path every copy has landed (both consumers waited for every slot).  After a
  // wait gave up, copies may still be in flight: give them time to land before the exit.
  if (*static_cast<volatile int*>(&g_wait_expired)) {
    const unsigned long long t0 = global_ns();
    while (global_ns() - t0 < 200000ull) {
    }
  }
  cluster_sync();  // neither CTA exits while the peer may still copy or arrive into it
}

template <int S>
float best_ms_multicast(const uint8_t* src, int ctas, size_t per_pair, int passes, uint8_t* flush,
                        size_t flush_bytes, cudaStream_t st) {
  const int smem = S * kChunk + 1024;
  if (cudaFuncSetAttribute(multicast_kernel<S>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
    return -1.f;
  }
  multicast_kernel<S><<<ctas, 64, smem, st>>>(src, per_pair, passes);
  cudaEvent_t a, b;
  cudaEventCreate(&a);
  cudaEventCreate(&b);
  float best = -1.f;
  for (int r = 0; r < 5; ++r) {
    if (flush) cudaMemsetAsync(flush, r, flush_bytes, st);
    cudaEventRecord(a, st);
    multicast_kernel<S><<<ctas, 64, smem, st>>>(src, per_pair, passes);
    cudaEventRecord(b, st);
    if (cudaEventSynchronize(b) != cudaSuccess) {
      best = -1.f;
      break;
    }
    float ms = 0.f;
    cudaEventElapsedTime(&ms, a, b);
    if (best < 0.f || ms < best) best = ms;
  }
  cudaEventDestroy(a);
  cudaEventDestroy(b);
  return best;
}

// Tiled tensor copies over `src` viewed as rows of 64 fp16 (128 bytes): unit u (a CTA, or a
// pair of CTAs with kMulticast) streams `passes` times over its `rows_per_unit` rows, 128 rows
// (16 KB) per slot.  Alone: one 128-row box per slot.  Multicast: CTA rank r loads rows
// 64r..64r+63 of the slot into both CTAs, as in multicast_kernel.
template <int S, bool kMulticast>
__device__ __forceinline__ void tensor_body(const CUtensorMap* tm, int rows_per_unit, int passes, int relaxed) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) unsigned long long bars[2 * S];  // full[S], then empty[S]
  constexpr int kHalf = kChunk / 2;
  const uint32_t ring = (static_cast<uint32_t>(__cvta_generic_to_shared(smem_raw)) + 1023u) & ~1023u;
  const uint32_t bar0 = static_cast<uint32_t>(__cvta_generic_to_shared(bars));
  const uint32_t rank = kMulticast ? cluster_rank() : 0u;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) bar_init(bar0 + 8u * s, 1);
    for (int s = 0; s < S; ++s) bar_init(bar0 + 8u * (S + s), kMulticast ? 2 : 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (kMulticast) {
    cluster_sync();
  } else {
    __syncthreads();
  }
  const int chunks = rows_per_unit / 128;
  const int n = chunks * passes;
  const int row0 = static_cast<int>(kMulticast ? blockIdx.x / 2 : blockIdx.x) * rows_per_unit;
  const uint64_t map = reinterpret_cast<uint64_t>(tm);
  if (threadIdx.x == 0) {
    for (int i = 0; i < n; ++i) {
      const int s = i % S;
      const uint32_t full = bar0 + 8u * s, empty = bar0 + 8u * (S + s);
      if (i >= S && !bar_wait(empty, static_cast<uint32_t>((i / S) - 1) & 1u)) break;
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(full), "r"(kChunk) : "memory");
      const int y = row0 + (i % chunks) * 128;
      if (kMulticast) {
        const uint16_t both = 0x3;
        asm volatile(
            "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster"
            " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(ring + static_cast<uint32_t>(s * kChunk) + rank * kHalf),
            "l"(map), "r"(full), "r"(0), "r"(y + static_cast<int>(rank) * 64), "h"(both)
            : "memory");
      } else {
        asm volatile(
            "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
            " [%0], [%1, {%3, %4}], [%2];" ::"r"(ring + static_cast<uint32_t>(s * kChunk)),
            "l"(map), "r"(full), "r"(0), "r"(y)
            : "memory");
      }
    }
  } else if (threadIdx.x == 32) {
    for (int i = 0; i < n; ++i) {
      const int s = i % S;
      if (!bar_wait(bar0 + 8u * s, static_cast<uint32_t>(i / S) & 1u)) break;
      const uint32_t empty = bar0 + 8u * (S + s);
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(empty) : "memory");
      if (kMulticast) {
        uint32_t remote;
        asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(empty), "r"(rank ^ 1u));
        if (relaxed) {
          asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote) : "memory");
        } else {
          asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote) : "memory");
        }
      }
    }
  }
  if (*static_cast<volatile int*>(&g_wait_expired)) {
    const unsigned long long t0 = global_ns();
    while (global_ns() - t0 < 200000ull) {
    }
  }
  if (kMulticast) {
    cluster_sync();
  } else {
    __syncthreads();
  }
}

template <int S>
__global__ void __launch_bounds__(64, 1) tensor_kernel(const __grid_constant__ CUtensorMap tm, int rows, int passes) {
  tensor_body<S, false>(&tm, rows, passes, 0);
}

template <int S>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(64, 1)
    tensor_multicast_kernel(const __grid_constant__ CUtensorMap tm, int rows, int passes, int relaxed) {
  tensor_body<S, true>(&tm, rows, passes, relaxed);
}

// Best of 5 timed launches of `launch()` (after one untimed), in ms, negative on a CUDA error.
template <typename F>
float best_ms_of(F launch, uint8_t* flush, size_t flush_bytes, cudaStream_t st) {
  launch();
  cudaEvent_t a, b;
  cudaEventCreate(&a);
  cudaEventCreate(&b);
  float best = -1.f;
  for (int r = 0; r < 5; ++r) {
    if (flush) cudaMemsetAsync(flush, r, flush_bytes, st);
    cudaEventRecord(a, st);
    launch();
    cudaEventRecord(b, st);
    if (cudaEventSynchronize(b) != cudaSuccess) {
      best = -1.f;
      break;
    }
    float ms = 0.f;
    cudaEventElapsedTime(&ms, a, b);
    if (best < 0.f || ms < best) best = ms;
  }
  cudaEventDestroy(a);
  cudaEventDestroy(b);
  return best;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// `src` (rows x 128 bytes) as a 2-D fp16 tensor map with boxes of 64 x box_rows, 128-B swizzle.
bool encode_rows(CUtensorMap* tm, void* src, uint64_t rows, uint32_t box_rows) {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || fn == nullptr) {
    return false;
  }
  const cuuint64_t dims[2] = {64, rows};
  const cuuint64_t strides[1] = {128};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return reinterpret_cast<EncodeTiledFn>(fn)(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, src, dims, strides, box, estr,
                                             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int S>
float best_ms_tensor(const CUtensorMap& tm, int mode, int ctas, int rows, int passes, uint8_t* flush,
                     size_t flush_bytes, cudaStream_t st) {
  const int smem = S * kChunk + 1024;
  if (cudaFuncSetAttribute(tensor_kernel<S>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
      cudaFuncSetAttribute(tensor_multicast_kernel<S>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
          cudaSuccess) {
    return -1.f;
  }
  if (mode > 0) {  // 1: multicast, release-ordered remote arrives; 2: relaxed ones
    const int relaxed = mode == 2;
    return best_ms_of([&] { tensor_multicast_kernel<S><<<ctas, 64, smem, st>>>(tm, rows, passes, relaxed); },
                      flush, flush_bytes, st);
  }
  return best_ms_of([&] { tensor_kernel<S><<<ctas, 64, smem, st>>>(tm, rows, passes); }, flush, flush_bytes, st);
}

// Best of 5 timed launches, in ms (negative on a CUDA error); `flush`, if given, is
// rewritten before every timed launch so the source comes from HBM.
template <int S>
float best_ms(const uint8_t* src, int ctas, size_t per_cta, int passes, uint8_t* flush, size_t flush_bytes,
              cudaStream_t st) {
  const int smem = S * kChunk + 1024;
  if (cudaFuncSetAttribute(stream_kernel<S>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
    return -1.f;
  }
  stream_kernel<S><<<ctas, 64, smem, st>>>(src, per_cta, passes);
  cudaEvent_t a, b;
  cudaEventCreate(&a);
  cudaEventCreate(&b);
  float best = -1.f;
  for (int r = 0; r < 5; ++r) {
    if (flush) cudaMemsetAsync(flush, r, flush_bytes, st);
    cudaEventRecord(a, st);
    stream_kernel<S><<<ctas, 64, smem, st>>>(src, per_cta, passes);
    cudaEventRecord(b, st);
    if (cudaEventSynchronize(b) != cudaSuccess) {
      best = -1.f;
      break;
    }
    float ms = 0.f;
    cudaEventElapsedTime(&ms, a, b);
    if (best < 0.f || ms < best) best = ms;
  }
  cudaEventDestroy(a);
  cudaEventDestroy(b);
  return best;
}

void print_rate(const char* key, double bytes, float ms, int ctas, bool last) {
  const double gbs = ms > 0.f ? bytes / (ms * 1e-3) / 1e9 : -1.0;
  std::printf("      \"%s\": {\"GB_s\": %.1f, \"GB_s_per_SM\": %.1f}%s\n", key, gbs, gbs / ctas, last ? "" : ",");
}

}  // namespace

int main() {
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0) != cudaSuccess || sms < 1) return 1;
  const size_t hbm_per_cta = 2ull << 20, l2_per_cta = 512ull << 10, flush_bytes = 256ull << 20;
  uint8_t* src = nullptr;
  uint8_t* flush = nullptr;
  if (cudaMalloc(&src, static_cast<size_t>(sms) * hbm_per_cta) != cudaSuccess ||
      cudaMalloc(&flush, flush_bytes) != cudaSuccess) {
    return 1;
  }
  cudaMemset(src, 1, static_cast<size_t>(sms) * hbm_per_cta);
  cudaStream_t st;
  cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking);
  const int counts[3] = {16, 64, sms};
  std::printf("{\n  \"chunk_bytes\": %d, \"unit\": \"GB/s\",\n", kChunk);
  std::printf("  \"hbm_2MB_per_cta_flushed\": {\n");
  for (int c = 0; c < 3; ++c) {
    const int ctas = counts[c];
    std::printf("    \"%d\": {\n", ctas);
    const double bytes = static_cast<double>(ctas) * hbm_per_cta;
    print_rate("ring_64KB", bytes, best_ms<4>(src, ctas, hbm_per_cta, 1, flush, flush_bytes, st), ctas, false);
    print_rate("ring_192KB", bytes, best_ms<12>(src, ctas, hbm_per_cta, 1, flush, flush_bytes, st), ctas, true);
    std::printf("    }%s\n", c == 2 ? "" : ",");
  }
  std::printf("  },\n  \"l2_resident_512KB_per_cta_8_passes\": {\n");
  for (int c = 0; c < 3; ++c) {
    const int ctas = counts[c];
    std::printf("    \"%d\": {\n", ctas);
    const double bytes = static_cast<double>(ctas) * l2_per_cta * 8;
    print_rate("ring_64KB", bytes, best_ms<4>(src, ctas, l2_per_cta, 8, nullptr, 0, st), ctas, false);
    print_rate("ring_192KB", bytes, best_ms<12>(src, ctas, l2_per_cta, 8, nullptr, 0, st), ctas, true);
    std::printf("    }%s\n", c == 2 ? "" : ",");
  }
  // Pairs of CTAs with multicast: each SM receives the pair's bytes (per pair: 2 MB from HBM, or
  // 512 KB 8 times from L2), so the received total is CTAs x that.
  std::printf("  },\n  \"multicast_pairs_hbm_2MB_per_pair_flushed\": {\n");
  for (int c = 0; c < 3; ++c) {
    const int ctas = counts[c] & ~1;  // whole clusters of two
    std::printf("    \"%d\": {\n", ctas);
    const double bytes = static_cast<double>(ctas) * hbm_per_cta;
    print_rate("ring_64KB", bytes, best_ms_multicast<4>(src, ctas, hbm_per_cta, 1, flush, flush_bytes, st), ctas,
               false);
    print_rate("ring_192KB", bytes, best_ms_multicast<12>(src, ctas, hbm_per_cta, 1, flush, flush_bytes, st), ctas,
               true);
    std::printf("    }%s\n", c == 2 ? "" : ",");
  }
  std::printf("  },\n  \"multicast_pairs_l2_resident_512KB_per_pair_8_passes\": {\n");
  for (int c = 0; c < 3; ++c) {
    const int ctas = counts[c] & ~1;  // whole clusters of two
    std::printf("    \"%d\": {\n", ctas);
    const double bytes = static_cast<double>(ctas) * l2_per_cta * 8;
    print_rate("ring_64KB", bytes, best_ms_multicast<4>(src, ctas, l2_per_cta, 8, nullptr, 0, st), ctas, false);
    print_rate("ring_192KB", bytes, best_ms_multicast<12>(src, ctas, l2_per_cta, 8, nullptr, 0, st), ctas, true);
    std::printf("    }%s\n", c == 2 ? "" : ",");
  }
  // Tiled tensor copies: each CTA's own rows (alone), or each pair's rows multicast (pairs).
  CUtensorMap tm128, tm64;
  const uint64_t total_rows = static_cast<uint64_t>(sms) * hbm_per_cta / 128;
  if (!encode_rows(&tm128, src, total_rows, 128) || !encode_rows(&tm64, src, total_rows, 64)) return 1;
  const int hbm_rows = static_cast<int>(hbm_per_cta / 128), l2_rows = static_cast<int>(l2_per_cta / 128);
  const char* mode_name[3] = {"alone", "multicast_pairs", "multicast_pairs_relaxed_arrive"};
  for (int mc = 0; mc < 3; ++mc) {
    const CUtensorMap& tm = mc ? tm64 : tm128;
    std::printf("  },\n  \"tensor_%s_hbm_2MB_flushed\": {\n", mode_name[mc]);
    for (int c = 0; c < 3; ++c) {
      const int ctas = counts[c] & ~1;
      std::printf("    \"%d\": {\n", ctas);
      const double bytes = static_cast<double>(ctas) * hbm_per_cta;
      print_rate("ring_64KB", bytes, best_ms_tensor<4>(tm, mc, ctas, hbm_rows, 1, flush, flush_bytes, st), ctas, false);
      print_rate("ring_192KB", bytes, best_ms_tensor<12>(tm, mc, ctas, hbm_rows, 1, flush, flush_bytes, st), ctas,
                 true);
      std::printf("    }%s\n", c == 2 ? "" : ",");
    }
    std::printf("  },\n  \"tensor_%s_l2_resident_512KB_8_passes\": {\n", mode_name[mc]);
    for (int c = 0; c < 3; ++c) {
      const int ctas = counts[c] & ~1;
      std::printf("    \"%d\": {\n", ctas);
      const double bytes = static_cast<double>(ctas) * l2_per_cta * 8;
      print_rate("ring_64KB", bytes, best_ms_tensor<4>(tm, mc, ctas, l2_rows, 8, nullptr, 0, st), ctas, false);
      print_rate("ring_192KB", bytes, best_ms_tensor<12>(tm, mc, ctas, l2_rows, 8, nullptr, 0, st), ctas, true);
      std::printf("    }%s\n", c == 2 ? "" : ",");
    }
  }
  int expired = 0;
  cudaMemcpyFromSymbol(&expired, g_wait_expired, sizeof(int));
  std::printf("  },\n  \"wait_expired\": %d\n}\n", expired);
  return (cudaGetLastError() == cudaSuccess && expired == 0) ? 0 : 1;
}
