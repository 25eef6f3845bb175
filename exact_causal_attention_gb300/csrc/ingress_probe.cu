// Shared-memory ingress probe (a measurement tool, not part of the library): C CTAs,
// one per SM, each stream bytes into a shared-memory ring of 16 KB slots with bulk
// copies (one producer lane issues `cp.async.bulk` into a slot once a consumer warp,
// which does nothing else, has released it).  Two sources: each CTA's own 2 MB of
// HBM with the L2 flushed before every timed launch, and each CTA's own 512 KB read 8
// times over (L2-resident after the first pass).  Every wait is bounded.  Prints one
// JSON object of GB/s, in all and per SM.  Built and run by `python bench.py --ingress`.
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
  int expired = 0;
  cudaMemcpyFromSymbol(&expired, g_wait_expired, sizeof(int));
  std::printf("  },\n  \"wait_expired\": %d\n}\n", expired);
  return (cudaGetLastError() == cudaSuccess && expired == 0) ? 0 : 1;
}
