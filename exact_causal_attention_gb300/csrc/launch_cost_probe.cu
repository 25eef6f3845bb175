// Launch-cost probe (a measurement tool, not part of the library): the time per
// launch of empty 384-thread kernels, one CTA per SM, launched back to back on one
// stream behind a spinning kernel and timed with CUDA events.  The kernels differ
// only in whether they store to global memory (one word per CTA) and whether they
// allocate tensor memory (512 columns, as the attention kernel does); each is
// launched in plain stream order, with programmatic dependent launch (the kernel
// waits for the grid ahead of it first and lets the next one start at once), and
// from a CUDA graph.  Prints one JSON object.  Built and run by
// `python bench.py --launch-cost`.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>

namespace {

constexpr int kMaxCtas = 1024;
constexpr int kLaunches = 200;
constexpr int kSmemBytes = 225 * 1024;  // reserved only (one CTA per SM), never touched

__device__ int g_out[kMaxCtas];

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

template <bool kWrite, bool kTmem, bool kPdl>
__global__ void __launch_bounds__(384, 1) probe_kernel(int flag) {
  __shared__ uint32_t tmem_base;
  if (kPdl) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  }
  const int warp = threadIdx.x / 32;
  if (kTmem && warp == 9) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(&tmem_base))),
                 "r"(512)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  if (kTmem && warp == 9) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(512) : "memory");
  }
  if (kWrite && threadIdx.x == 0 && blockIdx.x < kMaxCtas) g_out[blockIdx.x] = flag;
}

__global__ void spin_kernel(unsigned long long ns) {
  const unsigned long long t0 = global_ns();
  while (global_ns() - t0 < ns) {
  }
}

template <bool kWrite, bool kTmem, bool kPdl>
cudaError_t launch_one(int grid, cudaStream_t s, int flag) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(384);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = kPdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, probe_kernel<kWrite, kTmem, kPdl>, flag);
}

// Microseconds per launch, or a negative value on a CUDA error.
template <bool kWrite, bool kTmem, bool kPdl>
double us_per_launch(int grid, cudaStream_t s, bool graph) {
  if (cudaFuncSetAttribute(probe_kernel<kWrite, kTmem, kPdl>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kSmemBytes) != cudaSuccess) {
    return -1;
  }
  if (launch_one<kWrite, kTmem, kPdl>(grid, s, 0) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess) {
    return -1;
  }
  cudaGraphExec_t exec = nullptr;
  if (graph) {
    cudaGraph_t g = nullptr;
    if (cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal) != cudaSuccess) return -1;
    for (int i = 0; i < kLaunches; ++i) launch_one<kWrite, kTmem, kPdl>(grid, s, i);
    if (cudaStreamEndCapture(s, &g) != cudaSuccess || cudaGraphInstantiate(&exec, g, 0) != cudaSuccess) return -1;
    cudaGraphDestroy(g);
    if (cudaGraphLaunch(exec, s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess) return -1;
  }
  cudaEvent_t e0, e1;
  cudaEventCreate(&e0);
  cudaEventCreate(&e1);
  spin_kernel<<<1, 32, 0, s>>>(300000ull);  // every launch below is queued before the first runs
  cudaEventRecord(e0, s);
  if (graph) {
    cudaGraphLaunch(exec, s);
  } else {
    for (int i = 0; i < kLaunches; ++i) launch_one<kWrite, kTmem, kPdl>(grid, s, i);
  }
  cudaEventRecord(e1, s);
  double us = -1;
  if (cudaStreamSynchronize(s) == cudaSuccess) {
    float ms = 0;
    cudaEventElapsedTime(&ms, e0, e1);
    us = ms * 1000.0 / kLaunches;
  }
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (exec) cudaGraphExecDestroy(exec);
  return us;
}

template <bool kWrite, bool kTmem>
void row(const char* name, int grid, cudaStream_t s, bool last) {
  std::printf("    \"%s\": {\"stream\": %.2f, \"programmatic\": %.2f, \"graph\": %.2f}%s\n", name,
              us_per_launch<kWrite, kTmem, false>(grid, s, false), us_per_launch<kWrite, kTmem, true>(grid, s, false),
              us_per_launch<kWrite, kTmem, false>(grid, s, true), last ? "" : ",");
}

}  // namespace

int main() {
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0) != cudaSuccess || sms < 1 || sms > kMaxCtas) {
    std::printf("{\"error\": \"no usable device\"}\n");
    return 1;
  }
  cudaStream_t s;
  cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking);
  std::printf("{\n  \"ctas\": %d, \"launches\": %d, \"unit\": \"us per launch\",\n  \"kernels\": {\n", sms, kLaunches);
  row<false, false>("no store, no tensor memory", sms, s, false);
  row<true, false>("one store per CTA", sms, s, false);
  row<false, true>("tensor memory allocated", sms, s, false);
  row<true, true>("both", sms, s, true);
  std::printf("  }\n}\n");
  return cudaGetLastError() == cudaSuccess ? 0 : 1;
}
