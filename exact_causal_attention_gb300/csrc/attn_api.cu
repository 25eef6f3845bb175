// Host side of the C ABI declared in include/attn.h: argument checks, TMA tensor
// maps, launch on the caller's stream, and the device status word.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <functional>
#include <mutex>
#include <queue>
#include <utility>
#include <vector>

#include "attn.h"
#include "attn_fwd_kernel.cuh"
#include "paged_decode.cuh"
#include "row_softmax.cuh"
#include "splitkv_combine.cuh"

// Scratch of attn_fwd_splitkv_noalloc: one fixed array per device that loads this
// library, held until the process exits.  In host code this name only stands for
// the device array; its device address comes from cudaGetSymbolAddress.
constexpr unsigned long long kNoAllocScratchBytes = 64ull << 20;
static __device__ __align__(256) unsigned char g_splitkv_scratch[kNoAllocScratchBytes];

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxSplits = 64;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s per single wait

// Device status word: 0, or the code of the last bounded wait that gave up.
__device__ int g_device_status = 0;

// Work counters of the attention kernel, one 256-byte slot per launch, taken in
// turn: a launch hands its units out from slot[0] and counts finished CTAs in
// slot[32]; its last CTA sets both back to zero.  A slot is handed to a new
// launch only after the launch that last held it has finished: the new launch
// waits on the GPU for an event recorded after the old one (see SlotGuard), so
// more than 64 launches in flight at once queue up instead of sharing counters.
constexpr int kSchedSlots = 64;
__device__ int g_sched_pool[kSchedSlots * 64] = {};

// Counters of the paged decode's fused segment merge: one per (request, K/V head,
// head chunk), zero between launches (each group's last segment resets its
// counter).  Slots are taken in turn, guarded like the attention kernel's, so up
// to 8 launches run at once and a ninth waits for the first; larger launches use
// the separate merge kernel.
constexpr int kDecCounterSlots = 8;
constexpr int kDecCountersPerSlot = 4096;
__device__ unsigned g_dec_counters[kDecCounterSlots * kDecCountersPerSlot] = {};

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// Order of reuse of a pool of counter slots: before a launch takes a slot, its
// stream waits for the event recorded after the slot's previous launch (a no-op
// once that launch has finished), and the event is recorded again after the new
// launch.  Under stream capture no event is used: the slot is fixed in the
// graph when captured.
template <int kSlots>
struct SlotGuard {
  cudaEvent_t done[kSlots] = {};
  bool recorded[kSlots] = {};
  unsigned next = 0;

  // Takes the next slot for a launch on `stream`; ATTN_ERR_CUDA if an event call fails.
  int acquire(cudaStream_t stream, unsigned* slot, bool* capturing) {
    *slot = next++ % kSlots;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return ATTN_ERR_CUDA;
    *capturing = cs != cudaStreamCaptureStatusNone;
    if (*capturing || !recorded[*slot]) return ATTN_OK;
    return cudaStreamWaitEvent(stream, done[*slot], 0) == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
  }

  // Marks the slot busy until the work enqueued so far on `stream` has finished.
  int release(cudaStream_t stream, unsigned slot, bool capturing) {
    if (capturing) return ATTN_OK;
    if (done[slot] == nullptr && cudaEventCreateWithFlags(&done[slot], cudaEventDisableTiming) != cudaSuccess) {
      return ATTN_ERR_CUDA;
    }
    if (cudaEventRecord(done[slot], stream) != cudaSuccess) return ATTN_ERR_CUDA;
    recorded[slot] = true;
    return ATTN_OK;
  }
};

// Tensor maps already encoded, keyed by everything the encoding reads (address,
// element type and the [BH, N, D] extents with the box height), so a hit is
// exactly the map a new encoding would produce, whatever the caller freed or
// reallocated in between.  Least recently used entries are replaced.
struct MapCache {
  struct Entry {
    const void* ptr;
    uint64_t shape;  // D, N, BH, box rows, element type packed
    int BH;
    unsigned long long last_use;
    CUtensorMap map;
  };
  static constexpr int kEntries = 32;
  Entry e[kEntries] = {};
  unsigned long long clock = 0;

  static uint64_t pack(bool bf16, int D, int N, unsigned box_rows) {
    return (static_cast<uint64_t>(static_cast<uint32_t>(N)) << 32) | (static_cast<uint64_t>(D) << 16) |
           (static_cast<uint64_t>(box_rows) << 1) | (bf16 ? 1u : 0u);
  }
  // The cached map, or nullptr.
  const CUtensorMap* find(const void* ptr, uint64_t shape, int BH) {
    for (Entry& x : e) {
      if (x.last_use != 0 && x.ptr == ptr && x.shape == shape && x.BH == BH) {
        x.last_use = ++clock;
        return &x.map;
      }
    }
    return nullptr;
  }
  void insert(const void* ptr, uint64_t shape, int BH, const CUtensorMap& map) {
    Entry* victim = &e[0];
    for (Entry& x : e) {
      if (x.last_use < victim->last_use) victim = &x;
    }
    victim->ptr = ptr;
    victim->shape = shape;
    victim->BH = BH;
    victim->map = map;
    victim->last_use = ++clock;
  }
};

struct DeviceState {
  bool probed = false;
  bool sm103 = false;
  int sm_count = 0;
  int* status = nullptr;    // address of g_device_status on this device
  void* scratch = nullptr;  // address of g_splitkv_scratch on this device, set by its first use
  int* sched_pool = nullptr;  // address of g_sched_pool on this device
  SlotGuard<kSchedSlots> sched_slots;  // slots of the launches that take units from a counter
  unsigned* dec_counters = nullptr;  // address of g_dec_counters on this device
  SlotGuard<kDecCounterSlots> dec_slots;  // slots of the split decode launches that merge in the kernel
  MapCache maps;           // q/k/v/o tensor maps of recent attention launches
  unsigned configured = 0;  // bitmask of kernel instantiations with smem attribute set
  unsigned configured_decode = 0;
};

std::mutex g_mutex;
DeviceState g_devices[kMaxDevices];
EncodeTiledFn g_encode = nullptr;

int get_encode_fn(EncodeTiledFn* out) {
  if (g_encode == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr) {
      return ATTN_ERR_CUDA;
    }
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  *out = g_encode;
  return ATTN_OK;
}

// Per-device checks and the status word's device address; call with g_mutex held.
int device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  DeviceState& st = g_devices[dev];
  if (!st.probed) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
      return ATTN_ERR_CUDA;
    }
    st.sm103 = (major == 10 && minor == 3);
    if (cudaDeviceGetAttribute(&st.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        st.sm_count < 1) {
      return ATTN_ERR_CUDA;
    }
    if (st.sm103) {
      void* addr = nullptr;
      if (cudaGetSymbolAddress(&addr, g_device_status) != cudaSuccess) return ATTN_ERR_CUDA;
      st.status = static_cast<int*>(addr);
      if (cudaGetSymbolAddress(&addr, g_sched_pool) != cudaSuccess) return ATTN_ERR_CUDA;
      st.sched_pool = static_cast<int*>(addr);
      if (cudaGetSymbolAddress(&addr, g_dec_counters) != cudaSuccess) return ATTN_ERR_CUDA;
      st.dec_counters = static_cast<unsigned*>(addr);
    }
    st.probed = true;
  }
  if (!st.sm103) return ATTN_ERR_ARCH;
  *out = &st;
  return ATTN_OK;
}

// [B*H, N, D] 16-bit tensor as a rank-3 map (D, N, B*H) with 64 x 128 x 1 boxes,
// 128-byte swizzle; rows past N read as zero.
int encode_qkv_map(EncodeTiledFn encode, CUtensorMap* map, const void* ptr, bool bf16, int D, int N,
                   int BH, unsigned box_rows = 128) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(N),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                                 static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(D) * 2};
  const cuuint32_t box[3] = {64, box_rows, 1};
  const cuuint32_t elem_strides[3] = {1, 1, 1};
  const CUresult r =
      encode(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
             const_cast<void*>(ptr), dims, strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_INVALID_ARG;
}

// encode_qkv_map through the device's cache of recent maps.
int cached_qkv_map(MapCache& cache, EncodeTiledFn encode, CUtensorMap* map, const void* ptr, bool bf16, int D,
                   int N, int BH, unsigned box_rows = 128) {
  const uint64_t shape = MapCache::pack(bf16, D, N, box_rows);
  if (const CUtensorMap* hit = cache.find(ptr, shape, BH)) {
    *map = *hit;
    return ATTN_OK;
  }
  const int rc = encode_qkv_map(encode, map, ptr, bf16, D, N, BH, box_rows);
  if (rc == ATTN_OK) cache.insert(ptr, shape, BH, *map);
  return rc;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Do [a, a + na) and [b, b + nb) intersect?
bool overlaps(const void* a, uint64_t na, const void* b, uint64_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

// Checks that need no GPU.  Order: pointers, sizes, head dim, scale, alignment, overlap.
int check_args(const void* q, const void* k, const void* v, const void* o, const float* lse, int B,
               int H, int N, int D, float scale, int Hkv = 0) {
  if (Hkv == 0) Hkv = H;
  if (!q || !k || !v || !o) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || N < 1 || Hkv < 1 || H % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED_D;
  if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16)) return ATTN_ERR_UNALIGNED;
  if (lse && !aligned(lse, 4)) return ATTN_ERR_UNALIGNED;
  const uint64_t bh = static_cast<uint64_t>(B) * static_cast<uint64_t>(H);
  const uint64_t n_tiles = (static_cast<uint64_t>(N) + 127) / 128;
  const uint64_t n_pairs = (n_tiles + 1) / 2;
  // Grid (pairs x heads) and tensor-map extents must fit; byte sizes stay far below 2^63.
  if (bh > 0x7fffffffull || n_pairs * bh > 0x7fffffffull) return ATTN_ERR_INVALID_ARG;
  const uint64_t bytes = bh * static_cast<uint64_t>(N) * static_cast<uint64_t>(D) * 2;
  const uint64_t kv_bytes = bytes / static_cast<uint64_t>(H / Hkv);
  if (static_cast<uint64_t>(N) * D * 2 >= (1ull << 40) || bytes >= (1ull << 62)) return ATTN_ERR_INVALID_ARG;
  if (overlaps(o, bytes, q, bytes) || overlaps(o, bytes, k, kv_bytes) || overlaps(o, bytes, v, kv_bytes)) {
    return ATTN_ERR_INVALID_ARG;
  }
  return ATTN_OK;
}

// Split of the key tiles into segments: tiles per segment and the number of
// non-empty segments for a requested split count.
struct KeySplit {
  int seg_tiles;
  int splits;
};

// 128-row tiles of a sequence of N rows (N up to INT_MAX without overflow).
int tiles_of(int N) {
  return static_cast<int>((static_cast<long long>(N) + eca::kBlockN - 1) / eca::kBlockN);
}

KeySplit key_split(int N, int requested) {
  const int n_tiles = tiles_of(N);
  const int r = requested < 1 ? 1 : (requested > n_tiles ? n_tiles : requested);
  const int seg = (n_tiles + r - 1) / r;
  return KeySplit{seg, (n_tiles + seg - 1) / seg};
}

// Slices per group of the kernel's unit order: the smallest whole number of
// query heads sharing K/V heads that divides B*H and gives a group at least 1.5
// SMs' worth of units.  Small groups keep the CTAs' concurrent K/V reads within
// a few heads (so they stay in L2); equal groups of that size keep the
// heaviest-first order within each group enough to end the launch evenly.  When
// all of K and V fit in L2 anyway (64 MiB or less), one group.
int unit_group_heads(int BH, int q_per_kv, int units_per_slice, int sm_count, unsigned long long kv_bytes) {
  if (kv_bytes <= (64ull << 20)) return BH;
  const double target = 1.5 * sm_count / units_per_slice;
  for (int g = q_per_kv; g < BH; g += q_per_kv) {
    if (BH % g == 0 && g >= target) return g;
  }
  return BH;
}

// Split count with the shortest predicted time, from a replay of the kernel's
// schedule: units are taken in launch order by whichever CTA is free first, a
// unit costs the longer of its two tiles' key-tile counts (of its two halves with
// key-halves units) plus a fixed start/end cost, and a split adds the merge
// kernel's traffic.  The constants
// are rough (a key tile of both query tiles is about 1.2 us on a busy SM, a
// unit boundary about three of those, the merge about 4 TB/s); only their
// ratios matter.  Without a shortage of units the answer is 1.
int predicted_best_splits(int B, int H, int N, int D, int sm_count) {
  const int n_tiles = tiles_of(N);
  const int n_pairs = (n_tiles + 1) / 2;
  const long long bh = static_cast<long long>(B) * H;
  if (static_cast<long long>(n_pairs) * bh >= 2LL * sm_count) return 1;
  constexpr double kStepUs = 1.2, kUnitSteps = 3.0, kMergeBytesPerUs = 4.0e6, kMergeFixedUs = 4.0;
  int best = 1;
  double best_t = 0.0;
  int last_eff = 0;
  for (int req = 1; req <= kMaxSplits && req <= n_tiles; ++req) {
    const KeySplit ks = key_split(N, req);
    if (ks.splits == last_eff) continue;  // same segmentation as a smaller request
    last_eff = ks.splits;
    // The order within a group of slices does not change the costs: pairs heaviest
    // first, every slice and segment of a pair in turn.
    std::priority_queue<double, std::vector<double>, std::greater<double>> free_at;
    for (int c = 0; c < sm_count; ++c) free_at.push(0.0);
    double makespan = 0.0;
    if (ks.splits == 1 && static_cast<long long>(n_pairs) * bh < sm_count) {
      // Unsplit with fewer pair units than SMs: the kernel runs key-halves units,
      // one query tile each, its key tiles shared out between the CTA's two slots.
      for (int tile = n_tiles - 1; tile >= 0; --tile) {
        for (long long x = 0; x < bh; ++x) {
          const double t = free_at.top() + (tile + 2) / 2 + kUnitSteps;
          free_at.pop();
          free_at.push(t);
          if (t > makespan) makespan = t;
        }
      }
      best_t = makespan * kStepUs;
      continue;
    }
    for (int pair = n_pairs - 1; pair >= 0; --pair) {
      for (long long x = 0; x < bh; ++x) {
        for (int seg = 0; seg < ks.splits; ++seg) {
          const int kv0 = seg * ks.seg_tiles;
          const int kv_end = kv0 + ks.seg_tiles < n_tiles ? kv0 + ks.seg_tiles : n_tiles;
          const int need0 = 2 * pair + 1;
          const int need1 = 2 * pair + 1 < n_tiles ? 2 * pair + 2 : 0;
          const int n0 = (need0 < kv_end ? need0 : kv_end) - kv0;
          const int n1 = (need1 < kv_end ? need1 : kv_end) - kv0;
          const int n = n0 > n1 ? n0 : n1;
          if (n <= 0) continue;
          const double t = free_at.top() + n + kUnitSteps;
          free_at.pop();
          free_at.push(t);
          if (t > makespan) makespan = t;
        }
      }
    }
    double t = makespan * kStepUs;
    if (ks.splits > 1) {
      const double merge_bytes = static_cast<double>(bh) * N * D * (4.0 * ks.splits + 2.0);
      t += merge_bytes / kMergeBytesPerUs + kMergeFixedUs;
    }
    if (req == 1 || t < best_t) {
      best_t = t;
      best = ks.splits;
    }
  }
  return best;
}

uint64_t align256(uint64_t x) { return (x + 255) & ~static_cast<uint64_t>(255); }

// Launch with programmatic stream serialisation: the grid may be scheduled before
// the grid ahead of it on the stream has finished.  Only kernels that call
// grid_dependency_wait before touching global memory are launched this way.
// Between two back-to-back attention launches the second then starts as soon as
// the first completes, instead of after the full stream-ordered launch latency.
// ECA_PDL=0 in the environment (read once per process) launches in plain stream
// order instead, with the same results; it exists to measure the difference.
bool programmatic_launch_enabled() {
  static const bool enabled = [] {
    const char* v = std::getenv("ECA_PDL");
    return !(v != nullptr && v[0] == '0' && v[1] == '\0');
  }();
  return enabled;
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = programmatic_launch_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Workspace of a key split: fp32 partial outputs [splits, BH, N, D], then fp32
// partial log-sum-exp [splits, BH, N] at the next 256-byte boundary.
uint64_t splitkv_bytes(uint64_t bh, uint64_t N, uint64_t D, uint64_t splits, uint64_t* lse_offset) {
  const uint64_t o_bytes = splits * bh * N * D * 4;
  if (lse_offset) *lse_offset = align256(o_bytes);
  return align256(o_bytes) + align256(splits * bh * N * 4);
}

template <int D, bool BF16>
int launch(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Hkv, int N,
           int causal, float scale, cudaStream_t stream, DeviceState* st, EncodeTiledFn encode, const KeySplit& ks,
           float* part_o, float* part_lse) {
  const int BH = B * H;
  using L = eca::FwdSmem<D>;
  if (!(st->configured & (1u << ((D == 128 ? 2 : 0) + (BF16 ? 1 : 0))))) {
    // The three unit modes of this instantiation.
    if (cudaFuncSetAttribute(eca::attn_fwd_kernel<D, BF16, eca::kModePairs>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, L::kDynamicBytes) != cudaSuccess ||
        cudaFuncSetAttribute(eca::attn_fwd_kernel<D, BF16, eca::kModeDynamic>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, L::kDynamicBytes) != cudaSuccess ||
        cudaFuncSetAttribute(eca::attn_fwd_kernel<D, BF16, eca::kModeHalves>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, L::kDynamicBytes) != cudaSuccess) {
      return ATTN_ERR_CUDA;
    }
    // The fixed-assignment instances move registers between their warpgroups
    // (setmaxnreg); the counts they ask for must fit in what each block is launched
    // with, or a warpgroup would wait for registers forever.  Refuse a build where
    // they do not.
    const void* instances[2] = {reinterpret_cast<const void*>(eca::attn_fwd_kernel<D, BF16, eca::kModePairs>),
                                reinterpret_cast<const void*>(eca::attn_fwd_kernel<D, BF16, eca::kModeHalves>)};
    for (const void* fn : instances) {
      cudaFuncAttributes fa;
      if (cudaFuncGetAttributes(&fa, fn) != cudaSuccess) return ATTN_ERR_CUDA;
      if (fa.numRegs * eca::kThreads < 256 * eca::kRegsSoftmax + 128 * eca::kRegsControl) return ATTN_ERR_LAUNCH;
    }
    st->configured |= 1u << ((D == 128 ? 2 : 0) + (BF16 ? 1 : 0));
  }
  CUtensorMap tq, tk, tv, to;
  int rc = cached_qkv_map(st->maps, encode, &tq, q, BF16, D, N, BH);
  if (rc == ATTN_OK) rc = cached_qkv_map(st->maps, encode, &tk, k, BF16, D, N, B * Hkv);
  if (rc == ATTN_OK) rc = cached_qkv_map(st->maps, encode, &tv, v, BF16, D, N, B * Hkv);
  // Output: stored by each softmax warp in 32-row slabs.
  if (rc == ATTN_OK) rc = cached_qkv_map(st->maps, encode, &to, o, BF16, D, N, BH, 32);
  if (rc != ATTN_OK) return rc;

  eca::FwdParams p;
  p.o = o;
  p.lse = lse;
  p.part_o = part_o;
  p.part_lse = part_lse;
  p.status = st->status;
  p.N = N;
  static_assert(eca::kBlockM == eca::kBlockN, "query and key tiles have the same height");
  p.n_tiles = tiles_of(N);
  // Causal grouped heads pair two heads of a key/value group at one query tile:
  // both tiles then need the same key tiles.
  p.head_pair = (part_o == nullptr && causal && (H / Hkv) % 2 == 0) ? 1 : 0;
  p.n_pairs = p.head_pair ? p.n_tiles : (p.n_tiles + 1) / 2;
  p.BH = BH;
  p.H = H;
  p.Hkv = Hkv;
  p.splits = ks.splits;
  p.seg_tiles = ks.seg_tiles;
  p.n_units = p.n_pairs * (BH >> p.head_pair) * ks.splits;
  const unsigned long long kv_bytes = 4ull * static_cast<unsigned long long>(B) * Hkv * N * D;  // K and V, 16-bit
  p.group_heads = unit_group_heads(BH >> p.head_pair, (H / Hkv) >> p.head_pair, p.n_pairs * ks.splits,
                                   st->sm_count, kv_bytes);
  const bool dynamic = p.group_heads < (BH >> p.head_pair);
  // Fewer units than SMs (short sequences): a unit becomes one query tile whose key
  // tiles the CTA's two slots share out in halves, which doubles the units and
  // halves the longest chain of key steps.
  bool halves = false;
  if (part_o == nullptr && !dynamic && p.n_units < st->sm_count) {
    halves = true;
    p.head_pair = 0;
    p.n_pairs = p.n_tiles;
    p.n_units = p.n_tiles * BH;
    p.group_heads = BH;
  }
  // Only the dynamic instance touches its counters.
  unsigned slot = 0;
  bool capturing = false;
  if (dynamic) {
    const int rc_slot = st->sched_slots.acquire(stream, &slot, &capturing);
    if (rc_slot != ATTN_OK) return rc_slot;
  }
  p.sched = st->sched_pool + 64 * slot;
  // Divisors of the key-halves unit decoding (dividends are unit and slice indices,
  // below 2^31).
  const eca::HalvesDivs hd{eca::make_fast_div(BH), eca::make_fast_div(H), eca::make_fast_div(H / Hkv)};
  p.causal = causal ? 1 : 0;
  p.scale_log2e = scale * 1.4426950408889634f;
  p.wait_limit_ns = kWaitLimitNs;
  p.timeout_code = ATTN_ERR_TIMEOUT;
  // Persistent: one CTA per SM (the shared-memory footprint admits only one), never more than the units.
  const unsigned grid = static_cast<unsigned>(p.n_units < st->sm_count ? p.n_units : st->sm_count);
  const cudaError_t launched =
      dynamic ? launch_pdl(eca::attn_fwd_kernel<D, BF16, eca::kModeDynamic>, grid, eca::kThreads, L::kDynamicBytes,
                           stream, tq, tk, tv, to, p, hd)
      : halves ? launch_pdl(eca::attn_fwd_kernel<D, BF16, eca::kModeHalves>, grid, eca::kThreads, L::kDynamicBytes,
                            stream, tq, tk, tv, to, p, hd)
               : launch_pdl(eca::attn_fwd_kernel<D, BF16, eca::kModePairs>, grid, eca::kThreads, L::kDynamicBytes,
                            stream, tq, tk, tv, to, p, hd);
  if (launched != cudaSuccess) {
    cudaGetLastError();  // clear the error the failed launch recorded
    return ATTN_ERR_LAUNCH;
  }
  if (dynamic) {
    const int rc_slot = st->sched_slots.release(stream, slot, capturing);
    if (rc_slot != ATTN_OK) return rc_slot;
  }
  if (part_o == nullptr) return ATTN_OK;

  eca::CombineParams c;
  c.part_o = part_o;
  c.part_lse = part_lse;
  c.o = o;
  c.lse = lse;
  c.BH = BH;
  c.N = N;
  c.n_tiles = p.n_tiles;
  c.seg_tiles = ks.seg_tiles;
  c.splits = ks.splits;
  c.causal = p.causal;
  const long long rows = static_cast<long long>(BH) * N;
  const long long want = (rows + 7) / 8;  // 8 rows (warps) per 256-thread block
  const long long cap = static_cast<long long>(st->sm_count) * 8;
  if (launch_pdl(eca::splitkv_combine_kernel<D, BF16>, static_cast<unsigned>(want < cap ? want : cap), 256, 0, stream,
                 c) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_LAUNCH;
  }
  return ATTN_OK;
}

int attn_fwd_impl(bool bf16, const void* q, const void* k, const void* v, void* o, float* lse, int B,
                  int H, int N, int D, int causal, float scale, attn_stream_t stream, int kv_splits = 0,
                  void* workspace = nullptr, size_t workspace_bytes = 0, int Hkv = 0) {
  if (Hkv == 0) Hkv = H;
  int rc = check_args(q, k, v, o, lse, B, H, N, D, scale, Hkv);
  if (rc != ATTN_OK) return rc;
  KeySplit ks{tiles_of(N), 1};
  float* part_o = nullptr;
  float* part_lse = nullptr;
  if (kv_splits > 0) {
    if (kv_splits > kMaxSplits || workspace == nullptr) return ATTN_ERR_INVALID_ARG;
    if (!aligned(workspace, 256)) return ATTN_ERR_UNALIGNED;
    ks = key_split(N, kv_splits);
    const uint64_t bh = static_cast<uint64_t>(B) * static_cast<uint64_t>(H);
    uint64_t lse_off = 0;
    const uint64_t need = splitkv_bytes(bh, N, D, ks.splits, &lse_off);
    if (static_cast<uint64_t>(workspace_bytes) < need) return ATTN_ERR_INVALID_ARG;
    const uint64_t io_bytes = bh * static_cast<uint64_t>(N) * static_cast<uint64_t>(D) * 2;
    const uint64_t kv_bytes = io_bytes / static_cast<uint64_t>(H / Hkv);
    if (overlaps(workspace, need, q, io_bytes) || overlaps(workspace, need, k, kv_bytes) ||
        overlaps(workspace, need, v, kv_bytes) || overlaps(workspace, need, o, io_bytes)) {
      return ATTN_ERR_INVALID_ARG;
    }
    const uint64_t n_pairs = ((static_cast<uint64_t>(N) + 127) / 128 + 1) / 2;
    if (n_pairs * bh * static_cast<uint64_t>(ks.splits) > 0x7fffffffull) return ATTN_ERR_INVALID_ARG;
    part_o = static_cast<float*>(workspace);
    part_lse = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + lse_off);
  }
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState* st = nullptr;
  int r = device_state(&st);
  if (r != ATTN_OK) return r;
  EncodeTiledFn encode = nullptr;
  r = get_encode_fn(&encode);
  if (r != ATTN_OK) return r;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (D == 128) {
    return bf16 ? launch<128, true>(q, k, v, o, lse, B, H, Hkv, N, causal, scale, s, st, encode, ks, part_o,
                                    part_lse)
                : launch<128, false>(q, k, v, o, lse, B, H, Hkv, N, causal, scale, s, st, encode, ks, part_o,
                                     part_lse);
  }
  return bf16 ? launch<64, true>(q, k, v, o, lse, B, H, Hkv, N, causal, scale, s, st, encode, ks, part_o, part_lse)
              : launch<64, false>(q, k, v, o, lse, B, H, Hkv, N, causal, scale, s, st, encode, ks, part_o,
                                  part_lse);
}

// One thread waits on a barrier that nothing ever arrives on, with a bounded wait.
__global__ void watchdog_selftest_kernel(int* status, unsigned long long limit_ns, int code) {
  __shared__ __align__(8) uint64_t barrier;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    eca::mbar_init(eca::smem_u32(&barrier), 1);
    eca::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const eca::Watchdog wd{&abort_flag, status, limit_ns, code};
    wd.wait(eca::smem_u32(&barrier), 0);
  }
}

// ------------------------------------------------------------- paged decode

struct DecodeShape {
  int hc;          // query heads per CTA
  int head_chunks;
  int seg_pages;
  int splits;
};

DecodeShape decode_shape(int Hq, int Hkv, int page_size, int max_pages, int kv_splits) {
  const int group = Hq / Hkv;
  int hc = 8;
  while (group % hc != 0) hc /= 2;
  const int ppt = eca::kDecTile / page_size;
  int seg = (max_pages + kv_splits - 1) / kv_splits;
  seg = (seg + ppt - 1) / ppt * ppt;  // whole tiles per segment
  return DecodeShape{hc, group / hc, seg, (max_pages + seg - 1) / seg};
}

// Paged cache [P, 2, T, Hkv, D] as a rank-3 map (D, Hkv, P*2*T): one box is the
// T x 64 block of one head on one page, 128-byte swizzle.
int encode_cache_map(EncodeTiledFn encode, CUtensorMap* map, const void* cache, bool bf16, int D, int Hkv, int T,
                     int P) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(Hkv),
                              static_cast<cuuint64_t>(P) * 2 * static_cast<cuuint64_t>(T)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(Hkv) * D * 2};
  const cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(T)};
  const cuuint32_t elem_strides[3] = {1, 1, 1};
  const CUresult r =
      encode(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
             const_cast<void*>(cache), dims, strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_INVALID_ARG;
}

int check_paged_args(const void* cache, const int* block_table, const int* lengths, int B, int Hkv, int D,
                     int page_size, int max_pages, int num_pages) {
  if (!cache || !block_table || !lengths) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || Hkv < 1 || max_pages < 1 || num_pages < 1) return ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED_D;
  if (page_size != 8 && page_size != 16 && page_size != 32 && page_size != 64) return ATTN_ERR_INVALID_ARG;
  if (!aligned(cache, 16) || !aligned(block_table, 4) || !aligned(lengths, 4)) return ATTN_ERR_UNALIGNED;
  // The decode kernel addresses the cache's (page, kind, token) rows with a signed 32-bit tensor
  // coordinate, so there must be fewer than 2^31 of them.
  const uint64_t rows = static_cast<uint64_t>(num_pages) * 2 * static_cast<uint64_t>(page_size);
  if (rows > 0x7fffffffull || static_cast<uint64_t>(max_pages) * page_size > 0x7fffffffull) return ATTN_ERR_INVALID_ARG;
  if (static_cast<uint64_t>(B) * static_cast<uint64_t>(max_pages) > 0x7fffffffull) return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

uint64_t decode_ws_bytes(uint64_t B, uint64_t Hq, uint64_t D, uint64_t splits, uint64_t* lse_off) {
  const uint64_t o = splits * B * Hq * D * 4;
  if (lse_off) *lse_off = align256(o);
  return align256(o) + align256(splits * B * Hq * 4);
}

template <int D, bool BF16>
int launch_decode(const CUtensorMap& tm, eca::DecodeParams& p, const DecodeShape& sh, DeviceState* st,
                  cudaStream_t stream) {
  using L = eca::DecodeSmem<D>;
  const long long ctas = static_cast<long long>(p.B) * p.Hkv * sh.head_chunks * sh.splits;
  if (ctas > 0x7fffffffLL) return ATTN_ERR_INVALID_ARG;
  const unsigned grid = static_cast<unsigned>(ctas);
  auto run = [&](auto kernel, unsigned bit) -> int {
    if (!(st->configured_decode & bit)) {
      if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kDynamicBytes) !=
              cudaSuccess ||
          cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared) != cudaSuccess) {
        return ATTN_ERR_CUDA;
      }
      st->configured_decode |= bit;
    }
    if (launch_pdl(kernel, grid, eca::kDecThreads, L::kDynamicBytes, stream, tm, p) != cudaSuccess) {
      cudaGetLastError();
      return ATTN_ERR_LAUNCH;
    }
    return ATTN_OK;
  };
  const unsigned base = (D == 128 ? 0u : 8u) + (BF16 ? 4u : 0u);
  int rc;
  switch (sh.hc) {
    case 8: rc = run(eca::paged_decode_kernel<D, BF16, 8>, 1u << (base + 3)); break;
    case 4: rc = run(eca::paged_decode_kernel<D, BF16, 4>, 1u << (base + 2)); break;
    case 2: rc = run(eca::paged_decode_kernel<D, BF16, 2>, 1u << (base + 1)); break;
    default: rc = run(eca::paged_decode_kernel<D, BF16, 1>, 1u << base); break;
  }
  if (rc != ATTN_OK || p.part_o == nullptr || p.counters != nullptr) return rc;  // merged in the kernel
  const long long rows = static_cast<long long>(p.B) * p.Hq;
  const long long want = (rows + 7) / 8, cap = static_cast<long long>(st->sm_count) * 8;
  if (launch_pdl(eca::paged_decode_combine<D, BF16>, static_cast<unsigned>(want < cap ? want : cap), 256, 0, stream,
                 p) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_LAUNCH;
  }
  return ATTN_OK;
}

int decode_impl(bool bf16, const void* q, const void* cache, const int* block_table, const int* lengths, void* out,
                float* lse, int B, int Hq, int Hkv, int D, int page_size, int max_pages, int num_pages, float scale,
                int kv_splits, void* workspace, size_t workspace_bytes, attn_stream_t stream) {
  int rc = check_paged_args(cache, block_table, lengths, B, Hkv, D, page_size, max_pages, num_pages);
  if (rc != ATTN_OK) return rc;
  if (!q || !out || Hq < 1 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (kv_splits < 1 || kv_splits > kMaxSplits) return ATTN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(out, 16) || (lse && !aligned(lse, 4))) return ATTN_ERR_UNALIGNED;
  const uint64_t qbytes = static_cast<uint64_t>(B) * Hq * D * 2;
  if (overlaps(out, qbytes, q, qbytes)) return ATTN_ERR_INVALID_ARG;
  const DecodeShape sh = decode_shape(Hq, Hkv, page_size, max_pages, kv_splits);
  float* part_o = nullptr;
  float* part_lse = nullptr;
  if (sh.splits > 1) {
    if (workspace == nullptr) return ATTN_ERR_INVALID_ARG;
    if (!aligned(workspace, 256)) return ATTN_ERR_UNALIGNED;
    uint64_t lse_off = 0;
    const uint64_t need = decode_ws_bytes(B, Hq, D, sh.splits, &lse_off);
    if (static_cast<uint64_t>(workspace_bytes) < need) return ATTN_ERR_INVALID_ARG;
    if (overlaps(workspace, need, out, qbytes) || overlaps(workspace, need, q, qbytes)) return ATTN_ERR_INVALID_ARG;
    part_o = static_cast<float*>(workspace);
    part_lse = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + lse_off);
  }
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState* st = nullptr;
  rc = device_state(&st);
  if (rc != ATTN_OK) return rc;
  EncodeTiledFn encode = nullptr;
  rc = get_encode_fn(&encode);
  if (rc != ATTN_OK) return rc;
  CUtensorMap tm;
  rc = encode_cache_map(encode, &tm, cache, bf16, D, Hkv, page_size, num_pages);
  if (rc != ATTN_OK) return rc;
  eca::DecodeParams p;
  p.q = q;
  p.block_table = block_table;
  p.lengths = lengths;
  p.out = out;
  p.lse = lse;
  p.part_o = part_o;
  p.part_lse = part_lse;
  p.status = st->status;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.page_size = page_size;
  p.max_pages = max_pages;
  p.num_pages = num_pages;
  p.head_chunks = sh.head_chunks;
  p.splits = sh.splits;
  p.seg_pages = sh.seg_pages;
  p.scale_log2e = scale * 1.4426950408889634f;
  p.wait_limit_ns = kWaitLimitNs;
  p.timeout_code = ATTN_ERR_TIMEOUT;
  p.bad_index_code = ATTN_ERR_BAD_INDEX;
  p.counters = nullptr;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const long long groups = static_cast<long long>(B) * Hkv * sh.head_chunks;
  unsigned slot = 0;
  bool capturing = false;
  if (sh.splits > 1 && groups <= kDecCountersPerSlot) {
    rc = st->dec_slots.acquire(s, &slot, &capturing);
    if (rc != ATTN_OK) return rc;
    p.counters = st->dec_counters + static_cast<size_t>(slot) * kDecCountersPerSlot;
  }
  if (D == 128) {
    rc = bf16 ? launch_decode<128, true>(tm, p, sh, st, s) : launch_decode<128, false>(tm, p, sh, st, s);
  } else {
    rc = bf16 ? launch_decode<64, true>(tm, p, sh, st, s) : launch_decode<64, false>(tm, p, sh, st, s);
  }
  if (rc != ATTN_OK || p.counters == nullptr) return rc;
  return st->dec_slots.release(s, slot, capturing);
}

}  // namespace

extern "C" {

int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int D,
             int causal, float scale, attn_stream_t stream) {
  return attn_fwd_impl(false, q, k, v, o, lse, B, H, N, D, causal, scale, stream);
}

int attn_fwd_bf16(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
                  int D, int causal, float scale, attn_stream_t stream) {
  return attn_fwd_impl(true, q, k, v, o, lse, B, H, N, D, causal, scale, stream);
}

int attn_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Hkv,
                 int N, int D, int causal, float scale, attn_stream_t stream) {
  if (Hkv < 1) return ATTN_ERR_INVALID_ARG;
  return attn_fwd_impl(false, q, k, v, o, lse, B, H, N, D, causal, scale, stream, 0, nullptr, 0, Hkv);
}

int attn_fwd_gqa_bf16(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Hkv,
                      int N, int D, int causal, float scale, attn_stream_t stream) {
  if (Hkv < 1) return ATTN_ERR_INVALID_ARG;
  return attn_fwd_impl(true, q, k, v, o, lse, B, H, N, D, causal, scale, stream, 0, nullptr, 0, Hkv);
}

int attn_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
                     int D, int causal, float scale, int kv_splits, void* workspace, size_t workspace_bytes,
                     attn_stream_t stream) {
  if (kv_splits < 1) return ATTN_ERR_INVALID_ARG;
  return attn_fwd_impl(false, q, k, v, o, lse, B, H, N, D, causal, scale, stream, kv_splits, workspace,
                       workspace_bytes);
}

int attn_fwd_splitkv_bf16(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
                          int D, int causal, float scale, int kv_splits, void* workspace, size_t workspace_bytes,
                          attn_stream_t stream) {
  if (kv_splits < 1) return ATTN_ERR_INVALID_ARG;
  return attn_fwd_impl(true, q, k, v, o, lse, B, H, N, D, causal, scale, stream, kv_splits, workspace,
                       workspace_bytes);
}

int attn_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                             int N, int D, int causal, float scale, int kv_splits, attn_stream_t stream) {
  if (kv_splits < 1 || kv_splits > kMaxSplits) return ATTN_ERR_INVALID_ARG;
  const int rc = check_args(q, k, v, o, lse, B, H, N, D, scale);
  if (rc != ATTN_OK) return rc;
  const KeySplit ks = key_split(N, kv_splits);
  const uint64_t need =
      splitkv_bytes(static_cast<uint64_t>(B) * static_cast<uint64_t>(H), N, D, ks.splits, nullptr);
  if (need > kNoAllocScratchBytes) return ATTN_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState* st = nullptr;
    const int r = device_state(&st);
    if (r != ATTN_OK) return r;
    if (st->scratch == nullptr) {  // first use on this device: look the array's address up once
      void* ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, g_splitkv_scratch) != cudaSuccess || ptr == nullptr) return ATTN_ERR_CUDA;
      st->scratch = ptr;
    }
    scratch = st->scratch;
  }
  return attn_fwd_impl(false, q, k, v, o, lse, B, H, N, D, causal, scale, stream, kv_splits, scratch,
                       static_cast<size_t>(kNoAllocScratchBytes));
}

size_t attn_splitkv_workspace_bytes(int B, int H, int N, int D, int kv_splits) {
  if (B < 1 || H < 1 || N < 1 || (D != 64 && D != 128) || kv_splits < 1 || kv_splits > kMaxSplits) return 0;
  const KeySplit ks = key_split(N, kv_splits);
  return static_cast<size_t>(
      splitkv_bytes(static_cast<uint64_t>(B) * static_cast<uint64_t>(H), N, D, ks.splits, nullptr));
}

int attn_splitkv_default_splits(int B, int H, int N, int D) {
  if (B < 1 || H < 1 || N < 1 || (D != 64 && D != 128)) return ATTN_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState* st = nullptr;
  const int r = device_state(&st);
  if (r != ATTN_OK) return r;
  return predicted_best_splits(B, H, N, D, st->sm_count);
}

int attn_decode_paged(const void* q, const void* cache, const int* block_table, const int* lengths, void* out,
                      float* lse, int B, int Hq, int Hkv, int D, int page_size, int max_pages, int num_pages,
                      float scale, int kv_splits, void* workspace, size_t workspace_bytes, attn_stream_t stream) {
  return decode_impl(false, q, cache, block_table, lengths, out, lse, B, Hq, Hkv, D, page_size, max_pages, num_pages,
                     scale, kv_splits, workspace, workspace_bytes, stream);
}

int attn_decode_paged_bf16(const void* q, const void* cache, const int* block_table, const int* lengths, void* out,
                           float* lse, int B, int Hq, int Hkv, int D, int page_size, int max_pages, int num_pages,
                           float scale, int kv_splits, void* workspace, size_t workspace_bytes,
                           attn_stream_t stream) {
  return decode_impl(true, q, cache, block_table, lengths, out, lse, B, Hq, Hkv, D, page_size, max_pages, num_pages,
                     scale, kv_splits, workspace, workspace_bytes, stream);
}

size_t attn_decode_workspace_bytes(int B, int Hq, int D, int kv_splits) {
  if (B < 1 || Hq < 1 || (D != 64 && D != 128) || kv_splits < 1 || kv_splits > kMaxSplits) return 0;
  if (kv_splits == 1) return 0;
  return static_cast<size_t>(decode_ws_bytes(B, Hq, D, kv_splits, nullptr));
}

int attn_decode_default_splits(int B, int Hq, int Hkv, int page_size, int max_pages) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || max_pages < 1) return ATTN_ERR_INVALID_ARG;
  if (page_size != 8 && page_size != 16 && page_size != 32 && page_size != 64) return ATTN_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState* st = nullptr;
  const int r = device_state(&st);
  if (r != ATTN_OK) return r;
  const DecodeShape one = decode_shape(Hq, Hkv, page_size, max_pages, 1);
  const long long ctas = static_cast<long long>(B) * Hkv * one.head_chunks;
  const long long tiles = (static_cast<long long>(max_pages) * page_size + eca::kDecTile - 1) / eca::kDecTile;
  // About two CTAs per SM (measured best on the decode page's geometry, contexts
  // 1K-32K: fewer leave HBM idle, more add per-CTA start and merge costs).
  long long s = (2LL * st->sm_count + ctas / 2) / ctas;
  if (s > tiles) s = tiles;
  if (s > kMaxSplits) s = kMaxSplits;
  return s < 1 ? 1 : static_cast<int>(s);
}

int attn_paged_append(const void* new_kv, void* cache, const int* block_table, const int* lengths, int B, int Hkv,
                      int D, int page_size, int max_pages, int num_pages, attn_stream_t stream) {
  int rc = check_paged_args(cache, block_table, lengths, B, Hkv, D, page_size, max_pages, num_pages);
  if (rc != ATTN_OK) return rc;
  if (!new_kv) return ATTN_ERR_INVALID_ARG;
  if (!aligned(new_kv, 16)) return ATTN_ERR_UNALIGNED;
  DeviceState* st = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    rc = device_state(&st);
    if (rc != ATTN_OK) return rc;
  }
  eca::AppendParams p;
  p.new_kv = new_kv;
  p.cache = cache;
  p.block_table = block_table;
  p.lengths = lengths;
  p.status = st->status;
  p.B = B;
  p.Hkv = Hkv;
  p.D = D;
  p.page_size = page_size;
  p.max_pages = max_pages;
  p.num_pages = num_pages;
  p.bad_index_code = ATTN_ERR_BAD_INDEX;
  const long long rows = static_cast<long long>(B) * 2 * Hkv;
  const long long want = (rows + 7) / 8, cap = static_cast<long long>(st->sm_count) * 8;
  if (launch_pdl(eca::paged_append_kernel, static_cast<unsigned>(want < cap ? want : cap), 256, 0,
                 reinterpret_cast<cudaStream_t>(stream), p) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_LAUNCH;
  }
  return ATTN_OK;
}

int attn_row_softmax_f32(const float* x, float* y, long long M, int N, attn_stream_t stream) {
  if (!x || !y || M < 1 || N < 1) return ATTN_ERR_INVALID_ARG;
  if (!aligned(x, 4) || !aligned(y, 4)) return ATTN_ERR_UNALIGNED;
  const uint64_t bytes = static_cast<uint64_t>(M) * static_cast<uint64_t>(N) * 4;
  if (bytes >= (1ull << 62) || M > 0x7fffffffLL) return ATTN_ERR_INVALID_ARG;
  if (x != y && overlaps(x, bytes, y, bytes)) return ATTN_ERR_INVALID_ARG;  // in place is fine, partial overlap not
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState* st = nullptr;
    const int r = device_state(&st);
    if (r != ATTN_OK) return r;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool vec = (N % 4) == 0 && aligned(x, 16) && aligned(y, 16);
  const unsigned warp_blocks = static_cast<unsigned>((M + 7) / 8);  // 8 rows (warps) per block
  const unsigned row_blocks = static_cast<unsigned>(M);
  cudaError_t err;
#define ECA_ROWS(TPR, ITEMS, BLOCKS)                                                                   \
  err = vec ? launch_pdl(eca::row_softmax_cached<TPR, ITEMS, true>, BLOCKS, 256, 0, s, x, y, M, N)    \
            : launch_pdl(eca::row_softmax_cached<TPR, ITEMS, false>, BLOCKS, 256, 0, s, x, y, M, N)
  const unsigned pair_blocks = static_cast<unsigned>((M + 1) / 2);  // 2 rows (128 threads each) per block
  if (N <= 32 * 4) {
    ECA_ROWS(32, 4, warp_blocks);
  } else if (N <= 32 * 8) {
    ECA_ROWS(32, 8, warp_blocks);
  } else if (N <= 32 * 16) {
    ECA_ROWS(32, 16, warp_blocks);
  } else if (N <= 32 * 32) {
    ECA_ROWS(32, 32, warp_blocks);
  } else if (N <= 32 * 64) {
    ECA_ROWS(32, 64, warp_blocks);
  } else if (N <= 128 * 32) {
    // 128 threads per row: a short matrix (such as 1024 x 4096) fits in one wave.
    ECA_ROWS(128, 32, pair_blocks);
  } else if (N <= 256 * 32) {
    ECA_ROWS(256, 32, row_blocks);
  } else if (N <= 256 * 64) {
    ECA_ROWS(256, 64, row_blocks);
  } else {
    err = vec ? launch_pdl(eca::row_softmax_stream<true>, row_blocks, 256, 0, s, x, y, M, N)
              : launch_pdl(eca::row_softmax_stream<false>, row_blocks, 256, 0, s, x, y, M, N);
  }
#undef ECA_ROWS
  if (err != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_LAUNCH;
  }
  return ATTN_OK;
}

int attn_device_status(attn_stream_t stream) {
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState* st = nullptr;
  const int r = device_state(&st);
  if (r != ATTN_OK) return r;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return ATTN_ERR_CUDA;
  int value = 0;
  const int zero = 0;
  if (cudaMemcpy(&value, st->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return ATTN_ERR_CUDA;
  if (cudaMemcpy(st->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return ATTN_ERR_CUDA;
  return value == 0 ? ATTN_OK : value;
}

int attn_watchdog_selftest(unsigned int timeout_us, attn_stream_t stream) {
  if (timeout_us < 1 || timeout_us > 10000000u) return ATTN_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState* st = nullptr;
  const int r = device_state(&st);
  if (r != ATTN_OK) return r;
  watchdog_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      st->status, static_cast<unsigned long long>(timeout_us) * 1000ull, ATTN_ERR_TIMEOUT);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

int attn_anatomy_read(unsigned long long* out, size_t out_words, int reset) {
#ifdef ECA_ANATOMY
  constexpr size_t kWords = 2 * eca::kAnatomyCtas * eca::kAnatomyPoints;
  if (out == nullptr || out_words < kWords) return ATTN_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState* st = nullptr;
  const int r = device_state(&st);
  if (r != ATTN_OK) return r;
  if (cudaDeviceSynchronize() != cudaSuccess) return ATTN_ERR_CUDA;
  if (cudaMemcpyFromSymbol(out, eca::g_anatomy, kWords * sizeof(unsigned long long)) != cudaSuccess) {
    return ATTN_ERR_CUDA;
  }
  if (reset) {
    static const unsigned long long zeros[kWords] = {};
    const int zero = 0;
    if (cudaMemcpyToSymbol(eca::g_anatomy, zeros, sizeof(zeros)) != cudaSuccess ||
        cudaMemcpyToSymbol(eca::g_anatomy_launch, &zero, sizeof(int)) != cudaSuccess ||
        cudaMemcpyToSymbol(eca::g_anatomy_exited, &zero, sizeof(int)) != cudaSuccess) {
      return ATTN_ERR_CUDA;
    }
  }
  return ATTN_OK;
#else
  (void)out;
  (void)out_words;
  (void)reset;
  return ATTN_ERR_INVALID_ARG;  // not the anatomy build
#endif
}

const char* attn_status_string(int status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNALIGNED: return "tensor pointer not 16-byte aligned";
    case ATTN_ERR_UNSUPPORTED_D: return "unsupported head dimension (D must be 64 or 128)";
    case ATTN_ERR_ARCH: return "current device is not sm_103";
    case ATTN_ERR_LAUNCH: return "kernel launch failed";
    case ATTN_ERR_TIMEOUT: return "a bounded device wait timed out";
    case ATTN_ERR_CUDA: return "CUDA runtime/driver call failed";
    case ATTN_ERR_SCRATCH_LIMIT: return "the split needs more than the library's fixed 64 MiB scratch";
    case ATTN_ERR_BAD_INDEX: return "a block-table entry or a length was out of range (those tokens were skipped)";
    default: return "unknown status";
  }
}

int attn_version(void) { return 100; }

}  // extern "C"
