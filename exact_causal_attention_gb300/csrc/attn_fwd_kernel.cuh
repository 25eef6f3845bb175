// Fused attention forward for sm_103a: TMA-fed K/V ring, tcgen05 MMAs with TMEM
// accumulators for S = Q K^T and O += P V, FP32 online softmax.
//
// Method: "CUDA FlashAttention：从在线 Softmax 到长序列 IO 极限" (chengzipai.xyz):
// section 1 (the operation and its causal mask), section 4 (the online
// recurrence over key tiles: running max m, running sum l, unnormalised o,
// rescaled by exp(m_old - m_new) at every merge), section 5.1 (one CTA owns a
// block of query rows and streams K/V tiles so each tile is read once for all of
// them), section 6 (rescale the old O before adding this tile's P V; mask before
// the max; never form -inf - (-inf)), section 7 (skip key tiles entirely above
// the diagonal, mask element-wise only on the diagonal tile; keep the LSE).
//
// GB300 mapping (differs from the page's mma.sync / cp.async design):
//   * persistent CTAs, one per SM; a work unit is two consecutive 128-row query
//     tiles of one (batch, head).  A CTA takes the next unit of the launch from
//     a global counter when its producer warp is ready for one, and passes the
//     index to its other warps through a small shared-memory queue.  Units are
//     ordered by groups of heads (so the K/V tiles in use at any time stay in
//     L2), heaviest first within a group (causal work grows with the tile index).
//     Each query tile's next Q load starts as soon as that tile's last Q K^T MMA
//     is done, and its first P V only waits until that tile's epilogue has read
//     O, so unit boundaries overlap.  With a key split (long sequences, few
//     heads), a unit also names a segment of key tiles and its epilogue writes
//     the segment's normalised partial output and log-sum-exp in fp32 for a
//     separate merge ("CUDA KV Cache：分页存储与长上下文 Decode 极致优化",
//     section 6.4).  Grouped heads (same page, section 3.3): query head h
//     reads key/value head h / (H / Hkv) directly, with no copy.  Causal
//     unsplit launches with an even group pair two heads of a group at one query
//     tile instead of two consecutive tiles, so each K/V tile serves both query
//     heads in the CTA and both need the same key tiles; the heads of a group
//     are adjacent in the unit order so their K/V tiles come from L2.  When a
//     launch has fewer such units than SMs (short sequences), a unit is one query
//     tile whose key tiles are split in two halves, one per tile slot of the CTA
//     (key halves): the two slots run the same recurrence on their halves side by
//     side, each on ring items of its own, and the epilogue merges their (m, l, O)
//     with the online-softmax law (section 4's merge, the decode page's section
//     6.4), so the unit's chain of key steps is half as long.
//     384 threads:
//       warps 0-3  softmax for query tile 0     warps 4-7  softmax for query tile 1
//       warp 8     takes units; TMA producer of the ring items {V_j, K_j+1}
//       warp 9     TMEM owner; tcgen05.mma issuer for query tile 0
//       warp 10    tcgen05.mma issuer for query tile 1
//       warp 11    TMA loads of Q, per query tile
//     One issuing warp per query tile, run as a converged warp with an elected
//     lane issuing each MMA (operands stay warp-uniform; the same instructions
//     from a one-lane branch cost several times more issue time, and the pipe
//     then starves while a turn is being issued).  Each tile's P V -> Q K^T
//     order stays within one issuing lane, where tcgen05.mma executes in issue
//     order.  The two issuers pass a turn token (an mbarrier each), one turn per
//     ring item, tile 0 first, so each turn's MMAs are contiguous in the pipe
//     and the tiles alternate: one tile's softmax overlaps the other's MMAs.
//   * TMEM (512 columns x 128 lanes): S_t at column 128 t (128 fp32 columns),
//     O_t at column 256 + D t.  P_t (16-bit, two per column) is written over the
//     first 64 columns of S_t and read by the P V MMA straight from TMEM.
//   * a query row is a TMEM lane, so each softmax thread owns one full score row:
//     the row max and row sum need no shuffles.
//   * exp is computed as 2^(s * scale * log2 e - m) with the MUFU ex2.
//   * stale reference max: o and l share one reference m, and any reference
//     gives the same O and lse (exact algebra), so p is formed against the
//     current reference without first taking the new tile's row max.  No p may
//     overflow the 16-bit P: with fp16 a sum of at most 2^15 over keys 0-63 bounds
//     each of their p, and a max score of keys 64-127 at most 15 above the
//     reference bounds theirs (bf16, with fp32's exponent range, takes 2^30 and 30,
//     which only keep l and o in fp32 range).  Under the fixed assignment a unit whose first key tile is
//     unmasked starts from a guessed reference, kept only if the row's sum of p
//     over that tile is at least 1: then l >= 1 from the first tile on, as with
//     the row max as reference, so a p that lands in fp16's subnormal range
//     carries no more rounding relative to l than it would there.  Otherwise the
//     first key tile, the diagonal one and the rare rows that fail a check take
//     the row max, move the reference (rescaling O and l) and redo the tile from
//     S, still intact in TMEM.
//   * P reaches the issuer in two halves: the P V MMAs of keys 0-63 run while
//     the softmax exponentiates keys 64-127 (whose S columns it loaded while
//     exponentiating keys 0-63).
#pragma once
#include <cuda.h>
#include <cstdint>

#include "ptx.cuh"

namespace eca {

constexpr int kBlockM = 128;            // query rows per tile (one per TMEM lane)
constexpr int kBlockN = 128;            // keys per K/V tile
constexpr int kSubTileBytes = 128 * 128;  // 128 rows x 64 16-bit elements (one 128-B swizzle span)
constexpr int kThreads = 384;
constexpr int kTmemCols = 512;
// Bounds of the stale reference that keep every p in range of the 16-bit P: with
// fp16, a sum of at most 2^15 over keys 0-63 bounds each of their p, and keys
// 64-127 may score at most 15 above the reference.  bf16 has fp32's exponent range,
// so P cannot overflow there; its looser bounds (2^30, 30) only keep the fp32 l and
// o far from overflow (l stays below N 2^30), and let wide score distributions keep
// the reference longer.
template <bool BF16>
__host__ __device__ constexpr float max_row_sum() { return BF16 ? 1073741824.0f : 32768.0f; }
template <bool BF16>
__host__ __device__ constexpr float max_lead() { return BF16 ? 30.0f : 15.0f; }
constexpr float kGuessRef = 4.0f;       // first reference of a unit (scores times scale log2 e)
constexpr float kMinGuessSum = 1.0f;    // a guess is kept only if the first tile's sum of p reaches this
constexpr int kUnitQueue = 4;           // depth of the shared-memory queue of unit indices
constexpr int kUnitReaders = 11;        // warps that read each queue entry: 8 softmax, 2 issuers, Q loader
// Per-thread registers after the split (setmaxnreg): 256 softmax threads and 128
// control threads within what the block is launched with, kLaunchRegs per thread
// (the host checks the compiled count before the first launch).
constexpr int kLaunchRegs = 168;
constexpr int kRegsSoftmax = 208;
constexpr int kRegsControl = 80;
static_assert(256 * kRegsSoftmax + 128 * kRegsControl <= kThreads * kLaunchRegs,
              "the register split must fit in the registers the block is launched with");

// How a launch forms and assigns its work units (the kernel's third template argument).
constexpr int kModePairs = 0;    // two query tiles (or head pairs) per unit, fixed zig-zag assignment
constexpr int kModeDynamic = 1;  // the same units, taken from the launch's counter in head groups
constexpr int kModeHalves = 2;   // one query tile per unit, its key tiles in two halves; fixed assignment

// Division of an int in [0, 2^31) by a divisor d >= 1 fixed for the launch, as a
// multiply-high and two shifts: with l = ceil(log2 d) and m = ceil(2^(31 + l) / d)
// (below 2^32), floor(x / d) = floor(x m / 2^(31 + l)) = mulhi(2 x, m) >> l.  Exact:
// m d - 2^(31 + l) < d, so x m / 2^(31 + l) exceeds x / d by less than
// x / 2^(31 + l) < 2^-l <= 1 / d, which cannot carry floor(x / d) over an integer.
struct FastDiv {
  uint32_t m;
  uint32_t l;
  int d;
};

__host__ inline FastDiv make_fast_div(int d) {
  uint32_t l = 0;
  while ((1ull << l) < static_cast<unsigned long long>(d)) ++l;
  const unsigned long long two_s = 1ull << (31 + l);
  return FastDiv{static_cast<uint32_t>((two_s + static_cast<unsigned long long>(d) - 1) /
                                       static_cast<unsigned long long>(d)),
                 l, d};
}

__host__ __device__ __forceinline__ int fast_div(int x, const FastDiv& f) {
#ifdef __CUDA_ARCH__
  return static_cast<int>(__umulhi(static_cast<uint32_t>(x) << 1, f.m) >> f.l);
#else  // the same value on the host, for the host-side check of the divisors
  const unsigned long long hi = (static_cast<unsigned long long>(static_cast<uint32_t>(x) << 1) * f.m) >> 32;
  return static_cast<int>(static_cast<uint32_t>(hi) >> f.l);
#endif
}

// Divisors of the key-halves unit decoding.
struct HalvesDivs {
  FastDiv BH, H, q_per_kv;
};

// Anatomy build (compiled with ECA_ANATOMY, a separate library for measurement):
// every CTA records globaltimer stamps of its first unit's milestones, in one of two
// slots chosen by a launch counter, so two launches in a row can be compared.  In
// the normal build the stamps compile to nothing.
constexpr int kAnatomyCtas = 160;
constexpr int kAnatomyPoints = 10;
#ifdef ECA_ANATOMY
__device__ unsigned long long g_anatomy[2][kAnatomyCtas][kAnatomyPoints];
__device__ int g_anatomy_launch;
__device__ int g_anatomy_exited;
#define ECA_STAMP(slot, i)                                                                       \
  do {                                                                                           \
    if (blockIdx.x < kAnatomyCtas) g_anatomy[(slot)][blockIdx.x][(i)] = global_timer_ns();        \
  } while (0)
#else
#define ECA_STAMP(slot, i) \
  do {                     \
  } while (0)
#endif

struct FwdParams {
  void* o;        // [BH, N, D] 16-bit (unused when part_o is set)
  float* lse;     // [BH, N] or null (unused when part_o is set)
  float* part_o;  // key split: [splits, BH, N, D] fp32 partial outputs, else null
  float* part_lse;  // key split: [splits, BH, N] fp32 partial log-sum-exp
  int* status;    // device status word
  int N;
  int n_tiles;    // ceil(N / 128), for queries and keys alike
  int n_pairs;    // ceil(n_tiles / 2)
  int BH;
  int H;          // query heads per batch entry
  int Hkv;        // key/value heads per batch entry (H is a multiple)
  int splits;     // key segments (1 = no split)
  int seg_tiles;  // key tiles per segment
  int n_units;    // n_pairs * BH * splits
  int group_heads;  // slices per group in the unit order (the last group may be smaller)
  int head_pair;    // 1: a unit is one query tile of two heads of a key/value group (slices are head pairs)
  int* sched;     // [0]: next unit to hand out, [32]: CTAs finished; both back to 0 at exit
  int causal;
  float scale_log2e;  // scale * log2(e)
  unsigned long long wait_limit_ns;
  int timeout_code;
};

// Shared memory: Q of the unit's two query tiles, then a ring of stages.  A ring
// item is {V_j-1, K_j}: the V tile of step j-1 and the K tile of step j, which
// one step of each issuer consumes together (the first item of a unit holds K_0
// alone, the last V_last alone).  Each part lands on its own barrier: a step's
// P V MMAs need only V, so they go in while K is still arriving.
template <int D>
struct FwdSmem {
  static constexpr int kSub = D / 64;                      // 64-element column blocks per row
  static constexpr int kTileBytes = kSub * kSubTileBytes;  // one 128 x D tile
  static constexpr int kStageBytes = 2 * kTileBytes;       // V part, then K part
  static constexpr int kStages = D == 128 ? 2 : 4;
  static constexpr int kQOff = 0;
  static constexpr int kRingOff = 2 * kTileBytes;
  // Per query tile, 16 KB staging for the output: 128 rows x 64 columns of
  // 16-bit values in the 128-B swizzled box layout the TMA store reads, one
  // 32-row slab per softmax warp.
  static constexpr int kStageOutBytes = 128 * 128;
  static constexpr int kOutOff = kRingOff + kStages * kStageBytes;
  static constexpr int kBarOff = kOutOff + 2 * kStageOutBytes;
  // barrier indices
  static constexpr int kBarQFull = 0;                // + t: Q of tile t loaded
  static constexpr int kBarQFree = 2;                // + t: issuer t's last Q K^T of the unit done
  static constexpr int kBarFull = 4;                    // + slot: the item's V part landed (or it has none)
  static constexpr int kBarFullK = kBarFull + kStages;  // + slot: the item's K part landed (or it has none)
  static constexpr int kBarEmpty = kBarFullK + kStages;  // two arrivals: both issuers
  static constexpr int kBarS = kBarEmpty + kStages;  // + t: S_t computed
  static constexpr int kBarPa = kBarS + 2;           // + t: P_t of keys 0-63 written (and O_t rescaled)
  static constexpr int kBarPb = kBarPa + 2;          // + t: P_t of keys 64-127 written
  static constexpr int kBarO = kBarPb + 2;           // + t: last P V of the unit done
  static constexpr int kBarOFree = kBarO + 2;        // + t: epilogue has read O_t
  static constexpr int kBarDrain = kBarOFree + 2;    // + t: issuer t's MMAs all done
  static constexpr int kBarTurn = kBarDrain + 2;    // + t: issuer t may put its next turn into the pipe
  static constexpr int kBarUnitFull = kBarTurn + 2;          // + slot: queue entry written
  static constexpr int kBarUnitFree = kBarUnitFull + kUnitQueue;  // + slot: queue entry read by every reader
  static constexpr int kBarMerge = kBarUnitFree + kUnitQueue;     // key halves: slot 1's m and l published
  static constexpr int kNumBars = kBarMerge + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;  // TMEM base, abort flag, unit queue
  // Key halves: slot 1's final m and l per row, read by slot 0's epilogue.
  static constexpr int kMergeOff = (kMiscOff + 8 + 4 * kUnitQueue + 15) & ~15;
  static constexpr int kBytes = kMergeOff + 2 * kBlockM * 4;
  static constexpr int kDynamicBytes = kBytes + 1024;  // slack for 1024-B alignment
  static_assert(kDynamicBytes <= 227 * 1024, "shared memory exceeds the per-block limit");
};

// One work unit, against the key tiles kv0 .. kv0 + n_kv - 1 of key segment seg:
// query tiles 2*pair and 2*pair + 1 of slice bh; or, with head_pair set, query
// tile `pair` (tile0 = pair) of the two heads bh and bh + 1, which read the same
// key/value head; or, with key halves, query tile `pair` of slice bh in both
// slots, slot 0 against key tiles kv0 .. kv0 + n_kv0 - 1 and slot 1 against
// kv1 .. kv1 + n_kv1 - 1.
struct Unit {
  int bh;
  int kvh;  // key/value slice: query head h of batch b reads head h / (H / Hkv) of batch b
  int tile0;
  int seg;
  int kv0;           // first key tile of the segment (of slot 0's half with key halves)
  int kv1;           // first key tile of slot 1 (kv0 unless key halves)
  int n_kv0, n_kv1;  // key tiles each slot takes (0 = nothing to do)
  int n_max;
};

// Unit l of the launch.  Units are handed out in increasing l to whichever CTA
// asks next.  The order is by groups of group_heads slices (so the K/V tiles the
// CTAs read at any time belong to a few heads and stay in L2), then heaviest
// query-tile pair first (causal work grows with the tile index, so the light
// units come last in every group and the launch ends evenly), then slice, then
// key segment.
template <bool kHalves>
__device__ __forceinline__ void unit_from(int l, const FwdParams& p, const HalvesDivs& hd, Unit& u) {
  if constexpr (kHalves) {
    // One group of all BH slices, no key split, no head pairs: slice l mod BH, query
    // tile n_tiles - 1 - l / BH (heaviest first).  Decoded at the start of every
    // unit by every role, so with multiply-high divisions (short launches are
    // made of such starts).
    const int rq = fast_div(l, hd.BH);
    u.bh = l - rq * p.BH;
    const int b = fast_div(u.bh, hd.H);
    u.kvh = b * p.Hkv + fast_div(u.bh - b * p.H, hd.q_per_kv);
    u.seg = 0;
    u.tile0 = p.n_pairs - 1 - rq;
    u.kv0 = 0;
    const int need = p.causal ? u.tile0 + 1 : p.n_tiles;
    u.n_kv0 = (need + 1) / 2;
    u.n_kv1 = need - u.n_kv0;
    u.kv1 = u.n_kv0;
    u.n_max = u.n_kv0;
    return;
  }
  const int per_slice = p.n_pairs * p.splits;
  const int slices = p.BH >> p.head_pair;
  const int full_groups = slices / p.group_heads;
  int grp = l / (p.group_heads * per_slice);
  int g = p.group_heads;
  int local = l - grp * (p.group_heads * per_slice);
  if (grp >= full_groups) {  // the smaller last group
    grp = full_groups;
    g = slices - full_groups * p.group_heads;
    local = l - full_groups * (p.group_heads * per_slice);
  }
  u.seg = local % p.splits;
  const int r = local / p.splits;
  u.bh = (grp * p.group_heads + r % g) << p.head_pair;
  u.kvh = (u.bh / p.H) * p.Hkv + (u.bh % p.H) / (p.H / p.Hkv);
  const int pair = p.n_pairs - 1 - r / g;  // with head pairs, the query tile
  u.tile0 = p.head_pair ? pair : 2 * pair;
  u.kv0 = u.seg * p.seg_tiles;
  u.kv1 = u.kv0;
  const int kv_end = u.kv0 + p.seg_tiles < p.n_tiles ? u.kv0 + p.seg_tiles : p.n_tiles;
  const bool has1 = p.head_pair || u.tile0 + 1 < p.n_tiles;
  // key tiles each query tile needs in total, then the part inside this segment
  const int need0 = p.causal ? u.tile0 + 1 : p.n_tiles;
  const int need1 = has1 ? (p.causal ? u.tile0 + 2 - p.head_pair : p.n_tiles) : 0;
  const int e0 = need0 < kv_end ? need0 : kv_end;
  const int e1 = need1 < kv_end ? need1 : kv_end;
  u.n_kv0 = e0 > u.kv0 ? e0 - u.kv0 : 0;
  u.n_kv1 = e1 > u.kv0 ? e1 - u.kv0 : 0;
  u.n_max = u.n_kv0 > u.n_kv1 ? u.n_kv0 : u.n_kv1;
}

// S = Q K^T: A = Q (K-major, 128-B swizzle), B = K (K-major).  Descriptors are
// built once; stepping K by 16 elements adds 32 B (2 in the >>4 address field)
// inside a 128-B span and 16 KB (1024) across the 64-column blocks.
template <int D, bool BF16>
__device__ __forceinline__ void issue_qk(uint32_t s_tmem, uint64_t q_desc, uint64_t k_desc) {
  constexpr uint32_t idesc = idesc_f16_f32acc(kBlockM, kBlockN, BF16, false);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint64_t off = static_cast<uint64_t>((kk / 4) * (kSubTileBytes >> 4) + (kk % 4) * 2);
    mma_ss_warp(s_tmem, q_desc + off, k_desc + off, idesc, kk > 0 ? 1u : 0u);
  }
}

// O (+)= P V: A = P from TMEM (16 keys = 8 columns per step), B = V (MN-major,
// 16 keys = 16 rows of 128 B = 2048 B per step, 64-column blocks 16 KB apart).
template <int D, bool BF16>
__device__ __forceinline__ void issue_pv(uint32_t o_tmem, uint32_t p_tmem, uint64_t v_desc, bool accumulate, int k0 = 0,
                                         int k1 = kBlockN / 16) {
  constexpr uint32_t idesc = idesc_f16_f32acc(kBlockM, D, BF16, true);
#pragma unroll
  for (int kk = k0; kk < k1; ++kk) {
    mma_ts_warp(o_tmem, p_tmem + kk * 8, v_desc + static_cast<uint64_t>(kk * (2048 >> 4)), idesc,
           (accumulate || kk > 0) ? 1u : 0u);
  }
}

__device__ __forceinline__ uint32_t parity(int count) { return static_cast<uint32_t>(count) & 1u; }

// kMode: kModeDynamic takes units from the launch's counter and queues them to
// the CTA's warps (grouped head order); otherwise each warp follows the fixed
// zig-zag waves, of pair units or (kModeHalves) of key-halves units.
template <int D, bool BF16, int kMode>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                    const FwdParams p, const HalvesDivs hd) {
  using L = FwdSmem<D>;
  constexpr bool kDynamic = kMode == kModeDynamic;
  constexpr bool kHalves = kMode == kModeHalves;
  // The fixed-assignment instances move registers from the control warpgroup to the
  // softmax warpgroups (which then read O for the epilogue with fewer waits); the
  // dynamic instance measured about 1% slower at N = 8192 with the same split and
  // keeps one count for all warps.
  constexpr bool kSplitRegs = !kDynamic;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t sbase = (raw_base + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw_base);
  auto bar = [&](int i) -> uint32_t { return sbase + L::kBarOff + 8u * static_cast<uint32_t>(i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
  volatile int* unit_queue = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 8);

  // Broadcast from lane 0 so the compiler sees the role index (and the TMEM base
  // below) as warp-uniform.
  const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x / 32), 0);
  const int lane = threadIdx.x % 32;
#ifdef ECA_ANATOMY
  const unsigned long long an_entry = global_timer_ns();
#endif

  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(L::kBarQFull + t), 1);
      // With key halves both slots read Q from buffer 0, which is free again once
      // both issuers have finished their Q K^T of the unit.
      mbar_init(bar(L::kBarQFree + t), (kHalves && t == 0) ? 2 : 1);
    }
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(bar(L::kBarFull + s), 1);
      mbar_init(bar(L::kBarFullK + s), 1);
      mbar_init(bar(L::kBarEmpty + s), kHalves ? 1 : 2);  // the issuers that consume the item
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(L::kBarS + t), 1);
      mbar_init(bar(L::kBarPa + t), 4);
      mbar_init(bar(L::kBarPb + t), 4);
      mbar_init(bar(L::kBarO + t), 1);
      mbar_init(bar(L::kBarOFree + t), 4);
      mbar_init(bar(L::kBarDrain + t), 1);
      mbar_init(bar(L::kBarTurn + t), 1);
    }
    for (int q = 0; q < kUnitQueue; ++q) {
      mbar_init(bar(L::kBarUnitFull + q), 1);
      mbar_init(bar(L::kBarUnitFree + q), kUnitReaders);
    }
    mbar_init(bar(L::kBarMerge), 4);
    mbar_arrive(bar(L::kBarTurn + 0));  // issuer 0 takes the first turn
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  // Work that reads only the launch's own parameters, done before the wait for the
  // grid ahead: the tensor maps into the TMA unit's descriptor cache, and the
  // parameters the unit decoding reads into the constant cache (a decode of unit
  // 0 whose result goes to a queue entry that is written again before it is read).
  if (warp == 8 && lane == 0) {
    tma_prefetch_map(&tm_k);
    tma_prefetch_map(&tm_v);
  } else if (warp == 11 && lane == 0) {
    tma_prefetch_map(&tm_q);
    tma_prefetch_map(&tm_o);  // for the epilogue's first store, well before it
  } else if (warp == 10 && lane == 0) {
    Unit u;
    unit_from<kHalves>(0, p, hd, u);
    unit_queue[kUnitQueue - 1] = u.bh + u.kvh + u.tile0 + u.kv1 + u.n_max + p.N + p.causal;
  }
  // The k-th unit of this CTA under the fixed assignment: unit k G + c of wave k,
  // the waves dealt to the CTAs in alternating directions; -1 past the last.
  auto fixed_unit = [&](int k) -> int {
    const int c = static_cast<int>(blockIdx.x), G = static_cast<int>(gridDim.x);
    const long long l = static_cast<long long>(k) * G + ((k & 1) ? G - 1 - c : c);
    return l < p.n_units ? static_cast<int>(l) : -1;
  };
  // Next unit with work under the fixed assignment: 1 (in w) or 0 (no more).
  int units_fixed = 0;
  auto next_fixed = [&](Unit& w) -> int {
    while (true) {
      const int l = fixed_unit(units_fixed++);
      if (l < 0) return 0;
      unit_from<kHalves>(l, p, hd, w);
      if (w.n_max > 0) return 1;
    }
  };
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  // Set-up done.  The launch is made with programmatic stream serialisation: the
  // next launch on the stream may now start its own set-up on SMs this grid leaves
  // free, and nothing below touches global memory before the grid ahead of this
  // one has finished (every thread waits here, so no bounded wait starts its clock
  // earlier).
  grid_launch_dependents();
  grid_dependency_wait();
  const uint32_t tmem = __shfl_sync(0xffffffffu, *tmem_slot, 0);
#ifdef ECA_ANATOMY
  const int an_slot = *reinterpret_cast<volatile int*>(&g_anatomy_launch) & 1;
  if (threadIdx.x == 0 && blockIdx.x < kAnatomyCtas) g_anatomy[an_slot][blockIdx.x][0] = an_entry;  // entry
  if (threadIdx.x == 0) ECA_STAMP(an_slot, 1);  // set-up done and the grid ahead finished
  int an_units = 0;
#endif
  const Watchdog wd{abort_flag, p.status, p.wait_limit_ns, p.timeout_code};
  // Readers of the unit queue: entry n holds the n-th unit this CTA works on,
  // or -1 after the last.  `read_unit` is called by a whole warp (lane 0 alone
  // for the Q loader); it is false when a wait gave up.
  int units_read = 0;
  auto read_unit = [&](int& l, bool whole_warp) -> bool {
    const int q = units_read % kUnitQueue;
    bool got = wd.wait(bar(L::kBarUnitFull + q), parity(units_read / kUnitQueue));
    if (whole_warp) got = __all_sync(0xffffffffu, got) != 0;
    if (!got) return false;
    l = unit_queue[q];
    if (whole_warp) {
      __syncwarp();
      l = __reduce_max_sync(0xffffffffu, l);  // the same in every lane; warp-uniform for the compiler
    }
    if (lane == 0) mbar_arrive(bar(L::kBarUnitFree + q));
    ++units_read;
    return true;
  };
  // Next unit with work for a role: from the fixed assignment, or from the queue
  // under dynamic assignment.  1: got one in w; 0: no more; -1: a wait gave up.
  auto next_unit = [&](Unit& w, bool whole_warp) -> int {
    if (!kDynamic) return next_fixed(w);
    int l;
    if (!read_unit(l, whole_warp)) return -1;
    if (l < 0) return 0;
    unit_from<kHalves>(l, p, hd, w);
    return 1;
  };

  if (warp >= 8) {
    // Control warpgroup (producer, issuers, Q loader): gives registers to the softmax warps.
    if constexpr (kSplitRegs) setmaxnreg_dec<kRegsControl>();
    if (warp == 8) {
      // ------------------------------------------------------------ TMA producer
      if (lane == 0) {
        const uint64_t pol_kv = policy_evict_last();
        int it = 0;      // ring items issued
        int pushed = 0;  // unit queue entries written
        auto push_unit = [&](int l) -> bool {
          const int q = pushed % kUnitQueue;
          if (!wd.wait(bar(L::kBarUnitFree + q), parity(pushed / kUnitQueue) ^ 1u)) return false;
          unit_queue[q] = l;
          mbar_arrive(bar(L::kBarUnitFull + q));
          ++pushed;
          return true;
        };
        // Under dynamic assignment this warp takes the CTA's units from the launch's
        // counter (skipping key segments past a pair's last key tile, which have no
        // work) when it is about to load their items, and queues them for the other
        // warps; so a unit goes to the CTA that is free first.
        // A CTA's first unit is its own index (the grid never exceeds the units), so
        // the launch does not start with every CTA contending for the counter at once;
        // the counter then hands out units from the grid size on.
        bool first_claim = true;
        auto take_unit = [&]() -> int {
          while (true) {
            const int l = first_claim ? static_cast<int>(blockIdx.x) : atomicAdd(p.sched, 1) + static_cast<int>(gridDim.x);
            first_claim = false;
            if (l >= p.n_units) return -1;
            Unit u;
            unit_from<kHalves>(l, p, hd, u);
            if (u.n_max > 0) return l;
          }
        };
        bool ok = true;
        Unit w;
        while (ok) {
          if (kDynamic) {
            const int l = take_unit();
            if (!push_unit(l) || l < 0) break;
            unit_from<kHalves>(l, p, hd, w);
          } else if (next_unit(w, false) != 1) {
            break;
          }
          // Items i = 0 .. n_max: {V_(b+i-1) if 0 < i <= n, K_(b+i) if i < n}, with
          // b = kv0 and n = n_max shared by both slots; with key halves, one item of
          // each slot per i (slot 0 first), with that slot's b and n.
          const int per_i = kHalves ? 2 : 1;
          for (int i = 0; ok && i <= w.n_max; ++i) {
            for (int h = 0; h < per_i; ++h) {
              const int b = h ? w.kv1 : w.kv0;
              const int n = kHalves ? (h ? w.n_kv1 : w.n_kv0) : w.n_max;
              const int slot = it % L::kStages;
              if (!wd.wait(bar(L::kBarEmpty + slot), parity(it / L::kStages) ^ 1u)) {
                ok = false;
                break;
              }
              const uint32_t stage = sbase + L::kRingOff + slot * L::kStageBytes;
              // The V and K parts complete on barriers of their own, so the P V MMAs can
              // start before K has landed; a missing part is a plain arrival.
              const uint32_t full_v = bar(L::kBarFull + slot), full_k = bar(L::kBarFullK + slot);
              if (i > 0 && i <= n) {
                mbar_arrive_expect_tx(full_v, L::kTileBytes);
                for (int s = 0; s < L::kSub; ++s)
                  tma_load_3d(stage + s * kSubTileBytes, &tm_v, full_v, 64 * s, (b + i - 1) * kBlockN, w.kvh, pol_kv);
              } else {
                mbar_arrive(full_v);
              }
              if (i < n) {
                mbar_arrive_expect_tx(full_k, L::kTileBytes);
                for (int s = 0; s < L::kSub; ++s)
                  tma_load_3d(stage + L::kTileBytes + s * kSubTileBytes, &tm_k, full_k, 64 * s, (b + i) * kBlockN,
                              w.kvh, pol_kv);
              } else {
                mbar_arrive(full_k);
              }
#ifdef ECA_ANATOMY
              if (it == 0) ECA_STAMP(an_slot, 2);  // first K load issued
#endif
              ++it;
            }
          }
        }
        // Let every copy this thread started land before the block can exit.
        for (int x = (it > L::kStages ? it - L::kStages : 0); x < it; ++x) {
          wd.drain(bar(L::kBarFull + x % L::kStages), parity(x / L::kStages));
          wd.drain(bar(L::kBarFullK + x % L::kStages), parity(x / L::kStages));
        }
      }
    } else if (warp == 11) {
      // ------------------------------------------------------ Q loader, per query tile
      // Each tile's Q buffer is refilled as soon as that tile's last Q K^T of the
      // unit is done, so a tile that finishes first starts its next unit without
      // waiting for the other.
      if (lane == 0) {
        const uint64_t pol_q = policy_evict_first();
        int loads[2] = {0, 0};
        bool ok = true;
        Unit w;
        while (ok && next_unit(w, false) == 1) {
          // With key halves one Q tile serves both slots (slot 0 always has work).
          for (int t = 0; t < (kHalves ? 1 : 2); ++t) {
            if ((t ? w.n_kv1 : w.n_kv0) == 0) continue;
            if (loads[t] > 0 && !wd.wait(bar(L::kBarQFree + t), parity(loads[t] - 1))) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(bar(L::kBarQFull + t), L::kTileBytes);
            for (int s = 0; s < L::kSub; ++s) {
              tma_load_3d(sbase + L::kQOff + t * L::kTileBytes + s * kSubTileBytes, &tm_q, bar(L::kBarQFull + t),
                          64 * s, (w.tile0 + ((p.head_pair || kHalves) ? 0 : t)) * kBlockM,
                          w.bh + (p.head_pair ? t : 0), pol_q);
            }
            ++loads[t];
          }
        }
        // Let every copy this thread started land before the block can exit.
        for (int t = 0; t < 2; ++t) {
          if (loads[t] > 0) wd.drain(bar(L::kBarQFull + t), parity(loads[t] - 1));
        }
      }
    } else {
      // ------------------------------------------------- MMA issuer of query tile t
      // The whole warp runs this loop: waits are taken by every lane and decided by
      // a vote, descriptors are warp-uniform, and one elected lane issues each MMA
      // and commit.
      {
        const int t = warp - 9;
        const uint32_t s_tmem = tmem + 128u * t;                           // S_t, and P_t over it
        const uint32_t o_tmem = tmem + 256u + static_cast<uint32_t>(D) * t;  // O_t
        const int qb = kHalves ? 0 : t;  // Q buffer (and its barriers) of this issuer
        const uint64_t q_desc = smem_desc_sw128(sbase + L::kQOff + qb * L::kTileBytes, 16, 1024);
        const uint64_t ring_v_desc = smem_desc_sw128(sbase + L::kRingOff, kSubTileBytes, 1024);
        const uint64_t ring_k_desc = smem_desc_sw128(sbase + L::kRingOff + L::kTileBytes, 16, 1024);
        auto stage_off = [&](int item) {  // stage offset in the descriptors' >>4 address field
          return static_cast<uint64_t>((item % L::kStages) * (L::kStageBytes >> 4));
        };
        auto warp_wait = [&](uint32_t b, uint32_t ph) -> bool {
          return __all_sync(0xffffffffu, wd.wait(b, ph)) != 0;
        };
        // The issuers take turns, one per ring item each, tile 0 first: a turn's
        // MMAs stay contiguous in the pipe, so one tile's MMAs run while the other
        // tile's softmax works.
        int turns = 0;
        auto take_turn = [&]() -> bool { return warp_wait(bar(L::kBarTurn + t), parity(turns++)); };
        auto pass_turn = [&]() {
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(L::kBarTurn + (1 - t)));
        };
        int it = 0;       // ring items of the units done so far (both slots')
        int p_waits = 0;  // P_t handshakes consumed
        int used = 0;     // earlier units in which tile t existed (its O_t is read by an epilogue)
        int q_loads = 0;  // Q loads of tile t consumed
        bool ok = true;
        Unit w;
        while (ok) {
          const int got = next_unit(w, true);
          if (got != 1) {
            ok = got == 0;
            break;
          }
          const int n_kv = t ? w.n_kv1 : w.n_kv0;
          // Ring item of this issuer's step i: every item of the unit (both slots use
          // it), or with key halves every other one, starting with its own slot.
          const int base = it;
          auto item = [&](int i) { return kHalves ? base + 2 * i + t : base + i; };
          int x = item(0);
          // Item 0 (K_0).  Every item this issuer consumes is waited for and released
          // whether or not its tile uses it, so the ring's phases stay aligned (two
          // arrivals per item, or one with key halves).
          // With key halves Q is loaded once per unit, so both issuers count every load.
          const bool q_wait = n_kv > 0 && !warp_wait(bar(L::kBarQFull + qb), parity(q_loads));
          if (n_kv > 0 || kHalves) ++q_loads;
          if (q_wait || !warp_wait(bar(L::kBarFull + x % L::kStages), parity(x / L::kStages)) ||
              !warp_wait(bar(L::kBarFullK + x % L::kStages), parity(x / L::kStages))) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          if (!take_turn()) {
            ok = false;
            break;
          }
          if (n_kv > 0) issue_qk<D, BF16>(s_tmem, q_desc, ring_k_desc + stage_off(x));
#ifdef ECA_ANATOMY
          if (t == 0 && base == 0 && lane == 0) ECA_STAMP(an_slot, 3);  // first Q K^T issued
          if (t == 0 && lane == 0) ++an_units;
#endif
          pass_turn();
          if (n_kv > 0) tc_commit_warp(bar(L::kBarS + t));
          if (n_kv == 1) tc_commit_warp(bar(L::kBarQFree + qb));  // this tile's Q K^T are all issued
          // A key-halves slot with no keys releases the shared Q buffer at once: this
          // turn comes after the other issuer's first Q K^T of the unit, so the
          // buffer's previous phase is complete.
          if (kHalves && n_kv == 0) {
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(L::kBarQFree + qb));
          }
          tc_commit_warp(bar(L::kBarEmpty + x % L::kStages));
          for (int j = 0; j < w.n_max; ++j) {
            x = item(j + 1);
            if (!warp_wait(bar(L::kBarFull + x % L::kStages), parity(x / L::kStages))) {
              ok = false;
              break;
            }
            if (j < n_kv) {
              // O_t is overwritten by the first P V of a unit: the previous epilogue must have read it.
              if (j == 0 && used > 0 && !warp_wait(bar(L::kBarOFree + t), parity(used - 1))) {
                ok = false;
                break;
              }
              if (!warp_wait(bar(L::kBarPa + t), parity(p_waits))) {
                ok = false;
                break;
              }
              ++p_waits;
              tc_fence_after_sync();
            }
            if (!take_turn()) {
              ok = false;
              break;
            }
            if (j < n_kv) {
              // P V of keys 0-63 goes in while the softmax still works on keys 64-127.
              issue_pv<D, BF16>(o_tmem, s_tmem, ring_v_desc + stage_off(x), j > 0, 0, 4);
              if (!warp_wait(bar(L::kBarPb + t), parity(p_waits - 1))) {
                ok = false;
                break;
              }
              tc_fence_after_sync();
              issue_pv<D, BF16>(o_tmem, s_tmem, ring_v_desc + stage_off(x), true, 4, 8);
            }
            if (!warp_wait(bar(L::kBarFullK + x % L::kStages), parity(x / L::kStages))) {
              ok = false;
              break;
            }
            if (j + 1 < n_kv) {
              tc_fence_after_sync();
              issue_qk<D, BF16>(s_tmem, q_desc, ring_k_desc + stage_off(x));
            }
            pass_turn();
            if (j < n_kv) {
              if (j + 1 < n_kv) {
                tc_commit_warp(bar(L::kBarS + t));
                if (j + 2 == n_kv) tc_commit_warp(bar(L::kBarQFree + qb));
              } else {
                tc_commit_warp(bar(L::kBarO + t));
              }
            }
            tc_commit_warp(bar(L::kBarEmpty + x % L::kStages));
          }
          it = base + (kHalves ? 2 : 1) * (w.n_max + 1);
          used += n_kv > 0 ? 1 : 0;
        }
        // Every MMA issued above must finish before TMEM is released.
        tc_commit_warp(bar(L::kBarDrain + t));
        wd.drain(bar(L::kBarDrain + t), 0);
      }
    }
  } else {
    if constexpr (kSplitRegs) setmaxnreg_inc<kRegsSoftmax>();
    // ------------------------------------------------------------------ softmax
    const int t = warp / 4;
    const int wq = warp % 4;
    const int r_local = wq * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t t_s = tmem + lane_base + 128u * t;
    const uint32_t t_o = tmem + lane_base + 256u + static_cast<uint32_t>(D) * t;
    const float c = p.scale_log2e;
    const bool ragged_keys = !p.causal && (p.N % kBlockN) != 0;
    // Waits stay warp-uniform: the tcgen05.ld/st below are warp-collective.
    auto warp_wait = [&](uint32_t b, uint32_t ph) -> bool {
      const bool got = wd.wait(b, ph);
      return __all_sync(0xffffffffu, got) != 0;
    };
    float* merge_ml = reinterpret_cast<float*>(smem + L::kMergeOff);  // key halves: slot 1's m, then l
    int s_waits = 0, o_waits = 0;
    int merges = 0;  // slot 0 with key halves: units whose slot 1 had work
    bool ok = true;
    Unit w;
    while (ok) {
      const int got = next_unit(w, true);
      if (got != 1) {
        ok = got == 0;
        break;
      }
      const int n_kv = t ? w.n_kv1 : w.n_kv0;
      if (n_kv == 0) continue;
      const int kvb = t ? w.kv1 : w.kv0;  // this slot's first key tile
      const int tile = w.tile0 + ((p.head_pair || kHalves) ? 0 : t);
      const int head = w.bh + (p.head_pair ? t : 0);
      const int row = tile * kBlockM + r_local;
      // Reference max, base-2 domain (already multiplied by c).  Under the fixed
      // assignment a unit starts from a guess, kept on the first key tile only if
      // that tile's sum of p reaches 1 (a rejected guess is replaced, not kept).
      // (The dynamic instance starts from the first tile's max: with the guess it
      // measured 0.5-1% slower at N = 8192.)
      constexpr bool kGuessFirst = !kDynamic;
      float m_ref = kGuessFirst ? kGuessRef : -INFINITY;
      float l = 0.f;
      for (int j = 0; j < n_kv; ++j) {
        if (!warp_wait(bar(L::kBarS + t), parity(s_waits))) {
          ok = false;
          break;
        }
        ++s_waits;
#ifdef ECA_ANATOMY
        if (t == 0 && s_waits == 1 && wq == 0 && lane == 0) ECA_STAMP(an_slot, 4);  // first S ready
#endif
        tc_fence_after_sync();
        uint32_t s[4][32];
        // S of this key tile, masked: the diagonal tile (causal) or the ragged
        // last tile (non-causal).
        auto load_scores = [&]() {
#pragma unroll
          for (int q = 0; q < 4; ++q) tmem_ld_x32(t_s + 32u * q, s[q]);
#pragma unroll
          for (int q = 0; q < 4; ++q) tmem_wait_ld_x32(s[q]);
          if (p.causal && kvb + j == tile) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (32 * q + i > r_local) s[q][i] = __float_as_uint(-INFINITY);
          } else if (ragged_keys && kvb + j == p.n_tiles - 1) {
            const int valid = p.N - (kvb + j) * kBlockN;
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (32 * q + i >= valid) s[q][i] = __float_as_uint(-INFINITY);
          }
        };
        // p = 2^(s c - m_ref), packed for the P V MMA.
        uint32_t pk[2][32];
        // Columns 32 q0 .. 32 q1 - 1 of the row into acc; called with (0, 4), or
        // with (0, 2) then (2, 4) when keys 64-127 are still loading.
        auto exp_quarters = [&](int q0, int q1, float neg_m, float2 (&acc)[8]) {
          const float2 c2 = make_float2(c, c);
          const float2 nm2 = make_float2(neg_m, neg_m);
#pragma unroll
          for (int q = q0; q < q1; ++q) {
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              const float2 x = __ffma2_rn(make_float2(__uint_as_float(s[q][i]), __uint_as_float(s[q][i + 1])), c2, nm2);
              const float2 e = make_float2(ex2(x.x), ex2(x.y));
              acc[(i / 2) % 8] = __fadd2_rn(acc[(i / 2) % 8], e);  // eight short add chains
              pk[q / 2][(q % 2) * 16 + i / 2] = pack2<BF16>(e.x, e.y);
            }
          }
        };
        auto row_total = [](const float2 (&acc)[8]) -> float {
          const float2 a = __fadd2_rn(__fadd2_rn(__fadd2_rn(acc[0], acc[1]), __fadd2_rn(acc[2], acc[3])),
                                      __fadd2_rn(__fadd2_rn(acc[4], acc[5]), __fadd2_rn(acc[6], acc[7])));
          return a.x + a.y;
        };
        // p = 2^(s c - m_ref) for the whole row in registers; returns sum p.
        auto exponentiate = [&](float neg_m) -> float {
          float2 acc[8];
#pragma unroll
          for (int a = 0; a < 8; ++a) acc[a] = make_float2(0.f, 0.f);
          exp_quarters(0, 4, neg_m, acc);
          return row_total(acc);
        };

        float alpha = 1.f;
        float row_sum = 0.f;
        bool move = true;  // without a guess, the first key tile takes the row max
        if (kGuessFirst || j > 0) {
          const bool masked = (p.causal && kvb + j == tile) || (ragged_keys && kvb + j == p.n_tiles - 1);
          if (masked && j == 0) {
            // A masked first tile (the diagonal, or the only, ragged, key tile) holds a
            // row's first keys: take their max, as a guessed reference would round a
            // lone key's p in 16 bits where p = 1 is exact.
            move = true;
          } else if (masked) {
            load_scores();
            row_sum = exponentiate(-m_ref);
            move = !(row_sum <= max_row_sum<BF16>());  // (also an inf sum)
          } else {
            // Keys 64-127 load while keys 0-63 are exponentiated.
            tmem_ld_x32(t_s, s[0]);
            tmem_ld_x32(t_s + 32u, s[1]);
            tmem_wait_ld_x32(s[0]);
            tmem_wait_ld_x32(s[1]);
            tmem_ld_x32(t_s + 64u, s[2]);
            tmem_ld_x32(t_s + 96u, s[3]);
            float2 acc[8];
#pragma unroll
            for (int a = 0; a < 8; ++a) acc[a] = make_float2(0.f, 0.f);
            exp_quarters(0, 2, -m_ref, acc);
            const float sum_a = row_total(acc);
            tmem_wait_ld_x32(s[2]);
            tmem_wait_ld_x32(s[3]);
            float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              mx[0] = fmax3(mx[0], __uint_as_float(s[2][i]), __uint_as_float(s[2][i + 1]));
              mx[1] = fmax3(mx[1], __uint_as_float(s[3][i]), __uint_as_float(s[3][i + 1]));
            }
            // Keys 0-63 are handed over before keys 64-127 are exponentiated, so the
            // reference must hold for the whole row now: keys 0-63 are safe when
            // their sum of p is at most the bound, keys 64-127 when their max score
            // is at most the lead bound (log2 of the sum bound) above the reference.  A guess (first tile)
            // also needs the row's sum of p to reach 1, which keys 0-63 show by their
            // sum and keys 64-127 by a max score at or above the reference (p >= 1).
            const float top_b = fmaxf(mx[0], mx[1]) * c - m_ref;
            const bool fast = sum_a <= max_row_sum<BF16>() && top_b <= max_lead<BF16>() &&
                              (j > 0 || sum_a >= kMinGuessSum || top_b >= 0.f);
            if (__all_sync(0xffffffffu, fast)) {
              tmem_st_x32(t_s, pk[0]);
              tmem_wait_st();
              tc_fence_before_sync();
              __syncwarp();
              if (lane == 0) mbar_arrive(bar(L::kBarPa + t));
#pragma unroll
              for (int a = 0; a < 8; ++a) acc[a] = make_float2(0.f, 0.f);
              exp_quarters(2, 4, -m_ref, acc);
              tmem_st_x32(t_s + 32u, pk[1]);
              tmem_wait_st();
              tc_fence_before_sync();
              __syncwarp();
              if (lane == 0) mbar_arrive(bar(L::kBarPb + t));
              l += sum_a + row_total(acc);
              continue;
            }
            // A row that failed a bound, or whose guess fell short, takes the row max;
            // the other rows keep their reference, which the checks above showed to
            // hold for them (no second pass over the row to decide).
            move = !fast;
          }
        }
        if (__any_sync(0xffffffffu, move)) {
          load_scores();  // S is still intact in TMEM: P has not been stored yet
          if (move) {
            float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
#pragma unroll
              for (int q = 0; q < 4; ++q)
                mx[q] = fmax3(mx[q], __uint_as_float(s[q][i]), __uint_as_float(s[q][i + 1]));
            }
            const float m_tile = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * c;
            const float m_new = j == 0 ? m_tile : fmaxf(m_ref, m_tile);
            alpha = (j == 0 || m_ref == -INFINITY) ? 0.f : ex2(m_ref - m_new);
            m_ref = m_new;
          }
          row_sum = exponentiate(m_ref == -INFINITY ? 0.f : -m_ref);
        }
        l = l * alpha + row_sum;
        tmem_st_x32(t_s, pk[0]);
        tmem_st_x32(t_s + 32u, pk[1]);

        // Rescale the running O before this tile's P V is added (P V of tile j-1 is
        // complete: S of tile j was committed after it by the same issuer).
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          const float2 al2 = make_float2(alpha, alpha);
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t o[32];
            tmem_ld_x32(t_o + c0, o);
            tmem_wait_ld_x32(o);
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              const float2 v = __fmul2_rn(make_float2(__uint_as_float(o[i]), __uint_as_float(o[i + 1])), al2);
              o[i] = __float_as_uint(v.x);
              o[i + 1] = __float_as_uint(v.y);
            }
            tmem_st_x32(t_o + c0, o);
          }
        }
        tmem_wait_st();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar(L::kBarPa + t));
          mbar_arrive(bar(L::kBarPb + t));
        }
      }
      if (!ok || !warp_wait(bar(L::kBarO + t), parity(o_waits))) {
        ok = false;
        break;
      }
      ++o_waits;
#ifdef ECA_ANATOMY
      if (o_waits == 1 && wq == 0 && lane == 0) ECA_STAMP(an_slot, t == 0 ? 5 : 7);  // first unit's O ready
#endif
      tc_fence_after_sync();

      if (kHalves && t == 1) {
        // Key halves: slot 1 hands its m and l to slot 0, whose epilogue merges O_1
        // in and then releases it for the next unit.
        merge_ml[r_local] = m_ref;
        merge_ml[kBlockM + r_local] = l;
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(L::kBarMerge));
        continue;
      }
      // Key halves: merge slot 1's state with the online-softmax law, M = max(m0, m1),
      // L = l0 2^(m0 - M) + l1 2^(m1 - M), O = (O_0 2^(m0 - M) + O_1 2^(m1 - M)) / L.
      const bool merge = kHalves && w.n_kv1 > 0;
      float m_fin = m_ref, l_fin = l, w0 = 1.f, w1 = 0.f;
      if (merge) {
        if (!warp_wait(bar(L::kBarMerge), parity(merges)) || !warp_wait(bar(L::kBarO + 1), parity(merges))) {
          ok = false;
          break;
        }
        ++merges;
        tc_fence_after_sync();
        const float m1 = merge_ml[r_local], l1 = merge_ml[kBlockM + r_local];
        m_fin = fmaxf(m_ref, m1);
        w0 = m_ref == -INFINITY ? 0.f : ex2(m_ref - m_fin);
        w1 = m1 == -INFINITY ? 0.f : ex2(m1 - m_fin);
        l_fin = w0 * l + w1 * l1;
      }
      const uint32_t t_o1 = tmem + lane_base + 256u + static_cast<uint32_t>(D);  // O_1, merged in with key halves

      // Epilogue: O = o / l rounded to the output type, lse = (m + log2 l) ln 2;
      // with a key split, the segment's O in fp32 and its lse go to the workspace.
      const float inv_l = 1.f / l_fin;
      const float2 il2 = make_float2(w0 * inv_l, w0 * inv_l);
      const float2 il2b = make_float2(w1 * inv_l, w1 * inv_l);
      const float row_lse = (m_fin + log2f(l_fin)) * 0.69314718055994530942f;
      if (p.part_o != nullptr) {
        const size_t prow = (static_cast<size_t>(w.seg) * p.BH + head) * p.N + static_cast<size_t>(row);
        float* dst = p.part_o + prow * D;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t o[32];
          tmem_ld_x32(t_o + c0, o);
          tmem_wait_ld_x32(o);
          if (row < p.N) {
            float4* d4 = reinterpret_cast<float4*>(dst + c0);
#pragma unroll
            for (int v4 = 0; v4 < 8; ++v4) {
              const float2 a = __fmul2_rn(make_float2(__uint_as_float(o[4 * v4]), __uint_as_float(o[4 * v4 + 1])), il2);
              const float2 b = __fmul2_rn(make_float2(__uint_as_float(o[4 * v4 + 2]), __uint_as_float(o[4 * v4 + 3])), il2);
              d4[v4] = make_float4(a.x, a.y, b.x, b.y);
            }
          }
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(L::kBarOFree + t));
        if (row < p.N) p.part_lse[prow] = row_lse;
        continue;
      }
      // O = o / l rounded to the output type, 64 columns at a time.  Each warp
      // sends its 32 rows through its slab of the staging buffer with TMA stores
      // (rows past N are clipped by the tensor map).
      // With key halves slot 1 stores nothing, so slot 0 sends its two 64-column
      // blocks through both tiles' staging buffers and need not wait between them.
#pragma unroll
      for (int c64 = 0; c64 < D / 64; ++c64) {
        const uint32_t slab = sbase + L::kOutOff + (kHalves ? c64 : t) * L::kStageOutBytes + wq * 4096;
        // With the register split, the block's 64 columns (and with key halves O_1's)
        // are loaded with one wait.
        uint32_t h[32];
        if (merge) {
          uint32_t o[2][32], o1[2][32];
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            tmem_ld_x32(t_o + 64 * c64 + 32 * half, o[half]);
            tmem_ld_x32(t_o1 + 64 * c64 + 32 * half, o1[half]);
          }
          tmem_wait_ld_x32(o[0]);
          tmem_tie_x32(o[1]);
          tmem_tie_x32(o1[0]);
          tmem_tie_x32(o1[1]);
#pragma unroll
          for (int half = 0; half < 2; ++half) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float2 a = __fmul2_rn(
                  make_float2(__uint_as_float(o[half][2 * i]), __uint_as_float(o[half][2 * i + 1])), il2);
              const float2 v = __ffma2_rn(
                  make_float2(__uint_as_float(o1[half][2 * i]), __uint_as_float(o1[half][2 * i + 1])), il2b, a);
              h[16 * half + i] = pack2<BF16>(v.x, v.y);
            }
          }
        } else if constexpr (kSplitRegs) {
          uint32_t o[2][32];
          tmem_ld_x32(t_o + 64 * c64, o[0]);
          tmem_ld_x32(t_o + 64 * c64 + 32, o[1]);
          tmem_wait_ld_x32(o[0]);
          tmem_tie_x32(o[1]);
#pragma unroll
          for (int half = 0; half < 2; ++half) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float2 v = __fmul2_rn(
                  make_float2(__uint_as_float(o[half][2 * i]), __uint_as_float(o[half][2 * i + 1])), il2);
              h[16 * half + i] = pack2<BF16>(v.x, v.y);
            }
          }
        } else {
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t o[32];
            tmem_ld_x32(t_o + 64 * c64 + 32 * half, o);
            tmem_wait_ld_x32(o);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float2 v = __fmul2_rn(make_float2(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1])), il2);
              h[16 * half + i] = pack2<BF16>(v.x, v.y);
            }
          }
        }
        if (c64 == D / 64 - 1) {
          // O_t (and with key halves O_1) has been read: the next unit's first P V
          // may overwrite it.
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(bar(L::kBarOFree + t));
            if (merge) mbar_arrive(bar(L::kBarOFree + 1));
          }
        }
        // The slab's previous contents have been read (with key halves, the first
        // wait covers both slabs).
        if (lane == 0 && (!kHalves || c64 == 0)) bulk_wait_read_all();
        __syncwarp();
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          const uint32_t dst = slab + lane * 128 + ((ch ^ (lane & 7)) << 4);
          st_shared_v4(dst, h[4 * ch], h[4 * ch + 1], h[4 * ch + 2], h[4 * ch + 3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_3d(&tm_o, slab, 64 * c64, tile * kBlockM + wq * 32, head);
          bulk_commit_group();
        }
      }
      if (p.lse != nullptr && row < p.N) {
        p.lse[static_cast<size_t>(head) * p.N + row] = row_lse;
      }
#ifdef ECA_ANATOMY
      if (t == 0 && o_waits == 1 && wq == 0 && lane == 0) ECA_STAMP(an_slot, 6);  // first unit's output issued
#endif
    }
    // The staging slabs must stay valid until the stores have read them; the
    // writes themselves complete before the grid does.
    if (lane == 0) bulk_wait_read_all();
  }

  tc_fence_before_sync();
  __syncthreads();
  if (kDynamic && threadIdx.x == 0) {
    // The last CTA to finish returns the launch's counters to zero for the next launch.
    __threadfence();
    if (atomicAdd(p.sched + 32, 1) == static_cast<int>(gridDim.x) - 1) {
      atomicExch(p.sched, 0);
      atomicExch(p.sched + 32, 0);
    }
  }
  if (warp == 9) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
#ifdef ECA_ANATOMY
    if (lane == 0) {
      ECA_STAMP(an_slot, 8);  // exit
      if (blockIdx.x < kAnatomyCtas) g_anatomy[an_slot][blockIdx.x][9] = static_cast<unsigned long long>(an_units);
      __threadfence();
      if (atomicAdd(&g_anatomy_exited, 1) == static_cast<int>(gridDim.x) - 1) {
        g_anatomy_exited = 0;
        __threadfence();
        atomicAdd(&g_anatomy_launch, 1);
      }
    }
#endif
  }
}

}  // namespace eca
