/*
 * exact_causal_attention_gb300 -- C ABI of the attention forward library.
 *
 * The operation (page "CUDA FlashAttention：从在线 Softmax 到长序列 IO 极限",
 * chengzipai.xyz, section 1) is the exact scaled-dot-product attention forward
 *
 *     O = softmax(scale * Q K^T + M) V,     M_ij = 0 if j <= i, else -inf  (causal)
 *
 * computed with the tiled online-softmax recurrence of that page's section 4,
 * so the N x N score matrix is never written to memory.  It also returns the
 * natural-log log-sum-exp of every score row, lse_i = ln sum_j exp(s_ij) with
 * s_ij = scale * q_i . k_j over the unmasked j, which the page's section 7 says
 * training must keep.
 *
 * Layout (all tensors contiguous, row-major, last index fastest):
 *   q, k, v, o : [B, H, N, D] 16-bit elements (fp16 for attn_fwd, bf16 for
 *                attn_fwd_bf16); one N serves queries and keys.
 *   lse        : [B, H, N] fp32, or NULL to skip it.
 * The causal mask is the top-left square one (key j visible to query i iff
 * j <= i).  Arithmetic: fp16/bf16 products accumulated in fp32 on the tensor
 * cores, running max m, sum l and unnormalised output o kept in fp32 (the page's
 * section 2), probabilities rounded to the input type before the P V product,
 * O rounded to nearest even.  The kernel's m is a reference that may trail the
 * row's max as long as no probability can leave the 16-bit range, or start from
 * a fixed guess that is kept only when the first key tile's probabilities sum to
 * at least 1 (so the running sum l stays >= 1, as with the row max); the
 * recurrence gives the same O and lse for any reference, so this changes only
 * rounding.
 *
 * Ownership: every pointer is device memory owned by the caller; the library
 * allocates nothing per call and keeps no reference after the call returns.
 * Asynchrony: the call only enqueues work on `stream` (NULL = legacy default
 * stream) and never synchronises; a fault during execution surfaces at the
 * caller's next synchronisation.  Calls may come from several host threads (the
 * host side serialises them on one lock).
 *
 * Launch order: kernels are launched with programmatic stream serialisation
 * (programmatic dependent launch).  Stream order is kept for memory: a kernel's
 * CTAs may be scheduled while the work ahead of it on the stream still runs, but
 * they touch no global memory before it has completed.  The attention and
 * decode kernels also let the next such launch on the stream be scheduled once
 * their set-up is done (the row softmax at once), so back-to-back calls lose
 * less time between launches.
 * A kernel of the caller's that is launched with the same attribute right after
 * one of these calls must likewise wait for the grid ahead of it
 * (griddepcontrol.wait / cudaGridDependencySynchronize) before reading its
 * outputs.  ECA_PDL=0 in the environment, read once per process, launches in
 * plain stream order instead.
 *
 * Concurrency limits: launches whose key/value tensors together exceed 64 MiB
 * hand out their work from a device counter, taken from a pool of 64 per device
 * in turn; the split paged decode's in-kernel merge uses counters from a pool of
 * 8.  A counter is handed to a new launch only once the launch that last held
 * it has finished: the library makes the new launch's stream wait for an event
 * recorded after the old one, so more launches than the pool holds in flight at
 * once run one after another where they would share a counter, and are never
 * corrupted.  Under stream capture no event is used and a launch keeps the
 * counter it was captured with; two graphs whose captured launches hold the same
 * counter (captured 64, or 8, such launches apart) must not run at once.
 *
 * Bounded waits: every wait inside a kernel gives up after 2 s without progress
 * (a bug, or a kernel kept off the GPU that long).  The kernel then stops early
 * and leaves its outputs incomplete; the call that launched it has already
 * returned ATTN_OK, and only attn_device_status reports ATTN_ERR_TIMEOUT.  Call
 * attn_device_status after work whose results matter when a stall must not pass
 * unnoticed.
 *
 * Errors: arguments are checked before anything touches the GPU; an invalid
 * call returns a negative status and launches nothing (section 9 of the page:
 * unsupported shapes are rejected, never answered wrongly).
 */
#ifndef EXACT_CAUSAL_ATTENTION_GB300_ATTN_H_
#define EXACT_CAUSAL_ATTENTION_GB300_ATTN_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t, declared without the CUDA headers. */
typedef struct CUstream_st* attn_stream_t;

enum attn_status {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = -1,    /* NULL tensor pointer, B/H/N < 1, scale not finite and > 0,
                                   or sizes whose offsets overflow 64 bits / TMA limits */
  ATTN_ERR_UNALIGNED = -2,      /* a tensor pointer is not 16-byte aligned */
  ATTN_ERR_UNSUPPORTED_D = -3,  /* D is not 64 or 128 */
  ATTN_ERR_ARCH = -4,           /* the current device is not an sm_103 part */
  ATTN_ERR_LAUNCH = -5,         /* the CUDA runtime refused the launch, or the library was built with
                                   fewer registers per thread than its attention kernel's warpgroups
                                   move between them (checked before the first launch) */
  ATTN_ERR_TIMEOUT = -6,        /* a kernel's bounded wait expired (reported by attn_device_status) */
  ATTN_ERR_CUDA = -7,           /* another CUDA runtime/driver call failed */
  ATTN_ERR_SCRATCH_LIMIT = -8,  /* attn_fwd_splitkv_noalloc: the split needs more than its fixed scratch */
  ATTN_ERR_BAD_INDEX = -9       /* paged cache: a block-table entry or length out of range (reported by
                                   attn_device_status; those tokens were skipped, not read) */
};

/*
 * attn_fwd -- fp16 attention forward.
 *   q, k, v : device, [B, H, N, D] fp16, 16-byte aligned, read only.
 *   o       : device, [B, H, N, D] fp16, 16-byte aligned, written in full.
 *   lse     : device, [B, H, N] fp32, 4-byte aligned, written in full; or NULL.
 *   B, H, N : >= 1.   D : 64 or 128.   causal : 0 or nonzero.
 *   scale   : finite and > 0 (1/sqrt(D) for the usual attention).
 *   stream  : the caller's CUDA stream.
 * o must not overlap q, k or v.  Returns ATTN_OK or a negative attn_status.
 */
int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
             int D, int causal, float scale, attn_stream_t stream);

/* attn_fwd_bf16 -- the same operation and contract with bf16 q, k, v and o. */
int attn_fwd_bf16(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                  int N, int D, int causal, float scale, attn_stream_t stream);

/*
 * attn_fwd_gqa -- fp16 attention forward with grouped key/value heads (GQA; MQA
 * when Hkv = 1), page "CUDA KV Cache：分页存储与长上下文 Decode 极致优化", section
 * 3.3: with g = H / Hkv, query head h reads key/value head floor(h / g) of the
 * same batch entry, and K/V are not copied per query head.
 *   q, o : [B, H, N, D].    k, v : [B, Hkv, N, D].    lse : [B, H, N] or NULL.
 *   Hkv  : >= 1 and divides H.  Hkv = H is attn_fwd.
 * Everything else as attn_fwd.  Returns ATTN_ERR_INVALID_ARG when Hkv does not
 * divide H.
 */
int attn_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                 int Hkv, int N, int D, int causal, float scale, attn_stream_t stream);

/* attn_fwd_gqa_bf16 -- the same with bf16 q, k, v and o. */
int attn_fwd_gqa_bf16(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                      int Hkv, int N, int D, int causal, float scale, attn_stream_t stream);

/*
 * attn_fwd_splitkv -- the same operation with the key tiles split into
 * segments that run as separate work units (page "CUDA KV Cache：分页存储与长上下
 * 文 Decode 极致优化", section 6.4: when B x heads is too small to fill the GPU
 * and the sequence is long, each segment produces its own (m, l, o) and a second
 * kernel merges them with the online-softmax law).  Same arguments and result as
 * attn_fwd, plus:
 *   kv_splits       : requested segments, 1 .. 64 (fewer are used when N has
 *                     fewer 128-key tiles); see attn_splitkv_default_splits.
 *   workspace       : device memory owned by the caller, 256-byte aligned, at
 *                     least attn_splitkv_workspace_bytes(B, H, N, D, kv_splits)
 *                     bytes, not overlapping q, k, v or o.  It holds the fp32
 *                     partial outputs and log-sum-exps; its contents on entry do
 *                     not matter and are overwritten.  Two calls must not share
 *                     one workspace while both may be running.
 *   workspace_bytes : its size.
 * Returns ATTN_ERR_INVALID_ARG for kv_splits outside 1 .. 64, a NULL or too
 * small workspace, or overlap; ATTN_ERR_UNALIGNED for a misaligned workspace.
 */
int attn_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                     int N, int D, int causal, float scale, int kv_splits, void* workspace,
                     size_t workspace_bytes, attn_stream_t stream);

/* attn_fwd_splitkv_bf16 -- the same with bf16 q, k, v and o. */
int attn_fwd_splitkv_bf16(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                          int H, int N, int D, int causal, float scale, int kv_splits,
                          void* workspace, size_t workspace_bytes, attn_stream_t stream);

/*
 * attn_fwd_splitkv_noalloc -- attn_fwd_splitkv (fp16) for callers that cannot
 * allocate device memory: code whose device memory is all owned by a host
 * framework's own pool or budget, plugins that are handed only their input and
 * output buffers, and latency-bound callers that must not pay for an allocation
 * call on the hot path.  The pages have no counterpart of this entry point.
 *
 * The partial results live in one scratch array that the library declares at
 * file scope: 64 MiB per device, reserved on every GPU that loads the library
 * and held until the process exits.  The caller passes q, k, v, o and lse as
 * for attn_fwd_splitkv, but no workspace; nothing is allocated.  A call whose
 * split needs more than 64 MiB (see attn_splitkv_workspace_bytes) returns
 * ATTN_ERR_SCRATCH_LIMIT and launches nothing.
 * The first call on a device looks up the scratch array's device address (once
 * per device, with that device current); make that first call before any stream
 * capture.  Every call uses the same array, which keeps whatever the last call
 * left there; no part of it needs to start at zero, since each call writes every
 * value it later reads.  Calls whose kernels may overlap on the GPU (other
 * streams, other host threads) race on the array: order them.
 */
int attn_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                             int H, int N, int D, int causal, float scale, int kv_splits,
                             attn_stream_t stream);

/* Bytes of workspace attn_fwd_splitkv needs for these sizes; 0 for invalid sizes.
 * Needs no GPU. */
size_t attn_splitkv_workspace_bytes(int B, int H, int N, int D, int kv_splits);

/* A split count for the current device: 1 when there are at least two work
 * units (pairs of 128-row query tiles of one head) per SM; otherwise the count
 * whose predicted time is shortest, from a replay of the kernel's schedule
 * (units taken in order by whichever SM is free first) plus the merge kernel's
 * traffic (1 .. 64, at most the number of 128-key tiles).  Negative attn_status on bad sizes or a non-sm_103
 * device. */
int attn_splitkv_default_splits(int B, int H, int N, int D);

/*
 * attn_decode_paged -- one decode step of attention over a paged K/V cache with
 * grouped heads (page "CUDA KV Cache：分页存储与长上下文 Decode 极致优化": layout
 * and address rule of section 2, GQA head map of section 3.3, warp dataflow of
 * section 5, split-KV of section 6.4).  Request b's query (one token per head)
 * attends all lengths[b] tokens of its context:
 *     O[b, h] = softmax_t(scale * q[b, h] . K[b, t, h / g]) V[b, t, h / g],  g = Hq / Hkv,
 * where token t of request b lives on page block_table[b, t / page_size] at
 * offset t % page_size.
 *   q           : device, [B, Hq, D] fp16, 16-byte aligned.
 *   cache       : device, [num_pages, 2, page_size, Hkv, D] fp16 (index 0 = K,
 *                 1 = V), 16-byte aligned, read only.
 *   block_table : device, [B, max_pages] int32; entries past a request's last
 *                 page may be read (they lie inside the row) but are never
 *                 followed, so their values do not matter.
 *   lengths     : device, [B] int32, 0 .. max_pages * page_size.
 *   out         : device, [B, Hq, D] fp16, written in full.
 *   lse         : device, [B, Hq] fp32 natural-log log-sum-exp, or NULL.
 *   Hq % Hkv == 0.  D : 64 or 128.  page_size : 8, 16, 32 or 64.
 *   num_pages * 2 * page_size < 2^31 (the cache's token rows are addressed with
 *   32-bit tensor coordinates); max_pages * page_size < 2^31.
 *   scale       : finite and > 0.
 *   kv_splits   : 1 .. 64 segments of the context (see attn_decode_default_splits);
 *                 more than one needs `workspace` (256-byte aligned, at least
 *                 attn_decode_workspace_bytes(B, Hq, D, kv_splits) bytes,
 *                 contents on entry irrelevant); with 1 it may be NULL.
 * A request with length 0 gets O = 0 and lse = -inf.  A block-table entry
 * outside [0, num_pages) or a length outside [0, max_pages * page_size] is not
 * followed: the tokens it names are skipped and attn_device_status reports
 * ATTN_ERR_BAD_INDEX.  As in attn_fwd, P is rounded to the input's 16-bit type for
 * the P V product; scores, sums and O accumulate in fp32.
 */
int attn_decode_paged(const void* q, const void* cache, const int* block_table, const int* lengths,
                      void* out, float* lse, int B, int Hq, int Hkv, int D, int page_size,
                      int max_pages, int num_pages, float scale, int kv_splits, void* workspace,
                      size_t workspace_bytes, attn_stream_t stream);

/* attn_decode_paged_bf16 -- the same with bf16 q, cache and out. */
int attn_decode_paged_bf16(const void* q, const void* cache, const int* block_table,
                           const int* lengths, void* out, float* lse, int B, int Hq, int Hkv, int D,
                           int page_size, int max_pages, int num_pages, float scale, int kv_splits,
                           void* workspace, size_t workspace_bytes, attn_stream_t stream);

/* Workspace bytes of attn_decode_paged for kv_splits > 1 (0 when none is needed or
 * the sizes are invalid).  Needs no GPU. */
size_t attn_decode_workspace_bytes(int B, int Hq, int D, int kv_splits);

/* A context split for the current device: about two decode CTAs per SM (the
 * measured best at every context length of the page's benchmark geometry),
 * capped by the 64-token tiles of max_pages * page_size and by 64.  When the split
 * is used, the segments are merged inside the decode kernel (by each group's last
 * segment) unless B * Hkv * head chunks exceeds 4096, when a second kernel merges
 * them.  Negative attn_status on bad sizes or a non-sm_103 device. */
int attn_decode_default_splits(int B, int Hq, int Hkv, int page_size, int max_pages);

/*
 * attn_paged_append -- writes the newest token of every request into the paged
 * cache (the same page's section 4): row (b, kind, head) of new_kv
 * [B, 2, Hkv, D] (16-bit, 16-byte aligned) goes to
 * cache[block_table[b, t / page_size]][kind][t % page_size][head] with
 * t = lengths[b] - 1, as 16-byte stores.  Sizes and layout as attn_decode_paged;
 * element type does not matter (a copy of 16-bit values).  Out-of-range entries
 * are skipped and reported as ATTN_ERR_BAD_INDEX by attn_device_status.
 */
int attn_paged_append(const void* new_kv, void* cache, const int* block_table, const int* lengths,
                      int B, int Hkv, int D, int page_size, int max_pages, int num_pages,
                      attn_stream_t stream);

/*
 * attn_row_softmax_f32 -- row softmax of an fp32 matrix with the online (m, d)
 * recurrence of the page "Softmax kernels V1-V9" (lpnh.cn/news/2830604,
 * sections 4.4-4.9): y_ij = exp(x_ij - m_i) / sum_j exp(x_ij - m_i), m_i the row
 * max, in one pass over memory when a row fits on chip (N <= 16384), two passes
 * over the row otherwise.
 *   x : device, [M, N] fp32, rows contiguous, 4-byte aligned (16-byte aligned
 *       with N a multiple of 4 selects 16-byte accesses), read only.
 *   y : device, [M, N] fp32, written in full; y == x (in place) is allowed, any
 *       other overlap is rejected.
 *   M : 1 .. 2^31 - 1 rows.   N : >= 1.
 * Entries of -inf contribute nothing; a row of -inf only is written as zeros.
 * exp is the hardware approximation (__expf): elements stay within 1e-6 of the
 * exact result.  Returns ATTN_OK or a negative attn_status.
 */
int attn_row_softmax_f32(const float* x, float* y, long long M, int N, attn_stream_t stream);

/*
 * attn_device_status -- synchronises `stream`, then reads and clears the
 * library's device status word for the current device.  Returns ATTN_OK, or
 * ATTN_ERR_TIMEOUT if a kernel enqueued since the last call gave up on a
 * bounded wait (its outputs are then incomplete), or ATTN_ERR_CUDA if the
 * synchronisation itself failed.
 */
int attn_device_status(attn_stream_t stream);

/*
 * attn_watchdog_selftest -- launches one block whose thread waits on a
 * shared-memory barrier that nothing ever completes, with a limit of
 * `timeout_us` microseconds (1 .. 10,000,000).  The wait gives up, the kernel
 * records ATTN_ERR_TIMEOUT in the device status word and returns normally; a
 * following attn_device_status(stream) reports it.  Exists so that the
 * bounded-wait path can be tested without faulting or hanging a GPU.
 */
int attn_watchdog_selftest(unsigned int timeout_us, attn_stream_t stream);

/*
 * attn_anatomy_read -- measurement aid, no counterpart on the pages.  The library
 * also builds as libeca_attn_anatomy.so (compiled with ECA_ANATOMY), whose attention
 * kernel records, in every CTA, globaltimer stamps (ns) of its first unit's
 * milestones; two launches in a row land in two slots.  This call synchronises the
 * device and copies them to `out`: [2 slots][160 CTAs][10 words], words 0-8 the
 * stamps (entry, set-up done, first K load issued, first Q K^T issued, first S
 * ready, first unit's O ready for tile 0, its output issued, the same O for tile 1,
 * exit; 0 where a CTA has none) and word 9 the units the CTA processed; the slot
 * of a launch is the parity of the launches since the last reset.  reset != 0 then
 * zeroes the stamps and the launch count.  out_words must be at least 3200.
 * Returns ATTN_ERR_INVALID_ARG in the normal build.
 */
int attn_anatomy_read(unsigned long long* out, size_t out_words, int reset);

/* Text for a status code (static storage, never NULL). */
const char* attn_status_string(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
int attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* EXACT_CAUSAL_ATTENTION_GB300_ATTN_H_ */
