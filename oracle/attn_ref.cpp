// FP64 CPU oracle for exact scaled-dot-product attention forward.
//
// TEST INFRASTRUCTURE ONLY.  Nothing in the product library calls, links or
// includes this file; only the tests, the smoke check and the benchmark's CPU
// baseline leg load it.  It shares no code with the CUDA path.
//
// What it computes (page "CUDA FlashAttention：从在线 Softmax 到长序列 IO 极限",
// chengzipai.xyz, section 1): for Q, K, V of shape [B, H, N, D]
//
//     O = softmax(scale * Q K^T + M) V,   M_ij = 0 if j <= i else -inf (causal)
//
// plus the natural-log log-sum-exp of each score row,
//
//     lse_i = ln sum_j exp(s_ij)          (over the unmasked j).
//
// Two ways of reaching it, both in double precision:
//
//   mode 0 "two_pass": the safe-softmax definition written out -- scores,
//       row max, sum of exp(s - max), weighted sum of V, divide
//       (same page, section 3, the three stages of the plain path; the
//       double-precision stable softmax of the page "Softmax kernels V1-V9",
//       lpnh.cn, section 3.1).
//   mode 1 "online": the tiled online recurrence of the same page, section 4:
//       per tile the local max m~ and local sum l~, then m' = max(m, m~),
//       alpha = e^(m - m'), beta = e^(m~ - m'), l' = alpha*l + beta*l~,
//       o' = alpha*o + sum_j e^(s_j - m') v_j, and finally O = o / l.
//       The empty state is (-inf, 0); merging a tile whose max is -inf is
//       skipped, as the lpnh.cn page (section 4.6) requires so that
//       -inf - (-inf) never makes a NaN.
//
// Readings where the pages are silent:
//   * the mask is the top-left square one, j <= i (one N for queries and keys);
//   * lse is the natural log including the scale; a row with no unmasked key
//     (impossible for the square causal mask) gets O = 0 and lse = -inf;
//   * inputs arrive as fp16 / bf16 bit patterns and are decoded exactly to
//     double here, with a decoder written from the IEEE-754 binary16 and the
//     bfloat16 (truncated binary32) formats.
//
// Grouped heads (page "CUDA KV Cache：分页存储与长上下文 Decode 极致优化", section
// 3.3): with H query heads and Hkv key/value heads, g = H / Hkv, query head h
// reads key/value head floor(h / g) of the same batch entry.  Hkv = H is the
// ordinary one-to-one case.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

namespace {

double decode_fp16(uint16_t h) {
  const int sign = (h >> 15) & 1;
  const int exponent = (h >> 10) & 0x1f;
  const int mantissa = h & 0x3ff;
  double magnitude;
  if (exponent == 0) {
    magnitude = std::ldexp(static_cast<double>(mantissa), -24);  // subnormal: m * 2^-14 * 2^-10
  } else if (exponent == 31) {
    magnitude = mantissa == 0 ? std::numeric_limits<double>::infinity()
                              : std::numeric_limits<double>::quiet_NaN();
  } else {
    magnitude = std::ldexp(static_cast<double>(1024 + mantissa), exponent - 25);  // (1 + m/2^10) * 2^(e-15)
  }
  return sign ? -magnitude : magnitude;
}

double decode_bf16(uint16_t b) {
  const int sign = (b >> 15) & 1;
  const int exponent = (b >> 7) & 0xff;
  const int mantissa = b & 0x7f;
  double magnitude;
  if (exponent == 0) {
    magnitude = std::ldexp(static_cast<double>(mantissa), -133);  // m * 2^-126 * 2^-7
  } else if (exponent == 255) {
    magnitude = mantissa == 0 ? std::numeric_limits<double>::infinity()
                              : std::numeric_limits<double>::quiet_NaN();
  } else {
    magnitude = std::ldexp(static_cast<double>(128 + mantissa), exponent - 134);  // (1 + m/2^7) * 2^(e-127)
  }
  return sign ? -magnitude : magnitude;
}

struct Problem {
  const double* q;
  const double* k;
  const double* v;
  long B, H, N, D;
  int causal;
  double scale;
  long Hkv;  // key/value heads; H is a multiple of it
};

// Key/value slice read by query slice bh = b * H + h.
long kv_slice(const Problem& p, long bh) {
  const long b = bh / p.H, h = bh % p.H;
  return b * p.Hkv + h / (p.H / p.Hkv);
}

// Scores of query row i of slice bh against keys 0..last, written to s.
void score_row(const Problem& p, long bh, long i, long last, std::vector<double>& s) {
  const double* qi = p.q + (bh * p.N + i) * p.D;
  const double* kb = p.k + kv_slice(p, bh) * p.N * p.D;
  s.resize(last + 1);
  for (long j = 0; j <= last; ++j) {
    const double* kj = kb + j * p.D;
    double dot = 0.0;
    for (long d = 0; d < p.D; ++d) dot += qi[d] * kj[d];
    s[j] = p.scale * dot;
  }
}

// Definition, written out: safe softmax over the unmasked scores, then P V.
void row_two_pass(const Problem& p, long bh, long i, double* o, double* lse,
                  std::vector<double>& s) {
  const long last = p.causal ? i : p.N - 1;
  score_row(p, bh, i, last, s);
  double m = -std::numeric_limits<double>::infinity();
  for (long j = 0; j <= last; ++j) m = s[j] > m ? s[j] : m;
  for (long d = 0; d < p.D; ++d) o[d] = 0.0;
  if (last < 0 || m == -std::numeric_limits<double>::infinity()) {
    *lse = -std::numeric_limits<double>::infinity();
    return;
  }
  double l = 0.0;
  for (long j = 0; j <= last; ++j) l += std::exp(s[j] - m);
  const double* vb = p.v + kv_slice(p, bh) * p.N * p.D;
  for (long j = 0; j <= last; ++j) {
    const double w = std::exp(s[j] - m) / l;
    const double* vj = vb + j * p.D;
    for (long d = 0; d < p.D; ++d) o[d] += w * vj[d];
  }
  *lse = m + std::log(l);
}

// Online recurrence over key tiles of width `tile`, state (m, l, o).
void row_online(const Problem& p, long bh, long i, long tile, double* o, double* lse,
                std::vector<double>& s, std::vector<double>& acc) {
  const double neg_inf = -std::numeric_limits<double>::infinity();
  const long last = p.causal ? i : p.N - 1;
  score_row(p, bh, i, last, s);
  const double* vb = p.v + kv_slice(p, bh) * p.N * p.D;
  acc.assign(p.D, 0.0);
  double m = neg_inf;  // running max
  double l = 0.0;      // running sum of exp(s - m)
  for (long t0 = 0; t0 <= last; t0 += tile) {
    const long t1 = (t0 + tile - 1 < last) ? t0 + tile - 1 : last;
    double m_tile = neg_inf;
    for (long j = t0; j <= t1; ++j) m_tile = s[j] > m_tile ? s[j] : m_tile;
    if (m_tile == neg_inf) continue;  // empty tile: (-inf, 0) contributes nothing
    double l_tile = 0.0;
    for (long j = t0; j <= t1; ++j) l_tile += std::exp(s[j] - m_tile);
    const double m_new = m > m_tile ? m : m_tile;
    const double alpha = (m == neg_inf) ? 0.0 : std::exp(m - m_new);
    const double beta = std::exp(m_tile - m_new);
    l = alpha * l + beta * l_tile;
    for (long d = 0; d < p.D; ++d) acc[d] *= alpha;
    for (long j = t0; j <= t1; ++j) {
      const double w = std::exp(s[j] - m_new);
      const double* vj = vb + j * p.D;
      for (long d = 0; d < p.D; ++d) acc[d] += w * vj[d];
    }
    m = m_new;
  }
  if (m == neg_inf) {
    for (long d = 0; d < p.D; ++d) o[d] = 0.0;
    *lse = neg_inf;
    return;
  }
  for (long d = 0; d < p.D; ++d) o[d] = acc[d] / l;
  *lse = m + std::log(l);
}

int clamp_threads(int nthreads, long work) {
  int n = nthreads > 0 ? nthreads : static_cast<int>(std::thread::hardware_concurrency());
  if (n < 1) n = 1;
  if (work < n) n = static_cast<int>(work > 0 ? work : 1);
  return n;
}

// Runs f(r) for r in [0, count) split into contiguous ranges over threads.
template <typename F>
void parallel_rows(long count, int nthreads, F f) {
  const int n = clamp_threads(nthreads, count);
  if (n == 1) {
    f(0, count);
    return;
  }
  std::vector<std::thread> pool;
  const long chunk = (count + n - 1) / n;
  for (int t = 0; t < n; ++t) {
    const long lo = t * chunk;
    const long hi = lo + chunk < count ? lo + chunk : count;
    if (lo >= hi) break;
    pool.emplace_back([=]() { f(lo, hi); });
  }
  for (auto& th : pool) th.join();
}

bool valid(const Problem& p, int mode, long tile) {
  if (!p.q || !p.k || !p.v) return false;
  if (p.B < 1 || p.H < 1 || p.N < 1 || p.D < 1) return false;
  if (p.Hkv < 1 || p.H % p.Hkv != 0) return false;
  if (mode != 0 && mode != 1) return false;
  if (mode == 1 && tile < 1) return false;
  return true;
}

}  // namespace

extern "C" {

// Exact decode of n 16-bit patterns to double; dtype 0 = fp16, 1 = bf16.
int oracle_decode(const uint16_t* bits, double* out, long n, int dtype, int nthreads) {
  if (!bits || !out || n < 0 || (dtype != 0 && dtype != 1)) return -1;
  parallel_rows(n, nthreads, [&](long lo, long hi) {
    for (long x = lo; x < hi; ++x) out[x] = dtype == 0 ? decode_fp16(bits[x]) : decode_bf16(bits[x]);
  });
  return 0;
}

// Full forward: q, o are [B, H, N, D], k, v are [B, Hkv, N, D], lse is [B, H, N] (may be null).
// mode 0 = two-pass definition, mode 1 = online recurrence with key tiles of `tile`.
int oracle_attn_fwd(const double* q, const double* k, const double* v, double* o, double* lse,
                    long B, long H, long Hkv, long N, long D, int causal, double scale, int mode,
                    long tile, int nthreads) {
  Problem p{q, k, v, B, H, N, D, causal, scale, Hkv};
  if (!valid(p, mode, tile) || !o) return -1;
  parallel_rows(B * H * N, nthreads, [&](long lo, long hi) {
    std::vector<double> s, acc;
    for (long r = lo; r < hi; ++r) {
      const long bh = r / N, i = r % N;
      double l;
      if (mode == 0) {
        row_two_pass(p, bh, i, o + r * D, &l, s);
      } else {
        row_online(p, bh, i, tile, o + r * D, &l, s, acc);
      }
      if (lse) lse[r] = l;
    }
  });
  return 0;
}

// Selected rows only: rows holds nrows pairs (bh, i); o_rows is [nrows, D], lse_rows [nrows].
int oracle_attn_rows(const double* q, const double* k, const double* v, long B, long H, long Hkv,
                     long N, long D, int causal, double scale, const long* rows, long nrows,
                     double* o_rows, double* lse_rows, int nthreads) {
  Problem p{q, k, v, B, H, N, D, causal, scale, Hkv};
  if (!valid(p, 0, 1) || !rows || !o_rows || !lse_rows || nrows < 0) return -1;
  for (long r = 0; r < nrows; ++r) {
    if (rows[2 * r] < 0 || rows[2 * r] >= B * H || rows[2 * r + 1] < 0 || rows[2 * r + 1] >= N)
      return -1;
  }
  parallel_rows(nrows, nthreads, [&](long lo, long hi) {
    std::vector<double> s;
    for (long r = lo; r < hi; ++r) {
      row_two_pass(p, rows[2 * r], rows[2 * r + 1], o_rows + r * D, lse_rows + r, s);
    }
  });
  return 0;
}

}  // extern "C"
