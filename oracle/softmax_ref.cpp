// FP64 CPU oracle for the row softmax y_ij = exp(x_ij - m_i) / sum_j exp(x_ij - m_i),
// m_i = max_j x_ij, of an M x N matrix (rows contiguous).
//
// TEST INFRASTRUCTURE ONLY, like attn_ref.cpp next to it: nothing in the product
// library calls, links or includes it, and it shares no code with the CUDA path.
//
// Two ways of reaching the result, following the page "Softmax kernels V1-V9"
// (lpnh.cn/news/2830604):
//   mode 0: the double-precision stable softmax of its section 3.1 written out:
//           row max, then the sum of exp(x - max), then each exp(x - max) / sum.
//   mode 1: the online form: chunks of `tile` elements each run the one-pass
//           recurrence of section 4.4 (running max m and running sum d, d
//           rescaled by exp(m_old - m_new) whenever the max moves), and the
//           chunk states are merged left to right with the law of section 4.6,
//           m = max(m1, m2), d = d1 exp(m1 - m) + d2 exp(m2 - m), where an empty
//           state (-inf, 0) is skipped so that -inf - (-inf) never appears.
// A row whose entries are all -inf has no defined softmax; both modes return 0
// for it (reading: the empty state contributes nothing).
#include <cmath>
#include <limits>
#include <thread>
#include <vector>

namespace {

const double kNegInf = -std::numeric_limits<double>::infinity();

void row_two_pass(const double* x, double* y, long N) {
  double m = kNegInf;
  for (long j = 0; j < N; ++j) m = x[j] > m ? x[j] : m;
  if (m == kNegInf) {
    for (long j = 0; j < N; ++j) y[j] = 0.0;
    return;
  }
  double d = 0.0;
  for (long j = 0; j < N; ++j) d += std::exp(x[j] - m);
  for (long j = 0; j < N; ++j) y[j] = std::exp(x[j] - m) / d;
}

struct State {
  double m;
  double d;
};

// Section 4.4: one pass over a chunk, max and sum updated element by element.
State chunk_state(const double* x, long n) {
  State s{kNegInf, 0.0};
  for (long j = 0; j < n; ++j) {
    if (x[j] == kNegInf) continue;  // exp(-inf - m) = 0 adds nothing
    const double m_new = x[j] > s.m ? x[j] : s.m;
    s.d = (s.m == kNegInf ? 0.0 : s.d * std::exp(s.m - m_new)) + std::exp(x[j] - m_new);
    s.m = m_new;
  }
  return s;
}

// Section 4.6: merge of two partial states; the empty state is skipped.
State merge(State a, State b) {
  if (b.d == 0.0) return a;
  if (a.d == 0.0) return b;
  const double m = a.m > b.m ? a.m : b.m;
  return State{m, a.d * std::exp(a.m - m) + b.d * std::exp(b.m - m)};
}

void row_online(const double* x, double* y, long N, long tile) {
  State s{kNegInf, 0.0};
  for (long t0 = 0; t0 < N; t0 += tile) {
    const long n = t0 + tile <= N ? tile : N - t0;
    s = merge(s, chunk_state(x + t0, n));
  }
  if (s.d == 0.0) {
    for (long j = 0; j < N; ++j) y[j] = 0.0;
    return;
  }
  for (long j = 0; j < N; ++j) y[j] = std::exp(x[j] - s.m) / s.d;
}

}  // namespace

extern "C" {

// y = row softmax of x; both [M, N].  mode 0 = two-pass, mode 1 = online with chunks of `tile`.
int oracle_softmax(const double* x, double* y, long M, long N, int mode, long tile, int nthreads) {
  if (!x || !y || M < 1 || N < 1 || (mode != 0 && mode != 1) || (mode == 1 && tile < 1)) return -1;
  int n = nthreads > 0 ? nthreads : static_cast<int>(std::thread::hardware_concurrency());
  if (n < 1) n = 1;
  if (M < n) n = static_cast<int>(M);
  const long chunk = (M + n - 1) / n;
  auto work = [&](long lo, long hi) {
    for (long r = lo; r < hi; ++r) {
      if (mode == 0) {
        row_two_pass(x + r * N, y + r * N, N);
      } else {
        row_online(x + r * N, y + r * N, N, tile);
      }
    }
  };
  std::vector<std::thread> pool;
  for (int t = 0; t < n; ++t) {
    const long lo = t * chunk, hi = lo + chunk < M ? lo + chunk : M;
    if (lo >= hi) break;
    pool.emplace_back(work, lo, hi);
  }
  for (auto& th : pool) th.join();
  return 0;
}

}  // extern "C"
