// Dynamic chunk sizing for chunked prefill (host only).
//
// The SGLang pipeline-parallelism article ("SGLang Pipeline Parallelism: 1M-token
// context ...", TL;DR and the caption of its throughput figure) runs chunked prefill
// with dynamic chunking: an initial chunk of 12288 tokens and a smoothing factor of
// 0.65 ("DCK 12288 (sigma=0.65)").  The article stops before it gives the algorithm,
// so this is a reading of those two numbers:
//
//   cost(s, n)  the visible (query, key) pairs of chunk [s, s + n): row i sees i + 1 keys
//               under the causal mask (min(i + 1, W) with a window of W);
//   T           cost(0, n0), the first chunk's cost, n0 = min(initial, S);
//   n*(s)       the largest n >= 1 with cost(s, n) <= T (the chunk that costs what the
//               first one did; at least 1 token);
//   n_c         round(sigma * n*(s_c) + (1 - sigma) * n_{c-1}): exponential smoothing of
//               the equal-cost size, sigma being the smoothing factor; n_0 = n0;
//   then        n_c rounded down to a multiple of `align` (at least `align`), and the
//               last chunk clipped to the tokens left.
//
// Sizes never grow (n* falls as the prefix grows, and a smoothed value lies between n*
// and the previous size); sigma = 0 gives fixed chunks of n0, sigma = 1 the equal-cost
// partition.
#include <cmath>
#include <cstdint>
#include <vector>

#include "slope.h"

namespace {

// Visible pairs of rows [s, s + n): sum of min(i + 1, W) (or i + 1 without a window).  Exact in
// 64-bit integers: with s + n <= 2^30 every term stays below 2^61.
int64_t chunk_cost(int64_t s, int64_t n, int64_t window) {
  auto prefix = [window](int64_t m) -> int64_t {  // sum over rows i < m
    if (m <= 0) return 0;
    if (window <= 0 || m <= window) return m * (m + 1) / 2;
    return window * (window + 1) / 2 + (m - window) * window;
  };
  return prefix(s + n) - prefix(s);
}

// The largest n in [1, limit] with cost(s, n) <= target (1 if even one row costs more).
int64_t equal_cost_size(int64_t s, int64_t limit, int64_t target, int64_t window) {
  int64_t lo = 1, hi = limit;  // cost is increasing in n
  if (chunk_cost(s, hi, window) <= target) return hi;
  while (hi - lo > 1) {
    const int64_t mid = lo + (hi - lo) / 2;
    if (chunk_cost(s, mid, window) <= target)
      lo = mid;
    else
      hi = mid;
  }
  return lo;
}

}  // namespace

extern "C" SLOPE_API int64_t slope_dck_chunk_sizes(int64_t S, int64_t initial, double sigma, int64_t window,
                                                   int64_t align, int64_t* sizes, int64_t capacity) {
  if (S <= 0 || S > (int64_t(1) << 30) || initial <= 0 || window < 0 || align <= 0 || align > initial)
    return SLOPE_ERR_SHAPE;
  if (!(sigma >= 0.0 && sigma <= 1.0)) return SLOPE_ERR_SHAPE;
  if (capacity < 0 || (capacity > 0 && sizes == nullptr)) return SLOPE_ERR_NULL;
  const int64_t n0 = initial < S ? initial : S;
  const int64_t target = chunk_cost(0, n0, window);
  int64_t count = 0, s = 0, prev = n0;
  while (s < S) {
    int64_t n;
    if (count == 0) {
      n = n0;
    } else {
      const int64_t ideal = equal_cost_size(s, S - s, target, window);
      // both products rounded before the sum (no fused multiply-add), so the result does not
      // depend on the compiler's contraction choices
      const volatile double a = sigma * static_cast<double>(ideal);
      const volatile double b = (1.0 - sigma) * static_cast<double>(prev);
      const double smoothed = a + b;
      n = static_cast<int64_t>(std::floor(smoothed + 0.5));
      n = (n / align) * align;
      if (n < align) n = align;
    }
    if (n > S - s) n = S - s;
    if (count < capacity) sizes[count] = n;
    ++count;
    s += n;
    prev = n;
  }
  return count;
}
