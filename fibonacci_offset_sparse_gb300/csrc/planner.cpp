// Host planner for Depth-Staggered Fibonacci Spacing sparse attention.
//
// Follows "Depth-Staggered Fibonacci Spacing for Sparse Attention", Methodology:
//   "Attended set"  -- window of W keys plus sparse offsets from fib = [1, 2, 3, 5, ..., 987];
//   "Scaling"       -- d_k = alpha f_k, alpha in [0.5, 1.5] per layer;
//   "Implementation"-- non-integer d by linear interpolation between bracketing rows;
//   "Experimental variables" -- fixed / learned / staggered-linear / staggered-coprime;
//   "Controls"      -- reach-matched power-of-two base.
#include "planner.h"

#include <algorithm>
#include <cfenv>
#include <cmath>
#include <numeric>
#include <set>

namespace fibattn {

std::vector<int32_t> fibonacci_base(int32_t limit) {
  // 1, 2, 3, 5, ...: the Fibonacci sequence with its repeated leading 1 dropped.
  std::vector<int32_t> out;
  int64_t a = 1, b = 2;
  while (a <= limit) {
    out.push_back(static_cast<int32_t>(a));
    int64_t c = a + b;
    a = b;
    b = c;
  }
  return out;
}

std::vector<int32_t> pow2_base(int N) {
  std::vector<int32_t> out;
  for (int64_t p = 1; p < N; p *= 2) out.push_back(static_cast<int32_t>(p));
  return out;
}

static int gcd_int(int a, int b) {
  while (b) {
    int t = a % b;
    a = b;
    b = t;
  }
  return a < 0 ? -a : a;
}

bool schedule(int kind, int n_layers, int stride, std::vector<double>* out) {
  if (n_layers < 1) return false;
  out->assign(n_layers, 1.0);
  if (kind == 0) return true;  // fixed: alpha = 1 on every layer
  if (kind != 1 && kind != 2) return false;
  if (n_layers < 2) return false;
  std::vector<double> ramp(n_layers);
  // staggered linear: 0.5 at layer 0 rising to 1.5 at the last layer
  for (int l = 0; l < n_layers; ++l) ramp[l] = 0.5 + static_cast<double>(l) / static_cast<double>(n_layers - 1);
  if (kind == 1) {
    *out = ramp;
    return true;
  }
  // staggered coprime: layer l takes the ramp's value at (stride * l) mod L
  if (stride <= 0 || gcd_int(stride, n_layers) != 1) return false;
  for (int l = 0; l < n_layers; ++l)
    (*out)[l] = ramp[static_cast<int64_t>(stride) * l % n_layers];
  return true;
}

// nearbyint() rounds in the current mode; force round-to-nearest-even for the call.
static int64_t round_half_even(double x) {
  const int saved = std::fegetround();
  std::fesetround(FE_TONEAREST);
  const double r = std::nearbyint(x);
  std::fesetround(saved);
  return static_cast<int64_t>(r);
}

std::vector<int32_t> mask_distances(const int32_t* base, int n_base, double alpha, int W, int N) {
  std::set<int64_t> ds;
  for (int k = 0; k < n_base; ++k) {
    const int64_t d = round_half_even(alpha * static_cast<double>(base[k]));
    if (d >= W && d <= static_cast<int64_t>(N) - 1) ds.insert(d);
  }
  return std::vector<int32_t>(ds.begin(), ds.end());
}

std::vector<Rung> interp_rungs(const int32_t* base, int n_base, double alpha, int W, int N) {
  std::set<int32_t> fs(base, base + n_base);
  std::vector<Rung> out;
  for (int32_t f : fs) {
    const double d = alpha * static_cast<double>(f);
    if (d > static_cast<double>(W - 1) && d <= static_cast<double>(N - 1)) {
      const double lo = std::floor(d);
      out.push_back(Rung{f, static_cast<int32_t>(lo), static_cast<float>(d - lo)});
    }
  }
  return out;
}

void rope_tables(int n_max, double rope_base, std::vector<float>* lo, std::vector<float>* hi) {
  double theta[kHalf];
  for (int m = 0; m < kHalf; ++m) theta[m] = std::pow(rope_base, -2.0 * m / kHeadDim);
  lo->assign(static_cast<size_t>(kRopeSplit) * kHalf * 2, 0.f);
  for (int p = 0; p < kRopeSplit; ++p)
    for (int m = 0; m < kHalf; ++m) {
      const double a = static_cast<double>(p) * theta[m];
      (*lo)[(static_cast<size_t>(p) * kHalf + m) * 2 + 0] = static_cast<float>(std::cos(a));
      (*lo)[(static_cast<size_t>(p) * kHalf + m) * 2 + 1] = static_cast<float>(std::sin(a));
    }
  // distances up to n_max inclusive are looked up (an interp rung's second row sits at lo+1)
  const int n_hi = std::max(n_max, 1) / kRopeSplit + 1;
  hi->assign(static_cast<size_t>(n_hi) * kHalf * 2, 0.f);
  for (int p = 0; p < n_hi; ++p)
    for (int m = 0; m < kHalf; ++m) {
      const double a = static_cast<double>(p) * kRopeSplit * theta[m];
      (*hi)[(static_cast<size_t>(p) * kHalf + m) * 2 + 0] = static_cast<float>(std::cos(a));
      (*hi)[(static_cast<size_t>(p) * kHalf + m) * 2 + 1] = static_cast<float>(std::sin(a));
    }
}

}  // namespace fibattn
