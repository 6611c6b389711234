// Host-side planner: base lists, alpha schedules, per-layer distance/rung tables and the
// factored RoPE tables.  Pure C++ (no CUDA), so it runs and is tested without a GPU.
#pragma once
#include <cstdint>
#include <vector>

namespace fibattn {

constexpr int kHeadDim = 64;
constexpr int kHalf = kHeadDim / 2;   // rotate-half pairs (m, m + 32)
constexpr int kRopeSplit = 64;        // position p = hi * kRopeSplit + lo
constexpr int kMaxRungs = 32;
constexpr int kMaxWindow = 64;

// One interpolated rung: distance d = alpha * f, lo = floor(d), w = d - lo.
struct Rung {
  int32_t f;
  int32_t lo;
  float w;
};

// Base list ("Attended set": 1, 2, 3, 5, ..., 987; "Controls": {2^k : 2^k < N}).
std::vector<int32_t> fibonacci_base(int32_t limit = 987);
std::vector<int32_t> pow2_base(int N);

// Schedules ("Experimental variables"); returns false on invalid arguments.
bool schedule(int kind, int n_layers, int stride, std::vector<double>* out);

// Static distances: distinct round_half_even(alpha * f) with W <= d <= N-1, ascending.
std::vector<int32_t> mask_distances(const int32_t* base, int n_base, double alpha, int W, int N);

// Interpolated rungs: distinct f ascending with W-1 < alpha*f <= N-1.
std::vector<Rung> interp_rungs(const int32_t* base, int n_base, double alpha, int W, int N);

// Factored RoPE tables, float2-interleaved (cos, sin):
//   lo[pl * 32 + m] = e^{i pl theta_m},            pl < kRopeSplit
//   hi[ph * 32 + m] = e^{i ph * kRopeSplit theta_m}, ph <= n_max / kRopeSplit
// with theta_m = rope_base^(-2m/64), all angles and cos/sin evaluated in binary64.
void rope_tables(int n_max, double rope_base, std::vector<float>* lo, std::vector<float>* hi);

}  // namespace fibattn
