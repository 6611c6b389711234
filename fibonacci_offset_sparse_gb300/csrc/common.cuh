// Shared device-side pieces of the sm_103a kernels: the per-layer key table handed to
// every kernel by value, the CTA prologue that turns it into the layer's virtual keys,
// the relative-rotation (RoPE) factors, and row loaders.
//
// Conventions (all kernels): head dim 64; a "quad" of 4 consecutive threads owns one
// row; lane r of the quad holds the 8 rotate-half frequencies m = 8r .. 8r+7, i.e. dims
// [8r, 8r+8) in x[0..8) and their partners [32+8r, 32+8r+8) in x[8..16).  RoPE is then
// thread-local: pair (x[u], x[8+u]) is the complex number x_m + i x_{m+32}.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace fibattn {

constexpr int kD = 64;
constexpr int kFreq = 32;
constexpr int kSplit = 64;  // RoPE table split: p = hi * 64 + lo
constexpr int kMaxR = 32;
constexpr int kMaxW = 64;
constexpr int kMaxKeys = kMaxW + kMaxR;

// Per-layer attended-set description, passed by value.
//   MASK:   n entries of d[] (sorted distinct distances >= W).
//   INTERP: n rungs (lo[], w[], f[]) computed on the host from the binary64 alpha, or,
//           when alpha_dev != nullptr, n_base base values f[] from which the kernel
//           derives the rungs with alpha = alpha_dev[layer] (float32, exact in binary64).
struct LayerTable {
  int mode;  // 0 = mask, 1 = interp
  int W;
  int n;
  int layer;
  const float* alpha_dev;
  int32_t lo[kMaxR];
  float w[kMaxR];
  int32_t f[kMaxR];
};

// The side stream and events onto which the bf16 backward forks the second half of its
// (b, h) rows (owned by a plan, created with it).
struct BwdStreams {
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr;          // the caller's stream has reached the call
  cudaEvent_t first_q_done = nullptr;  // the first half's dQ grid has completed
  cudaEvent_t join = nullptr;          // the second half has completed
};

// Virtual keys of a layer, built in shared memory by the CTA prologue.
struct KeySmem {
  int nv;              // window + rungs
  int nr;              // rungs
  int lo[kMaxKeys];    // distance of the first (or only) row
  int need[kMaxKeys];  // query i attends key c iff i >= need[c]
  float w[kMaxKeys];   // weight of the second row (i - lo - 1); 0 for window and mask keys
  int f[kMaxKeys];     // base value of an interp rung (for dalpha); 0 otherwise
};

__device__ __forceinline__ void build_keys(const LayerTable& t, int N, KeySmem* ks) {
  const int tid = threadIdx.x;
  if (tid < 32) {
    int keep = 0, lo = 0, f = 0;
    float w = 0.f;
    if (t.mode == 0) {
      if (tid < t.n) {
        lo = t.lo[tid];
        keep = 1;
      }
    } else if (t.alpha_dev == nullptr) {
      if (tid < t.n) {
        lo = t.lo[tid];
        w = t.w[tid];
        f = t.f[tid];
        keep = 1;
      }
    } else if (tid < t.n) {
      // d = alpha * f is exact in binary64 (24-bit alpha times an integer < 2^29)
      const double a = static_cast<double>(__ldg(t.alpha_dev + t.layer));
      f = t.f[tid];
      const double d = a * static_cast<double>(f);
      keep = (d > static_cast<double>(t.W - 1)) && (d <= static_cast<double>(N - 1));
      const double fl = floor(d);
      lo = static_cast<int>(fl);
      w = static_cast<float>(d - fl);
    }
    const unsigned mask = __ballot_sync(0xffffffffu, keep);
    if (keep) {
      const int pos = __popc(mask & ((1u << tid) - 1u));
      const int c = t.W + pos;
      ks->lo[c] = lo;
      ks->w[c] = w;
      ks->f[c] = f;
      ks->need[c] = lo + (w > 0.f ? 1 : 0);
    }
    if (tid == 0) {
      ks->nr = __popc(mask);
      ks->nv = t.W + __popc(mask);
    }
  }
  for (int c = tid; c < t.W; c += blockDim.x) {
    ks->lo[c] = c;
    ks->need[c] = c;
    ks->w[c] = 0.f;
    ks->f[c] = 0;
  }
}

// e^{i delta theta_m} from the factored binary64-built float32 tables.
__device__ __forceinline__ float2 rope_factor(const float2* __restrict__ lo_tab,
                                              const float2* __restrict__ hi_tab, int delta,
                                              int m) {
  const float2 a = __ldg(hi_tab + (delta / kSplit) * kFreq + m);
  const float2 b = __ldg(lo_tab + (delta % kSplit) * kFreq + m);
  return make_float2(a.x * b.x - a.y * b.y, a.x * b.y + a.y * b.x);
}

// Relative-rotation factors of the layer's keys into shared memory:
//   fac[c * 32 + m]           = e^{i lo_c theta_m}          for c < nv
//   fac[(nv + r) * 32 + m]    = e^{i (lo_c + 1) theta_m}    for interp rung r = c - W
// (q'_i . k'_j = Re sum_m qhat_m conj(khat_m) e^{i (i-j) theta_m} for raw q, k.)
__device__ __forceinline__ int n_factor_slots(const KeySmem* ks, int mode) {
  return ks->nv + (mode == 1 ? ks->nr : 0);
}
__device__ __forceinline__ void build_factors(const KeySmem* ks, int mode, int W,
                                              const float2* lo_tab, const float2* hi_tab,
                                              float2* fac) {
  const int slots = n_factor_slots(ks, mode);
  for (int idx = threadIdx.x; idx < slots * kFreq; idx += blockDim.x) {
    const int s = idx / kFreq, m = idx % kFreq;
    const int delta = s < ks->nv ? ks->lo[s] : ks->lo[W + (s - ks->nv)] + 1;
    fac[idx] = rope_factor(lo_tab, hi_tab, delta, m);
  }
}

// ------------------------------------------------------------------ row part loaders --
__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

__device__ __forceinline__ void load_part(const float* __restrict__ row, int r, float (&x)[16]) {
  const float4* a = reinterpret_cast<const float4*>(row + 8 * r);
  const float4* b = reinterpret_cast<const float4*>(row + kFreq + 8 * r);
  const float4 a0 = __ldg(a), a1 = __ldg(a + 1), b0 = __ldg(b), b1 = __ldg(b + 1);
  x[0] = a0.x; x[1] = a0.y; x[2] = a0.z; x[3] = a0.w;
  x[4] = a1.x; x[5] = a1.y; x[6] = a1.z; x[7] = a1.w;
  x[8] = b0.x; x[9] = b0.y; x[10] = b0.z; x[11] = b0.w;
  x[12] = b1.x; x[13] = b1.y; x[14] = b1.z; x[15] = b1.w;
}

__device__ __forceinline__ void load_part(const __nv_bfloat16* __restrict__ row, int r,
                                          float (&x)[16]) {
  const uint4 a = __ldg(reinterpret_cast<const uint4*>(row + 8 * r));
  const uint4 b = __ldg(reinterpret_cast<const uint4*>(row + kFreq + 8 * r));
  x[0] = bf_lo(a.x); x[1] = bf_hi(a.x); x[2] = bf_lo(a.y); x[3] = bf_hi(a.y);
  x[4] = bf_lo(a.z); x[5] = bf_hi(a.z); x[6] = bf_lo(a.w); x[7] = bf_hi(a.w);
  x[8] = bf_lo(b.x); x[9] = bf_hi(b.x); x[10] = bf_lo(b.y); x[11] = bf_hi(b.y);
  x[12] = bf_lo(b.z); x[13] = bf_hi(b.z); x[14] = bf_lo(b.w); x[15] = bf_hi(b.w);
}

__device__ __forceinline__ void store_part(float* __restrict__ row, int r, const float (&x)[16]) {
  float4* a = reinterpret_cast<float4*>(row + 8 * r);
  float4* b = reinterpret_cast<float4*>(row + kFreq + 8 * r);
  a[0] = make_float4(x[0], x[1], x[2], x[3]);
  a[1] = make_float4(x[4], x[5], x[6], x[7]);
  b[0] = make_float4(x[8], x[9], x[10], x[11]);
  b[1] = make_float4(x[12], x[13], x[14], x[15]);
}

__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);  // round-to-nearest-even
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ void store_part(__nv_bfloat16* __restrict__ row, int r,
                                           const float (&x)[16]) {
  uint4 a, b;
  a.x = pack_bf2(x[0], x[1]); a.y = pack_bf2(x[2], x[3]);
  a.z = pack_bf2(x[4], x[5]); a.w = pack_bf2(x[6], x[7]);
  b.x = pack_bf2(x[8], x[9]); b.y = pack_bf2(x[10], x[11]);
  b.z = pack_bf2(x[12], x[13]); b.w = pack_bf2(x[14], x[15]);
  *reinterpret_cast<uint4*>(row + 8 * r) = a;
  *reinterpret_cast<uint4*>(row + kFreq + 8 * r) = b;
}

// Re sum_{u<8} (q_u * e_u) conj(k_u): the quad-partial RoPE'd dot at relative distance
// with factors e (8 consecutive float2 in shared memory, 16-byte aligned).
__device__ __forceinline__ float rel_dot(const float (&q)[16], const float (&k)[16],
                                         const float2* __restrict__ e) {
  const float4* e4 = reinterpret_cast<const float4*>(e);
  float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    const float4 f = e4[h];
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      const int u = 2 * h + s;
      const float c = s ? f.z : f.x, sn = s ? f.w : f.y;
      const float zr = q[u] * c - q[8 + u] * sn;
      const float zi = q[u] * sn + q[8 + u] * c;
      if (s) {
        acc1 = fmaf(zr, k[u], acc1);
        acc1 = fmaf(zi, k[8 + u], acc1);
      } else {
        acc0 = fmaf(zr, k[u], acc0);
        acc0 = fmaf(zi, k[8 + u], acc0);
      }
    }
  }
  return acc0 + acc1;
}

// Rotate x by e^{-i delta theta} (conj factor) or e^{+i delta theta}, in place.
__device__ __forceinline__ void rotate_part(float (&x)[16], const float2* __restrict__ e,
                                            bool conj) {
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const float2 f = e[u];
    const float s = conj ? -f.y : f.y;
    const float a = x[u], b = x[8 + u];
    x[u] = a * f.x - b * s;
    x[8 + u] = a * s + b * f.x;
  }
}

__device__ __forceinline__ float quad_sum(float x) {
  x += __shfl_xor_sync(0xffffffffu, x, 1);
  x += __shfl_xor_sync(0xffffffffu, x, 2);
  return x;
}

// Codes a kernel records in the plan's status word (the fib_status values of the C ABI).
constexpr int kStatusTimeout = 5;       // a bounded wait gave up
constexpr int kStatusDeviceAssert = 6;  // a device-side check of the rung table failed
constexpr int kStatusRange = 7;         // a value does not fit the float16 operands

// Nonzero when either float16 half of w is infinite or NaN (exponent bits all ones).
__device__ __forceinline__ uint32_t h2_nonfinite(uint32_t w) {
  return static_cast<uint32_t>((~w & 0x7c00u) == 0u) | static_cast<uint32_t>((~w & 0x7c000000u) == 0u);
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

}  // namespace fibattn
