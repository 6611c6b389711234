// Single-token decode against a KV cache (sm_103a).
//
// The new token at position pos attends exactly the set a forward pass gives row pos
// ("Depth-Staggered Fibonacci Spacing for Sparse Attention", Methodology > "Attended set",
// "Scaling", "Implementation"): window rows pos-t (t < W) and, per kept rung, row pos-d or
// the blend of rows pos-lo and pos-lo-1.  Key results 2 ("Efficiency") compares the
// inference latency of the interpolated and the mask path; this kernel serves both.
//
// One CTA of 32 quads per (b, h): quad c takes keys c, c+32, ... (every key of a usual
// layer in one round), issuing all of its loads -- the RoPE factors, the K and V rows, the
// partner rows of an interpolated key -- before it uses any, so that a decode step waits
// for about one memory round trip.  Each quad keeps an online softmax over its keys (lane t
// of a quad holds the dims D_t, see common.cuh); the 32 quads then merge through shared
// memory in a fixed order (max, rescale, sum).  RoPE is applied in relative form from the
// factored tables, so the cache holds raw (unrotated) K rows.
#include "common.cuh"

namespace fibattn {

constexpr int kDecQuads = 32;
constexpr int kDecThreads = 4 * kDecQuads;

struct DecArgs {
  LayerTable t;
  int N;    // sequence length the key table is built for (the cache length)
  int pos;  // position of the new token, < N
  int BH;
  const void* q;  // [B*H, 64]
  const void* k;  // [B*H, N, 64]
  const void* v;
  void* o;        // [B*H, 64]
  float* lse;     // [B*H] or null
  const float2* rope_lo;
  const float2* rope_hi;
};

// Re sum_u (q_u e_u) conj(k_u) with the 8 factors in registers.
__device__ __forceinline__ float rel_dot_reg(const float (&q)[16], const float (&k)[16],
                                             const float2 (&e)[8]) {
  float acc = 0.f;
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const float zr = q[u] * e[u].x - q[8 + u] * e[u].y;
    const float zi = q[u] * e[u].y + q[8 + u] * e[u].x;
    acc = fmaf(zr, k[u], acc);
    acc = fmaf(zi, k[8 + u], acc);
  }
  return acc;
}

template <typename DT>
__global__ void __launch_bounds__(kDecThreads) decode_kernel(const __grid_constant__ DecArgs a) {
  __shared__ KeySmem ks;
  __shared__ float s_m[kDecQuads], s_l[kDecQuads];
  __shared__ float s_o[kDecQuads][kD];
  const int bh = blockIdx.x;
  const int tid = threadIdx.x;
  const int quad = tid >> 2, t = tid & 3;
  const int i = a.pos;
  const DT* Q = static_cast<const DT*>(a.q) + static_cast<size_t>(bh) * kD;
  const DT* K = static_cast<const DT*>(a.k) + static_cast<size_t>(bh) * a.N * kD;
  const DT* V = static_cast<const DT*>(a.v) + static_cast<size_t>(bh) * a.N * kD;
  float q[16];
  load_part(Q, t, q);  // independent of the key table: in flight during its build
  // The key table: read from the launch parameters where the distances are known on the
  // host (every mask layer, and interp with the plan's alpha), so that the cache loads issue
  // at once; built in shared memory from the device alpha otherwise.
  const bool host_keys = a.t.mode == 0 || a.t.alpha_dev == nullptr;  // uniform
  if (!host_keys) {
    build_keys(a.t, a.N, &ks);
    __syncthreads();
  }
  const int W = a.t.W;
#pragma unroll
  for (int u = 0; u < 16; ++u) q[u] *= kLog2e / 8.0f;
  float o[16];
#pragma unroll
  for (int u = 0; u < 16; ++u) o[u] = 0.f;
  float m = -INFINITY, l = 0.f;
  const int nv = host_keys ? W + a.t.n : ks.nv;
  // the same trip count in every quad, so that the quad shuffles stay warp-uniform
  for (int c0 = 0; c0 < nv; c0 += kDecQuads) {
    const int c = c0 + quad;
    // key c: window key c (c < W) or rung c - W, as build_keys lays the table out
    int klo = 0, kneed = 0;
    float kw = 0.f;
    if (c < nv) {
      if (!host_keys) {
        klo = ks.lo[c];
        kw = ks.w[c];
        kneed = ks.need[c];
      } else if (c < W) {
        klo = kneed = c;
      } else {
        klo = a.t.lo[c - W];
        kw = a.t.mode == 1 ? a.t.w[c - W] : 0.f;
        kneed = klo + (kw > 0.f ? 1 : 0);
      }
    }
    const bool ok = c < nv && i >= kneed;
    const int lo = ok ? klo : 0;
    const float w = ok ? kw : 0.f;
    const bool two = w > 0.f;
    // every load of this key first: factors, K and V rows (and the partner rows)
    float2 e0[8], e1[8];
    float k0[16], k1[16], v0[16], v1[16];
    if (ok) {
#pragma unroll
      for (int u = 0; u < 8; ++u) e0[u] = rope_factor(a.rope_lo, a.rope_hi, lo, 8 * t + u);
      load_part(K + static_cast<size_t>(i - lo) * kD, t, k0);
      load_part(V + static_cast<size_t>(i - lo) * kD, t, v0);
      if (two) {
#pragma unroll
        for (int u = 0; u < 8; ++u) e1[u] = rope_factor(a.rope_lo, a.rope_hi, lo + 1, 8 * t + u);
        load_part(K + static_cast<size_t>(i - lo - 1) * kD, t, k1);
        load_part(V + static_cast<size_t>(i - lo - 1) * kD, t, v1);
      }
    }
    float s = 0.f;
    if (ok) {
      s = rel_dot_reg(q, k0, e0);
      if (two) s = (1.f - w) * s + w * rel_dot_reg(q, k1, e1);
    }
    s = quad_sum(s);
    if (!ok) continue;  // after the shuffles; no further warp-wide operation in this trip
    const float mn = fmaxf(m, s);
    const float corr = exp2f(m - mn);
    const float p = exp2f(s - mn);
    l = l * corr + p;
    const float p0 = p * (1.f - w);
#pragma unroll
    for (int u = 0; u < 16; ++u) o[u] = fmaf(p0, v0[u], o[u] * corr);
    if (two) {
      const float p1 = p * w;
#pragma unroll
      for (int u = 0; u < 16; ++u) o[u] = fmaf(p1, v1[u], o[u]);
    }
    m = mn;
  }
  // merge the quads in a fixed order: the largest max, then every quad rescaled to it
  if (t == 0) s_m[quad] = m;
  __syncthreads();
  float mall = -INFINITY;
  for (int qd = 0; qd < kDecQuads; ++qd) mall = fmaxf(mall, s_m[qd]);
  const float sc = (m == -INFINITY) ? 0.f : exp2f(m - mall);  // a quad that saw no key
  if (t == 0) s_l[quad] = l * sc;
  // lane t holds dims [8t, 8t+8) in o[0..8) and [32+8t, 32+8t+8) in o[8..16)
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    s_o[quad][8 * t + u] = o[u] * sc;
    s_o[quad][32 + 8 * t + u] = o[8 + u] * sc;
  }
  __syncthreads();
  if (tid < kD) {
    float acc = 0.f, lsum = 0.f;
    for (int qd = 0; qd < kDecQuads; ++qd) {
      acc += s_o[qd][tid];
      lsum += s_l[qd];
    }
    const float outv = acc / lsum;
    if constexpr (sizeof(DT) == 4) {
      static_cast<float*>(a.o)[static_cast<size_t>(bh) * kD + tid] = outv;
    } else {
      static_cast<__nv_bfloat16*>(a.o)[static_cast<size_t>(bh) * kD + tid] = __float2bfloat16_rn(outv);
    }
    if (tid == 0 && a.lse != nullptr) a.lse[bh] = (mall + log2f(lsum)) * kLn2;
  }
}

cudaError_t launch_decode(const LayerTable& t, int B, int H, int N, int pos, int dtype,
                          const void* q, const void* k, const void* v, void* o, float* lse,
                          const float2* lo_tab, const float2* hi_tab, cudaStream_t stream) {
  DecArgs a;
  a.t = t;
  a.N = N;
  a.pos = pos;
  a.BH = B * H;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.rope_lo = lo_tab;
  a.rope_hi = hi_tab;
  const int blocks = a.BH;
  if (dtype == 0)
    decode_kernel<float><<<blocks, kDecThreads, 0, stream>>>(a);
  else
    decode_kernel<__nv_bfloat16><<<blocks, kDecThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace fibattn
