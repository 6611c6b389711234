// Single-token decode against a KV cache (sm_103a).
//
// The new token at position pos attends exactly the set a forward pass gives row pos
// ("Depth-Staggered Fibonacci Spacing for Sparse Attention", Methodology > "Attended set",
// "Scaling", "Implementation"): window rows pos-t (t < W) and, per kept rung, row pos-d or
// the blend of rows pos-lo and pos-lo-1.  Key results 2 ("Efficiency") compares the
// inference latency of the interpolated and the mask path; this kernel serves both.
//
// One warp per (b, h): its 8 quads take the W + R keys round-robin, each quad keeps its own
// online softmax over the keys it saw (lane t of a quad holds the dims D_t, see
// common.cuh), then the quads merge (max, rescale, sum) with shuffles.  RoPE is applied in
// relative form from the factored tables, so the cache holds raw (unrotated) K rows.
#include "common.cuh"

namespace fibattn {

constexpr int kDecWarps = 4;

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
__global__ void __launch_bounds__(32 * kDecWarps) decode_kernel(DecArgs a) {
  __shared__ KeySmem ks;
  build_keys(a.t, a.N, &ks);
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.x * kDecWarps + warp;
  if (bh >= a.BH) return;  // whole warps only: the shuffles below stay full-warp
  const int quad = lane >> 2, t = lane & 3;
  const int i = a.pos;
  const DT* Q = static_cast<const DT*>(a.q) + static_cast<size_t>(bh) * kD;
  const DT* K = static_cast<const DT*>(a.k) + static_cast<size_t>(bh) * a.N * kD;
  const DT* V = static_cast<const DT*>(a.v) + static_cast<size_t>(bh) * a.N * kD;

  float q[16];
  load_part(Q, t, q);
#pragma unroll
  for (int u = 0; u < 16; ++u) q[u] *= kLog2e / 8.0f;
  float o[16];
#pragma unroll
  for (int u = 0; u < 16; ++u) o[u] = 0.f;
  float m = -INFINITY, l = 0.f;
  const int nv = ks.nv;
  // every quad runs the same trip count, so the quad shuffles stay uniform
  for (int c0 = 0; c0 < nv; c0 += 8) {
    const int c = c0 + quad;
    const bool ok = c < nv && i >= ks.need[c];
    float s = 0.f;
    int lo = 0;
    float w = 0.f;
    if (ok) {
      lo = ks.lo[c];
      w = ks.w[c];
      float2 e[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) e[u] = rope_factor(a.rope_lo, a.rope_hi, lo, 8 * t + u);
      float kx[16];
      load_part(K + static_cast<size_t>(i - lo) * kD, t, kx);
      s = rel_dot_reg(q, kx, e);
      if (w > 0.f) {
#pragma unroll
        for (int u = 0; u < 8; ++u) e[u] = rope_factor(a.rope_lo, a.rope_hi, lo + 1, 8 * t + u);
        load_part(K + static_cast<size_t>(i - lo - 1) * kD, t, kx);
        s = (1.f - w) * s + w * rel_dot_reg(q, kx, e);
      }
    }
    s = quad_sum(s);
    if (ok) {
      const float mn = fmaxf(m, s);
      const float corr = exp2f(m - mn);
      const float p = exp2f(s - mn);
      l = l * corr + p;
      float vx[16];
      load_part(V + static_cast<size_t>(i - lo) * kD, t, vx);
      const float p0 = p * (1.f - w);
#pragma unroll
      for (int u = 0; u < 16; ++u) o[u] = fmaf(p0, vx[u], o[u] * corr);
      if (w > 0.f) {
        load_part(V + static_cast<size_t>(i - lo - 1) * kD, t, vx);
        const float p1 = p * w;
#pragma unroll
        for (int u = 0; u < 16; ++u) o[u] = fmaf(p1, vx[u], o[u]);
      }
      m = mn;
    }
  }
  // merge the 8 quads (lanes with equal t hold the same dims)
  float mall = m;
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) mall = fmaxf(mall, __shfl_xor_sync(0xffffffffu, mall, off));
  const float sc = (m == -INFINITY) ? 0.f : exp2f(m - mall);  // a quad that saw no key
  l *= sc;
#pragma unroll
  for (int u = 0; u < 16; ++u) o[u] *= sc;
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    l += __shfl_xor_sync(0xffffffffu, l, off);
#pragma unroll
    for (int u = 0; u < 16; ++u) o[u] += __shfl_xor_sync(0xffffffffu, o[u], off);
  }
  if (quad == 0) {
    const float inv = 1.f / l;
#pragma unroll
    for (int u = 0; u < 16; ++u) o[u] *= inv;
    store_part(static_cast<DT*>(a.o) + static_cast<size_t>(bh) * kD, t, o);
    if (t == 0 && a.lse != nullptr) a.lse[bh] = (mall + log2f(l)) * kLn2;
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
  const int blocks = (a.BH + kDecWarps - 1) / kDecWarps;
  if (dtype == 0)
    decode_kernel<float><<<blocks, 32 * kDecWarps, 0, stream>>>(a);
  else
    decode_kernel<__nv_bfloat16><<<blocks, 32 * kDecWarps, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace fibattn
