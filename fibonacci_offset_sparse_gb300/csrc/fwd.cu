// Forward kernels of Depth-Staggered Fibonacci Spacing sparse attention (sm_103a).
//
// "Depth-Staggered Fibonacci Spacing for Sparse Attention", Methodology > "Attended set",
// "Scaling", "Implementation": query i attends the window rows i-t (t < W) and, per kept
// rung, row i-d (MASK) or the blend (1-w) row(i-lo) + w row(i-lo-1) (INTERP), with RoPE
// applied to Q and K before the gather.
//
// Design.  One CTA = one (b, h) and a tile of 64 consecutive queries; a quad of threads
// owns a query and splits the 64 dims by rotate-half frequency (see common.cuh).  Every
// key is a shifted row of the same (b, h), so a warp's 8 queries read 8 consecutive rows
// = one contiguous 1 KB (bf16) run per key: coalesced without staging.  RoPE is applied
// in relative form: q'_i . k'_j = Re sum_m qhat_m conj(khat_m) e^{i (i-j) theta_m}, and
// i-j is the same for every query of a key slot, so the CTA precomputes one factor row
// per slot and Q/K are read raw.  Softmax is online over chunks of 4 keys, in log2 units.
#include "common.cuh"

namespace fibattn {

constexpr int kTile = 64;     // queries per CTA
constexpr int kThreads = 256; // 4 threads per query
constexpr int kChunk = 4;

struct FwdArgs {
  LayerTable t;
  int N;
  int tiles;  // ceil(N / kTile)
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  const float2* rope_lo;
  const float2* rope_hi;
  float qscale;  // log2(e) / sqrt(D)
};

template <typename DT>
__global__ void __launch_bounds__(kThreads) fwd_kernel(FwdArgs a) {
  __shared__ KeySmem ks;
  extern __shared__ float4 smem_dyn[];
  float2* fac = reinterpret_cast<float2*>(smem_dyn);

  const int bh = blockIdx.x / a.tiles;
  const int tile = blockIdx.x - bh * a.tiles;
  build_keys(a.t, a.N, &ks);
  __syncthreads();
  build_factors(&ks, a.t.mode, a.t.W, a.rope_lo, a.rope_hi, fac);
  __syncthreads();

  const int qi = threadIdx.x >> 2, r = threadIdx.x & 3;
  const int i_raw = tile * kTile + qi;
  const bool active = i_raw < a.N;
  const int i = active ? i_raw : a.N - 1;  // ragged tail: compute a valid row, store nothing
  const size_t base = static_cast<size_t>(bh) * a.N * kD;
  const DT* __restrict__ Q = static_cast<const DT*>(a.q) + base;
  const DT* __restrict__ K = static_cast<const DT*>(a.k) + base;
  const DT* __restrict__ V = static_cast<const DT*>(a.v) + base;

  float q[16];
  load_part(Q + static_cast<size_t>(i) * kD, r, q);
#pragma unroll
  for (int u = 0; u < 16; ++u) q[u] *= a.qscale;

  float o[16];
#pragma unroll
  for (int u = 0; u < 16; ++u) o[u] = 0.f;
  float m = -INFINITY, l = 0.f;
  const int nv = ks.nv;
  const int W = a.t.W;

  for (int c0 = 0; c0 < nv; c0 += kChunk) {
    float s[kChunk];
#pragma unroll
    for (int cc = 0; cc < kChunk; ++cc) {
      const int c = c0 + cc;
      float sc = 0.f;
      bool ok = false;
      if (c < nv && i >= ks.need[c]) {
        ok = true;
        float kx[16];
        const int j0 = i - ks.lo[c];
        load_part(K + static_cast<size_t>(j0) * kD, r, kx);
        sc = rel_dot(q, kx, fac + c * kFreq + 8 * r);
        const float w = ks.w[c];
        if (w > 0.f) {
          float kx1[16];
          load_part(K + static_cast<size_t>(j0 - 1) * kD, r, kx1);
          const float s1 = rel_dot(q, kx1, fac + (nv + (c - W)) * kFreq + 8 * r);
          sc = (1.f - w) * sc + w * s1;
        }
      }
      sc = quad_sum(sc);
      s[cc] = ok ? sc : -INFINITY;
    }
    float mc = m;
#pragma unroll
    for (int cc = 0; cc < kChunk; ++cc) mc = fmaxf(mc, s[cc]);
    const float corr = exp2f(m - mc);  // m = -inf only before the first chunk (key 0 is
                                       // the query itself, always attended)
    l *= corr;
#pragma unroll
    for (int u = 0; u < 16; ++u) o[u] *= corr;
    m = mc;
#pragma unroll
    for (int cc = 0; cc < kChunk; ++cc) {
      const int c = c0 + cc;
      const float p = exp2f(s[cc] - m);
      l += p;
      if (p > 0.f) {
        float vx[16];
        const int j0 = i - ks.lo[c];
        load_part(V + static_cast<size_t>(j0) * kD, r, vx);
        const float w = ks.w[c];
        const float p0 = p * (1.f - w);
#pragma unroll
        for (int u = 0; u < 16; ++u) o[u] = fmaf(p0, vx[u], o[u]);
        if (w > 0.f) {
          load_part(V + static_cast<size_t>(j0 - 1) * kD, r, vx);
          const float p1 = p * w;
#pragma unroll
          for (int u = 0; u < 16; ++u) o[u] = fmaf(p1, vx[u], o[u]);
        }
      }
    }
  }
  if (active) {
    const float inv = 1.f / l;
#pragma unroll
    for (int u = 0; u < 16; ++u) o[u] *= inv;
    DT* O = static_cast<DT*>(a.o) + base + static_cast<size_t>(i) * kD;
    store_part(O, r, o);
    if (r == 0 && a.lse != nullptr)
      a.lse[static_cast<size_t>(bh) * a.N + i] = (m + log2f(l)) * kLn2;
  }
}

// Attended index sets from the same key table: out[(i - i0) * (W + 32) + slot].
__global__ void debug_indices_kernel(LayerTable t, int N, int i0, int i1, int32_t* out,
                                     float* w_out) {
  __shared__ KeySmem ks;
  build_keys(t, N, &ks);
  __syncthreads();
  const int stride = t.W + kMaxR;
  const int rows = i1 - i0;
  for (int idx = blockIdx.x * blockDim.x + threadIdx.x; idx < rows * stride;
       idx += gridDim.x * blockDim.x) {
    const int row = idx / stride, slot = idx % stride;
    const int i = i0 + row;
    int val = -1;
    if (slot < t.W) {
      if (i >= ks.need[slot]) val = i - ks.lo[slot];
    } else {
      const int c = t.W + (slot - t.W);
      if (slot - t.W < ks.nr && i >= ks.need[c]) val = i - ks.lo[c];
    }
    out[idx] = val;
  }
  if (blockIdx.x == 0 && w_out != nullptr)
    for (int rr = threadIdx.x; rr < kMaxR; rr += blockDim.x)
      w_out[rr] = rr < ks.nr ? ks.w[t.W + rr] : 0.f;
}

static size_t fwd_smem_bytes(const LayerTable& t) {
  // factor slots: window + rungs (+ second row per interp rung)
  const int slots = t.W + kMaxR + (t.mode == 1 ? kMaxR : 0);
  return static_cast<size_t>(slots) * kFreq * sizeof(float2);
}

cudaError_t launch_fwd(const LayerTable& t, int B, int H, int N, int dtype, const void* q,
                       const void* k, const void* v, void* o, float* lse, const float2* lo_tab,
                       const float2* hi_tab, cudaStream_t stream) {
  FwdArgs a;
  a.t = t;
  a.N = N;
  a.tiles = (N + kTile - 1) / kTile;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.rope_lo = lo_tab;
  a.rope_hi = hi_tab;
  a.qscale = kLog2e / 8.0f;  // 1/sqrt(64) = 0.125 exactly
  const size_t smem = fwd_smem_bytes(t);
  const long long blocks = static_cast<long long>(a.tiles) * B * H;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  if (dtype == 0) {
    fwd_kernel<float><<<static_cast<unsigned>(blocks), kThreads, smem, stream>>>(a);
  } else {
    fwd_kernel<__nv_bfloat16><<<static_cast<unsigned>(blocks), kThreads, smem, stream>>>(a);
  }
  return cudaGetLastError();
}

cudaError_t launch_debug_indices(const LayerTable& t, int N, int i0, int i1, int32_t* out,
                                 float* w_out, cudaStream_t stream) {
  const long long total = static_cast<long long>(i1 - i0) * (t.W + kMaxR);
  int blocks = static_cast<int>((total + 255) / 256);
  if (blocks < 1) blocks = 1;
  if (blocks > 4096) blocks = 4096;
  debug_indices_kernel<<<blocks, 256, 0, stream>>>(t, N, i0, i1, out, w_out);
  return cudaGetLastError();
}

}  // namespace fibattn
