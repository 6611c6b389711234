// Backward kernels of Depth-Staggered Fibonacci Spacing sparse attention (sm_103a).
//
// Gradients of l = sum(O * dO) for one layer.  "Depth-Staggered Fibonacci Spacing for
// Sparse Attention", Methodology > "Implementation": the interpolated rows give alpha a
// gradient; here dw/dalpha = f with lo held fixed (the right derivative at integer d).
//
//   Delta_i = dO_i . O_i                                  (bwd_pre_kernel)
//   P = exp(s - LSE), dP = dO . v~, dS = P (dP - Delta)
//   dq_i  = scale sum_c dS_c k~_c rotated back to position i         (bwd_dq_kernel,
//   dalpha partial per CTA                                            query-owned)
//   dk_j, dv_j: every (query, key-slot) that reads row j, with its blend weight
//                                                          (bwd_dkdv_kernel, key-owned:
//                                                           no atomics)
//   dalpha = fixed-order sum of the CTA partials          (dalpha_reduce_kernel)
// Both main kernels recompute scores from raw Q/K with the relative RoPE factors
// (see fwd.cu), so no attention matrix is stored.
#include "common.cuh"

namespace fibattn {

constexpr int kBTile = 64;
constexpr int kBThreads = 256;

struct BwdArgs {
  LayerTable t;
  int N;
  int tiles;
  const void* q;
  const void* k;
  const void* v;
  const void* o;
  const float* lse;
  const void* dO;
  void* dq;
  void* dk;
  void* dv;
  float* delta;     // [B*H*N] workspace
  float* partials;  // [blocks] workspace
  const float2* rope_lo;
  const float2* rope_hi;
};

template <typename DT>
__global__ void __launch_bounds__(kBThreads) bwd_pre_kernel(BwdArgs a, long long rows) {
  const long long row = (static_cast<long long>(blockIdx.x) * kBThreads + threadIdx.x) >> 2;
  const int r = threadIdx.x & 3;
  const bool ok = row < rows;
  const long long rr = ok ? row : rows - 1;
  float x[16], y[16];
  load_part(static_cast<const DT*>(a.dO) + rr * kD, r, x);
  load_part(static_cast<const DT*>(a.o) + rr * kD, r, y);
  float s = 0.f;
#pragma unroll
  for (int u = 0; u < 16; ++u) s = fmaf(x[u], y[u], s);
  s = quad_sum(s);
  if (ok && r == 0) a.delta[rr] = s;
}

__device__ __forceinline__ float dot16(const float (&x)[16], const float (&y)[16]) {
  float a0 = 0.f, a1 = 0.f;
#pragma unroll
  for (int u = 0; u < 16; u += 2) {
    a0 = fmaf(x[u], y[u], a0);
    a1 = fmaf(x[u + 1], y[u + 1], a1);
  }
  return a0 + a1;
}

template <typename DT>
__global__ void __launch_bounds__(kBThreads) bwd_dq_kernel(BwdArgs a) {
  __shared__ KeySmem ks;
  __shared__ float red[kBThreads / 32];
  extern __shared__ float4 smem_dyn[];
  float2* fac = reinterpret_cast<float2*>(smem_dyn);
  const int bh = blockIdx.x / a.tiles;
  const int tile = blockIdx.x - bh * a.tiles;
  build_keys(a.t, a.N, &ks);
  __syncthreads();
  build_factors(&ks, a.t.mode, a.t.W, a.rope_lo, a.rope_hi, fac);
  __syncthreads();

  const int qi = threadIdx.x >> 2, r = threadIdx.x & 3;
  const int i_raw = tile * kBTile + qi;
  const bool active = i_raw < a.N;
  const int i = active ? i_raw : a.N - 1;
  const size_t base = static_cast<size_t>(bh) * a.N * kD;
  const DT* Q = static_cast<const DT*>(a.q) + base;
  const DT* K = static_cast<const DT*>(a.k) + base;
  const DT* V = static_cast<const DT*>(a.v) + base;
  const DT* dO = static_cast<const DT*>(a.dO) + base;
  const float qs = kLog2e / 8.0f;

  float q[16], g[16], dq[16];
  load_part(Q + static_cast<size_t>(i) * kD, r, q);
  load_part(dO + static_cast<size_t>(i) * kD, r, g);
#pragma unroll
  for (int u = 0; u < 16; ++u) {
    q[u] *= qs;
    dq[u] = 0.f;
  }
  const float lse2 = a.lse[static_cast<size_t>(bh) * a.N + i] * kLog2e;
  const float delta = a.delta[static_cast<size_t>(bh) * a.N + i];
  const int nv = ks.nv, W = a.t.W;
  float dalpha = 0.f;

  for (int c = 0; c < nv; ++c) {
    const bool ok = i >= ks.need[c];
    const float w = ks.w[c];
    const int f = ks.f[c];
    const int j0 = i - ks.lo[c];
    // the second row is read for a blend (w > 0) and, for an interp rung, for dalpha
    const bool two = ok && (f != 0) && (j0 - 1 >= 0);
    float k0[16], k1[16], v0[16], v1[16];
    float s0 = 0.f, s1 = 0.f, p0d = 0.f, p1d = 0.f;
    if (ok) {
      load_part(K + static_cast<size_t>(j0) * kD, r, k0);
      load_part(V + static_cast<size_t>(j0) * kD, r, v0);
      s0 = rel_dot(q, k0, fac + c * kFreq + 8 * r);
      p0d = dot16(g, v0);
    }
    if (two) {
      load_part(K + static_cast<size_t>(j0 - 1) * kD, r, k1);
      load_part(V + static_cast<size_t>(j0 - 1) * kD, r, v1);
      s1 = rel_dot(q, k1, fac + (nv + (c - W)) * kFreq + 8 * r);
      p1d = dot16(g, v1);
    }
    s0 = quad_sum(s0);
    s1 = quad_sum(s1);
    p0d = quad_sum(p0d);
    p1d = quad_sum(p1d);
    if (ok) {
      const float s = (1.f - w) * s0 + w * s1;   // log2 units
      const float P = exp2f(s - lse2);
      const float dP = (1.f - w) * p0d + w * p1d;
      const float dS = P * (dP - delta);
      // dq += scale dS ((1-w) rot(k0, -lo) + w rot(k1, -(lo+1)))
      const float c0 = 0.125f * dS * (1.f - w);
      rotate_part(k0, fac + c * kFreq + 8 * r, true);
#pragma unroll
      for (int u = 0; u < 16; ++u) dq[u] = fmaf(c0, k0[u], dq[u]);
      if (two) {
        if (w > 0.f) {
          const float c1 = 0.125f * dS * w;
          float kr[16];
#pragma unroll
          for (int u = 0; u < 16; ++u) kr[u] = k1[u];
          rotate_part(kr, fac + (nv + (c - W)) * kFreq + 8 * r, true);
#pragma unroll
          for (int u = 0; u < 16; ++u) dq[u] = fmaf(c1, kr[u], dq[u]);
        }
        // dl/dw = dS (s1 - s0) [natural units] + P (dO.v1 - dO.v0); dw/dalpha = f
        if (r == 0 && active)
          dalpha += static_cast<float>(f) * (dS * (s1 - s0) * kLn2 + P * (p1d - p0d));
      }
    }
  }
  if (active) {
    DT* out = static_cast<DT*>(a.dq) + base + static_cast<size_t>(i) * kD;
    store_part(out, r, dq);
  }
  // CTA partial of dalpha, fixed order: warp tree, then warps in index order
  for (int off = 16; off > 0; off >>= 1) dalpha += __shfl_xor_sync(0xffffffffu, dalpha, off);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = dalpha;
  __syncthreads();
  if (threadIdx.x == 0) {
    float s = 0.f;
    for (int wp = 0; wp < kBThreads / 32; ++wp) s += red[wp];
    a.partials[blockIdx.x] = s;
  }
}

template <typename DT>
__global__ void __launch_bounds__(kBThreads) bwd_dkdv_kernel(BwdArgs a) {
  __shared__ KeySmem ks;
  extern __shared__ float4 smem_dyn[];
  float2* fac = reinterpret_cast<float2*>(smem_dyn);
  const int bh = blockIdx.x / a.tiles;
  const int tile = blockIdx.x - bh * a.tiles;
  build_keys(a.t, a.N, &ks);
  __syncthreads();
  build_factors(&ks, a.t.mode, a.t.W, a.rope_lo, a.rope_hi, fac);
  __syncthreads();

  const int ji = threadIdx.x >> 2, r = threadIdx.x & 3;
  const int j_raw = tile * kBTile + ji;
  const bool active = j_raw < a.N;
  const int j = active ? j_raw : a.N - 1;
  const size_t base = static_cast<size_t>(bh) * a.N * kD;
  const DT* Q = static_cast<const DT*>(a.q) + base;
  const DT* K = static_cast<const DT*>(a.k) + base;
  const DT* V = static_cast<const DT*>(a.v) + base;
  const DT* dO = static_cast<const DT*>(a.dO) + base;
  const float* lse = a.lse + static_cast<size_t>(bh) * a.N;
  const float* dlt = a.delta + static_cast<size_t>(bh) * a.N;
  const float qs = kLog2e / 8.0f;
  const int nv = ks.nv, W = a.t.W;

  float dk[16], dv[16];
#pragma unroll
  for (int u = 0; u < 16; ++u) {
    dk[u] = 0.f;
    dv[u] = 0.f;
  }
  // role 0: row j is the first row (i - lo) of key c for query i = j + lo, weight 1-w
  // role 1: row j is the second row (i - lo - 1) of key c for query i = j + lo + 1, weight w
  for (int c = 0; c < nv; ++c) {
    const float w = ks.w[c];
    for (int role = 0; role < 2; ++role) {
      if (role == 1 && !(w > 0.f)) break;
      const int i = j + ks.lo[c] + role;
      const bool ok = (i < a.N) && (i >= ks.need[c]);
      float qx[16], g[16], ka[16], kb[16], va[16], vb[16];
      float sa = 0.f, sb = 0.f, pa = 0.f, pb = 0.f;
      const int ra = i - ks.lo[c];  // first row of the key for query i
      if (ok) {
        load_part(Q + static_cast<size_t>(i) * kD, r, qx);
        load_part(dO + static_cast<size_t>(i) * kD, r, g);
#pragma unroll
        for (int u = 0; u < 16; ++u) qx[u] *= qs;
        load_part(K + static_cast<size_t>(ra) * kD, r, ka);
        load_part(V + static_cast<size_t>(ra) * kD, r, va);
        sa = rel_dot(qx, ka, fac + c * kFreq + 8 * r);
        pa = dot16(g, va);
        if (w > 0.f) {
          load_part(K + static_cast<size_t>(ra - 1) * kD, r, kb);
          load_part(V + static_cast<size_t>(ra - 1) * kD, r, vb);
          sb = rel_dot(qx, kb, fac + (nv + (c - W)) * kFreq + 8 * r);
          pb = dot16(g, vb);
        }
      }
      sa = quad_sum(sa);
      sb = quad_sum(sb);
      pa = quad_sum(pa);
      pb = quad_sum(pb);
      if (ok) {
        const float s = (1.f - w) * sa + w * sb;
        const float P = exp2f(s - lse[i] * kLog2e);
        const float dP = (1.f - w) * pa + w * pb;
        const float dS = P * (dP - dlt[i]);
        const float wt = role == 0 ? (1.f - w) : w;
        // dk_j += wt * scale * dS * rot(q_i, +(i - j)); dv_j += wt * P * dO_i
        const float cq = wt * 0.125f * dS / qs;  // qx carries qs; undo it
        const float2* e = role == 0 ? fac + c * kFreq + 8 * r : fac + (nv + (c - W)) * kFreq + 8 * r;
        rotate_part(qx, e, false);
        const float cv = wt * P;
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          dk[u] = fmaf(cq, qx[u], dk[u]);
          dv[u] = fmaf(cv, g[u], dv[u]);
        }
      }
    }
  }
  if (active) {
    store_part(static_cast<DT*>(a.dk) + base + static_cast<size_t>(j) * kD, r, dk);
    store_part(static_cast<DT*>(a.dv) + base + static_cast<size_t>(j) * kD, r, dv);
  }
}

__global__ void dalpha_reduce_kernel(const float* partials, int n, float* dalpha, int mode) {
  __shared__ float red[256];
  float s = 0.f;
  for (int idx = threadIdx.x; idx < n; idx += 256) s += partials[idx];
  red[threadIdx.x] = s;
  __syncthreads();
  for (int off = 128; off > 0; off >>= 1) {
    if (threadIdx.x < off) red[threadIdx.x] += red[threadIdx.x + off];
    __syncthreads();
  }
  if (threadIdx.x == 0) *dalpha = mode == 1 ? red[0] : 0.f;
}

size_t bwd_workspace_bytes(int B, int H, int N) {
  const size_t rows = static_cast<size_t>(B) * H * N;
  const size_t tiles = (static_cast<size_t>(N) + kBTile - 1) / kBTile * B * H;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  return up(rows * sizeof(float)) + up(tiles * sizeof(float));
}

cudaError_t launch_bwd(const LayerTable& t, int B, int H, int N, int dtype, const void* q,
                       const void* k, const void* v, const void* o, const float* lse,
                       const void* dO, void* dq, void* dk, void* dv, float* dalpha,
                       void* ws, const float2* lo_tab, const float2* hi_tab,
                       cudaStream_t stream) {
  BwdArgs a;
  a.t = t;
  a.N = N;
  a.tiles = (N + kBTile - 1) / kBTile;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.dO = dO;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  const size_t rows = static_cast<size_t>(B) * H * N;
  a.delta = static_cast<float*>(ws);
  a.partials = reinterpret_cast<float*>(static_cast<char*>(ws) + (rows * sizeof(float) + 255) / 256 * 256);
  a.rope_lo = lo_tab;
  a.rope_hi = hi_tab;
  const int slots = t.W + kMaxR + (t.mode == 1 ? kMaxR : 0);
  const size_t smem = static_cast<size_t>(slots) * kFreq * sizeof(float2);
  const long long blocks = static_cast<long long>(a.tiles) * B * H;
  const long long pre_blocks = (static_cast<long long>(rows) * 4 + kBThreads - 1) / kBThreads;
  if (blocks > 0x7fffffffLL || pre_blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  if (dtype == 0) {
    bwd_pre_kernel<float><<<static_cast<unsigned>(pre_blocks), kBThreads, 0, stream>>>(a, static_cast<long long>(rows));
    bwd_dq_kernel<float><<<static_cast<unsigned>(blocks), kBThreads, smem, stream>>>(a);
    bwd_dkdv_kernel<float><<<static_cast<unsigned>(blocks), kBThreads, smem, stream>>>(a);
  } else {
    bwd_pre_kernel<__nv_bfloat16><<<static_cast<unsigned>(pre_blocks), kBThreads, 0, stream>>>(a, static_cast<long long>(rows));
    bwd_dq_kernel<__nv_bfloat16><<<static_cast<unsigned>(blocks), kBThreads, smem, stream>>>(a);
    bwd_dkdv_kernel<__nv_bfloat16><<<static_cast<unsigned>(blocks), kBThreads, smem, stream>>>(a);
  }
  dalpha_reduce_kernel<<<1, 256, 0, stream>>>(a.partials, static_cast<int>(blocks), dalpha, t.mode);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------------------
// Backward without any allocation: the scratch lives in a fixed, file-scope device array.
//
// Some callers must not allocate device memory on the call path: a plugin inside a host
// framework that owns the whole device heap, or a real-time loop with a no-allocation
// rule.  They cannot hand fib_attn_bwd a workspace of their own, so fib_attn_bwd_noalloc
// uses the array below instead.  The array is kNoAllocScratchBytes (8 MiB) on every device
// that loads the library, held until the process exits.  Every call shares it and it keeps
// the last call's contents; nothing in it needs to start at zero (Delta and the dalpha
// partials are fully written before they are read).  Two calls whose kernels overlap on the
// GPU (different streams without ordering) race on the array.
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;
static __device__ __align__(256) unsigned char g_bwd_scratch[kNoAllocScratchBytes];

// Device address of the scratch array on the current device.  In host code the array's
// name is only a host-side stand-in, never a device address, so every call looks the
// address up with cudaGetSymbolAddress (with the caller's device current) and checks the
// result.  Nothing is cached, so a context torn down and created again (cudaDeviceReset)
// never leaves a stale address behind.
cudaError_t noalloc_scratch(void** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_bwd_scratch);
  if (e != cudaSuccess) return e;
  if (p == nullptr) return cudaErrorInvalidSymbol;
  *out = p;
  return cudaSuccess;
}

size_t noalloc_scratch_bytes() { return kNoAllocScratchBytes; }

}  // namespace fibattn
