// bf16 backward (sm_103a) on tensor cores: gradients of l = sum(O * dO) for one layer,
// "Depth-Staggered Fibonacci Spacing for Sparse Attention", Methodology > "Implementation"
// (the interpolated rows give alpha a gradient; dw/dalpha = f with lo held fixed, the right
// derivative at an integer distance).
//
// Scores are recomputed, never stored.  With q'_i = R(i) q_i, k'_j = R(j) k_j (RoPE at the
// rows' own positions), s = q'.k'/8 (blended over the two rows of an interpolated key),
// P = exp(s - LSE), dP = dO . v~, Delta_i = dO_i . O_i and dS = P (dP - Delta):
//   dq_i = R(i)^T sum dS wt k'_j / 8      dk_j = R(j)^T sum dS wt q'_i / 8      dv_j = sum P wt dO_i
// over the (query, key row) pairs with blend weight wt (1 for window and mask keys).
//
// The (b, h) rows run as two halves (one when B*H = 1), the second on a side stream, each
// as three launches:
//   * bwd_prep_kernel: Q's = RoPE(q) log2(e)/8, K' = RoPE(k), V' = v and dO' = dO, all f16
//     with the chunk swizzle of fwd_tc.cu, and Delta (float32), each row read once.
//   * bwd_q_kernel (query-owned, 64 queries a CTA): the forward's structure, with dP =
//     dO'.V'^T beside S = Q's.K'^T and dq' += dS K' in place of O += P V'.  Rungs are
//     diagonals of 16x16 blocks, as in the forward (interp: one 24-row band per operand
//     gives the row and its partner).  It also writes P and dS of every attended (query,
//     key slot) -- W + R float pairs a query, the sparse pattern makes that small; stored
//     slot-major, so that a slot's run of consecutive queries is contiguous -- and each
//     CTA's dalpha partial.
//   * bwd_kv_kernel (key-owned, 64 keys a CTA, no atomics): a gather, no score is
//     recomputed.  The queries that read the CTA's keys stream through a ring (the 80-row
//     block [j0, j0+80) of Q's and dO' for the window band, then per rung the query slab
//     [j0+lo, j0+lo+65) with its run of stored P and dS), dk' += dS^T Q's and dv += P^T dO'.
//     In the half that sums it, its CTA 0 also adds the dalpha partials of both halves'
//     dQ grids in a fixed order.
// Precision as the forward: f16 operands (Q's, K', V', dO', P, dS), f32 accumulation.
#include <algorithm>
#include <type_traits>

#include "tc_common.cuh"

namespace fibattn {

constexpr int kBWarps = 4;                 // compute warps of a backward CTA (16 rows each)
constexpr int kBTileT = 16 * kBWarps;      // queries (bwd_q) or keys (bwd_kv) per CTA
constexpr int kBCons = 32 * kBWarps;
constexpr int kBThreadsT = kBCons + 32;    // + one producer warp
constexpr int kBSlots = 3;
constexpr int kKvQRows = kBTileT + 16;     // query rows a kv stage holds (window block: 80)
constexpr int kBWinMax = 16;               // widest window of the tensor-core backward
constexpr int kKvPdsBytes = 68 * 8;        // a kv rung stage's (P, dS) run: 65 queries, rounded

struct BtcArgs {
  LayerTable t;
  int N;
  int tiles;
  int bh;
  int slab_rows;   // bwd_q: rows of a rung slab region (64, interp 72)
  int slot_bytes;
  const __half* qs;   // Q's rows
  const __half* dos;  // dO' rows
  const __half* kp;   // K' rows
  const __half* vp;   // V' rows
  const float* lse;
  const float* delta;
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  float* partials;
  int n_partials;   // CTAs of bwd_q_kernel
  float* dalpha;    // written by bwd_kv_kernel's CTA 0: the fixed-order sum of the partials
  float2* pds;      // (P, dS) of every attended (query, key slot): [B*H][pds_stride][N], slot-major
                    // (a rung's slot of consecutive queries is contiguous: coalesced in both kernels)
  int pds_stride;   // W + rungs of the layer table
  const float2* rope_lo;
  const float2* rope_hi;
  int* status;
  unsigned long long wait_ns;
};

__device__ __forceinline__ void bcons_sync() {
  asm volatile("bar.sync 1, %0;\n" ::"n"(kBCons) : "memory");
}

// e^{i p theta_m} for m = 8nt + 2t + e (nt < 4, e < 2): the frequencies whose dims a lane
// holds in the natural accumulator layout (dims 8nt+2t+e and their partners 32 + those).
__device__ __forceinline__ void rope_natural(const float2* __restrict__ lo_tab, const float2* __restrict__ hi_tab,
                                             int p, int t, float2 (&e)[8]) {
  const float2* hr = hi_tab + (p / kSplit) * kFreq;
  const float2* lr = lo_tab + (p % kSplit) * kFreq;
#pragma unroll
  for (int nt = 0; nt < 4; ++nt) {
    const float4 x = __ldg(reinterpret_cast<const float4*>(hr + 8 * nt + 2 * t));
    const float4 y = __ldg(reinterpret_cast<const float4*>(lr + 8 * nt + 2 * t));
    e[2 * nt] = make_float2(x.x * y.x - x.y * y.y, x.x * y.y + x.y * y.x);
    e[2 * nt + 1] = make_float2(x.z * y.z - x.w * y.w, x.z * y.w + x.w * y.z);
  }
}

// Row h (0: g, 1: g+8) of a natural-layout accumulator rotated back by R(p)^T, times scale,
// stored as bf16: dims 8nt+2t+e (nt < 4) pair with 32 + the same.
__device__ __forceinline__ void store_rotated_back(__nv_bfloat16* row, const float (&acc)[8][4], int h, int t,
                                                   const float2 (&e)[8], float scale) {
  uint32_t* out = reinterpret_cast<uint32_t*>(row);
#pragma unroll
  for (int nt = 0; nt < 4; ++nt) {
    float lo2[2], hi2[2];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const float a = acc[nt][2 * h + c], b = acc[nt + 4][2 * h + c];
      const float2 f = e[2 * nt + c];
      lo2[c] = (a * f.x + b * f.y) * scale;   // dq_m     =  cos g'_m + sin g'_{m+32}
      hi2[c] = (b * f.x - a * f.y) * scale;   // dq_{m+32} = -sin g'_m + cos g'_{m+32}
    }
    out[4 * nt + t] = pack_bf2_rn(lo2[0], lo2[1]);
    out[16 + 4 * nt + t] = pack_bf2_rn(hi2[0], hi2[1]);
  }
}

__device__ __forceinline__ void store_plain(__nv_bfloat16* row, const float (&acc)[8][4], int h, int t) {
  uint32_t* out = reinterpret_cast<uint32_t*>(row);
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) out[4 * nt + t] = pack_bf2_rn(acc[nt][2 * h], acc[nt][2 * h + 1]);
}

// ------------------------------------------------------------------ preparation
// One thread per (row, quarter u), frequencies m = 8u .. 8u+7 (chunks u and u+4 of a row):
// the four f16 arrays, and Delta by a quad reduction.  Without KV (K' and V' prepared by the
// layer's forward and handed over), only Q's, dO' and Delta.
constexpr int kBPrepThreads = 128;  // four threads a row (128: measured best of 64-512)

template <bool KV>
__global__ void __launch_bounds__(kBPrepThreads) bwd_prep_kernel(const __nv_bfloat16* __restrict__ q,
                                                       const __nv_bfloat16* __restrict__ k,
                                                       const __nv_bfloat16* __restrict__ v,
                                                       const __nv_bfloat16* __restrict__ o,
                                                       const __nv_bfloat16* __restrict__ dO, __half* __restrict__ qs,
                                                       __half* __restrict__ kp, __half* __restrict__ vp,
                                                       __half* __restrict__ dos, float* __restrict__ delta,
                                                       const float2* __restrict__ lo_tab,
                                                       const float2* __restrict__ hi_tab, int N, long long rows,
                                                       float qscale, int* __restrict__ status) {
  // The dependent dQ grid may launch at once (its CTAs take the SMs as this grid drains);
  // it waits for the whole of this grid before it reads what this grid writes.
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  const long long gid = static_cast<long long>(blockIdx.x) * kBPrepThreads + threadIdx.x;
  const long long row = gid >> 2;
  const unsigned active = __ballot_sync(0xffffffffu, row < rows);  // whole quads
  if (row >= rows) return;
  const int u = static_cast<int>(gid & 3);
  const int p = static_cast<int>(row % N);
  const size_t off = static_cast<size_t>(row) * kD;
  auto ld = [&](const __nv_bfloat16* base, int c) { return __ldcs(reinterpret_cast<const uint4*>(base + off) + c); };
  const uint4 qa = ld(q, u), qb = ld(q, u + 4), ga = ld(dO, u), gb = ld(dO, u + 4);
  const uint4 oa = ld(o, u), ob = ld(o, u + 4);
  uint4 ka, kb, va, vb;
  if (KV) ka = ld(k, u), kb = ld(k, u + 4), va = ld(v, u), vb = ld(v, u + 4);
  float2 e[8];
  rope_row(lo_tab, hi_tab, p, u, e);
  auto rotate = [&](const uint4& xa4, const uint4& xb4, float sc, uint4& ya4, uint4& yb4) {
    const uint32_t xa[4] = {xa4.x, xa4.y, xa4.z, xa4.w}, xb[4] = {xb4.x, xb4.y, xb4.z, xb4.w};
    uint32_t ya[4], yb[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const float x1 = bf_lo(xa[c]) * sc, y1 = bf_hi(xa[c]) * sc, x2 = bf_lo(xb[c]) * sc, y2 = bf_hi(xb[c]) * sc;
      const float2 e0 = e[2 * c], e1 = e[2 * c + 1];
      ya[c] = pack_h2(x1 * e0.x - x2 * e0.y, y1 * e1.x - y2 * e1.y);
      yb[c] = pack_h2(x1 * e0.y + x2 * e0.x, y1 * e1.y + y2 * e1.x);
    }
    ya4 = make_uint4(ya[0], ya[1], ya[2], ya[3]);
    yb4 = make_uint4(yb[0], yb[1], yb[2], yb[3]);
  };
  auto to_h = [&](const uint4& x4) {
    return make_uint4(pack_h2(bf_lo(x4.x), bf_hi(x4.x)), pack_h2(bf_lo(x4.y), bf_hi(x4.y)),
                      pack_h2(bf_lo(x4.z), bf_hi(x4.z)), pack_h2(bf_lo(x4.w), bf_hi(x4.w)));
  };
  const int sw = swz(p);
  auto put = [&](__half* base, const uint4& lo4, const uint4& hi4) {
    uint4* r4 = reinterpret_cast<uint4*>(base + off);
    r4[u ^ sw] = lo4;
    r4[(u + 4) ^ sw] = hi4;
  };
  // A value beyond the float16 range (|x| > 65504 after rotation and scaling) cannot be held
  // in the prepared rows: record it (the gradients of this call are then unspecified).
  uint32_t bad = 0;
  auto chk = [&](const uint4& x) { bad |= h2_nonfinite(x.x) | h2_nonfinite(x.y) | h2_nonfinite(x.z) | h2_nonfinite(x.w); };
  uint4 ya, yb;
  rotate(qa, qb, qscale, ya, yb);
  chk(ya); chk(yb);
  put(qs, ya, yb);
  if (KV) {
    rotate(ka, kb, 1.f, ya, yb);
    chk(ya); chk(yb);
    put(kp, ya, yb);
    const uint4 vha = to_h(va), vhb = to_h(vb);
    chk(vha); chk(vhb);
    put(vp, vha, vhb);
  }
  const uint4 gha = to_h(ga), ghb = to_h(gb);
  chk(gha); chk(ghb);
  put(dos, gha, ghb);
  if (bad) atomicExch(status, kStatusRange);
  // Delta = dO . O over the row (float32 from the bf16 values)
  float d = 0.f;
  const uint32_t g4[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
  const uint32_t o4[8] = {oa.x, oa.y, oa.z, oa.w, ob.x, ob.y, ob.z, ob.w};
#pragma unroll
  for (int c = 0; c < 8; ++c) d = fmaf(bf_lo(g4[c]), bf_lo(o4[c]), fmaf(bf_hi(g4[c]), bf_hi(o4[c]), d));
  d += __shfl_xor_sync(active, d, 1);
  d += __shfl_xor_sync(active, d, 2);
  if (u == 0) delta[row] = d;
}

// ------------------------------------------------------------------ query-owned: dq, dalpha
template <int MODE>
__global__ void __launch_bounds__(kBThreadsT, 3) bwd_q_kernel(BtcArgs a) {
  __shared__ KeySmem ks;
  __shared__ __align__(8) uint64_t full_bar[kBSlots];
  __shared__ __align__(8) uint64_t empty_bar[kBSlots];
  __shared__ volatile int s_err;
  __shared__ float red[kBWarps];
  extern __shared__ __align__(128) unsigned char smem[];
  const int SR = a.slab_rows;
  unsigned char* ring = smem;
  constexpr int kI = MODE == 1 ? 1 : 0;

  const int bh = blockIdx.x % a.bh;
  const int tile = a.tiles - 1 - static_cast<int>(blockIdx.x / a.bh);  // heaviest first
  const int i0 = tile * kBTileT;
  const int N = a.N;
  const int tid = threadIdx.x;
  const size_t base = static_cast<size_t>(bh) * N * kD;
  const int i_last = min(i0 + kBTileT, N) - 1;
  const int w0 = max(i0 - 16, 0);

  build_keys(a.t, N, &ks);
  if (tid == 0) {
    s_err = 0;
    for (int s = 0; s < kBSlots; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kBWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncthreads();
  const int W = a.t.W;
  const int nr = ks.nr;
  const int warp = tid >> 5, lane = tid & 31;
  const unsigned attended = __ballot_sync(0xffffffffu, lane < nr && ks.need[W + lane] <= i_last);
  const int nrt = 32 - __clz(static_cast<int>(attended));
  const int n_stages = 3 + nrt;  // Q's + dO', window K', window V', then one per rung

  // ===================================================================== producer
  if (warp == kBWarps) {
    if (lane != 0) return;
    int last_n[kBSlots];
#pragma unroll
    for (int s = 0; s < kBSlots; ++s) last_n[s] = -1;
    for (int n = 0; n < n_stages; ++n) {
      if (s_err) break;
      const int slot = n % kBSlots;
      if (!mbar_wait_backoff(&empty_bar[slot], ((n / kBSlots) & 1) ^ 1, a.wait_ns)) {
        s_err = 1;
        break;
      }
      unsigned char* dst = ring + slot * a.slot_bytes;
      if (n == 0) {  // Q's and dO' rows [i0, i_last]
        // every array read from here on comes from the preparation grid launched just
        // before this one (programmatic dependent launch): wait for it and its writes
        asm volatile("griddepcontrol.wait;\n" ::: "memory");
        const uint32_t bytes = static_cast<uint32_t>(i_last - i0 + 1) * kRowBytes;
        mbar_arrive_tx(&full_bar[slot], 2 * bytes);
        bulk_g2s(dst, a.qs + base + static_cast<size_t>(i0) * kD, bytes, &full_bar[slot]);
        bulk_g2s(dst + SR * kRowBytes, a.dos + base + static_cast<size_t>(i0) * kD, bytes, &full_bar[slot]);
      } else if (n <= 2) {  // window rows [w0, i_last] of K' (n = 1) or V' (n = 2)
        const uint32_t bytes = static_cast<uint32_t>(i_last + 1 - w0) * kRowBytes;
        mbar_arrive_tx(&full_bar[slot], bytes);
        bulk_g2s(dst + (w0 - (i0 - 16)) * kRowBytes, (n == 1 ? a.kp : a.vp) + base + static_cast<size_t>(w0) * kD,
                 bytes, &full_bar[slot]);
      } else {  // rung slab rows [first, first + SR) of K', then of V', where inside [0, N)
        const int lo = ks.lo[W + n - 3];
        const int first = i0 - lo - kI;
        const int r0 = max(first, 0);
        const int r1 = i_last - lo + 1;
        const uint32_t bytes = r1 > r0 ? static_cast<uint32_t>(r1 - r0) * kRowBytes : 0u;
        mbar_arrive_tx(&full_bar[slot], 2 * bytes);
        if (bytes) {
          bulk_g2s(dst + (r0 - first) * kRowBytes, a.kp + base + static_cast<size_t>(r0) * kD, bytes, &full_bar[slot]);
          bulk_g2s(dst + (SR + r0 - first) * kRowBytes, a.vp + base + static_cast<size_t>(r0) * kD, bytes,
                   &full_bar[slot]);
        }
      }
      last_n[slot] = n;
    }
#pragma unroll
    for (int s = 0; s < kBSlots; ++s)
      if (last_n[s] >= 0) mbar_wait(&full_bar[s], (last_n[s] / kBSlots) & 1, a.wait_ns);
    if (s_err) atomicExch(a.status, kStatusTimeout);
    return;
  }

  // ===================================================================== compute warps
  const int g = lane >> 2, t = lane & 3;
  const int mi = lane >> 3, rl = lane & 7;
  const int q0 = i0 + 16 * warp;
  int irow[2], ic[2];
  float lse2[2], dlt[2];
  asm volatile("griddepcontrol.wait;\n" ::: "memory");  // Delta comes from the preparation grid
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    irow[h] = q0 + g + 8 * h;
    ic[h] = irow[h] < N ? irow[h] : N - 1;
    lse2[h] = __ldg(a.lse + static_cast<size_t>(bh) * N + ic[h]) * kLog2e;
    dlt[h] = __ldg(a.delta + static_cast<size_t>(bh) * N + ic[h]);
  }
  auto wait_stage = [&](int n) {
    if (!s_err && !mbar_wait(&full_bar[n % kBSlots], (n / kBSlots) & 1, a.wait_ns)) {
      s_err = 1;
      atomicExch(a.status, kStatusTimeout);
    }
  };
  auto release_stage = [&](int n) {
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_bar[n % kBSlots]);
  };
  auto slot_of = [&](int n) { return ring + (n % kBSlots) * a.slot_bytes; };

  // ---- stage 0: A fragments of Q's and dO' (dims D_t of rows g, g+8)
  uint32_t qa[2][2][4], da[2][2][4];
  wait_stage(0);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int row = ic[h] - i0;
    lds_kfrag(reinterpret_cast<const uint4*>(slot_of(0) + row * kRowBytes), t, ic[h], qa[h][0], qa[h][1]);
    lds_kfrag(reinterpret_cast<const uint4*>(slot_of(0) + (SR + row) * kRowBytes), t, ic[h], da[h][0], da[h][1]);
  }
  release_stage(0);

  // ---- window: S = Q's K'^T, dP = dO' V'^T over keys [q0-16, q0+16); dq' += dS K'
  float2* wst = reinterpret_cast<float2*>(ring + kBSlots * a.slot_bytes) + warp * 16 * kBWinMax;  // [slot][row]
  float acc[8][4];  // dq' in the natural accumulator layout
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
  const uint4* Ks = reinterpret_cast<const uint4*>(slot_of(1));
  const uint4* Vs = reinterpret_cast<const uint4*>(slot_of(2));
  float S[4][4], D[4][4];
  wait_stage(1);
  wait_stage(2);
#pragma unroll
  for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
    for (int c = 0; c < 4; ++c) S[nt][c] = D[nt][c] = 0.f;
    const int row = 16 * warp + 8 * nt + g;
    uint32_t kl[4], kh[4], vl[4], vh[4];
    lds_kfrag(Ks + row * 8, t, i0 - 16 + row, kl, kh);
    lds_kfrag(Vs + row * 8, t, i0 - 16 + row, vl, vh);
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      mma16816(S[nt], qa[0][0][s], qa[1][0][s], qa[0][1][s], qa[1][1][s], kl[s], kh[s]);
      mma16816(D[nt], da[0][0][s], da[1][0][s], da[0][1][s], da[1][1][s], vl[s], vh[s]);
    }
  }
  release_stage(2);
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int c = 8 * nt + 2 * t + e;
        const int dist = g + 8 * h + 16 - c;
        const bool ok = dist >= 0 && dist < W && q0 - 16 + c >= 0;
        // keys outside the copied window rows (before position 0, or after the tile's last
        // row) were computed from stale shared memory: they are replaced, never multiplied,
        // so that no stale NaN or infinity can reach dS through a product with p = 0
        const float p = ok ? exp2f(S[nt][2 * h + e] - lse2[h]) : 0.f;
        S[nt][2 * h + e] = ok ? p * (D[nt][2 * h + e] - dlt[h]) : 0.f;  // dS
        // slot d of query row g + 8h (the key i - d), staged so that the warp writes each slot's
        // 16 queries as one contiguous run below; every (slot < W, row) is one element here
        if (dist >= 0 && dist < W) wst[dist * 16 + g + 8 * h] = make_float2(p, S[nt][2 * h + e]);
      }
  __syncwarp();
  for (int d0 = 0; d0 < W; d0 += 2) {  // two slots a store: lanes 0-15 slot d0, 16-31 slot d0 + 1
    const int d = d0 + (lane >> 4), r = lane & 15;
    if (d < W && q0 + r < N) a.pds[(static_cast<size_t>(bh) * a.pds_stride + d) * N + q0 + r] = wst[d * 16 + r];
  }
#pragma unroll
  for (int s2 = 0; s2 < 2; ++s2) {
    const uint32_t pa0 = pack_h2(S[2 * s2][0], S[2 * s2][1]);
    const uint32_t pa1 = pack_h2(S[2 * s2][2], S[2 * s2][3]);
    const uint32_t pa2 = pack_h2(S[2 * s2 + 1][0], S[2 * s2 + 1][1]);
    const uint32_t pa3 = pack_h2(S[2 * s2 + 1][2], S[2 * s2 + 1][3]);
    const int pc = min(max(q0 - 16 + 16 * s2 + (mi & 1) * 8 + rl, w0), i_last);
    const unsigned char* krow = reinterpret_cast<const unsigned char*>(Ks) + (pc - (i0 - 16)) * kRowBytes;
    const int sw = swz(pc);
#pragma unroll
    for (int nd = 0; nd < 8; nd += 2) {
      uint32_t b[4];
      ldsm_x4_trans(b, krow + ((nd + (mi >> 1)) ^ sw) * 16);
      mma16816(acc[nd], pa0, pa1, pa2, pa3, b[0], b[1]);
      mma16816(acc[nd + 1], pa0, pa1, pa2, pa3, b[2], b[3]);
    }
  }
  release_stage(1);

  // ---- rungs (one per step): diagonal S and dP, dS, dalpha; dq' += diag(dS wt) K'_slab
  const int src_lane = 4 * g + (g >> 1);
  const float sel_lo = (t == (g >> 1) && !(g & 1)) ? 1.f : 0.f;
  const float sel_hi = (t == (g >> 1) && (g & 1)) ? 1.f : 0.f;
  const int lcop = i_last - i0 + kI;
  float dal = 0.f;
  for (int r = 0; r < nrt; ++r) {
    const int n = 3 + r;
    wait_stage(n);
    const int c = W + r;
    const int lo = ks.lo[c];
    const float w = MODE == 1 ? ks.w[c] : 0.f;
    const int first = i0 - lo - kI;
    const int fcop = max(0, lo - i0 + kI);
    bool ok[2];
    int rowu[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      ok[h] = !s_err && irow[h] < N && ic[h] >= ks.need[c];  // rows past N are not counted twice
      rowu[h] = ok[h] ? ic[h] - i0 + kI : fcop;
    }
    if (__any_sync(0xffffffffu, ok[0] || ok[1])) {
      const uint4* kst = reinterpret_cast<const uint4*>(slot_of(n));
      const uint4* vst = reinterpret_cast<const uint4*>(slot_of(n) + SR * kRowBytes);
      // scores and dP of the row (slab row rowu) and, interp, of its partner (rowu - 1),
      // broadcast to the row's quad
      float sc[2][2], dp[2][2];  // [part][h]
      if (MODE == 0) {
        float C[2][4], E[2][4];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int row = rowu[h];
          uint32_t kl[4], kh[4], vl[4], vh[4];
          lds_kfrag(kst + row * 8, t, first + row, kl, kh);
          lds_kfrag(vst + row * 8, t, first + row, vl, vh);
#pragma unroll
          for (int u = 0; u < 4; ++u) C[h][u] = E[h][u] = 0.f;
#pragma unroll
          for (int s = 0; s < 4; ++s) {
            mma16816(C[h], qa[0][0][s], qa[1][0][s], qa[0][1][s], qa[1][1][s], kl[s], kh[s]);
            mma16816(E[h], da[0][0][s], da[1][0][s], da[0][1][s], da[1][1][s], vl[s], vh[s]);
          }
        }
        sc[0][0] = __shfl_sync(0xffffffffu, (g & 1) ? C[0][1] : C[0][0], src_lane);
        sc[0][1] = __shfl_sync(0xffffffffu, (g & 1) ? C[1][3] : C[1][2], src_lane);
        dp[0][0] = __shfl_sync(0xffffffffu, (g & 1) ? E[0][1] : E[0][0], src_lane);
        dp[0][1] = __shfl_sync(0xffffffffu, (g & 1) ? E[1][3] : E[1][2], src_lane);
      } else {
        // Banded, as in the forward: column g of key n-tile nt holds slab row R0 + 8nt + g,
        // R0 = 16 warp + kI - 8, so the row of query g + 8h is column g of n-tile h + 1 and its
        // partner column (g + 7) & 7 of n-tile h + (g + 7) / 8: 12 MMAs for both diagonals of
        // S, 12 for dP.  Rows outside [fcop, lcop] are read from the nearest copied row; no
        // attending query picks those columns.
        const int R0 = 16 * warp + kI - 8;
        const int pc = (g + 7) & 7;
        const int plane = 4 * g + (pc >> 1);  // lane holding the partner entries of rows g, g+8
        const bool lo_tile = g == 0;          // partner in column 7 of the n-tile before
#pragma unroll
        for (int op = 0; op < 2; ++op) {  // 0: S from K', 1: dP from V'
          const uint4* bst = op == 0 ? kst : vst;
          float C[3][4];
#pragma unroll
          for (int nt = 0; nt < 3; ++nt) {
            const int row = min(max(R0 + 8 * nt + g, fcop), lcop);
            uint32_t bl[4], bh[4];
            lds_kfrag(bst + row * 8, t, first + row, bl, bh);
            C[nt][0] = C[nt][1] = C[nt][2] = C[nt][3] = 0.f;
#pragma unroll
            for (int s = 0; s < 4; ++s) {
              if (op == 0)
                mma16816(C[nt], qa[0][0][s], qa[1][0][s], qa[0][1][s], qa[1][1][s], bl[s], bh[s]);
              else
                mma16816(C[nt], da[0][0][s], da[1][0][s], da[0][1][s], da[1][1][s], bl[s], bh[s]);
            }
          }
          float (&out)[2][2] = op == 0 ? sc : dp;
          out[0][0] = __shfl_sync(0xffffffffu, (g & 1) ? C[1][1] : C[1][0], src_lane);
          out[0][1] = __shfl_sync(0xffffffffu, (g & 1) ? C[2][3] : C[2][2], src_lane);
          const float v0 = lo_tile ? ((pc & 1) ? C[0][1] : C[0][0]) : ((pc & 1) ? C[1][1] : C[1][0]);
          const float v1 = lo_tile ? ((pc & 1) ? C[1][3] : C[1][2]) : ((pc & 1) ? C[2][3] : C[2][2]);
          out[1][0] = __shfl_sync(0xffffffffu, v0, plane);
          out[1][1] = __shfl_sync(0xffffffffu, v1, plane);
        }
      }
      float ds[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float s = MODE == 1 ? (1.f - w) * sc[0][h] + w * sc[1][h] : sc[0][h];
        const float dpp = MODE == 1 ? (1.f - w) * dp[0][h] + w * dp[1][h] : dp[0][h];
        const float P = ok[h] ? exp2f(s - lse2[h]) : 0.f;
        ds[h] = P * (dpp - dlt[h]);
        if (ok[h] && t == 0)  // slot W + r of query i (blended P and dS of the rung key)
          a.pds[(static_cast<size_t>(bh) * a.pds_stride + c) * N + irow[h]] = make_float2(P, ds[h]);
        if (MODE == 1) {
          // dl/dw = dS (s1 - s0) + P (dO.v1 - dO.v0) (natural units), dw/dalpha = f; the
          // partner row i-lo-1 must exist (it only does not when w = 0 and i = lo)
          const bool two = ok[h] && ic[h] - lo - 1 >= 0 && t == 0;
          if (two) dal += static_cast<float>(ks.f[c]) * (ds[h] * (sc[1][h] - sc[0][h]) * kLn2 + P * (dp[1][h] - dp[0][h]));
        }
      }
      // dq' += diag(dS (1-w)) K'[slab rows] (+ diag(dS w) K'[rows - 1])
#pragma unroll
      for (int part = 0; part < (MODE == 1 ? 2 : 1); ++part) {
        if (part == 1 && !(w > 0.f)) continue;  // uniform
        const float f = MODE == 1 ? (part == 0 ? 1.f - w : w) : 1.f;
        const float x0 = ds[0] * f, x1 = ds[1] * f;
        const uint32_t a0 = pack_h2(x0 * sel_lo, x0 * sel_hi);
        const uint32_t a3 = pack_h2(x1 * sel_lo, x1 * sel_hi);
        const int kr = min(max(16 * warp + (mi & 1) * 8 + rl + kI - part, fcop), lcop);
        const unsigned char* krow = slot_of(n) + kr * kRowBytes;
        const int sw = swz(first + kr);
#pragma unroll
        for (int nd = 0; nd < 8; nd += 2) {
          uint32_t b[4];
          ldsm_x4_trans(b, krow + ((nd + (mi >> 1)) ^ sw) * 16);
          mma16816(acc[nd], a0, 0u, 0u, a3, b[0], b[1]);
          mma16816(acc[nd + 1], a0, 0u, 0u, a3, b[2], b[3]);
        }
      }
    }
    release_stage(n);
  }

  // ---- epilogue: the CTA's dalpha partial (fixed order), then dq = R(i)^T dq' / 8
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) dal += __shfl_xor_sync(0xffffffffu, dal, off);
  if (lane == 0) red[warp] = dal;
  bcons_sync();
  if (tid == 0) {
    float s = 0.f;
    for (int wp = 0; wp < kBWarps; ++wp) s += red[wp];
    a.partials[blockIdx.x] = s;
  }
  if (s_err) {
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    return;
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    if (irow[h] >= N) continue;
    float2 e[8];
    rope_natural(a.rope_lo, a.rope_hi, irow[h], t, e);
    store_rotated_back(a.dq + base + static_cast<size_t>(irow[h]) * kD, acc, h, t, e, 0.125f);
  }
  // this thread's outputs (dq, P and dS, the partial) are written: the dependent kv grid may
  // launch (it waits for this whole grid before it reads them)
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

// ------------------------------------------------------------------ key-owned: dk, dv
// Stage 0 brings the window block's Q's and dO' rows [j0, j0+80), stage 1+r the query slab
// of rung r: rows [j0+lo, j0+lo+65), and those queries' (P, dS) of the rung's slot (one
// contiguous run in the slot-major array, copied from the even element at or before it, so
// that the copy starts and ends on 16 bytes).  P and dS come from bwd_q_kernel.
template <int MODE>
__global__ void __launch_bounds__(kBThreadsT, 3) bwd_kv_kernel(BtcArgs a) {
  __shared__ KeySmem ks;
  __shared__ __align__(8) uint64_t full_bar[kBSlots];
  __shared__ __align__(8) uint64_t empty_bar[kBSlots];
  __shared__ volatile int s_err;
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* ring = smem;
  constexpr int kQ2 = kKvQRows * kRowBytes;  // dO' rows after the Q's rows

  const int bh = blockIdx.x % a.bh;
  const int tile = static_cast<int>(blockIdx.x / a.bh);  // an early key is read by more rungs
  const int j0 = tile * kBTileT;
  const int N = a.N;
  const int tid = threadIdx.x;
  const size_t base = static_cast<size_t>(bh) * N * kD;
  const int j_last = min(j0 + kBTileT, N) - 1;

  build_keys(a.t, N, &ks);
  if (tid == 0) {
    s_err = 0;
    for (int s = 0; s < kBSlots; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kBWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncthreads();
  const int W = a.t.W;
  const int nr = ks.nr;
  const int warp = tid >> 5, lane = tid & 31;
  // rungs whose first query j0 + lo exists (ascending lo: a prefix)
  const unsigned reach = __ballot_sync(0xffffffffu, lane < nr && j0 + ks.lo[W + lane] < N);
  const int nrk = 32 - __clz(static_cast<int>(reach));
  const int n_stages = 1 + nrk;

  // ===================================================================== producer
  if (warp == kBWarps) {
    if (blockIdx.x == 0 && a.dalpha != nullptr) {
      // dalpha of the layer: the dQ grids' partials, summed in a fixed order (lane l takes
      // partials l, l+32, ... in turn, then a fixed shuffle tree)
      asm volatile("griddepcontrol.wait;\n" ::: "memory");
      float acc = 0.f;
      for (int idx = lane; idx < a.n_partials; idx += 32) acc += a.partials[idx];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      if (lane == 0) *a.dalpha = MODE == 1 ? acc : 0.f;
    }
    if (lane != 0) return;
    int last_n[kBSlots];
#pragma unroll
    for (int s = 0; s < kBSlots; ++s) last_n[s] = -1;
    for (int n = 0; n < n_stages; ++n) {
      if (s_err) break;
      const int slot = n % kBSlots;
      if (!mbar_wait_backoff(&empty_bar[slot], ((n / kBSlots) & 1) ^ 1, a.wait_ns)) {
        s_err = 1;
        break;
      }
      unsigned char* dst = ring + slot * a.slot_bytes;
      const int qfirst = n == 0 ? j0 : j0 + ks.lo[W + n - 1];   // first query row of the stage
      const int qrows = n == 0 ? kKvQRows : kBTileT + 1;
      const int q1 = min(qfirst + qrows, N);
      const uint32_t qbytes = q1 > qfirst ? static_cast<uint32_t>(q1 - qfirst) * kRowBytes : 0u;
      uint32_t pbytes = 0;
      size_t p0 = 0;
      if (n > 0 && qbytes) {
        // P and dS are written by the dQ grid launched just before: wait for it (stage 0
        // holds only rows of the preparation, which completed before this grid launched)
        if (n == 1) asm volatile("griddepcontrol.wait;\n" ::: "memory");
        const size_t e0 = (static_cast<size_t>(bh) * a.pds_stride + W + n - 1) * N + qfirst;
        p0 = e0 & ~static_cast<size_t>(1);
        pbytes = static_cast<uint32_t>(((e0 + (q1 - qfirst) + 1) & ~static_cast<size_t>(1)) - p0) * sizeof(float2);
      }
      mbar_arrive_tx(&full_bar[slot], 2 * qbytes + pbytes);
      if (qbytes) {
        bulk_g2s(dst, a.qs + base + static_cast<size_t>(qfirst) * kD, qbytes, &full_bar[slot]);
        bulk_g2s(dst + kQ2, a.dos + base + static_cast<size_t>(qfirst) * kD, qbytes, &full_bar[slot]);
      }
      if (pbytes) bulk_g2s(dst + 2 * kQ2, a.pds + p0, pbytes, &full_bar[slot]);
      last_n[slot] = n;
    }
#pragma unroll
    for (int s = 0; s < kBSlots; ++s)
      if (last_n[s] >= 0) mbar_wait(&full_bar[s], (last_n[s] / kBSlots) & 1, a.wait_ns);
    if (s_err) atomicExch(a.status, kStatusTimeout);
    return;
  }

  // ===================================================================== compute warps
  const int g = lane >> 2, t = lane & 3;
  const int mi = lane >> 3, rl = lane & 7;
  const int k0 = j0 + 16 * warp;  // the warp's first key
  auto wait_stage = [&](int n) {
    if (!s_err && !mbar_wait(&full_bar[n % kBSlots], (n / kBSlots) & 1, a.wait_ns)) {
      s_err = 1;
      atomicExch(a.status, kStatusTimeout);
    }
  };
  auto release_stage = [&](int n) {
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_bar[n % kBSlots]);
  };
  auto slot_of = [&](int n) { return ring + (n % kBSlots) * a.slot_bytes; };
  // P and dS come from the dQ grid launched just before (programmatic dependent launch):
  // wait for it, and its writes, before the first load of them
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  const float2* pds = a.pds + static_cast<size_t>(bh) * N * a.pds_stride;

  float dK[8][4], dV[8][4];  // natural accumulator layout, rows = keys g, g+8
#pragma unroll
  for (int nt = 0; nt < 8; ++nt)
#pragma unroll
    for (int c = 0; c < 4; ++c) dK[nt][c] = dV[nt][c] = 0.f;

  // ---- window band: queries [k0, k0+32) of the warp's 16 keys (query = key + d, d < W).
  // C-layout element (key row g + 8h, query column c = 8nt + 2t + e): slot d = c - (g + 8h).
  {
    float S[4][4], D[4][4];  // dS^T and P^T
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int c = 8 * nt + 2 * t + e;
          const int d = c - (g + 8 * h);
          const bool ok = d >= 0 && d < W && k0 + c < N && k0 + g + 8 * h < N;
          const float2 v = ok ? __ldg(pds + static_cast<size_t>(d) * N + (k0 + c)) : make_float2(0.f, 0.f);
          D[nt][2 * h + e] = v.x;
          S[nt][2 * h + e] = v.y;
        }
    wait_stage(0);
    const unsigned char* qst = slot_of(0);
    const int qlast = min(j0 + kKvQRows, N) - 1;  // last copied query row of the block
    // dk' += dS^T Q's, dv += P^T dO' over the 32 queries (k-steps of 16)
#pragma unroll
    for (int s2 = 0; s2 < 2; ++s2) {
      const uint32_t sa0 = pack_h2(S[2 * s2][0], S[2 * s2][1]), sa1 = pack_h2(S[2 * s2][2], S[2 * s2][3]);
      const uint32_t sa2 = pack_h2(S[2 * s2 + 1][0], S[2 * s2 + 1][1]), sa3 = pack_h2(S[2 * s2 + 1][2], S[2 * s2 + 1][3]);
      const uint32_t pa0 = pack_h2(D[2 * s2][0], D[2 * s2][1]), pa1 = pack_h2(D[2 * s2][2], D[2 * s2][3]);
      const uint32_t pa2 = pack_h2(D[2 * s2 + 1][0], D[2 * s2 + 1][1]), pa3 = pack_h2(D[2 * s2 + 1][2], D[2 * s2 + 1][3]);
      const int qp = min(k0 + 16 * s2 + (mi & 1) * 8 + rl, qlast);  // rows past the block: weight 0
      const unsigned char* qrow = qst + (qp - j0) * kRowBytes;
      const int sw = swz(qp);
#pragma unroll
      for (int nd = 0; nd < 8; nd += 2) {
        uint32_t b[4], c4[4];
        ldsm_x4_trans(b, qrow + ((nd + (mi >> 1)) ^ sw) * 16);
        ldsm_x4_trans(c4, qrow + kQ2 + ((nd + (mi >> 1)) ^ sw) * 16);
        mma16816(dK[nd], sa0, sa1, sa2, sa3, b[0], b[1]);
        mma16816(dK[nd + 1], sa0, sa1, sa2, sa3, b[2], b[3]);
        mma16816(dV[nd], pa0, pa1, pa2, pa3, c4[0], c4[1]);
        mma16816(dV[nd + 1], pa0, pa1, pa2, pa3, c4[2], c4[3]);
      }
    }
    release_stage(0);
  }

  // ---- rungs: key j is read by query i = j + lo + role, as the first (role 0, weight
  // 1-w) or, interp, the second (role 1, weight w) row of that query's rung key; slab row
  // of query i: i - (j0 + lo).  dk' += diag(wt dS) Q's[slab], dv += diag(wt P) dO'[slab].
  const float sel_lo = (t == (g >> 1) && !(g & 1)) ? 1.f : 0.f;
  const float sel_hi = (t == (g >> 1) && (g & 1)) ? 1.f : 0.f;
  for (int r = 0; r < nrk; ++r) {
    const int n = 1 + r;
    const int c = W + r;
    const int lo = ks.lo[c];
    const int need = ks.need[c];
    const float w = MODE == 1 ? ks.w[c] : 0.f;
    const int qfirst = j0 + lo;
    const int xlast = min(qfirst + kBTileT, N - 1) - qfirst;  // last copied slab row
    // the stage's (P, dS) run starts one element early when the query's is odd
    const int par = static_cast<int>(((static_cast<size_t>(bh) * a.pds_stride + c) * N + qfirst) & 1);
    wait_stage(n);
    const unsigned char* qst = slot_of(n);
    const float2* sp = reinterpret_cast<const float2*>(qst + 2 * kQ2) + par;
    // stored (P, dS) of the query i of key k0 + g + 8h for each role; entries of queries
    // before the rung's first attending one or past N are not the dQ grid's: never used
    float2 v[2][2];  // [role][h]
#pragma unroll
    for (int role = 0; role < 2; ++role)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int x = 16 * warp + g + 8 * h + role;  // slab row of query i = qfirst + x
        const int i = qfirst + x;
        const bool ok = (role == 0 || MODE == 1) && k0 + g + 8 * h <= j_last && i < N && i >= need;
        v[role][h] = ok ? sp[x] : make_float2(0.f, 0.f);
      }
#pragma unroll
    for (int role = 0; role < (MODE == 1 ? 2 : 1); ++role) {
      if (role == 1 && !(w > 0.f)) continue;  // uniform: weight 0
      const float wt = MODE == 1 ? (role == 0 ? 1.f - w : w) : 1.f;
      const float xs0 = wt * v[role][0].y, xs1 = wt * v[role][1].y;
      const float xp0 = wt * v[role][0].x, xp1 = wt * v[role][1].x;
      if (!__any_sync(0xffffffffu, xs0 != 0.f || xs1 != 0.f || xp0 != 0.f || xp1 != 0.f)) continue;
      const uint32_t s0 = pack_h2(xs0 * sel_lo, xs0 * sel_hi), s3 = pack_h2(xs1 * sel_lo, xs1 * sel_hi);
      const uint32_t p0 = pack_h2(xp0 * sel_lo, xp0 * sel_hi), p3 = pack_h2(xp1 * sel_lo, xp1 * sel_hi);
      const int x = min(16 * warp + (mi & 1) * 8 + rl + role, xlast);
      const unsigned char* qrow = qst + x * kRowBytes;
      const int sw = swz(qfirst + x);
#pragma unroll
      for (int nd = 0; nd < 8; nd += 2) {
        uint32_t b[4], c4[4];
        ldsm_x4_trans(b, qrow + ((nd + (mi >> 1)) ^ sw) * 16);
        ldsm_x4_trans(c4, qrow + kQ2 + ((nd + (mi >> 1)) ^ sw) * 16);
        mma16816(dK[nd], s0, 0u, 0u, s3, b[0], b[1]);
        mma16816(dK[nd + 1], s0, 0u, 0u, s3, b[2], b[3]);
        mma16816(dV[nd], p0, 0u, 0u, p3, c4[0], c4[1]);
        mma16816(dV[nd + 1], p0, 0u, 0u, p3, c4[2], c4[3]);
      }
    }
    release_stage(n);
  }

  // ---- epilogue: dk = R(j)^T dk' ln2 (dk' accumulated against Q's = q' log2(e)/8), dv
  if (s_err) return;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int j = k0 + g + 8 * h;
    if (j > j_last) continue;
    float2 e[8];
    rope_natural(a.rope_lo, a.rope_hi, j, t, e);
    store_rotated_back(a.dk + base + static_cast<size_t>(j) * kD, dK, h, t, e, kLn2);
    store_plain(a.dv + base + static_cast<size_t>(j) * kD, dV, h, t);
  }
}

// ------------------------------------------------------------------ launch
bool bwd_tc_supported(const LayerTable& t) { return t.W <= kBWinMax; }

namespace {
size_t up256(size_t x) { return (x + 255) / 256 * 256; }
// The scratch of one half of the (b, h) rows: Q's, dO', K', V' rows, Delta, (P, dS) pairs.
size_t half_bytes(long long bh, int N, int W) {
  const size_t rows = static_cast<size_t>(bh) * N;
  return 4 * up256(rows * kRowBytes) + up256(rows * sizeof(float)) +
         up256(rows * (W + kMaxR) * sizeof(float2) + 16);  // + the dK/dV copies' rounding
}
// The rows of the first half: the (b, h) rows split in two when there are two or more.
long long first_half(long long bh) { return bh >= 2 ? bh / 2 : bh; }
}  // namespace

size_t bwd_tc_workspace_bytes(int B, int H, int N, int W) {
  const long long bh = static_cast<long long>(B) * H;
  const size_t tiles = (static_cast<size_t>(N) + kBTileT - 1) / kBTileT * bh;
  const long long bh0 = first_half(bh);
  return up256(tiles * sizeof(float)) + half_bytes(bh0, N, W) + (bh > bh0 ? half_bytes(bh - bh0, N, W) : 0);
}

namespace {
// The three launches of the (b, h) rows [off, off + n) on one stream.  The dQ grid writes its
// CTAs' dalpha partials at partials + n_before; the dK/dV grid sums partials[0 .. n_sum) into
// dalpha when dalpha is not null.  record_after_q, when given, is recorded between the dQ and
// the dK/dV launch (it marks the end of the dQ grid for the other half); wait_before_kv, when
// given, is an event the dK/dV launch waits for first (the other half's dQ grid, whose
// partials it sums too).  kv_k, kv_v: the whole call's K' and V' rows prepared by the layer's
// forward (the half's rows are read at its offset), or null to prepare them here.
cudaError_t launch_half(const LayerTable& t, long long off, long long n, int N, const void* q, const void* k,
                        const void* v, const __half* kv_k, const __half* kv_v, const void* o, const float* lse,
                        const void* dO, void* dq, void* dk, void* dv,
                        float* partials, long long n_before, long long n_sum, float* dalpha, unsigned char* w,
                        const float2* lo_tab, const float2* hi_tab, int* status, unsigned long long wait_ns,
                        cudaEvent_t record_after_q, cudaEvent_t wait_before_kv, cudaStream_t stream) {
  const long long rows = n * N;
  const size_t eo = static_cast<size_t>(off) * N * kD;  // element offset of the half's rows
  auto bf = [&](const void* x) { return static_cast<const __nv_bfloat16*>(x) + eo; };
  auto bfo = [&](void* x) { return static_cast<__nv_bfloat16*>(x) + eo; };
  const size_t arr = up256(static_cast<size_t>(rows) * kRowBytes);
  BtcArgs a;
  a.t = t;
  a.N = N;
  a.tiles = (N + kBTileT - 1) / kBTileT;
  a.bh = static_cast<int>(n);
  a.qs = reinterpret_cast<const __half*>(w);
  a.dos = reinterpret_cast<const __half*>(w + arr);
  a.kp = kv_k != nullptr ? kv_k + eo : reinterpret_cast<const __half*>(w + 2 * arr);
  a.vp = kv_v != nullptr ? kv_v + eo : reinterpret_cast<const __half*>(w + 3 * arr);
  float* delta = reinterpret_cast<float*>(w + 4 * arr);
  a.delta = delta;
  a.pds = reinterpret_cast<float2*>(w + 4 * arr + up256(static_cast<size_t>(rows) * sizeof(float)));
  a.pds_stride = t.W + t.n;  // the kernels keep at most t.n rungs
  a.lse = lse + static_cast<size_t>(off) * N;
  a.dq = bfo(dq);
  a.dk = bfo(dk);
  a.dv = bfo(dv);
  a.rope_lo = lo_tab;
  a.rope_hi = hi_tab;
  a.status = status;
  a.wait_ns = wait_ns;
  const long long blocks = static_cast<long long>(a.tiles) * n;
  const long long prep_blocks = (rows * 4 + kBPrepThreads - 1) / kBPrepThreads;
  if (blocks > 0x7fffffffLL || prep_blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  if (kv_k == nullptr)
    bwd_prep_kernel<true><<<static_cast<unsigned>(prep_blocks), kBPrepThreads, 0, stream>>>(
        bf(q), bf(k), bf(v), bf(o), bf(dO), const_cast<__half*>(a.qs), const_cast<__half*>(a.kp),
        const_cast<__half*>(a.vp), const_cast<__half*>(a.dos), delta, lo_tab, hi_tab, N, rows, kLog2e / 8.0f, status);
  else
    bwd_prep_kernel<false><<<static_cast<unsigned>(prep_blocks), kBPrepThreads, 0, stream>>>(
        bf(q), nullptr, nullptr, bf(o), bf(dO), const_cast<__half*>(a.qs), nullptr, nullptr,
        const_cast<__half*>(a.dos), delta, lo_tab, hi_tab, N, rows, kLog2e / 8.0f, status);
  cudaError_t e;
  // query-owned: dq and the dalpha partials
  a.partials = partials + n_before;
  a.slab_rows = t.mode == 1 ? kBTileT + 8 : kBTileT;
  a.slot_bytes = 2 * a.slab_rows * kRowBytes;
  {
    // a programmatic dependent of the preparation grid: the CTAs' prologue overlaps its tail
    const int smem = kBSlots * a.slot_bytes + kBWarps * 16 * kBWinMax * static_cast<int>(sizeof(float2));
    void (*kern)(BtcArgs) = t.mode == 0 ? bwd_q_kernel<0> : bwd_q_kernel<1>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(kBThreadsT);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, a);
    if (e != cudaSuccess) return e;
  }
  if (record_after_q != nullptr) {
    e = cudaEventRecord(record_after_q, stream);
    if (e != cudaSuccess) return e;
  }
  if (wait_before_kv != nullptr) {
    e = cudaStreamWaitEvent(stream, wait_before_kv, 0);
    if (e != cudaSuccess) return e;
  }
  // key-owned: dk, dv, and dalpha (CTA 0), launched as a programmatic dependent of the dQ
  // grid: its prologue and first copies (of rows the preparation wrote) overlap that grid's
  // tail; it waits for the grid before it reads P, dS and the partials.  The dQ CTAs signal
  // only at their end, after each of their threads waited for the preparation grid, so that
  // grid has completed before this one launches.
  a.slab_rows = kKvQRows;
  a.slot_bytes = 2 * kKvQRows * kRowBytes + kKvPdsBytes;
  a.partials = partials;
  a.n_partials = static_cast<int>(n_sum);
  a.dalpha = dalpha;
  {
    const int smem = kBSlots * a.slot_bytes;
    void (*kern)(BtcArgs) = t.mode == 0 ? bwd_kv_kernel<0> : bwd_kv_kernel<1>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(kBThreadsT);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, a);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_bwd_tc(const LayerTable& t, int B, int H, int N, const void* q, const void* k, const void* v,
                          const void* kv_prepared, const void* o, const float* lse, const void* dO, void* dq,
                          void* dk, void* dv, float* dalpha, void* ws, const float2* lo_tab, const float2* hi_tab,
                          int* status, unsigned long long wait_ns, cudaStream_t stream, const BwdStreams& side) {
  // The (b, h) rows run as two halves, the second on the side stream (forked from and joined
  // back to `stream` with events): each half's grids then fill the SMs that the other half's
  // last, partly filled wave of CTAs leaves idle.  The first half's dK/dV grid leaves dalpha
  // alone; the second half's waits for the first half's dQ grid too and sums every partial
  // of both, in one fixed order.
  const long long bh = static_cast<long long>(B) * H;
  const long long bh0 = first_half(bh);
  const long long tiles = (N + kBTileT - 1) / kBTileT;
  unsigned char* w = static_cast<unsigned char*>(ws);
  float* partials = reinterpret_cast<float*>(w);
  unsigned char* w0 = w + up256(static_cast<size_t>(tiles * bh) * sizeof(float));
  unsigned char* w1 = w0 + half_bytes(bh0, N, t.W);
  // the layer's forward workspace, when handed over: K' rows of the whole call, then its V'
  const __half* kv_k = static_cast<const __half*>(kv_prepared);
  const __half* kv_v = kv_k != nullptr ? kv_k + static_cast<size_t>(bh) * N * kD : nullptr;
  if (bh == bh0)
    return launch_half(t, 0, bh, N, q, k, v, kv_k, kv_v, o, lse, dO, dq, dk, dv, partials, 0, tiles * bh, dalpha, w0, lo_tab,
                       hi_tab, status, wait_ns, nullptr, nullptr, stream);
  cudaError_t e = cudaEventRecord(side.fork, stream);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(side.stream, side.fork, 0);
  if (e == cudaSuccess)
    e = launch_half(t, 0, bh0, N, q, k, v, kv_k, kv_v, o, lse, dO, dq, dk, dv, partials, 0, 0, nullptr, w0, lo_tab, hi_tab,
                    status, wait_ns, side.first_q_done, nullptr, stream);
  if (e == cudaSuccess)
    e = launch_half(t, bh0, bh - bh0, N, q, k, v, kv_k, kv_v, o, lse, dO, dq, dk, dv, partials, tiles * bh0, tiles * bh, dalpha,
                    w1, lo_tab, hi_tab, status, wait_ns, nullptr, side.first_q_done, side.stream);
  if (e == cudaSuccess) e = cudaEventRecord(side.join, side.stream);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, side.join, 0);
  return e;
}

}  // namespace fibattn
