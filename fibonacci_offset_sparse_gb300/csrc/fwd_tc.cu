// bf16 forward kernel (sm_103a): window band on tensor cores, rungs on CUDA cores, every
// K/V row staged into shared memory by the bulk-copy engine.
//
// Same operation as fwd.cu ("Depth-Staggered Fibonacci Spacing for Sparse Attention",
// Methodology > "Attended set", "Scaling", "Implementation"), split by where the work is
// dense:
//   * window band: for a warp's 16 consecutive queries every window key lies in the
//     32-row block [q0-16, q0+16) (W <= 16), so S = Q' K'^T and O = P V run as
//     mma.sync m16n8k16 (f16 operands, f32 accumulation).  Q' and K' are RoPE-rotated at
//     their own positions once per staged row; V is staged as f16.
//   * rungs: a rung is a shifted diagonal (query i reads row i-d); it has no dense block,
//     so those pairs run on the CUDA cores with packed f32x2 arithmetic, applying RoPE in
//     relative form: q'_i . k'_{i-d} = sum_m z_m . k_m with z_m the raw query pair rotated
//     by d theta_m and k_m the raw key pair (rotate-half pairs (m, m+32)).
//   * data movement: a CTA owns 64 consecutive queries of one (b,h) and is warp-specialised:
//     4 consumer warps compute, 1 producer thread streams every row they read through a
//     4-slot shared-memory ring with cp.async.bulk (mbarrier completion): the Q rows, the
//     raw window K and V rows [i0-16, i0+64), then per rung the slab rows [i0-d, i0-d+64)
//     of K and V (two contiguous runs).  The producer runs up to 4 slots ahead and refills a
//     slot as soon as the 4 consumer warps release it; the window rows are converted in
//     place inside their slots, so the ring is nearly all of the CTA's shared memory and 3
//     CTAs fit on an SM.  Every mbarrier wait is bounded in time; a wait that gives up
//     records FIB_ERR_TIMEOUT in the plan's status word, the consumers stop, and the producer
//     lets its copies in flight land before the CTA exits.
// Register layout: lane (g = lane/4, t = lane%4) owns query rows g and g+8 of its warp's 16
// and the dims D_t = [8t, 8t+8) u [32+8t, 32+8t+8) (RoPE partners in the same lane).  The
// MMA k-order is permuted so that a lane's A/B fragments hold exactly D_t, and V's columns
// are permuted so that its O accumulator fragment is D_t too: the CUDA-core rung updates
// and the tensor-core window update share the O registers.
#include <cuda_fp16.h>

#include "common.cuh"

namespace fibattn {

#ifndef FIB_TC_WARPS
#define FIB_TC_WARPS 4
#endif
constexpr int kTcWarps = FIB_TC_WARPS;         // consumer warps (16 queries each)
constexpr int kTcTile = 16 * kTcWarps;         // queries per CTA
constexpr int kConsumers = 32 * kTcWarps;
constexpr int kTcThreads = kConsumers + 32;    // + one producer warp
constexpr int kWinRows = kTcTile + 16;         // window rows [i0-16, i0+64)
constexpr int kTcMaxW = 16;
constexpr int kSlots = 4;                      // ring slots
constexpr int kRungChunk = 2;                  // rungs per online-softmax step
constexpr int kRowBytes = kD * 2;              // one bf16 row

struct TcArgs {
  LayerTable t;
  int N;
  int tiles;
  int bh;  // B * H
  int slab_rows;   // rows of a rung slab region: 64 (mask) or 72 (interp: 65 used)
  int slot_bytes;  // 2 * slab_rows * 128
  int fac_stride;  // rungs per factor table (second table for interp rows lo+1)
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  __nv_bfloat16* o;
  float* lse;
  const float2* rope_lo;
  const float2* rope_hi;
  float qscale;                // log2(e)/sqrt(D)
  int* status;                 // plan status word (FIB_ERR_TIMEOUT on a wait that gave up)
  unsigned long long wait_ns;  // bound of every mbarrier wait
  int skip_first_rung_copy;    // test hook: never arrive on rung 0's stage
  // Rung factors cos / sin of (lo theta_m) and, for interp, of ((lo+1) theta_m), built in
  // binary64 by the plan: table 0 at fac_dev[r*64 + {0..31: cos, 32..63: sin}], table 1 at
  // fac_dev[(kMaxR + r)*64 + ...].  Null: computed here from the RoPE tables.
  const float* fac_dev;
};

// ------------------------------------------------------------------ small PTX helpers
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Wait for the phase of parity `parity` of `bar`, giving up after `limit_ns`.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned long long limit_ns) {
  if (mbar_try(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (true) {
    if (mbar_try(bar, parity)) return true;
    if (global_ns() - t0 > limit_ns) return false;
  }
}
// The producer's wait: like mbar_wait, but it backs off with __nanosleep between polls so
// that a waiting producer leaves the issue slots to the consumer warps of its SM.
__device__ __forceinline__ bool mbar_wait_backoff(uint64_t* bar, uint32_t parity, unsigned long long limit_ns) {
  if (mbar_try(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  unsigned sleep_ns = 32;
  while (true) {
    __nanosleep(sleep_ns);
    if (mbar_try(bar, parity)) return true;
    if (sleep_ns < 512) sleep_ns *= 2;
    if (global_ns() - t0 > limit_ns) return false;
  }
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ float2 bf2(uint32_t w) { return make_float2(bf_lo(w), bf_hi(w)); }

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], const void* smem_row) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_addr(smem_row)));
}

// Read the 16 dims D_t of a 128-byte bf16 row in shared memory as two 16-byte words;
// odd rows read their halves in the opposite order, so the 8 lanes of a phase (two rows
// x four t) hit 8 distinct bank groups.
__device__ __forceinline__ void lds_row_part(const unsigned char* row, int t, bool odd, uint4& lo,
                                             uint4& hi) {
  const uint4* r4 = reinterpret_cast<const uint4*>(row);
  if (odd) {
    hi = r4[t + 4];
    lo = r4[t];
  } else {
    lo = r4[t];
    hi = r4[t + 4];
  }
}

// Score partial of one row: sum over the lane's 4 frequency pairs of z1 k1 + z2 k2 with
// z = q e^{i d theta} (cs = cos, sn = sin of d theta for the lane's frequencies).
__device__ __forceinline__ float rung_dot(const float2 (&q1)[4], const float2 (&q2)[4],
                                          const float2 (&cs)[4], const float2 (&sn)[4],
                                          const float2 (&ns)[4], const uint4& ka, const uint4& kb) {
  const uint32_t xa[4] = {ka.x, ka.y, ka.z, ka.w}, xb[4] = {kb.x, kb.y, kb.z, kb.w};
  float2 acc1 = make_float2(0.f, 0.f), acc2 = make_float2(0.f, 0.f);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 k1 = bf2(xa[j]), k2 = bf2(xb[j]);
    // z = q e^{i d theta}: z1 = c q1 - s q2, z2 = s q1 + c q2
    const float2 z1 = __ffma2_rn(ns[j], q2[j], __fmul2_rn(cs[j], q1[j]));
    const float2 z2 = __ffma2_rn(cs[j], q2[j], __fmul2_rn(sn[j], q1[j]));
    acc1 = __ffma2_rn(z1, k1, acc1);
    acc2 = __ffma2_rn(z2, k2, acc2);
  }
  return (acc1.x + acc2.x) + (acc1.y + acc2.y);
}

__device__ __forceinline__ void load_fac(const float* f, int t, float2 (&cs)[4], float2 (&sn)[4]) {
  const float4* f4 = reinterpret_cast<const float4*>(f);
  const float4 ca = f4[2 * t], cb = f4[2 * t + 1], sa = f4[8 + 2 * t], sb = f4[8 + 2 * t + 1];
  cs[0] = make_float2(ca.x, ca.y);
  cs[1] = make_float2(ca.z, ca.w);
  cs[2] = make_float2(cb.x, cb.y);
  cs[3] = make_float2(cb.z, cb.w);
  sn[0] = make_float2(sa.x, sa.y);
  sn[1] = make_float2(sa.z, sa.w);
  sn[2] = make_float2(sb.x, sb.y);
  sn[3] = make_float2(sb.z, sb.w);
}

__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;\n" ::"n"(kConsumers) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_addr(bar)) : "memory");
}

template <int MODE>
__global__ void __launch_bounds__(kTcThreads, kTcWarps == 4 ? (MODE == 0 ? 3 : 2) : (MODE == 0 ? 5 : 4))
    fwd_tc_kernel(TcArgs a) {
  __shared__ KeySmem ks;
  __shared__ __align__(8) uint64_t full_bar[kSlots];
  __shared__ __align__(8) uint64_t empty_bar[kSlots];
  __shared__ volatile int s_err;
  extern __shared__ __align__(128) unsigned char smem[];
  const int SR = a.slab_rows;
  unsigned char* ring = smem;
  float* fac = reinterpret_cast<float*>(smem + kSlots * a.slot_bytes);  // cos[32], sin[32] per rung

  // Heaviest tiles first: a later tile attends more rungs (d <= i), so launching the tiles
  // from the end of the sequence backwards leaves the light ones for the last partial wave.
  const int bh = blockIdx.x % a.bh;
  const int tile = a.tiles - 1 - static_cast<int>(blockIdx.x / a.bh);
  const int i0 = tile * kTcTile;
  const int N = a.N;
  const int tid = threadIdx.x;
  const size_t base = static_cast<size_t>(bh) * N * kD;
  const __nv_bfloat16* __restrict__ Q = a.q + base;
  const __nv_bfloat16* __restrict__ K = a.k + base;
  const __nv_bfloat16* __restrict__ V = a.v + base;
  const int i_last = min(i0 + kTcTile, N) - 1;  // last real query of the tile

  build_keys(a.t, N, &ks);
  if (tid == 0) {
    s_err = 0;
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kTcWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncthreads();  // the only block-wide barrier: the roles split below
  const int W = a.t.W;
  const int nr = ks.nr;

  const int warp = tid >> 5, lane = tid & 31;
  // Rungs are kept in ascending distance; the tile streams rungs [0, nrt), up to the last one
  // that some row of it attends (a later tile attends more).
  const unsigned attended = __ballot_sync(0xffffffffu, lane < nr && ks.need[W + lane] <= i_last);
  const int nrt = 32 - __clz(static_cast<int>(attended));
  const int n_stages = 3 + nrt;  // Q, window K, window V, then one per streamed rung

  // ===================================================================== producer
  if (warp == kTcWarps) {
    if (lane != 0) return;
    int last_n[kSlots];
#pragma unroll
    for (int s = 0; s < kSlots; ++s) last_n[s] = -1;
    const int w0 = max(i0 - 16, 0);
    for (int n = 0; n < n_stages; ++n) {
      if (s_err) break;
      const int slot = n % kSlots;
      if (!mbar_wait_backoff(&empty_bar[slot], ((n / kSlots) & 1) ^ 1, a.wait_ns)) {
        s_err = 1;
        break;
      }
      unsigned char* dst = ring + slot * a.slot_bytes;
      if (n == 0) {  // Q rows [i0, i_last]; then the plan's rung factor tables, if any
        const uint32_t bytes = static_cast<uint32_t>(i_last - i0 + 1) * kRowBytes;
        const uint32_t fbytes = a.fac_dev != nullptr ? static_cast<uint32_t>(nr) * 256u : 0u;
        mbar_arrive_tx(&full_bar[slot], bytes + (MODE == 1 ? 2 : 1) * fbytes);
        bulk_g2s(dst, Q + static_cast<size_t>(i0) * kD, bytes, &full_bar[slot]);
        if (fbytes) {
          bulk_g2s(dst + kTcTile * kRowBytes, a.fac_dev, fbytes, &full_bar[slot]);
          if (MODE == 1)  // table 1 packed right after table 0
            bulk_g2s(dst + kTcTile * kRowBytes + fbytes, a.fac_dev + kMaxR * 64, fbytes, &full_bar[slot]);
        }
      } else if (n <= 2) {  // raw window rows [max(i0-16, 0), i_last] of K (n = 1) or V (n = 2)
        const uint32_t bytes = static_cast<uint32_t>(i_last + 1 - w0) * kRowBytes;
        mbar_arrive_tx(&full_bar[slot], bytes);
        bulk_g2s(dst + (w0 - (i0 - 16)) * kRowBytes, (n == 1 ? K : V) + static_cast<size_t>(w0) * kD, bytes,
                 &full_bar[slot]);
      } else {  // rung slab: rows [first, first + SR) of K, then of V, where inside [0, N)
        const int r = n - 3;
        if (r == 0 && a.skip_first_rung_copy) continue;  // test hook: this stage never completes
        const int lo = ks.lo[W + r];
        const int first = i0 - lo - (MODE == 1 ? 1 : 0);
        const int r0 = max(first, 0);
        const int r1 = i_last - lo + 1;
        const uint32_t bytes = r1 > r0 ? static_cast<uint32_t>(r1 - r0) * kRowBytes : 0u;
        mbar_arrive_tx(&full_bar[slot], 2 * bytes);
        if (bytes) {
          bulk_g2s(dst + (r0 - first) * kRowBytes, K + static_cast<size_t>(r0) * kD, bytes, &full_bar[slot]);
          bulk_g2s(dst + (SR + r0 - first) * kRowBytes, V + static_cast<size_t>(r0) * kD, bytes,
                   &full_bar[slot]);
        }
      }
      last_n[slot] = n;
    }
    // let every copy issued land before the CTA can exit (a completed phase returns at once)
#pragma unroll
    for (int s = 0; s < kSlots; ++s)
      if (last_n[s] >= 0) mbar_wait(&full_bar[s], (last_n[s] / kSlots) & 1, a.wait_ns);
    if (s_err) atomicExch(a.status, 5 /* FIB_ERR_TIMEOUT */);
    return;
  }

  // ===================================================================== consumers
  const int g = lane >> 2, t = lane & 3;
  const int q0 = i0 + 16 * warp;
  // Every factor load is issued here, before the first stage wait, so that its latency
  // overlaps the first copies.  (1) rung factors e^{i lo theta} into shared memory, from the
  // kernel parameters when the host built them, else from the RoPE tables;
  for (int idx = a.fac_dev != nullptr ? nr * kFreq : tid; idx < nr * kFreq; idx += kConsumers) {
    const int r = idx / kFreq, m = idx % kFreq;
    const int lo = ks.lo[W + r];
    const float2 e = rope_factor(a.rope_lo, a.rope_hi, lo, m);
    fac[r * 64 + m] = e.x;
    fac[r * 64 + 32 + m] = e.y;
    if (MODE == 1) {
      const float2 e1 = rope_factor(a.rope_lo, a.rope_hi, lo + 1, m);
      fac[(a.fac_stride + r) * 64 + m] = e1.x;
      fac[(a.fac_stride + r) * 64 + 32 + m] = e1.y;
    }
  }
  // (2) window rotation factors.  Q' and K' are rotated by their offset from the tile base
  // p0 = i0 - 16 instead of their absolute position: the common e^{i p0 theta} cancels in
  // q'_i . k'_j, and the offsets (< 80) need only the small lo table (plus hi row 1).
  // Rows of this thread: Q rows g, g+8 of the warp (offsets 16 + 16 warp + g (+8)) and the
  // K' conversion tasks (row tid/4 + (consumers/4) k, frequencies 8t..8t+7 since tid % 4 == t).
  constexpr int kKTasks = (kWinRows * 4 + kConsumers - 1) / kConsumers;  // K' tasks per thread
  float2 eq[2][8], ek[kKTasks][8];
  {
    float2 h1[8];  // e^{i 64 theta_m}
    const float4* h4 = reinterpret_cast<const float4*>(a.rope_hi + kFreq + 8 * t);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float4 x = __ldg(h4 + u);
      h1[2 * u] = make_float2(x.x, x.y);
      h1[2 * u + 1] = make_float2(x.z, x.w);
    }
    auto rel = [&](int off, float2 (&e)[8]) {
      const int o = off < kWinRows ? off : 0;
      const float4* l4 = reinterpret_cast<const float4*>(a.rope_lo + (o & 63) * kFreq + 8 * t);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float4 x = __ldg(l4 + u);
        e[2 * u] = make_float2(x.x, x.y);
        e[2 * u + 1] = make_float2(x.z, x.w);
      }
      if (o >= 64) {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float2 b = e[u];
          e[u] = make_float2(h1[u].x * b.x - h1[u].y * b.y, h1[u].x * b.y + h1[u].y * b.x);
        }
      }
    };
#pragma unroll
    for (int h = 0; h < 2; ++h) rel(16 + 16 * warp + g + 8 * h, eq[h]);
#pragma unroll
    for (int k = 0; k < kKTasks; ++k) rel((tid >> 2) + (kConsumers / 4) * k, ek[k]);
  }
  auto wait_stage = [&](int n) {
    if (!s_err && !mbar_wait(&full_bar[n % kSlots], (n / kSlots) & 1, a.wait_ns)) {
      s_err = 1;
      atomicExch(a.status, 5 /* FIB_ERR_TIMEOUT */);
    }
  };
  auto release_stage = [&](int n) {
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_bar[n % kSlots]);
  };

  // ---- stage 0: Q rows -> raw q (for the rungs) and rotated f16 A fragments (window)
  int irow[2], ic[2];
  float2 q1[2][4], q2[2][4];  // raw q * qscale: (dims 8t+2j, 8t+2j+1) and their partners
  uint32_t qa[2][2][4];       // A fragments: [row h][dim half][k-step]
  wait_stage(0);
  {
    const unsigned char* qst = ring;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      irow[h] = q0 + g + 8 * h;
      ic[h] = irow[h] < N ? irow[h] : N - 1;
      const int row = ic[h] - i0;
      float x[16];
      if (!s_err) {
        uint4 wa, wb;
        lds_row_part(qst + row * kRowBytes, t, row & 1, wa, wb);
        const uint32_t xa[4] = {wa.x, wa.y, wa.z, wa.w}, xb[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          x[2 * j] = bf_lo(xa[j]) * a.qscale;
          x[2 * j + 1] = bf_hi(xa[j]) * a.qscale;
          x[8 + 2 * j] = bf_lo(xb[j]) * a.qscale;
          x[8 + 2 * j + 1] = bf_hi(xb[j]) * a.qscale;
        }
      } else {
#pragma unroll
        for (int u = 0; u < 16; ++u) x[u] = 0.f;
      }
      const float2(&e)[8] = eq[h];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        q1[h][j] = make_float2(x[2 * j], x[2 * j + 1]);
        q2[h][j] = make_float2(x[8 + 2 * j], x[8 + 2 * j + 1]);
      }
      float y[16];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        y[u] = x[u] * e[u].x - x[8 + u] * e[u].y;
        y[8 + u] = x[u] * e[u].y + x[8 + u] * e[u].x;
      }
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        qa[h][0][s] = pack_h2(y[2 * s], y[2 * s + 1]);
        qa[h][1][s] = pack_h2(y[8 + 2 * s], y[8 + 2 * s + 1]);
      }
    }
  }
  if (a.fac_dev != nullptr) {  // the factor tables rode in after the Q rows
    const float* src = reinterpret_cast<const float*>(ring + kTcTile * kRowBytes);
    for (int idx = tid; idx < nr * 64; idx += kConsumers) {
      fac[idx] = src[idx];
      if (MODE == 1) fac[a.fac_stride * 64 + idx] = src[nr * 64 + idx];
    }
  }
  release_stage(0);

  // ---- stages 1, 2: window rows, converted in place: K -> K' f16 rotated (chunk c of row
  // r at c ^ 4(r&1)), V -> f16 with columns in pi order (chunk ^ (r&7))
  uint4* Ks = reinterpret_cast<uint4*>(ring + 1 * a.slot_bytes);
  uint4* Vs = reinterpret_cast<uint4*>(ring + 2 * a.slot_bytes);
  wait_stage(1);
#pragma unroll
  for (int k = 0; k < kKTasks; ++k) {
    const int task = tid + k * kConsumers;
    if (task >= kWinRows * 4) break;
    const int row = task >> 2, c = task & 3;
    const int p = i0 - 16 + row;
    uint4 lo4 = make_uint4(0, 0, 0, 0), hi4 = make_uint4(0, 0, 0, 0);
    if (p >= 0 && p < N && !s_err) {
      const uint4 wa = Ks[row * 8 + c], wb = Ks[row * 8 + c + 4];
      const uint32_t xa[4] = {wa.x, wa.y, wa.z, wa.w}, xb[4] = {wb.x, wb.y, wb.z, wb.w};
      const float2(&e)[8] = ek[k];
      uint32_t ya[4], yb[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 k1 = bf2(xa[j]), k2 = bf2(xb[j]);
        const float2 e0 = e[2 * j], e1 = e[2 * j + 1];
        ya[j] = pack_h2(k1.x * e0.x - k2.x * e0.y, k1.y * e1.x - k2.y * e1.y);
        yb[j] = pack_h2(k1.x * e0.y + k2.x * e0.x, k1.y * e1.y + k2.y * e1.x);
      }
      lo4 = make_uint4(ya[0], ya[1], ya[2], ya[3]);
      hi4 = make_uint4(yb[0], yb[1], yb[2], yb[3]);
    }
    const int sw = (row & 1) * 4;  // this thread read exactly chunks c and c+4 of this row
    Ks[row * 8 + (c ^ sw)] = lo4;
    Ks[row * 8 + ((c + 4) ^ sw)] = hi4;
  }
  wait_stage(2);
  {
    constexpr int kVTasks = kWinRows * 8 / kConsumers;  // 5 (4 warps) or 6 (2 warps)
    static_assert(kVTasks * kConsumers == kWinRows * 8, "V conversion tasks must divide evenly");
    uint32_t w[kVTasks][4];
#pragma unroll
    for (int k = 0; k < kVTasks; ++k) {
      const int task = tid + k * kConsumers;
      const int row = task >> 3, c8 = task & 7;
      const int p = i0 - 16 + row;
      w[k][0] = w[k][1] = w[k][2] = w[k][3] = 0u;
      if (p >= 0 && p < N && !s_err) {
        const uint4 raw = Vs[row * 8 + c8];
        const uint32_t rw[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) w[k][j] = pack_h2(bf_lo(rw[j]), bf_hi(rw[j]));
      }
    }
    consumer_sync();  // every raw V chunk is in registers (and K' is complete)
#pragma unroll
    for (int k = 0; k < kVTasks; ++k) {
      const int task = tid + k * kConsumers;
      const int row = task >> 3, c8 = task & 7;
      const int hh = c8 >> 2, tt = c8 & 3;
      uint32_t* vrow = reinterpret_cast<uint32_t*>(Vs + row * 8);
      // dim 32hh + 8tt + u  ->  column 8 (4hh + u/2) + 2tt + (u%2)
#pragma unroll
      for (int j = 0; j < 4; ++j) vrow[((4 * hh + j) ^ (row & 7)) * 4 + tt] = w[k][j];
    }
    consumer_sync();
  }

  // ---- window: S = Q' K'^T over keys [q0-16, q0+16)
  float S[4][4];
#pragma unroll
  for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
    for (int u = 0; u < 4; ++u) S[nt][u] = 0.f;
    const int row = 16 * warp + 8 * nt + g;
    const int sw = (row & 1) * 4;
    const uint4 klo = Ks[row * 8 + (t ^ sw)];
    const uint4 khi = Ks[row * 8 + ((t + 4) ^ sw)];
    const uint32_t kl[4] = {klo.x, klo.y, klo.z, klo.w};
    const uint32_t kh[4] = {khi.x, khi.y, khi.z, khi.w};
#pragma unroll
    for (int s = 0; s < 4; ++s)
      mma16816(S[nt], qa[0][0][s], qa[1][0][s], qa[0][1][s], qa[1][1][s], kl[s], kh[s]);
  }
  release_stage(1);
  // mask: query row rr = g + 8h, key column c = 8nt + 2t + e  ->  distance rr + 16 - c
  float m[2], lw[2], lr[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float mx = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int c = 8 * nt + 2 * t + e;
        const int dist = g + 8 * h + 16 - c;
        const bool ok = dist >= 0 && dist < W && q0 - 16 + c >= 0;
        float& s = S[nt][2 * h + e];
        s = ok ? s : -INFINITY;
        mx = fmaxf(mx, s);
      }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    m[h] = mx;  // finite: distance 0 (the query itself) is always in the block
    float sum = 0.f;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float& s = S[nt][2 * h + e];
        s = exp2f(s - mx);
        sum += s;
      }
    lw[h] = sum;  // lane-partial window sum
    lr[h] = 0.f;  // rung sum (the same in the 4 lanes of a quad)
  }
  // ---- window: O = P V
  float2 O[8][2];  // [n-tile nd][row h] = dims (2nd, 2nd+1) of D_t
#pragma unroll
  for (int nd = 0; nd < 8; ++nd) O[nd][0] = O[nd][1] = make_float2(0.f, 0.f);
  {
    const int mi = lane >> 3, rl = lane & 7;
#pragma unroll
    for (int s2 = 0; s2 < 2; ++s2) {
      const uint32_t pa0 = pack_h2(S[2 * s2][0], S[2 * s2][1]);
      const uint32_t pa1 = pack_h2(S[2 * s2][2], S[2 * s2][3]);
      const uint32_t pa2 = pack_h2(S[2 * s2 + 1][0], S[2 * s2 + 1][1]);
      const uint32_t pa3 = pack_h2(S[2 * s2 + 1][2], S[2 * s2 + 1][3]);
      const int vrow = 16 * warp + 16 * s2 + (mi & 1) * 8 + rl;
#pragma unroll
      for (int nd = 0; nd < 8; nd += 2) {
        const int ch = (nd + (mi >> 1)) ^ (vrow & 7);
        uint32_t b[4];
        ldsm_x4_trans(b, Vs + vrow * 8 + ch);
        float c0[4] = {O[nd][0].x, O[nd][0].y, O[nd][1].x, O[nd][1].y};
        float c1[4] = {O[nd + 1][0].x, O[nd + 1][0].y, O[nd + 1][1].x, O[nd + 1][1].y};
        mma16816(c0, pa0, pa1, pa2, pa3, b[0], b[1]);
        mma16816(c1, pa0, pa1, pa2, pa3, b[2], b[3]);
        O[nd][0] = make_float2(c0[0], c0[1]);
        O[nd][1] = make_float2(c0[2], c0[3]);
        O[nd + 1][0] = make_float2(c1[0], c1[1]);
        O[nd + 1][1] = make_float2(c1[2], c1[3]);
      }
    }
  }
  release_stage(2);

  // ---- rungs: chunks of kRungChunk, online softmax; rung r is stage 3 + r.
  // The slab row of query i is i - i0 (+1 for interp) for every rung.  Inside a warp the
  // arithmetic is branch-free: a row that does not attend the rung reads the slab's first
  // copied row instead (finite data) and gets p = 0; a warp none of whose rows attends the
  // rung skips it as a whole (a uniform branch).
  int srow[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) srow[h] = ic[h] - i0 + (MODE == 1 ? 1 : 0);
  for (int r0 = 0; r0 < nrt; r0 += kRungChunk) {
#pragma unroll
    for (int cc = 0; cc < kRungChunk; ++cc)
      if (r0 + cc < nrt) wait_stage(3 + r0 + cc);
    float sc[2][kRungChunk];
    bool act[kRungChunk];
    int rowu[2][kRungChunk], fcop[kRungChunk];
#pragma unroll
    for (int cc = 0; cc < kRungChunk; ++cc) {
      const int r = r0 + cc < nrt ? r0 + cc : r0;
      const int c = W + r;
      const int lo = ks.lo[c];
      const bool in = (r0 + cc < nrt) && !s_err;
      bool ok[2];
      // first copied row of this slab (slab rows start at global row i0 - lo - interp)
      const int first_copied = max(0, lo - i0 + (MODE == 1 ? 1 : 0));
      fcop[cc] = first_copied;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        ok[h] = in && ic[h] >= ks.need[c];
        rowu[h][cc] = ok[h] ? srow[h] : first_copied;
      }
      act[cc] = __any_sync(0xffffffffu, ok[0] || ok[1]);
      sc[0][cc] = sc[1][cc] = -INFINITY;
      if (act[cc]) {
        const unsigned char* kst = ring + ((3 + r) % kSlots) * a.slot_bytes;
        float2 cs[4], sn[4], ns[4];
        load_fac(fac + r * 64, t, cs, sn);
#pragma unroll
        for (int j = 0; j < 4; ++j) ns[j] = make_float2(-sn[j].x, -sn[j].y);
        float part[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int row = rowu[h][cc];
          uint4 ka, kb;
          lds_row_part(kst + row * kRowBytes, t, row & 1, ka, kb);
          part[h] = rung_dot(q1[h], q2[h], cs, sn, ns, ka, kb);
        }
        if (MODE == 1) {
          const float w = ks.w[c];
          if (w > 0.f) {  // uniform: w belongs to the rung
            float2 c2[4], s2[4], n2[4];
            load_fac(fac + (a.fac_stride + r) * 64, t, c2, s2);
#pragma unroll
            for (int j = 0; j < 4; ++j) n2[j] = make_float2(-s2[j].x, -s2[j].y);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int row = max(rowu[h][cc] - 1, first_copied);
              uint4 ka, kb;
              lds_row_part(kst + row * kRowBytes, t, row & 1, ka, kb);
              part[h] = (1.f - w) * part[h] + w * rung_dot(q1[h], q2[h], c2, s2, n2, ka, kb);
            }
          }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          part[h] += __shfl_xor_sync(0xffffffffu, part[h], 1);
          part[h] += __shfl_xor_sync(0xffffffffu, part[h], 2);
          sc[h][cc] = ok[h] ? part[h] : -INFINITY;
        }
      }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float mc = m[h];
#pragma unroll
      for (int cc = 0; cc < kRungChunk; ++cc) mc = fmaxf(mc, sc[h][cc]);
      const float corr = exp2f(m[h] - mc);
      m[h] = mc;
      lw[h] *= corr;
      lr[h] *= corr;
      const float2 corr2 = make_float2(corr, corr);
#pragma unroll
      for (int nd = 0; nd < 8; ++nd) O[nd][h] = __fmul2_rn(O[nd][h], corr2);
    }
#pragma unroll
    for (int cc = 0; cc < kRungChunk; ++cc) {
      if (!act[cc]) continue;  // uniform
      const int r = r0 + cc;
      const float w = MODE == 1 ? ks.w[W + r] : 0.f;
      const unsigned char* vst = ring + ((3 + r) % kSlots) * a.slot_bytes + SR * kRowBytes;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float p = exp2f(sc[h][cc] - m[h]);  // 0 for a row that does not attend
        lr[h] += p;
        const int row = rowu[h][cc];
        uint4 va, vb;
        lds_row_part(vst + row * kRowBytes, t, row & 1, va, vb);
        const uint32_t xa[4] = {va.x, va.y, va.z, va.w}, xb[4] = {vb.x, vb.y, vb.z, vb.w};
        const float p0 = p * (1.f - w);
        const float2 pp = make_float2(p0, p0);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          O[j][h] = __ffma2_rn(pp, bf2(xa[j]), O[j][h]);
          O[4 + j][h] = __ffma2_rn(pp, bf2(xb[j]), O[4 + j][h]);
        }
        if (MODE == 1 && w > 0.f) {
          const int row1 = max(row - 1, fcop[cc]);
          lds_row_part(vst + row1 * kRowBytes, t, row1 & 1, va, vb);
          const uint32_t ya[4] = {va.x, va.y, va.z, va.w}, yb[4] = {vb.x, vb.y, vb.z, vb.w};
          const float2 pw = make_float2(p * w, p * w);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            O[j][h] = __ffma2_rn(pw, bf2(ya[j]), O[j][h]);
            O[4 + j][h] = __ffma2_rn(pw, bf2(yb[j]), O[4 + j][h]);
          }
        }
      }
    }
#pragma unroll
    for (int cc = 0; cc < kRungChunk; ++cc)
      if (r0 + cc < nrt) release_stage(3 + r0 + cc);
  }

  // ---- epilogue (nothing is written after a wait gave up; the producer reports it)
  if (s_err) return;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float l = lw[h];
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    l += lr[h];
    const int i = irow[h];
    if (i < N) {
      const float inv = 1.f / l;
      float ov[16];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        ov[2 * j] = O[j][h].x * inv;
        ov[2 * j + 1] = O[j][h].y * inv;
        ov[8 + 2 * j] = O[4 + j][h].x * inv;
        ov[8 + 2 * j + 1] = O[4 + j][h].y * inv;
      }
      store_part(a.o + base + static_cast<size_t>(i) * kD, t, ov);
      if (t == 0 && a.lse != nullptr) a.lse[static_cast<size_t>(bh) * N + i] = (m[h] + log2f(l)) * kLn2;
    }
  }
}

bool tc_supported(const LayerTable& t) { return t.W <= kTcMaxW; }

cudaError_t launch_fwd_tc(const LayerTable& t, int B, int H, int N, const void* q, const void* k,
                          const void* v, void* o, float* lse, const float2* lo_tab,
                          const float2* hi_tab, int* status, unsigned long long wait_ns,
                          int skip_first_rung_copy, const float* fac_dev, cudaStream_t stream) {
  TcArgs a;
  // the Q rows (8 KB) and the factor tables (256 B per rung, two tables for interp) share a slot
  const int slot = 2 * (t.mode == 1 ? kTcTile + 8 : kTcTile) * kRowBytes;
  const bool fits = kTcTile * kRowBytes + (t.mode == 1 ? 2 : 1) * t.n * 256 <= slot;
  a.fac_dev = fits ? fac_dev : nullptr;
  a.t = t;
  a.N = N;
  a.tiles = (N + kTcTile - 1) / kTcTile;
  a.bh = B * H;
  a.slab_rows = t.mode == 1 ? kTcTile + 8 : kTcTile;
  a.slot_bytes = 2 * a.slab_rows * kRowBytes;
  a.fac_stride = t.n > 0 ? t.n : 1;  // rungs kept <= t.n (device-alpha interp may keep fewer)
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.k = static_cast<const __nv_bfloat16*>(k);
  a.v = static_cast<const __nv_bfloat16*>(v);
  a.o = static_cast<__nv_bfloat16*>(o);
  a.lse = lse;
  a.rope_lo = lo_tab;
  a.rope_hi = hi_tab;
  a.qscale = kLog2e / 8.0f;
  a.status = status;
  a.wait_ns = wait_ns;
  a.skip_first_rung_copy = skip_first_rung_copy;
  const long long blocks = static_cast<long long>(a.tiles) * B * H;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const size_t smem = static_cast<size_t>(kSlots) * a.slot_bytes +
                      static_cast<size_t>(t.mode == 1 ? 2 : 1) * a.fac_stride * 64 * sizeof(float);
  // The opt-in limit is a property of the kernel function, not of a launch: launches that a
  // CUDA graph captured earlier replay under whatever limit was set last.  So it is always
  // set to the largest size any launch of this kernel can ask for (all kMaxR rungs).
  const int smem_max = kSlots * 2 * (t.mode == 1 ? kTcTile + 8 : kTcTile) * kRowBytes +
                       (t.mode == 1 ? 2 : 1) * kMaxR * 64 * static_cast<int>(sizeof(float));
  cudaError_t e;
  if (t.mode == 0) {
    e = cudaFuncSetAttribute(fwd_tc_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max);
    if (e != cudaSuccess) return e;
    fwd_tc_kernel<0><<<static_cast<unsigned>(blocks), kTcThreads, smem, stream>>>(a);
  } else {
    e = cudaFuncSetAttribute(fwd_tc_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max);
    if (e != cudaSuccess) return e;
    fwd_tc_kernel<1><<<static_cast<unsigned>(blocks), kTcThreads, smem, stream>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace fibattn
