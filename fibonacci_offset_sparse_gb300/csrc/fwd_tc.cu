// bf16 forward (sm_103a): RoPE'd keys and f16 values prepared once per layer, then the
// window band and every rung on tensor cores, every row staged in shared memory by the
// bulk-copy engine.
//
// Same operation as fwd.cu ("Depth-Staggered Fibonacci Spacing for Sparse Attention",
// Methodology > "Attended set", "Scaling", "Implementation"), in two launches:
//   * prep_kv_kernel streams K and V once: K' = RoPE(K) at each row's own position and
//     V' = V, both rounded to f16, rows stored chunk-swizzled (below).  A key row is read
//     by its window band and by one query per rung, so rotating and converting it once
//     here replaces a rotation and a conversion per (query, rung) in the attention kernel.
//   * fwd_tc_kernel: a CTA owns 64 consecutive queries of one (b,h): 4 compute warps of 16
//     queries plus one producer thread that streams the rows they read through a 3-slot
//     shared-memory ring with cp.async.bulk (mbarrier completion): the Q rows, the "near
//     block" rows [i0-64, i0+64) of K' and of V', then per remaining rung the slab rows
//     [i0-d, i0-d+64) of K' and V'.  The near block holds the window band and the slab of
//     every rung with d <= 64 (up to 5, interp 4, of them), so those rungs need no copy of
//     their own and are computed together with the window.  The producer refills a slot
//     once the 4 compute warps release it; with one streamed rung per online-softmax step
//     the next two stages are in flight while a rung is being computed.  The producer
//     issues the Q copy before the block barrier.  3 slots of 16 KB and 96 registers a
//     thread let 4 CTAs share an SM.  Every mbarrier wait is bounded in time; a wait that
//     gives up records FIB_ERR_TIMEOUT in the plan's status word, the warps stop, and the
//     producer lets its copies in flight land before the CTA exits.
//   * window band: for a warp's 16 queries every window key lies in the 32-row block
//     [q0-16, q0+16) (W <= 16): S = Q' K'^T and O = P V' as mma.sync m16n8k16 (f16
//     operands, f32 accumulation), Q' rotated at its own position and scaled by
//     log2(e)/sqrt(D) so that scores are in log2 units.
//   * rungs: query i reads slab row i - i0 (+1 for interp), so a rung is the diagonal of a
//     16x16 block: S_r = diag(Q' K'_slab^T) takes 8 MMAs (2 key n-tiles x 4 k-steps) whose
//     diagonal entries sit in one "holder" lane per row, and O += diag(P) V'_slab takes 8
//     more (A = diag(P) in f16).  Interp reads a 24-row band instead, whose two adjacent
//     diagonals are the row and its partner (12 MMAs).  The tensor pipe does 16x the needed
//     products, but a warp-rung costs those MMAs and about a hundred other instructions
//     where the CUDA cores would need ~250 (RoPE of the query, bf16 unpacking, dot
//     products, axpys).
// Register layout: lane (g = lane/4, t = lane%4) owns query rows g and g+8 of its warp.  For
// the score MMAs the k-order is permuted so that a lane's A fragments hold the dims
// D_t = [8t, 8t+8) u [32+8t, 32+8t+8) (RoPE partners in the same lane) and its B fragments
// the same dims of one key row (two 16-byte chunks).  O is in the natural accumulator
// layout: n-tile nt of row g holds dims 8nt+2t, 8nt+2t+1.
// Shared/global row layout of K' and V': the 16-byte chunk c (dims 8c..8c+7) of the row of
// sequence position p sits at chunk c ^ swz(p), swz(p) = 4(p&1) | ((p>>1)&3).  Eight
// consecutive rows put a given chunk in 8 distinct bank groups (ldmatrix of V'), and two
// consecutive rows put chunks {0..3} in opposite halves (the 16-byte loads of K').
#include <cuda_fp16.h>

#include "tc_common.cuh"

namespace fibattn {

#ifndef FIB_TC_WARPS
#define FIB_TC_WARPS 4
#endif
constexpr int kTcWarps = FIB_TC_WARPS;         // compute warps (16 queries each)
constexpr int kTcTile = 16 * kTcWarps;         // queries per CTA
constexpr int kConsumers = 32 * kTcWarps;
constexpr int kTcThreads = kConsumers + 32;    // + one producer warp
constexpr int kTcMaxW = 16;
#ifndef FIB_TC_SLOTS
#define FIB_TC_SLOTS 3
#endif
#ifndef FIB_TC_MIN_CTAS
#define FIB_TC_MIN_CTAS 4
#endif
#ifndef FIB_TC_MIN_CTAS_INTERP
#define FIB_TC_MIN_CTAS_INTERP 4
#endif
constexpr int kSlots = FIB_TC_SLOTS;           // ring slots
constexpr int kNear = 64;     // the near block holds K'/V' rows [i0 - kNear, i0 + kTcTile)
// Q, the near K' and the near V' are in flight at once, and a near block fills one slot
// (a slot holds 2 * kTcTile rows, interp 2 * (kTcTile + 1)).
static_assert(kSlots >= 3, "the first three stages need their own slots");
static_assert(kNear <= kTcTile, "the near block must fit a ring slot");
static_assert(kTcWarps >= 1 && kTcWarps <= 8, "compute warps per CTA");

struct TcArgs {
  LayerTable t;
  int N;
  int tiles;
  int bh;          // B * H
  int slab_rows;   // rows of a rung slab region: 64 (mask) or 65 (interp)
  int slot_bytes;  // 2 * slab_rows * 128
  const __nv_bfloat16* q;
  const __half* kp;  // K' rows (prep_kv_kernel)
  const __half* vp;  // V' rows
  __nv_bfloat16* o;
  float* lse;
  const float2* rope_lo;
  const float2* rope_hi;
  float qscale;                // log2(e)/sqrt(D)
  int* status;                 // plan status word: timeout, rung-table check, float16 range
  unsigned long long wait_ns;  // bound of every mbarrier wait
  int skip_first_rung_copy;    // test hook: never arrive on rung 0's stage
};

// ------------------------------------------------------------------ K', V' preparation
// A warp prepares 8 * kPrepIters consecutive rows: lane (j8 = lane/4, u = lane%4) handles rows
// base + 8i + j8 (i < kPrepIters) and the frequencies m = 8u .. 8u+7, i.e. chunks u (dims
// 8u..) and u+4 (their rotate-half partners 32+8u..) of the K row, and the same two chunks
// of V.  Every load of the warp is issued first.  The RoPE factors e^{i p theta_m} of the
// first row come from the factored tables; each later row of the lane sits 8 positions
// further, so its factors are the previous ones times e^{i 8 theta_m} (one complex product
// each, relative error ~1e-7 a step, far below the float16 rounding of K'), unless a new
// sequence began in between (position < 8), where the tables are read again.  This keeps
// the table reads at a few bytes a row instead of 128.
constexpr int kPrepIters = 3;
constexpr int kPrepThreads = 128;
constexpr int kPrepRowsPerBlock = kPrepThreads / 4 * kPrepIters;  // 96

__global__ void __launch_bounds__(kPrepThreads) prep_kv_kernel(const __nv_bfloat16* __restrict__ k,
                                                               const __nv_bfloat16* __restrict__ v,
                                                               __half* __restrict__ kp, __half* __restrict__ vp,
                                                               const float2* __restrict__ lo_tab,
                                                               const float2* __restrict__ hi_tab, int N,
                                                               long long rows, int* __restrict__ status) {
  // The dependent attention grid may launch at once: its CTAs take the SMs as this grid
  // drains and load and rotate their Q rows meanwhile; each waits for the whole of this grid
  // (griddepcontrol.wait) before it reads K'/V'.
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int u = lane & 3, j8 = lane >> 2;
  const long long base = static_cast<long long>(blockIdx.x) * kPrepRowsPerBlock + (threadIdx.x >> 5) * (8 * kPrepIters) + j8;
  uint4 ka[kPrepIters], kb[kPrepIters], va[kPrepIters], vb[kPrepIters];
#pragma unroll
  for (int i = 0; i < kPrepIters; ++i) {
    const long long row = base + 8 * i;
    if (row < rows) {
      const uint4* k4 = reinterpret_cast<const uint4*>(k + row * kD);
      const uint4* v4 = reinterpret_cast<const uint4*>(v + row * kD);
      ka[i] = __ldcs(k4 + u);
      kb[i] = __ldcs(k4 + u + 4);
      va[i] = __ldcs(v4 + u);
      vb[i] = __ldcs(v4 + u + 4);
    }
  }
  float2 step[8];  // e^{i 8 theta_m}: row 8 of the low table
  {
    const float4* s4 = reinterpret_cast<const float4*>(lo_tab + 8 * kFreq + 8 * u);
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float4 x = __ldg(s4 + w);
      step[2 * w] = make_float2(x.x, x.y);
      step[2 * w + 1] = make_float2(x.z, x.w);
    }
  }
  float2 e[8];
  uint32_t bad = 0;
#pragma unroll
  for (int i = 0; i < kPrepIters; ++i) {
    const long long row = base + 8 * i;
    if (row >= rows) break;
    const int p = static_cast<int>(row % N);
    if (i == 0 || p < 8) {
      rope_row(lo_tab, hi_tab, p, u, e);
    } else {
#pragma unroll
      for (int w = 0; w < 8; ++w)
        e[w] = make_float2(e[w].x * step[w].x - e[w].y * step[w].y, e[w].x * step[w].y + e[w].y * step[w].x);
    }
    const uint32_t xa[4] = {ka[i].x, ka[i].y, ka[i].z, ka[i].w}, xb[4] = {kb[i].x, kb[i].y, kb[i].z, kb[i].w};
    uint32_t ya[4], yb[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      // (k_m, k_{m+32}) -> (k_m cos - k_{m+32} sin, k_m sin + k_{m+32} cos), m = 8u + 2c (+1)
      const float k1x = bf_lo(xa[c]), k1y = bf_hi(xa[c]), k2x = bf_lo(xb[c]), k2y = bf_hi(xb[c]);
      const float2 e0 = e[2 * c], e1 = e[2 * c + 1];
      ya[c] = pack_h2(k1x * e0.x - k2x * e0.y, k1y * e1.x - k2y * e1.y);
      yb[c] = pack_h2(k1x * e0.y + k2x * e0.x, k1y * e1.y + k2y * e1.x);
    }
    const uint32_t wa[4] = {va[i].x, va[i].y, va[i].z, va[i].w}, wb[4] = {vb[i].x, vb[i].y, vb[i].z, vb[i].w};
    uint32_t za[4], zb[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      za[c] = pack_h2(bf_lo(wa[c]), bf_hi(wa[c]));
      zb[c] = pack_h2(bf_lo(wb[c]), bf_hi(wb[c]));
    }
    // A rotated key or a value beyond the float16 range (|x| > 65504) cannot be represented
    // in the prepared rows: record it (the outputs of this call are then unspecified).
#pragma unroll
    for (int c = 0; c < 4; ++c) bad |= h2_nonfinite(ya[c]) | h2_nonfinite(yb[c]) | h2_nonfinite(za[c]) | h2_nonfinite(zb[c]);
    const int sw = swz(p);
    uint4* ko = reinterpret_cast<uint4*>(kp + row * kD);
    uint4* vo = reinterpret_cast<uint4*>(vp + row * kD);
    ko[u ^ sw] = make_uint4(ya[0], ya[1], ya[2], ya[3]);
    ko[(u + 4) ^ sw] = make_uint4(yb[0], yb[1], yb[2], yb[3]);
    vo[u ^ sw] = make_uint4(za[0], za[1], za[2], za[3]);
    vo[(u + 4) ^ sw] = make_uint4(zb[0], zb[1], zb[2], zb[3]);
  }
  if (bad) atomicExch(status, kStatusRange);
}

// ------------------------------------------------------------------ attention kernel
template <int MODE>
__global__ void __launch_bounds__(kTcThreads, MODE == 0 ? FIB_TC_MIN_CTAS : FIB_TC_MIN_CTAS_INTERP) fwd_tc_kernel(const __grid_constant__ TcArgs a) {
  __shared__ KeySmem ks;
  __shared__ __align__(8) uint64_t full_bar[kSlots];
  __shared__ __align__(8) uint64_t empty_bar[kSlots];
  __shared__ volatile int s_err;
  extern __shared__ __align__(128) unsigned char smem[];
  const int SR = a.slab_rows;
  unsigned char* ring = smem;
  constexpr int kI = MODE == 1 ? 1 : 0;  // interp: the slab starts one row earlier

  // Heaviest tiles first: a later tile attends more rungs (d <= i), so launching the tiles
  // from the end of the sequence backwards leaves the light ones for the last partial wave.
  const int bh = blockIdx.x % a.bh;
  const int tile = a.tiles - 1 - static_cast<int>(blockIdx.x / a.bh);
  const int i0 = tile * kTcTile;
  const int N = a.N;
  const int tid = threadIdx.x;
  const size_t base = static_cast<size_t>(bh) * N * kD;
  const __nv_bfloat16* __restrict__ Q = a.q + base;
  const __half* __restrict__ Kp = a.kp + base;
  const __half* __restrict__ Vp = a.vp + base;
  const int i_last = min(i0 + kTcTile, N) - 1;  // last real query of the tile
  const int w0 = max(i0 - 16, 0);                // first copied window row

  // The producer lane initialises the mbarriers and issues stage 0 (the Q rows, an input of
  // this grid) before the block barrier, so that the copy overlaps the prologue.
  if (tid == kConsumers) {
    s_err = 0;
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kTcWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    const uint32_t bytes = static_cast<uint32_t>(i_last - i0 + 1) * kRowBytes;
    mbar_arrive_tx(&full_bar[0], bytes);
    bulk_g2s(ring, Q + static_cast<size_t>(i0) * kD, bytes, &full_bar[0]);
  }
  // Rung table: the mask path reads it from the launch parameters (its distances are known
  // on the host), so no thread builds it before the block barrier; the interp path builds it
  // in shared memory (from the device alpha when the caller passes one).  (Reading the
  // host-known interp table from the parameters too measured slower.)
  constexpr bool host_keys = MODE == 0;
  if (!host_keys) build_keys(a.t, N, &ks);
  __syncthreads();  // the only block-wide barrier: the roles split below
  const int W = a.t.W;
  const int nr = host_keys ? a.t.n : ks.nr;
  auto rung_lo = [&](int r) { return host_keys ? a.t.lo[r] : ks.lo[W + r]; };
  auto rung_w = [&](int r) { return MODE == 1 ? (host_keys ? a.t.w[r] : ks.w[W + r]) : 0.f; };
  auto rung_need = [&](int r) { return host_keys ? rung_lo(r) + (rung_w(r) > 0.f ? 1 : 0) : ks.need[W + r]; };

  const int warp = tid >> 5, lane = tid & 31;
  // Device-side check of the rung table before any rung row is copied: every kept rung
  // must lie beyond the window and inside the sequence (mask: W <= d <= N-1, strictly
  // ascending; interp: W-1 < d = lo + w <= N-1, lo non-decreasing).  A table that breaks
  // this records FIB_ERR_DEVICE_ASSERT and the CTA returns without writing output (the
  // producer first lets its Q copy land).
  {
    bool bad = false;
    if (lane < nr) {
      const int lo = rung_lo(lane);
      const float w = rung_w(lane);
      const int prev = lane > 0 ? rung_lo(lane - 1) : -1;
      if (MODE == 0) bad = lo < W || lo > N - 1 || lo <= prev;
      else bad = lo < W - 1 || !(w >= 0.f && w < 1.f) || (lo == W - 1 && w == 0.f) || rung_need(lane) > N - 1 || lo < prev;
    }
    if (__any_sync(0xffffffffu, bad)) {  // the same vote in every warp
      if (tid == kConsumers) {
        mbar_wait(&full_bar[0], 0, a.wait_ns);
        atomicExch(a.status, kStatusDeviceAssert);
      }
      return;
    }
  }
  // Rungs are kept in ascending distance; the tile streams rungs [0, nrt), up to the last one
  // that some row of it attends (a later tile attends more).
  const unsigned attended = __ballot_sync(0xffffffffu, lane < nr && rung_need(lane) <= i_last);
  const int nrt = 32 - __clz(static_cast<int>(attended));
  // Rungs whose slab lies inside the near block (ascending distances: a prefix) are served
  // from it, up to kMaxNear of them (per path, set by measurement: each near rung holds its
  // scores in registers until the window's P.V, which costs more on the interpolated path,
  // where the rung step already holds more); every other rung streams its own slab.
  constexpr int kMaxNear = MODE == 0 ? 4 : 1;
  const int n_near = min(kMaxNear, __popc(__ballot_sync(0xffffffffu, lane < nrt && rung_lo(lane) + kI <= kNear)));
  const int n_stages = 3 + nrt - n_near;  // Q, near K', near V', then one per streamed rung

  // ===================================================================== producer
  if (warp == kTcWarps) {
    if (lane != 0) return;
    int last_n[kSlots];
#pragma unroll
    for (int s = 0; s < kSlots; ++s) last_n[s] = -1;
    last_n[0] = 0;  // stage 0 was issued before the block barrier
    for (int n = 1; n < n_stages; ++n) {
      if (s_err) break;
      const int slot = n % kSlots;
      if (!mbar_wait_backoff(&empty_bar[slot], ((n / kSlots) & 1) ^ 1, a.wait_ns)) {
        s_err = 1;
        break;
      }
      unsigned char* dst = ring + slot * a.slot_bytes;
      if (n <= 2) {  // near-block rows [nb0, i_last] of K' (n = 1) or V' (n = 2)
        // K'/V' come from the preparation grid launched just before this one (programmatic
        // dependent launch): wait for it, and its writes, before the first copy of them
        if (n == 1) asm volatile("griddepcontrol.wait;\n" ::: "memory");
        if (n == 2 && a.skip_first_rung_copy) continue;  // test hook: this stage never completes
        const int nb0 = max(i0 - kNear, 0);
        const uint32_t bytes = static_cast<uint32_t>(i_last + 1 - nb0) * kRowBytes;
        mbar_arrive_tx(&full_bar[slot], bytes);
        bulk_g2s(dst + (nb0 - (i0 - kNear)) * kRowBytes, (n == 1 ? Kp : Vp) + static_cast<size_t>(nb0) * kD,
                 bytes, &full_bar[slot]);
      } else {  // rung slab: rows [first, first + SR) of K', then of V', where inside [0, N)
        const int r = n_near + n - 3;
        const int lo = rung_lo(r);
        const int first = i0 - lo - kI;
        const int r0 = max(first, 0);
        const int r1 = i_last - lo + 1;
        const uint32_t bytes = r1 > r0 ? static_cast<uint32_t>(r1 - r0) * kRowBytes : 0u;
        mbar_arrive_tx(&full_bar[slot], 2 * bytes);
        if (bytes) {
          bulk_g2s(dst + (r0 - first) * kRowBytes, Kp + static_cast<size_t>(r0) * kD, bytes, &full_bar[slot]);
          bulk_g2s(dst + (SR + r0 - first) * kRowBytes, Vp + static_cast<size_t>(r0) * kD, bytes,
                   &full_bar[slot]);
        }
      }
      last_n[slot] = n;
    }
    // let every copy issued land before the CTA can exit (a completed phase returns at once)
#pragma unroll
    for (int s = 0; s < kSlots; ++s)
      if (last_n[s] >= 0) mbar_wait(&full_bar[s], (last_n[s] / kSlots) & 1, a.wait_ns);
    if (s_err) atomicExch(a.status, kStatusTimeout);
    return;
  }

  // ===================================================================== compute warps
  const int g = lane >> 2, t = lane & 3;
  const int q0 = i0 + 16 * warp;
  int irow[2], ic[2];
  float2 eq[2][8];  // e^{i p theta_m} of the lane's two query rows (loads overlap the copies)
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    irow[h] = q0 + g + 8 * h;
    ic[h] = irow[h] < N ? irow[h] : N - 1;
    rope_row(a.rope_lo, a.rope_hi, ic[h], t, eq[h]);
  }
  auto wait_stage = [&](int n) {
    if (!s_err && !mbar_wait(&full_bar[n % kSlots], (n / kSlots) & 1, a.wait_ns)) {
      s_err = 1;
      atomicExch(a.status, kStatusTimeout);
    }
  };
  auto release_stage = [&](int n) {
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_bar[n % kSlots]);
  };

  // ---- stage 0: Q rows -> Q' = RoPE(q) * log2(e)/sqrt(D) as f16 A fragments
  uint32_t qa[2][2][4];  // [row h][dim half][k-step]
  wait_stage(0);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int row = ic[h] - i0;
    float x[16];
    if (!s_err) {
      uint4 wa, wb;
      lds_row_part(ring + row * kRowBytes, t, row & 1, wa, wb);
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
  {
    uint32_t bad = 0;  // a scaled, rotated query beyond the float16 range
#pragma unroll
    for (int s = 0; s < 4; ++s) bad |= h2_nonfinite(qa[0][0][s]) | h2_nonfinite(qa[0][1][s]) | h2_nonfinite(qa[1][0][s]) | h2_nonfinite(qa[1][1][s]);
    if (bad) atomicExch(a.status, kStatusRange);
  }
  release_stage(0);

  // ---- near block: K'/V' rows [i0 - kNear, i0 + 64) (index = position - (i0 - kNear); rows
  // outside [max(i0 - kNear, 0), i_last] hold stale data and are masked or clamped below).
  // It serves the window band and the first n_near rungs in the same two stages.
  const uint4* Ks = reinterpret_cast<const uint4*>(ring + 1 * a.slot_bytes);
  const unsigned char* Vs = ring + 2 * a.slot_bytes;
  constexpr int kWin = kNear - 16;  // index of the window block's first row (position i0 - 16)
  const int mi = lane >> 3, rl = lane & 7;
  // Rung layout.  Slab row of query i: i - i0 + kI (global row i - lo; interp: its partner
  // i - lo - 1 is the row before).  Rows that a query does not attend are read from the slab's
  // first copied row (finite data) and get p = 0; a warp none of whose rows attends a rung
  // skips it as a whole (a uniform branch).
  // Diagonal: query g's score sits in lane (g, g>>1) of key n-tile 0, element g&1; query
  // g+8's in the same lane of n-tile 1, element 2 + (g&1).  Only that "holder" lane keeps a
  // rung's score (the other three take -inf, so p = 0 there), and it holds the nonzero
  // entries of A = diag(P) as well: row g in a0, row g+8 in a3, each in half g&1.  So the
  // rung part of the softmax sum accumulates in the holder lane and joins the quad sum at
  // the end, and the reference m, the same in the four lanes of a quad, moves only through
  // a rescale that broadcasts the holder's value.
  const bool holder = t == (g >> 1);
  const int src_lane = 4 * g + (g >> 1);
  const int lcop = i_last - i0 + kI;  // last copied slab row of every rung
  int srow[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) srow[h] = ic[h] - i0 + kI;
  const int vbase = 16 * warp + (mi & 1) * 8 + rl + kI;  // ldmatrix row of this lane, before clamping
  // A rung's metadata does not depend on the staged rows (it is computed for the next
  // streamed rung while the current one's products are in flight).
  int first = 0, fcop = 0, rowu[2] = {0, 0};
  bool ok[2] = {false, false}, act = false;
  float wr = 0.f;
  auto meta = [&](int r) {
    const int lo = rung_lo(r);
    const int need = rung_need(r);
    first = i0 - lo - kI;          // global row of slab row 0
    fcop = max(0, lo - i0 + kI);   // first copied slab row (<= lcop: the tile attends r)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      ok[h] = ic[h] >= need;
      rowu[h] = ok[h] ? srow[h] : fcop;
    }
    act = __any_sync(0xffffffffu, ok[0] || ok[1]);
    if (MODE == 1) wr = rung_w(r);
  };
  // The rung's diagonal scores (holder lanes; -inf elsewhere) from the K' rows at kst (slab
  // row 0), for the current metadata.
  auto rung_scores = [&](const uint4* kst, float (&sc)[2]) {
    float d[2];
    if (MODE == 0) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t kl[4], kh[4];
        lds_kfrag(kst + rowu[h] * 8, t, first + rowu[h], kl, kh);
        // two independent halves of the k-sum: MMA dependency chains of two, not four
        float ca[4] = {0.f, 0.f, 0.f, 0.f}, cb[4] = {0.f, 0.f, 0.f, 0.f};
        mma16816(ca, qa[0][0][0], qa[1][0][0], qa[0][1][0], qa[1][1][0], kl[0], kh[0]);
        mma16816(cb, qa[0][0][2], qa[1][0][2], qa[0][1][2], qa[1][1][2], kl[2], kh[2]);
        mma16816(ca, qa[0][0][1], qa[1][0][1], qa[0][1][1], qa[1][1][1], kl[1], kh[1]);
        mma16816(cb, qa[0][0][3], qa[1][0][3], qa[0][1][3], qa[1][1][3], kl[3], kh[3]);
        d[h] = (g & 1) ? ca[2 * h + 1] + cb[2 * h + 1] : ca[2 * h] + cb[2 * h];
      }
    } else {
      // Interp, banded: column g of key n-tile nt holds slab row R0 + 8nt + g, R0 = 16 warp +
      // kI - 8, so that the row of query g + 8h is column g of n-tile h + 1 and its partner
      // (the row before) column (g + 7) & 7 of n-tile h + (g + 7) / 8: 12 MMAs give both
      // diagonals.  Rows outside [fcop, lcop] are read from the nearest copied row; no
      // attending query picks those columns.
      const int R0 = 16 * warp + kI - 8;
      float C[3][4];
#pragma unroll
      for (int nt = 0; nt < 3; ++nt) {
        const int row = min(max(R0 + 8 * nt + g, fcop), lcop);
        uint32_t kl[4], kh[4];
        lds_kfrag(kst + row * 8, t, first + row, kl, kh);
        C[nt][0] = C[nt][1] = C[nt][2] = C[nt][3] = 0.f;
#pragma unroll
        for (int s = 0; s < 4; ++s)
          mma16816(C[nt], qa[0][0][s], qa[1][0][s], qa[0][1][s], qa[1][1][s], kl[s], kh[s]);
      }
      d[0] = (g & 1) ? C[1][1] : C[1][0];  // the holder lane's diagonal entries
      d[1] = (g & 1) ? C[2][3] : C[2][2];
      if (wr > 0.f) {  // uniform: w belongs to the rung
        // the partner entry sits in lane (g, pc >> 1) of the quad: fetch it from there
        const int pc = (g + 7) & 7;
        const bool lo_tile = g == 0;  // column 7 of the n-tile before
        float v0 = lo_tile ? ((pc & 1) ? C[0][1] : C[0][0]) : ((pc & 1) ? C[1][1] : C[1][0]);
        float v1 = lo_tile ? ((pc & 1) ? C[1][3] : C[1][2]) : ((pc & 1) ? C[2][3] : C[2][2]);
        v0 = __shfl_sync(0xffffffffu, v0, 4 * g + (pc >> 1));
        v1 = __shfl_sync(0xffffffffu, v1, 4 * g + (pc >> 1));
        d[0] = (1.f - wr) * d[0] + wr * v0;
        d[1] = (1.f - wr) * d[1] + wr * v1;
      }
    }
    sc[0] = holder && ok[0] ? d[0] : -INFINITY;
    sc[1] = holder && ok[1] ? d[1] : -INFINITY;
  };
  // O += diag(p (1-w)) V'[slab rows of the 16 queries]; interp: + diag(p w) V'[rows - 1], the
  // V' rows at vst (slab row 0), for the current metadata.
  auto rung_pv = [&](const unsigned char* vst, const float (&p)[2], float (&O)[8][4]) {
#pragma unroll
    for (int part = 0; part < (MODE == 1 ? 2 : 1); ++part) {
      if (part == 1 && !(wr > 0.f)) break;  // uniform
      const float f = MODE == 1 ? (part == 0 ? 1.f - wr : wr) : 1.f;
      const float x0 = p[0] * f, x1 = p[1] * f;
      const uint32_t a0 = (g & 1) ? pack_h2(0.f, x0) : pack_h2(x0, 0.f);
      const uint32_t a3 = (g & 1) ? pack_h2(0.f, x1) : pack_h2(x1, 0.f);
      const int vr = min(max(vbase - part, fcop), lcop);
      const unsigned char* vrow = vst + vr * kRowBytes;
      const int sw = swz(first + vr);
#pragma unroll
      for (int nd = 0; nd < 8; nd += 2) {
        uint32_t b[4];
        ldsm_x4_trans(b, vrow + ((nd + (mi >> 1)) ^ sw) * 16);
        mma16816(O[nd], a0, 0u, 0u, a3, b[0], b[1]);
        mma16816(O[nd + 1], a0, 0u, 0u, a3, b[2], b[3]);
      }
    }
  };

  // ---- window band S = Q' K'^T over keys [q0-16, q0+16), and the near rungs' scores
  float S[4][4];
  float pn[kMaxNear][2];  // near rungs: scores, then probabilities
  wait_stage(1);
#pragma unroll
  for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
    for (int u = 0; u < 4; ++u) S[nt][u] = 0.f;
    const int row = 16 * warp + 8 * nt + g;
    uint32_t kl[4], kh[4];
    lds_kfrag(Ks + (kWin + row) * 8, t, i0 - 16 + row, kl, kh);
#pragma unroll
    for (int s = 0; s < 4; ++s)
      mma16816(S[nt], qa[0][0][s], qa[1][0][s], qa[0][1][s], qa[1][1][s], kl[s], kh[s]);
  }
#pragma unroll
  for (int j = 0; j < kMaxNear; ++j) {
    pn[j][0] = pn[j][1] = -INFINITY;
    if (j < n_near) {  // uniform
      meta(j);
      if (act) rung_scores(Ks + (first - (i0 - kNear)) * 8, pn[j]);  // uniform
    }
  }
  release_stage(1);
  // mask: query row rr = g + 8h, key column c = 8nt + 2t + e  ->  distance rr + 16 - c.  The
  // reference m is the exact maximum over the window band and the near rungs.
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
#pragma unroll
    for (int j = 0; j < kMaxNear; ++j) mx = fmaxf(mx, pn[j][h]);
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
    float rs = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxNear; ++j) {
      pn[j][h] = exp2f(pn[j][h] - mx);  // 0 outside the holder lanes and for absent rungs
      rs += pn[j][h];
    }
    lr[h] = rs;  // rung sum (nonzero in the holder lane of the quad only)
  }
  // ---- O = P V' over the window band, then the near rungs.  Window: ldmatrix lane l supplies
  // row (l&7) of matrix l>>3: keys 16 s2 + 8 ((l>>3)&1) + (l&7), chunk nd + (l>>4).  Rows
  // outside [w0, i_last] (P = 0 there) are read from the nearest copied row, so that no stale
  // value can turn 0 * x into NaN.
  float O[8][4];  // [n-tile nt]: (row g: dims 8nt+2t, +1), (row g+8: the same dims)
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) O[nt][0] = O[nt][1] = O[nt][2] = O[nt][3] = 0.f;
  wait_stage(2);
#pragma unroll
  for (int s2 = 0; s2 < 2; ++s2) {
    const uint32_t pa0 = pack_h2(S[2 * s2][0], S[2 * s2][1]);
    const uint32_t pa1 = pack_h2(S[2 * s2][2], S[2 * s2][3]);
    const uint32_t pa2 = pack_h2(S[2 * s2 + 1][0], S[2 * s2 + 1][1]);
    const uint32_t pa3 = pack_h2(S[2 * s2 + 1][2], S[2 * s2 + 1][3]);
    const int pc = min(max(q0 - 16 + 16 * s2 + (mi & 1) * 8 + rl, w0), i_last);
    const unsigned char* vrow = Vs + (pc - (i0 - kNear)) * kRowBytes;
    const int sw = swz(pc);
#pragma unroll
    for (int nd = 0; nd < 8; nd += 2) {
      uint32_t b[4];
      ldsm_x4_trans(b, vrow + ((nd + (mi >> 1)) ^ sw) * 16);
      mma16816(O[nd], pa0, pa1, pa2, pa3, b[0], b[1]);
      mma16816(O[nd + 1], pa0, pa1, pa2, pa3, b[2], b[3]);
    }
  }
#pragma unroll
  for (int j = 0; j < kMaxNear; ++j) {
    if (j < n_near) {  // uniform
      meta(j);
      if (act) rung_pv(Vs + (first - (i0 - kNear)) * kRowBytes, pn[j], O);  // uniform
    }
  }
  release_stage(2);

  // ---- streamed rungs: one per online-softmax step; rung r is stage 3 + r - n_near.
  // Ring slot and phase parity of the current stage (stage n sits in slot n % kSlots, phase
  // n / kSlots), advanced as the loop runs.
  int slot = 3 % kSlots;
  uint32_t par = (3 / kSlots) & 1;
  if (n_near < nrt) meta(n_near);
  for (int r = n_near; r < nrt; ++r) {
    if (!s_err && !mbar_wait(&full_bar[slot], par, a.wait_ns)) {
      s_err = 1;
      atomicExch(a.status, kStatusTimeout);
    }
    const unsigned char* st = ring + slot * a.slot_bytes;
    float sc[2] = {-INFINITY, -INFINITY};
    if (act) rung_scores(reinterpret_cast<const uint4*>(st), sc);  // uniform
    // Online softmax with a lazy reference: m only moves when a score passes it by more
    // than 8 (log2 units), so p = 2^(s - m) <= 256 (exact in f16 range) and O and the sums
    // are rescaled only then.
    if (__any_sync(0xffffffffu, sc[0] > m[0] + 8.f || sc[1] > m[1] + 8.f)) {  // uniform
      float corr[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float mc = __shfl_sync(0xffffffffu, fmaxf(m[h], sc[h]), src_lane);
        corr[h] = exp2f(m[h] - mc);
        m[h] = mc;
        lw[h] *= corr[h];
        lr[h] *= corr[h];
      }
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        O[nt][0] *= corr[0];
        O[nt][1] *= corr[0];
        O[nt][2] *= corr[1];
        O[nt][3] *= corr[1];
      }
    }
    if (act) {  // uniform
      float p[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        p[h] = exp2f(sc[h] - m[h]);  // 0 outside the holder lanes and for rows that do not attend
        lr[h] += p[h];
      }
      rung_pv(st + SR * kRowBytes, p, O);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_bar[slot]);
    if (r + 1 < nrt) meta(r + 1);  // uniform
    if (++slot == kSlots) {
      slot = 0;
      par ^= 1u;
    }
  }

  // ---- epilogue (nothing is written after a wait gave up; the producer reports it)
  if (s_err) return;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float l = lw[h] + lr[h];  // lane partial: its window terms, and the rung terms in the holder
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    const int i = irow[h];
    if (i < N) {
      const float inv = 1.f / l;
      uint32_t* orow = reinterpret_cast<uint32_t*>(a.o + base + static_cast<size_t>(i) * kD);
#pragma unroll
      for (int nt = 0; nt < 8; ++nt)
        orow[4 * nt + t] = pack_bf2_rn(O[nt][2 * h] * inv, O[nt][2 * h + 1] * inv);
      if (t == 0 && a.lse != nullptr) a.lse[static_cast<size_t>(bh) * N + i] = (m[h] + log2f(l)) * kLn2;
    }
  }
}

bool tc_supported(const LayerTable& t) { return t.W <= kTcMaxW; }

size_t fwd_tc_workspace_bytes(int B, int H, int N) {
  return static_cast<size_t>(B) * H * N * kD * 2 * sizeof(__half);
}

cudaError_t launch_prep_kv(int B, int H, int N, const void* k, const void* v, const float2* lo_tab,
                           const float2* hi_tab, void* workspace, int* status, cudaStream_t stream) {
  const long long rows = static_cast<long long>(B) * H * N;
  __half* kp = static_cast<__half*>(workspace);
  __half* vp = kp + rows * kD;
  const long long blocks = (rows + kPrepRowsPerBlock - 1) / kPrepRowsPerBlock;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  prep_kv_kernel<<<static_cast<unsigned>(blocks), kPrepThreads, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(k), static_cast<const __nv_bfloat16*>(v), kp, vp, lo_tab, hi_tab, N,
      rows, status);
  return cudaGetLastError();
}

cudaError_t launch_fwd_tc(const LayerTable& t, int B, int H, int N, const void* q, const void* workspace,
                          void* o, float* lse, const float2* lo_tab, const float2* hi_tab, int* status,
                          unsigned long long wait_ns, int skip_first_rung_copy, bool after_prep,
                          cudaStream_t stream) {
  const long long rows = static_cast<long long>(B) * H * N;
  TcArgs a;
  a.t = t;
  a.N = N;
  a.tiles = (N + kTcTile - 1) / kTcTile;
  a.bh = B * H;
  a.slab_rows = t.mode == 1 ? kTcTile + 1 : kTcTile;  // interp reads one row more
  a.slot_bytes = 2 * a.slab_rows * kRowBytes;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.kp = static_cast<const __half*>(workspace);
  a.vp = a.kp + rows * kD;
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
  const int smem = kSlots * a.slot_bytes;
  void (*kern)(TcArgs) = t.mode == 0 ? fwd_tc_kernel<0> : fwd_tc_kernel<1>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // After this layer's own preparation grid (after_prep) the launch is a programmatic
  // dependent of it: the CTAs may start (build their key table, load and rotate Q) while
  // that grid drains, and wait for it before they read K'/V'.  Q is read before that wait,
  // which is safe only because the preparation writes nothing but the workspace; after any
  // other grid (the split entry point) the launch is an ordinary one.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = after_prep ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, kern, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace fibattn
