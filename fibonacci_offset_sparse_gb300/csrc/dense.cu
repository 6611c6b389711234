// Dense causal attention with the same RoPE, bf16 (sm_103a): the dense control of
// "Depth-Staggered Fibonacci Spacing for Sparse Attention", Methodology > "Controls" (a dense
// model of the same architecture as the upper bound) and Key results 3 (dense attention at
// 4x the training length).  Every query i attends every key j <= i; scores are
// RoPE(q_i).RoPE(k_j)/sqrt(D), the same reading of RoPE as the sparse path.
//
// Two launches, like the sparse bf16 forward: prep_kv_kernel (fwd_tc.cu) writes K rotated at
// each row's own position and V as float16 chunk-swizzled rows into the workspace, then
// dense_fwd_kernel: a CTA owns 64 consecutive queries of one (b, h) (4 compute warps of 16
// and one producer warp) and streams the 64-row key blocks 0 .. its own diagonal block
// through a ring of 16 KB slots (K' block + V' block, cp.async.bulk with mbarrier
// completion).  Per warp and key block: S = Q' K'^T (32 mma.sync m16n8k16, f16 operands,
// f32 accumulation), an online softmax with an exact running maximum, O += P V' (32 more).
// Q' = RoPE(q) log2(e)/8 is formed in registers, so scores are in log2 units.  Tiles launch
// heaviest first (a later tile reads more key blocks).  Every mbarrier wait is bounded; a
// wait that gives up records FIB_ERR_TIMEOUT and the CTA writes nothing.
#include <cuda_fp16.h>

#include "tc_common.cuh"

namespace fibattn {

constexpr int kDnWarps = 4;
constexpr int kDnTile = 16 * kDnWarps;          // queries per CTA
constexpr int kDnBlock = 64;                    // keys per ring stage
constexpr int kDnCons = 32 * kDnWarps;
constexpr int kDnThreads = kDnCons + 32;        // + one producer warp
constexpr int kDnSlots = 4;
constexpr int kDnSlotBytes = 2 * kDnBlock * kRowBytes;  // K' block, then V' block
constexpr int kDnQBytes = kDnTile * kRowBytes;
static_assert(kDnTile == kDnBlock, "a CTA's diagonal block is one key block");

struct DenseArgs {
  int N;
  int tiles;
  int bh;
  const __nv_bfloat16* q;
  const __half* kp;
  const __half* vp;
  __nv_bfloat16* o;
  float* lse;
  const float2* rope_lo;
  const float2* rope_hi;
  float qscale;  // log2(e)/sqrt(D)
  int* status;
  unsigned long long wait_ns;
  int after_prep;  // launched as a programmatic dependent of the preparation grid
};

__global__ void __launch_bounds__(kDnThreads, 3) dense_fwd_kernel(const __grid_constant__ DenseArgs a) {
  __shared__ __align__(8) uint64_t full_bar[kDnSlots];
  __shared__ __align__(8) uint64_t empty_bar[kDnSlots];
  __shared__ __align__(8) uint64_t q_bar;
  __shared__ volatile int s_err;
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* qbuf = smem;
  unsigned char* ring = smem + kDnQBytes;

  const int bh = blockIdx.x % a.bh;
  const int tile = a.tiles - 1 - static_cast<int>(blockIdx.x / a.bh);
  const int i0 = tile * kDnTile;
  const int N = a.N;
  const int tid = threadIdx.x;
  const size_t base = static_cast<size_t>(bh) * N * kD;
  const int i_last = min(i0 + kDnTile, N) - 1;
  const int nblocks = tile + 1;  // key blocks 0 .. tile (the last one is the diagonal block)

  if (tid == kDnCons) {
    s_err = 0;
    for (int s = 0; s < kDnSlots; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kDnWarps);
    }
    mbar_init(&q_bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    const uint32_t bytes = static_cast<uint32_t>(i_last - i0 + 1) * kRowBytes;
    mbar_arrive_tx(&q_bar, bytes);
    bulk_g2s(qbuf, a.q + base + static_cast<size_t>(i0) * kD, bytes, &q_bar);
  }
  __syncthreads();
  const int warp = tid >> 5, lane = tid & 31;

  // ===================================================================== producer
  if (warp == kDnWarps) {
    if (lane != 0) return;
    int last_n[kDnSlots];
#pragma unroll
    for (int s = 0; s < kDnSlots; ++s) last_n[s] = -1;
    for (int n = 0; n < nblocks; ++n) {
      if (s_err) break;
      const int slot = n % kDnSlots;
      if (!mbar_wait_backoff(&empty_bar[slot], ((n / kDnSlots) & 1) ^ 1, a.wait_ns)) {
        s_err = 1;
        break;
      }
      // K'/V' come from the preparation grid launched just before this one: wait for it
      if (n == 0 && a.after_prep) asm volatile("griddepcontrol.wait;\n" ::: "memory");
      const int r0 = n * kDnBlock;
      const int rows = min(kDnBlock, i_last + 1 - r0);
      const uint32_t bytes = static_cast<uint32_t>(rows) * kRowBytes;
      unsigned char* dst = ring + slot * kDnSlotBytes;
      mbar_arrive_tx(&full_bar[slot], 2 * bytes);
      bulk_g2s(dst, a.kp + base + static_cast<size_t>(r0) * kD, bytes, &full_bar[slot]);
      bulk_g2s(dst + kDnBlock * kRowBytes, a.vp + base + static_cast<size_t>(r0) * kD, bytes, &full_bar[slot]);
      last_n[slot] = n;
    }
    mbar_wait(&q_bar, 0, a.wait_ns);
#pragma unroll
    for (int s = 0; s < kDnSlots; ++s)
      if (last_n[s] >= 0) mbar_wait(&full_bar[s], (last_n[s] / kDnSlots) & 1, a.wait_ns);
    if (s_err) atomicExch(a.status, kStatusTimeout);
    return;
  }

  // ===================================================================== compute warps
  const int g = lane >> 2, t = lane & 3;
  const int q0 = i0 + 16 * warp;
  int irow[2], ic[2];
  float2 eq[2][8];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    irow[h] = q0 + g + 8 * h;
    ic[h] = irow[h] < N ? irow[h] : N - 1;
    rope_row(a.rope_lo, a.rope_hi, ic[h], t, eq[h]);
  }
  auto fail = [&]() {
    s_err = 1;
    atomicExch(a.status, kStatusTimeout);
  };
  // Q' = RoPE(q) * log2(e)/sqrt(D) as f16 A fragments (dims D_t of rows g and g+8)
  uint32_t qa[2][2][4];
  if (!mbar_wait(&q_bar, 0, a.wait_ns)) fail();
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int row = ic[h] - i0;
    float x[16];
    if (!s_err) {
      uint4 wa, wb;
      lds_row_part(qbuf + row * kRowBytes, t, row & 1, wa, wb);
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
    for (int s = 0; s < 4; ++s)
      bad |= h2_nonfinite(qa[0][0][s]) | h2_nonfinite(qa[0][1][s]) | h2_nonfinite(qa[1][0][s]) | h2_nonfinite(qa[1][1][s]);
    if (bad) atomicExch(a.status, kStatusRange);
  }

  const int mi = lane >> 3, rl = lane & 7;
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
  float O[8][4];
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) O[nt][0] = O[nt][1] = O[nt][2] = O[nt][3] = 0.f;
  int slot = 0;
  uint32_t par = 0;
  for (int n = 0; n < nblocks; ++n) {
    if (!s_err && !mbar_wait(&full_bar[slot], par, a.wait_ns)) fail();
    if (s_err) break;
    const unsigned char* st = ring + slot * kDnSlotBytes;
    const uint4* Ks = reinterpret_cast<const uint4*>(st);
    const unsigned char* Vs = st + kDnBlock * kRowBytes;
    const int r0 = n * kDnBlock;
    const int rows = min(kDnBlock, i_last + 1 - r0);  // copied rows of this block
    // ---- S = Q' K'^T over the block's 64 keys (key column 8nt + g of the lane's B fragment)
    float S[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int u = 0; u < 4; ++u) S[nt][u] = 0.f;
      const int row = min(8 * nt + g, rows - 1);
      uint32_t kl[4], kh[4];
      lds_kfrag(Ks + row * 8, t, r0 + row, kl, kh);
#pragma unroll
      for (int s = 0; s < 4; ++s)
        mma16816(S[nt], qa[0][0][s], qa[1][0][s], qa[0][1][s], qa[1][1][s], kl[s], kh[s]);
    }
    // ---- causal mask (keys after the query; this also covers the uncopied rows of the
    // diagonal block, which lie after every query of the tile), online softmax
    const bool diag = n == nblocks - 1;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float mx = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float& s = S[nt][2 * h + e];
          if (diag && r0 + 8 * nt + 2 * t + e > ic[h]) s = -INFINITY;
          mx = fmaxf(mx, s);
        }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float mn = fmaxf(m[h], mx);  // finite: key 0 <= every query
      const float corr = exp2f(m[h] - mn);
      m[h] = mn;
      float sum = 0.f;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float& s = S[nt][2 * h + e];
          s = exp2f(s - mn);
          sum += s;
        }
      l[h] = l[h] * corr + sum;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        O[nt][2 * h] *= corr;
        O[nt][2 * h + 1] *= corr;
      }
    }
    // ---- O += P V' (k-step s2 covers keys 16 s2 .. 16 s2 + 15; ldmatrix rows outside the
    // copied ones read the last copied row, where P = 0, so that stale data never meets a 0)
#pragma unroll
    for (int s2 = 0; s2 < 4; ++s2) {
      const uint32_t pa0 = pack_h2(S[2 * s2][0], S[2 * s2][1]);
      const uint32_t pa1 = pack_h2(S[2 * s2][2], S[2 * s2][3]);
      const uint32_t pa2 = pack_h2(S[2 * s2 + 1][0], S[2 * s2 + 1][1]);
      const uint32_t pa3 = pack_h2(S[2 * s2 + 1][2], S[2 * s2 + 1][3]);
      const int vr = min(16 * s2 + (mi & 1) * 8 + rl, rows - 1);
      const unsigned char* vrow = Vs + vr * kRowBytes;
      const int sw = swz(r0 + vr);
#pragma unroll
      for (int nd = 0; nd < 8; nd += 2) {
        uint32_t b[4];
        ldsm_x4_trans(b, vrow + ((nd + (mi >> 1)) ^ sw) * 16);
        mma16816(O[nd], pa0, pa1, pa2, pa3, b[0], b[1]);
        mma16816(O[nd + 1], pa0, pa1, pa2, pa3, b[2], b[3]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_bar[slot]);
    if (++slot == kDnSlots) {
      slot = 0;
      par ^= 1u;
    }
  }
  if (s_err) return;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float lt = l[h];
    lt += __shfl_xor_sync(0xffffffffu, lt, 1);
    lt += __shfl_xor_sync(0xffffffffu, lt, 2);
    const int i = irow[h];
    if (i < N) {
      const float inv = 1.f / lt;
      uint32_t* orow = reinterpret_cast<uint32_t*>(a.o + base + static_cast<size_t>(i) * kD);
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) orow[4 * nt + t] = pack_bf2_rn(O[nt][2 * h] * inv, O[nt][2 * h + 1] * inv);
      if (t == 0 && a.lse != nullptr) a.lse[static_cast<size_t>(bh) * N + i] = (m[h] + log2f(lt)) * kLn2;
    }
  }
}

cudaError_t launch_dense_fwd(int B, int H, int N, const void* q, const void* workspace, void* o, float* lse,
                             const float2* lo_tab, const float2* hi_tab, int* status, unsigned long long wait_ns,
                             bool after_prep, cudaStream_t stream) {
  const long long rows = static_cast<long long>(B) * H * N;
  DenseArgs a;
  a.N = N;
  a.tiles = (N + kDnTile - 1) / kDnTile;
  a.bh = B * H;
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
  a.after_prep = after_prep ? 1 : 0;
  const long long blocks = static_cast<long long>(a.tiles) * B * H;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const int smem = kDnQBytes + kDnSlots * kDnSlotBytes;
  cudaError_t e = cudaFuncSetAttribute(dense_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(kDnThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = after_prep ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, dense_fwd_kernel, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace fibattn
