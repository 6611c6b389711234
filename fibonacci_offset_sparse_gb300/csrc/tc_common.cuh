// Device helpers shared by the tensor-core kernels (fwd_tc.cu, bwd_tc.cu): mbarrier waits
// bounded in time, bulk copies, mma.sync / ldmatrix wrappers, the row swizzle of the
// prepared f16 rows, and RoPE factors from the factored tables.
#pragma once
#include <cuda_fp16.h>

#include "common.cuh"

namespace fibattn {

constexpr int kRowBytes = kD * 2;  // one row of 16-bit values

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
// that a waiting producer leaves the issue slots to the compute warps of its SM.
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
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack_bf2_rn(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm(
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

// Chunk swizzle of the K'/V' row of sequence position p (p >= 0 where it matters).
__device__ __forceinline__ int swz(int p) { return ((p & 1) << 2) | ((p >> 1) & 3); }

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

// The dims D_t of the swizzled K' row of position p, as the B fragments of the 4 k-steps.
__device__ __forceinline__ void lds_kfrag(const uint4* row, int t, int p, uint32_t (&lo)[4],
                                          uint32_t (&hi)[4]) {
  const int s = swz(p);
  const uint4 a = row[t ^ s], b = row[(t + 4) ^ s];
  lo[0] = a.x; lo[1] = a.y; lo[2] = a.z; lo[3] = a.w;
  hi[0] = b.x; hi[1] = b.y; hi[2] = b.z; hi[3] = b.w;
}

// e^{i p theta_m} for the lane's frequencies m = 8t .. 8t+7, from the factored tables.
__device__ __forceinline__ void rope_row(const float2* __restrict__ lo_tab, const float2* __restrict__ hi_tab,
                                         int p, int t, float2 (&e)[8]) {
  const float4* h4 = reinterpret_cast<const float4*>(hi_tab + (p / kSplit) * kFreq + 8 * t);
  const float4* l4 = reinterpret_cast<const float4*>(lo_tab + (p % kSplit) * kFreq + 8 * t);
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const float4 x = __ldg(h4 + u), y = __ldg(l4 + u);
    e[2 * u] = make_float2(x.x * y.x - x.y * y.y, x.x * y.y + x.y * y.x);
    e[2 * u + 1] = make_float2(x.z * y.z - x.w * y.w, x.z * y.w + x.w * y.z);
  }
}

}  // namespace fibattn
