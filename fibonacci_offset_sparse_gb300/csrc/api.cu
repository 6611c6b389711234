// C ABI of libfibattn.so (declared in include/fib_attn.h): argument checking, the plan
// (host tables + device RoPE tables + status word) and kernel launches.  Every device
// entry point only enqueues work on the caller's stream.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>
#include <set>
#include <vector>

#include "../../include/fib_attn.h"
#include "common.cuh"
#include "planner.h"

namespace fibattn {
cudaError_t launch_fwd(const LayerTable& t, int B, int H, int N, int dtype, const void* q,
                       const void* k, const void* v, void* o, float* lse, const float2* lo_tab,
                       const float2* hi_tab, cudaStream_t stream);
bool tc_supported(const LayerTable& t);
size_t fwd_tc_workspace_bytes(int B, int H, int N);
cudaError_t launch_prep_kv(int B, int H, int N, const void* k, const void* v, const float2* lo_tab,
                           const float2* hi_tab, void* workspace, int* status, cudaStream_t stream);
cudaError_t launch_fwd_tc(const LayerTable& t, int B, int H, int N, const void* q, const void* workspace,
                          void* o, float* lse, const float2* lo_tab, const float2* hi_tab, int* status,
                          unsigned long long wait_ns, int skip_first_rung_copy, bool after_prep,
                          cudaStream_t stream);
cudaError_t launch_debug_indices(const LayerTable& t, int N, int i0, int i1, int32_t* out,
                                 float* w_out, cudaStream_t stream);
size_t bwd_workspace_bytes(int B, int H, int N);
bool bwd_tc_supported(const LayerTable& t);
size_t bwd_tc_workspace_bytes(int B, int H, int N, int W);
cudaError_t launch_bwd_tc(const LayerTable& t, int B, int H, int N, const void* q, const void* k, const void* v,
                          const void* kv_prepared, const void* o, const float* lse, const void* dO, void* dq,
                          void* dk, void* dv, float* dalpha, void* ws, const float2* lo_tab, const float2* hi_tab,
                          int* status, unsigned long long wait_ns, cudaStream_t stream, const BwdStreams& side);
cudaError_t launch_bwd(const LayerTable& t, int B, int H, int N, int dtype, const void* q,
                       const void* k, const void* v, const void* o, const float* lse,
                       const void* dO, void* dq, void* dk, void* dv, float* dalpha, void* ws,
                       const float2* lo_tab, const float2* hi_tab, cudaStream_t stream);
cudaError_t launch_decode(const LayerTable& t, int B, int H, int N, int pos, int dtype,
                          const void* q, const void* k, const void* v, void* o, float* lse,
                          const float2* lo_tab, const float2* hi_tab, cudaStream_t stream);
cudaError_t launch_dense_fwd(int B, int H, int N, const void* q, const void* workspace, void* o, float* lse,
                             const float2* lo_tab, const float2* hi_tab, int* status, unsigned long long wait_ns,
                             bool after_prep, cudaStream_t stream);
cudaError_t noalloc_scratch(void** out);
size_t noalloc_scratch_bytes();
}  // namespace fibattn

using namespace fibattn;

namespace {
// Test hook: every CTA takes a whole SM's shared memory and fills it with `pattern`, so that
// the kernels launched next on those SMs start from known stale contents.
__global__ void fill_shared_kernel(uint32_t pattern, int words) {
  extern __shared__ uint32_t fill_smem[];
  for (int i = threadIdx.x; i < words; i += blockDim.x) fill_smem[i] = pattern;
  __syncthreads();
  // keep the stores: make them observable through a value no thread will ever see
  if (fill_smem[(threadIdx.x * 7) % words] == pattern + 1u && pattern == 0xffffffffu) fill_smem[0] = 0u;
}
}  // namespace

struct fib_attn_plan_s {
  int base_kind = 0;
  std::vector<int32_t> custom;
  std::vector<double> alpha;
  int W = 0, N_max = 0, D = 0, mode = 0;
  double rope_base = 10000.0;
  int device = -1;
  float2* d_lo = nullptr;
  float2* d_hi = nullptr;
  int* d_status = nullptr;
  unsigned long long wait_ns = 1000000000ULL;  // bound of every device-side wait (1 s)
  int skip_first_rung_copy = 0;                // test hooks, see fib_attn_plan_set_debug
  int corrupt_rung_table = 0;
  BwdStreams side;                             // the bf16 backward's second-half stream
  std::mutex side_mu;                          // one backward at a time forks onto it
};

namespace {

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Frees what a plan holds on the device (each handle may be null).
void release_device_state(fib_attn_plan_s* p) {
  cudaFree(p->d_lo);
  cudaFree(p->d_hi);
  cudaFree(p->d_status);
  if (p->side.join) cudaEventDestroy(p->side.join);
  if (p->side.first_q_done) cudaEventDestroy(p->side.first_q_done);
  if (p->side.fork) cudaEventDestroy(p->side.fork);
  if (p->side.stream) cudaStreamDestroy(p->side.stream);
}

std::vector<int32_t> plan_base(const fib_attn_plan_s* p, int N) {
  if (p->base_kind == FIB_BASE_FIBONACCI) return fibonacci_base(987);
  if (p->base_kind == FIB_BASE_POW2) return pow2_base(N);
  return p->custom;
}

// Per-layer key table for a call at sequence length N.
int make_table(const fib_attn_plan_s* p, int layer, int N, const float* alpha_dev,
               LayerTable* t) {
  std::memset(t, 0, sizeof(*t));
  t->mode = p->mode;
  t->W = p->W;
  t->layer = layer;
  const std::vector<int32_t> base = plan_base(p, N);
  if (p->mode == FIB_MODE_MASK) {
    const std::vector<int32_t> d = mask_distances(base.data(), static_cast<int>(base.size()),
                                                  p->alpha[layer], p->W, N);
    if (d.size() > static_cast<size_t>(kMaxR)) return FIB_ERR_UNSUPPORTED;
    t->n = static_cast<int>(d.size());
    for (int r = 0; r < t->n; ++r) t->lo[r] = d[r];
  } else if (alpha_dev == nullptr) {
    const std::vector<Rung> rs = interp_rungs(base.data(), static_cast<int>(base.size()),
                                              p->alpha[layer], p->W, N);
    if (rs.size() > static_cast<size_t>(kMaxR)) return FIB_ERR_UNSUPPORTED;
    t->n = static_cast<int>(rs.size());
    for (int r = 0; r < t->n; ++r) {
      t->lo[r] = rs[r].lo;
      t->w[r] = rs[r].w;
      t->f[r] = rs[r].f;
    }
  } else {
    const std::set<int32_t> fs(base.begin(), base.end());
    if (fs.size() > static_cast<size_t>(kMaxR)) return FIB_ERR_UNSUPPORTED;
    t->n = 0;
    for (int32_t f : fs) t->f[t->n++] = f;
    t->alpha_dev = alpha_dev;
  }
  return FIB_OK;
}

// Test hook of the tensor-core forward only (the one kernel family that checks its rung
// table on the device): the first rung of a host-built table is moved to distance 0, inside
// the window.  That row is the query's own, so the corrupted table still addresses only rows
// of the sequence; the kernel's check rejects it before any rung row is copied.
void corrupt_for_test(const fib_attn_plan_s* p, LayerTable* t) {
  if (p->corrupt_rung_table && t->n > 0 && t->alpha_dev == nullptr) {
    t->lo[0] = 0;
    t->w[0] = 0.f;
  }
}

int check_device(const fib_attn_plan_s* p) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return FIB_ERR_CUDA;
  if (dev != p->device) return FIB_ERR_INVALID_ARG;
  return FIB_OK;
}

int check_tensor(const void* ptr) {
  if (ptr == nullptr || !aligned(ptr, 16)) return FIB_ERR_INVALID_ARG;
  return FIB_OK;
}

int check_shape(const fib_attn_plan_s* p, int layer, int B, int H, int N, int dtype) {
  if (p == nullptr) return FIB_ERR_INVALID_ARG;
  if (layer < 0 || layer >= static_cast<int>(p->alpha.size())) return FIB_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || N < 1 || N > p->N_max) return FIB_ERR_INVALID_ARG;
  if (dtype != FIB_DTYPE_F32 && dtype != FIB_DTYPE_BF16) return FIB_ERR_INVALID_ARG;
  const long long rows = static_cast<long long>(B) * H * N;
  if (rows > (1LL << 40) / kD) return FIB_ERR_INVALID_ARG;
  return FIB_OK;
}

int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return FIB_OK;
  if (e == cudaErrorMemoryAllocation) return FIB_ERR_NOMEM;
  return FIB_ERR_CUDA;
}

}  // namespace

extern "C" {

const char* fib_attn_error_string(int code) {
  switch (code) {
    case FIB_OK: return "ok";
    case FIB_ERR_INVALID_ARG: return "invalid argument";
    case FIB_ERR_UNSUPPORTED: return "unsupported configuration";
    case FIB_ERR_CUDA: return "CUDA runtime error";
    case FIB_ERR_NOMEM: return "out of memory";
    case FIB_ERR_TIMEOUT: return "device wait timed out";
    case FIB_ERR_DEVICE_ASSERT: return "device-side check failed";
    case FIB_ERR_RANGE: return "value outside the float16 range of the bf16 tensor-core path";
    default: return "unknown status";
  }
}

int fib_attn_base(int base_kind, int N, int32_t* out, int cap, int* n_out) {
  if (n_out == nullptr || cap < 0 || (cap > 0 && out == nullptr)) return FIB_ERR_INVALID_ARG;
  std::vector<int32_t> b;
  if (base_kind == FIB_BASE_FIBONACCI) {
    b = fibonacci_base(987);
  } else if (base_kind == FIB_BASE_POW2) {
    if (N < 2) return FIB_ERR_INVALID_ARG;
    b = pow2_base(N);
  } else {
    return FIB_ERR_INVALID_ARG;
  }
  *n_out = static_cast<int>(b.size());
  for (int i = 0; i < cap && i < static_cast<int>(b.size()); ++i) out[i] = b[i];
  return FIB_OK;
}

int fib_attn_schedule(int kind, int n_layers, int stride, double* alpha_out) {
  if (alpha_out == nullptr || n_layers < 1 || n_layers > FIB_MAX_LAYERS) return FIB_ERR_INVALID_ARG;
  std::vector<double> a;
  if (!schedule(kind, n_layers, stride, &a)) return FIB_ERR_INVALID_ARG;
  for (int l = 0; l < n_layers; ++l) alpha_out[l] = a[l];
  return FIB_OK;
}

static int check_base_args(const int32_t* base, int n_base, double alpha, int W, int N) {
  if (n_base < 0 || (n_base > 0 && base == nullptr)) return FIB_ERR_INVALID_ARG;
  if (!std::isfinite(alpha) || alpha <= 0.0 || W < 1 || N < 1) return FIB_ERR_INVALID_ARG;
  for (int k = 0; k < n_base; ++k)
    if (base[k] < 1) return FIB_ERR_INVALID_ARG;
  return FIB_OK;
}

int fib_attn_mask_distances(const int32_t* base, int n_base, double alpha, int W, int N,
                            int32_t* out, int cap, int* n_out) {
  if (n_out == nullptr || cap < 0 || (cap > 0 && out == nullptr)) return FIB_ERR_INVALID_ARG;
  const int st = check_base_args(base, n_base, alpha, W, N);
  if (st != FIB_OK) return st;
  const std::vector<int32_t> d = mask_distances(base, n_base, alpha, W, N);
  *n_out = static_cast<int>(d.size());
  for (int i = 0; i < cap && i < static_cast<int>(d.size()); ++i) out[i] = d[i];
  return FIB_OK;
}

int fib_attn_interp_rungs(const int32_t* base, int n_base, double alpha, int W, int N,
                          int32_t* f_out, int32_t* lo_out, float* w_out, int cap, int* n_out) {
  if (n_out == nullptr || cap < 0) return FIB_ERR_INVALID_ARG;
  if (cap > 0 && (f_out == nullptr || lo_out == nullptr || w_out == nullptr)) return FIB_ERR_INVALID_ARG;
  const int st = check_base_args(base, n_base, alpha, W, N);
  if (st != FIB_OK) return st;
  const std::vector<Rung> rs = interp_rungs(base, n_base, alpha, W, N);
  *n_out = static_cast<int>(rs.size());
  for (int i = 0; i < cap && i < static_cast<int>(rs.size()); ++i) {
    f_out[i] = rs[i].f;
    lo_out[i] = rs[i].lo;
    w_out[i] = rs[i].w;
  }
  return FIB_OK;
}

int fib_attn_plan_create(fib_attn_plan_t* out, int base_kind, const int32_t* custom_base,
                         int n_custom, const double* alpha, int n_layers, int W, int N_max,
                         int D, int mode, double rope_base) {
  if (out == nullptr) return FIB_ERR_INVALID_ARG;
  *out = nullptr;
  if (base_kind < FIB_BASE_FIBONACCI || base_kind > FIB_BASE_CUSTOM) return FIB_ERR_INVALID_ARG;
  if (base_kind == FIB_BASE_CUSTOM) {
    if (custom_base == nullptr || n_custom < 1 || n_custom > kMaxR) return FIB_ERR_INVALID_ARG;
    for (int k = 0; k < n_custom; ++k)
      if (custom_base[k] < 1) return FIB_ERR_INVALID_ARG;
  }
  if (alpha == nullptr || n_layers < 1 || n_layers > FIB_MAX_LAYERS) return FIB_ERR_INVALID_ARG;
  for (int l = 0; l < n_layers; ++l)
    if (!std::isfinite(alpha[l]) || alpha[l] <= 0.0) return FIB_ERR_INVALID_ARG;
  if (W < 1 || W > kMaxW || N_max < 1 || N_max > (1 << 20)) return FIB_ERR_INVALID_ARG;
  if (mode != FIB_MODE_MASK && mode != FIB_MODE_INTERP) return FIB_ERR_INVALID_ARG;
  if (!std::isfinite(rope_base) || rope_base <= 1.0) return FIB_ERR_INVALID_ARG;
  if (D != kD) return FIB_ERR_UNSUPPORTED;

  fib_attn_plan_s* p = new (std::nothrow) fib_attn_plan_s();
  if (p == nullptr) return FIB_ERR_NOMEM;
  p->base_kind = base_kind;
  if (base_kind == FIB_BASE_CUSTOM) p->custom.assign(custom_base, custom_base + n_custom);
  p->alpha.assign(alpha, alpha + n_layers);
  p->W = W;
  p->N_max = N_max;
  p->D = D;
  p->mode = mode;
  p->rope_base = rope_base;
  // every layer's table must fit at the largest N
  for (int l = 0; l < n_layers; ++l) {
    LayerTable t;
    const int st = make_table(p, l, N_max, nullptr, &t);
    if (st != FIB_OK) {
      delete p;
      return st;
    }
  }
  if (cudaGetDevice(&p->device) != cudaSuccess) {
    delete p;
    return FIB_ERR_CUDA;
  }
  std::vector<float> lo, hi;
  rope_tables(N_max, rope_base, &lo, &hi);
  cudaError_t e = cudaMalloc(&p->d_lo, lo.size() * sizeof(float));
  if (e == cudaSuccess) e = cudaMalloc(&p->d_hi, hi.size() * sizeof(float));
  if (e == cudaSuccess) e = cudaMalloc(&p->d_status, sizeof(int));
  if (e == cudaSuccess) e = cudaMemcpy(p->d_lo, lo.data(), lo.size() * sizeof(float), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(p->d_hi, hi.data(), hi.size() * sizeof(float), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemset(p->d_status, 0, sizeof(int));
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p->side.stream, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->side.fork, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->side.first_q_done, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->side.join, cudaEventDisableTiming);
  if (e != cudaSuccess) {
    release_device_state(p);
    delete p;
    return cuda_status(e);
  }
  *out = p;
  return FIB_OK;
}

int fib_attn_plan_destroy(fib_attn_plan_t p) {
  if (p == nullptr) return FIB_OK;
  int prev = -1;
  cudaGetDevice(&prev);
  if (p->device >= 0) cudaSetDevice(p->device);
  cudaDeviceSynchronize();
  release_device_state(p);
  if (prev >= 0) cudaSetDevice(prev);
  delete p;
  return FIB_OK;
}

int fib_attn_plan_distances(fib_attn_plan_t p, int layer, int N, int32_t* out, int cap,
                            int* n_out) {
  if (p == nullptr || n_out == nullptr || cap < 0 || (cap > 0 && out == nullptr)) return FIB_ERR_INVALID_ARG;
  if (layer < 0 || layer >= static_cast<int>(p->alpha.size()) || N < 1 || N > p->N_max) return FIB_ERR_INVALID_ARG;
  LayerTable t;
  const int st = make_table(p, layer, N, nullptr, &t);
  if (st != FIB_OK) return st;
  *n_out = t.n;
  for (int i = 0; i < cap && i < t.n; ++i) out[i] = t.lo[i];
  return FIB_OK;
}

size_t fib_attn_fwd_workspace_size(fib_attn_plan_t p, int B, int H, int N, int dtype) {
  if (p == nullptr || B < 1 || H < 1 || N < 1 || dtype != FIB_DTYPE_BF16 || p->W > 16) return 0;
  return fwd_tc_workspace_bytes(B, H, N);
}

int fib_attn_fwd(fib_attn_plan_t p, int layer, int B, int H, int N, int dtype, const void* q,
                 const void* k, const void* v, void* o, float* lse, const float* alpha_dev,
                 void* workspace, size_t ws_bytes, void* stream) {
  int st = check_shape(p, layer, B, H, N, dtype);
  if (st != FIB_OK) return st;
  const size_t need = fib_attn_fwd_workspace_size(p, B, H, N, dtype);
  if (need > 0 && (workspace == nullptr || !aligned(workspace, 256) || ws_bytes < need))
    return FIB_ERR_INVALID_ARG;
  if (need > 0 && (workspace == q || workspace == k || workspace == v || workspace == o))
    return FIB_ERR_INVALID_ARG;
  if (check_tensor(q) || check_tensor(k) || check_tensor(v) || check_tensor(o)) return FIB_ERR_INVALID_ARG;
  if (o == q || o == k || o == v) return FIB_ERR_INVALID_ARG;
  if (lse != nullptr && !aligned(lse, 4)) return FIB_ERR_INVALID_ARG;
  if (alpha_dev != nullptr && !aligned(alpha_dev, 4)) return FIB_ERR_INVALID_ARG;
  st = check_device(p);
  if (st != FIB_OK) return st;
  LayerTable t;
  st = make_table(p, layer, N, p->mode == FIB_MODE_INTERP ? alpha_dev : nullptr, &t);
  if (st != FIB_OK) return st;
  // bf16 with a window of at most 16 keys: K'/V' preparation plus the tensor-core kernel
  // (fwd_tc.cu); otherwise the CUDA-core kernel (fwd.cu), which also serves float32 exactly.
  if (dtype == FIB_DTYPE_BF16 && tc_supported(t)) {
    corrupt_for_test(p, &t);
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    const cudaError_t e = launch_prep_kv(B, H, N, k, v, p->d_lo, p->d_hi, workspace, p->d_status, s);
    if (e != cudaSuccess) return cuda_status(e);
    return cuda_status(launch_fwd_tc(t, B, H, N, q, workspace, o, lse, p->d_lo, p->d_hi, p->d_status,
                                     p->wait_ns, p->skip_first_rung_copy, true, s));
  }
  return cuda_status(launch_fwd(t, B, H, N, dtype, q, k, v, o, lse, p->d_lo, p->d_hi,
                                static_cast<cudaStream_t>(stream)));
}

int fib_attn_fwd_prepare_kv(fib_attn_plan_t p, int B, int H, int N, int dtype, const void* k,
                            const void* v, void* workspace, size_t ws_bytes, void* stream) {
  int st = check_shape(p, 0, B, H, N, dtype);
  if (st != FIB_OK) return st;
  const size_t need = fib_attn_fwd_workspace_size(p, B, H, N, dtype);
  if (need == 0) return FIB_ERR_UNSUPPORTED;
  if (check_tensor(k) || check_tensor(v)) return FIB_ERR_INVALID_ARG;
  if (workspace == nullptr || !aligned(workspace, 256) || ws_bytes < need) return FIB_ERR_INVALID_ARG;
  if (workspace == k || workspace == v) return FIB_ERR_INVALID_ARG;
  st = check_device(p);
  if (st != FIB_OK) return st;
  return cuda_status(launch_prep_kv(B, H, N, k, v, p->d_lo, p->d_hi, workspace, p->d_status,
                                    static_cast<cudaStream_t>(stream)));
}

int fib_attn_fwd_attend(fib_attn_plan_t p, int layer, int B, int H, int N, int dtype, const void* q,
                        const void* workspace, size_t ws_bytes, void* o, float* lse,
                        const float* alpha_dev, void* stream) {
  int st = check_shape(p, layer, B, H, N, dtype);
  if (st != FIB_OK) return st;
  const size_t need = fib_attn_fwd_workspace_size(p, B, H, N, dtype);
  if (need == 0) return FIB_ERR_UNSUPPORTED;
  if (check_tensor(q) || check_tensor(o) || o == q) return FIB_ERR_INVALID_ARG;
  if (workspace == nullptr || !aligned(workspace, 256) || ws_bytes < need) return FIB_ERR_INVALID_ARG;
  if (workspace == q || workspace == o) return FIB_ERR_INVALID_ARG;
  if (lse != nullptr && !aligned(lse, 4)) return FIB_ERR_INVALID_ARG;
  if (alpha_dev != nullptr && !aligned(alpha_dev, 4)) return FIB_ERR_INVALID_ARG;
  st = check_device(p);
  if (st != FIB_OK) return st;
  LayerTable t;
  st = make_table(p, layer, N, p->mode == FIB_MODE_INTERP ? alpha_dev : nullptr, &t);
  if (st != FIB_OK) return st;
  corrupt_for_test(p, &t);
  return cuda_status(launch_fwd_tc(t, B, H, N, q, workspace, o, lse, p->d_lo, p->d_hi, p->d_status,
                                   p->wait_ns, p->skip_first_rung_copy, false,
                                   static_cast<cudaStream_t>(stream)));
}

size_t fib_attn_dense_fwd_workspace_size(fib_attn_plan_t p, int B, int H, int N, int dtype) {
  if (p == nullptr || B < 1 || H < 1 || N < 1 || dtype != FIB_DTYPE_BF16) return 0;
  return fwd_tc_workspace_bytes(B, H, N);
}

int fib_attn_dense_fwd(fib_attn_plan_t p, int B, int H, int N, int dtype, const void* q, const void* k,
                       const void* v, void* o, float* lse, void* workspace, size_t ws_bytes, void* stream) {
  int st = check_shape(p, 0, B, H, N, dtype);
  if (st != FIB_OK) return st;
  if (dtype != FIB_DTYPE_BF16) return FIB_ERR_UNSUPPORTED;
  const size_t need = fib_attn_dense_fwd_workspace_size(p, B, H, N, dtype);
  if (workspace == nullptr || !aligned(workspace, 256) || ws_bytes < need) return FIB_ERR_INVALID_ARG;
  if (workspace == q || workspace == k || workspace == v || workspace == o) return FIB_ERR_INVALID_ARG;
  if (check_tensor(q) || check_tensor(k) || check_tensor(v) || check_tensor(o)) return FIB_ERR_INVALID_ARG;
  if (o == q || o == k || o == v) return FIB_ERR_INVALID_ARG;
  if (lse != nullptr && !aligned(lse, 4)) return FIB_ERR_INVALID_ARG;
  st = check_device(p);
  if (st != FIB_OK) return st;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const cudaError_t e = launch_prep_kv(B, H, N, k, v, p->d_lo, p->d_hi, workspace, p->d_status, s);
  if (e != cudaSuccess) return cuda_status(e);
  return cuda_status(launch_dense_fwd(B, H, N, q, workspace, o, lse, p->d_lo, p->d_hi, p->d_status, p->wait_ns,
                                      true, s));
}

int fib_attn_decode(fib_attn_plan_t p, int layer, int B, int H, int N, int pos, int dtype,
                    const void* q, const void* k_cache, const void* v_cache, void* o, float* lse,
                    const float* alpha_dev, void* stream) {
  int st = check_shape(p, layer, B, H, N, dtype);
  if (st != FIB_OK) return st;
  if (pos < 0 || pos >= N) return FIB_ERR_INVALID_ARG;
  if (check_tensor(q) || check_tensor(k_cache) || check_tensor(v_cache) || check_tensor(o))
    return FIB_ERR_INVALID_ARG;
  if (o == q || o == k_cache || o == v_cache) return FIB_ERR_INVALID_ARG;
  if (lse != nullptr && !aligned(lse, 4)) return FIB_ERR_INVALID_ARG;
  if (alpha_dev != nullptr && !aligned(alpha_dev, 4)) return FIB_ERR_INVALID_ARG;
  st = check_device(p);
  if (st != FIB_OK) return st;
  LayerTable t;
  st = make_table(p, layer, N, p->mode == FIB_MODE_INTERP ? alpha_dev : nullptr, &t);
  if (st != FIB_OK) return st;
  return cuda_status(launch_decode(t, B, H, N, pos, dtype, q, k_cache, v_cache, o, lse, p->d_lo,
                                   p->d_hi, static_cast<cudaStream_t>(stream)));
}

size_t fib_attn_bwd_workspace_size(fib_attn_plan_t p, int B, int H, int N) {
  if (p == nullptr || B < 1 || H < 1 || N < 1) return 0;
  // one size for both dtypes: the bf16 tensor-core path (W <= 16) needs the prepared rows
  if (p->W <= 16) return std::max(bwd_workspace_bytes(B, H, N), bwd_tc_workspace_bytes(B, H, N, p->W));
  return bwd_workspace_bytes(B, H, N);
}

int fib_attn_bwd(fib_attn_plan_t p, int layer, int B, int H, int N, int dtype, const void* q,
                 const void* k, const void* v, const void* o, const float* lse, const void* dO,
                 void* dq, void* dk, void* dv, float* dalpha, const float* alpha_dev,
                 void* workspace, size_t ws_bytes, void* stream) {
  int st = check_shape(p, layer, B, H, N, dtype);
  if (st != FIB_OK) return st;
  if (check_tensor(q) || check_tensor(k) || check_tensor(v) || check_tensor(o) ||
      check_tensor(dO) || check_tensor(dq) || check_tensor(dk) || check_tensor(dv))
    return FIB_ERR_INVALID_ARG;
  if (lse == nullptr || !aligned(lse, 4) || dalpha == nullptr || !aligned(dalpha, 4)) return FIB_ERR_INVALID_ARG;
  if (alpha_dev != nullptr && !aligned(alpha_dev, 4)) return FIB_ERR_INVALID_ARG;
  if (workspace == nullptr || !aligned(workspace, 256) || ws_bytes < fib_attn_bwd_workspace_size(p, B, H, N))
    return FIB_ERR_INVALID_ARG;
  const void* ins[] = {q, k, v, o, dO};
  const void* outs[] = {dq, dk, dv};
  for (const void* a : outs)
    for (const void* b : ins)
      if (a == b) return FIB_ERR_INVALID_ARG;
  if (dq == dk || dq == dv || dk == dv) return FIB_ERR_INVALID_ARG;
  st = check_device(p);
  if (st != FIB_OK) return st;
  LayerTable t;
  st = make_table(p, layer, N, p->mode == FIB_MODE_INTERP ? alpha_dev : nullptr, &t);
  if (st != FIB_OK) return st;
  // bf16 with a window of at most 16 keys: prepared rows + tensor-core kernels (bwd_tc.cu);
  // otherwise the CUDA-core kernels (bwd.cu), which also serve float32
  if (dtype == FIB_DTYPE_BF16 && bwd_tc_supported(t)) {
    std::lock_guard<std::mutex> lock(p->side_mu);
    return cuda_status(launch_bwd_tc(t, B, H, N, q, k, v, nullptr, o, lse, dO, dq, dk, dv, dalpha, workspace,
                                     p->d_lo, p->d_hi, p->d_status, p->wait_ns, static_cast<cudaStream_t>(stream),
                                     p->side));
  }
  return cuda_status(launch_bwd(t, B, H, N, dtype, q, k, v, o, lse, dO, dq, dk, dv, dalpha,
                                workspace, p->d_lo, p->d_hi, static_cast<cudaStream_t>(stream)));
}

// Backward from the forward's prepared K' and V' rows (bf16 tensor-core path only): the same
// checks and kernels as fib_attn_bwd, minus the preparation of K' and V'.
int fib_attn_bwd_prepared(fib_attn_plan_t p, int layer, int B, int H, int N, int dtype, const void* q,
                          const void* kv_prepared, size_t kv_bytes, const void* o, const float* lse,
                          const void* dO, void* dq, void* dk, void* dv, float* dalpha, const float* alpha_dev,
                          void* workspace, size_t ws_bytes, void* stream) {
  int st = check_shape(p, layer, B, H, N, dtype);
  if (st != FIB_OK) return st;
  if (check_tensor(q) || check_tensor(o) || check_tensor(dO) || check_tensor(dq) || check_tensor(dk) ||
      check_tensor(dv))
    return FIB_ERR_INVALID_ARG;
  if (lse == nullptr || !aligned(lse, 4) || dalpha == nullptr || !aligned(dalpha, 4)) return FIB_ERR_INVALID_ARG;
  if (alpha_dev != nullptr && !aligned(alpha_dev, 4)) return FIB_ERR_INVALID_ARG;
  if (workspace == nullptr || !aligned(workspace, 256) || ws_bytes < fib_attn_bwd_workspace_size(p, B, H, N))
    return FIB_ERR_INVALID_ARG;
  const size_t kv_need = fib_attn_fwd_workspace_size(p, B, H, N, dtype);
  if (kv_need == 0) return FIB_ERR_UNSUPPORTED;  // float32, or a window wider than 16
  if (kv_prepared == nullptr || !aligned(kv_prepared, 256) || kv_bytes < kv_need) return FIB_ERR_INVALID_ARG;
  const void* ins[] = {q, o, dO, kv_prepared};
  const void* outs[] = {dq, dk, dv};
  for (const void* a : outs)
    for (const void* b : ins)
      if (a == b) return FIB_ERR_INVALID_ARG;
  if (dq == dk || dq == dv || dk == dv) return FIB_ERR_INVALID_ARG;
  if (kv_prepared == workspace) return FIB_ERR_INVALID_ARG;
  st = check_device(p);
  if (st != FIB_OK) return st;
  LayerTable t;
  st = make_table(p, layer, N, p->mode == FIB_MODE_INTERP ? alpha_dev : nullptr, &t);
  if (st != FIB_OK) return st;
  if (!bwd_tc_supported(t)) return FIB_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(p->side_mu);
  return cuda_status(launch_bwd_tc(t, B, H, N, q, nullptr, nullptr, kv_prepared, o, lse, dO, dq, dk, dv, dalpha,
                                   workspace, p->d_lo, p->d_hi, p->d_status, p->wait_ns,
                                   static_cast<cudaStream_t>(stream), p->side));
}

// Backward for callers that cannot allocate device memory: the same checks and kernels as
// fib_attn_bwd, but the scratch is the library's fixed device array (bwd.cu), so the caller
// passes no workspace and nothing is allocated here.
int fib_attn_bwd_noalloc(fib_attn_plan_t p, int layer, int B, int H, int N, int dtype,
                         const void* q, const void* k, const void* v, const void* o,
                         const float* lse, const void* dO, void* dq, void* dk, void* dv,
                         float* dalpha, const float* alpha_dev, void* stream) {
  int st = check_shape(p, layer, B, H, N, dtype);
  if (st != FIB_OK) return st;
  if (check_tensor(q) || check_tensor(k) || check_tensor(v) || check_tensor(o) ||
      check_tensor(dO) || check_tensor(dq) || check_tensor(dk) || check_tensor(dv))
    return FIB_ERR_INVALID_ARG;
  if (lse == nullptr || !aligned(lse, 4) || dalpha == nullptr || !aligned(dalpha, 4)) return FIB_ERR_INVALID_ARG;
  if (alpha_dev != nullptr && !aligned(alpha_dev, 4)) return FIB_ERR_INVALID_ARG;
  const void* ins[] = {q, k, v, o, dO};
  const void* outs[] = {dq, dk, dv};
  for (const void* a : outs)
    for (const void* b : ins)
      if (a == b) return FIB_ERR_INVALID_ARG;
  if (dq == dk || dq == dv || dk == dv) return FIB_ERR_INVALID_ARG;
  // the whole scratch of this call must fit the fixed array
  if (bwd_workspace_bytes(B, H, N) > noalloc_scratch_bytes()) return FIB_ERR_INVALID_ARG;
  st = check_device(p);
  if (st != FIB_OK) return st;
  LayerTable t;
  st = make_table(p, layer, N, p->mode == FIB_MODE_INTERP ? alpha_dev : nullptr, &t);
  if (st != FIB_OK) return st;
  void* scratch = nullptr;
  const cudaError_t e = noalloc_scratch(&scratch);
  if (e != cudaSuccess) return cuda_status(e);
  return cuda_status(launch_bwd(t, B, H, N, dtype, q, k, v, o, lse, dO, dq, dk, dv, dalpha,
                                scratch, p->d_lo, p->d_hi, static_cast<cudaStream_t>(stream)));
}

int fib_attn_debug_indices(fib_attn_plan_t p, int layer, int N, int i_begin, int i_end,
                           int32_t* out_dev, float* w_out_dev, const float* alpha_dev,
                           void* stream) {
  if (p == nullptr || out_dev == nullptr || !aligned(out_dev, 4)) return FIB_ERR_INVALID_ARG;
  if (layer < 0 || layer >= static_cast<int>(p->alpha.size()) || N < 1 || N > p->N_max) return FIB_ERR_INVALID_ARG;
  if (i_begin < 0 || i_end > N || i_begin >= i_end) return FIB_ERR_INVALID_ARG;
  if (w_out_dev != nullptr && !aligned(w_out_dev, 4)) return FIB_ERR_INVALID_ARG;
  int st = check_device(p);
  if (st != FIB_OK) return st;
  LayerTable t;
  st = make_table(p, layer, N, p->mode == FIB_MODE_INTERP ? alpha_dev : nullptr, &t);
  if (st != FIB_OK) return st;
  return cuda_status(launch_debug_indices(t, N, i_begin, i_end, out_dev, w_out_dev,
                                          static_cast<cudaStream_t>(stream)));
}

int fib_attn_plan_set_debug(fib_attn_plan_t p, int debug_flags, long long wait_ns) {
  if (p == nullptr || wait_ns < 1000 || wait_ns > 60LL * 1000000000LL) return FIB_ERR_INVALID_ARG;
  if (debug_flags & ~(FIB_DEBUG_SKIP_COPY | FIB_DEBUG_CORRUPT_TABLE)) return FIB_ERR_INVALID_ARG;
  p->skip_first_rung_copy = (debug_flags & FIB_DEBUG_SKIP_COPY) ? 1 : 0;
  p->corrupt_rung_table = (debug_flags & FIB_DEBUG_CORRUPT_TABLE) ? 1 : 0;
  p->wait_ns = static_cast<unsigned long long>(wait_ns);
  return FIB_OK;
}

int fib_attn_debug_fill_shared(uint32_t pattern, void* stream) {
  int dev = 0, sms = 0, smem = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(fill_shared_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return cuda_status(e);
  // two waves of one CTA per SM, so that every SM is reached
  fill_shared_kernel<<<2 * sms, 1024, static_cast<size_t>(smem), static_cast<cudaStream_t>(stream)>>>(
      pattern, smem / 4);
  return cuda_status(cudaGetLastError());
}

int fib_attn_last_device_status(fib_attn_plan_t p) {
  if (p == nullptr) return FIB_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return FIB_ERR_CUDA;
  int h = 0;
  if (cudaMemcpy(&h, p->d_status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return FIB_ERR_CUDA;
  if (cudaMemset(p->d_status, 0, sizeof(int)) != cudaSuccess) return FIB_ERR_CUDA;
  return h;
}

}  // extern "C"
