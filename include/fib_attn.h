/*
 * fib_attn.h -- C ABI of the GB300 (sm_103a) Depth-Staggered Fibonacci Spacing sparse
 * attention library (libfibattn.so).
 *
 * The operation ("Depth-Staggered Fibonacci Spacing for Sparse Attention: Static
 * Schedules Beat Learned Dilation and Extrapolate Where Dense Attention Fails",
 * Methodology > "Attended set", "Scaling", "Implementation"):
 *   each causal query i of a layer attends to a dense local window of W keys
 *   (distances 0..W-1, the query itself included) plus sparse keys at distances
 *   d_k = alpha_l * f_k, f the Fibonacci list 1, 2, 3, 5, ..., 987 (or the power-of-two
 *   control base), alpha_l one scalar per layer in [0.5, 1.5].  RoPE is applied to Q and
 *   K before the gather.  Integer distances take the boolean-mask path (MASK); non-integer
 *   ones are served by linear interpolation between the two bracketing K/V rows, which
 *   gives alpha a gradient (INTERP).
 *
 * Readings where the pages are silent:
 *   - a static non-integer distance is rounded half-to-even (binary64 product alpha*f);
 *     MASK keeps the distinct distances d >= W, INTERP keeps rungs with d > W-1;
 *   - a rung is attended by query i iff d <= i (no padding, no clamping);
 *   - softmax scale 1/sqrt(D); RoPE rotate-half pairs (m, m+D/2), positions 0..N-1,
 *     angle p * rope_base^(-2m/D); V is not rotated;
 *   - INTERP blends the rotated rows: k~ = (1-w) k'[i-lo] + w k'[i-lo-1], lo = floor(d),
 *     w = d - lo; dalpha is the right derivative (lo held fixed, dw/dalpha = f), the
 *     term is zero where row i-lo-1 does not exist.
 *
 * Conventions for every entry point:
 *   - Return value: a fib_status code; no function aborts, prints or exits.
 *   - Tensors are caller-owned device buffers, contiguous [B, H, N, D] row-major with
 *     D = 64, 16-byte aligned.  Q/K/V/O/dO/dQ/dK/dV share one dtype (fib_dtype); LSE
 *     ([B, H, N]) and dalpha are float32.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Device entry points
 *     only enqueue work on it and never synchronise, except fib_attn_last_device_status.
 *   - The library owns only the plan (host struct + its small device RoPE tables and
 *     status word, allocated by fib_attn_plan_create on the device current at that time;
 *     every device call must run with that same device current).
 *   - There is no CPU fallback: without a CUDA device the device entry points return
 *     FIB_ERR_CUDA.
 */
#ifndef FIB_ATTN_H
#define FIB_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct fib_attn_plan_s* fib_attn_plan_t;

enum fib_status {
  FIB_OK = 0,
  FIB_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size, out-of-range index   */
  FIB_ERR_UNSUPPORTED = 2,   /* valid request the library does not implement (D != 64) */
  FIB_ERR_CUDA = 3,          /* a CUDA runtime call failed (incl. no device)            */
  FIB_ERR_NOMEM = 4,         /* host or device allocation failed                        */
  FIB_ERR_TIMEOUT = 5,       /* a bounded device wait gave up (see last_device_status)  */
  FIB_ERR_DEVICE_ASSERT = 6, /* a device-side check recorded a violated invariant       */
  FIB_ERR_RANGE = 7          /* an input value does not fit the float16 operands of the
                                bf16 tensor-core path (see fib_attn_fwd)                */
};

/* Test hooks of fib_attn_plan_set_debug (bit flags). */
enum fib_debug_flag { FIB_DEBUG_SKIP_COPY = 1, FIB_DEBUG_CORRUPT_TABLE = 2 };

enum fib_base_kind { FIB_BASE_FIBONACCI = 0, FIB_BASE_POW2 = 1, FIB_BASE_CUSTOM = 2 };
enum fib_schedule_kind { FIB_SCHED_FIXED = 0, FIB_SCHED_LINEAR = 1, FIB_SCHED_COPRIME = 2 };
enum fib_mode { FIB_MODE_MASK = 0, FIB_MODE_INTERP = 1 };
enum fib_dtype { FIB_DTYPE_F32 = 0, FIB_DTYPE_BF16 = 1 };

#define FIB_HEAD_DIM 64   /* the only head dimension built */
#define FIB_MAX_RUNGS 32  /* rungs per layer, after dedup */
#define FIB_MAX_WINDOW 64 /* largest window W */
#define FIB_MAX_LAYERS 256

/* Human-readable name of a status code (static storage; never NULL).  No counterpart in
 * the paper. */
const char* fib_attn_error_string(int code);

/* ---------------------------------------------------------------- host-only planner --
 * These run on the CPU only and need no GPU.                                           */

/* Base list f ("Attended set" / "Controls").  FIBONACCI: 1, 2, 3, 5, ..., 987 (15
 * entries, the repeated leading 1 dropped).  POW2: {2^k : 2^k < N} (reach-matched
 * control; N >= 2).  Writes min(count, cap) entries to out, the full count to *n_out.
 * FIB_ERR_INVALID_ARG on a bad kind, N < 2 for POW2, cap < 0 or null n_out.            */
int fib_attn_base(int base_kind, int N, int32_t* out, int cap, int* n_out);

/* Per-layer alpha ("Experimental variables").  FIXED: 1.  LINEAR: 0.5 + l/(L-1) in
 * binary64 (0.5 at layer 0, 1.5 at the last; L >= 2).  COPRIME: alpha_lin[(stride*l)
 * mod L] with gcd(stride, L) = 1 (the pages use stride 7, L = 16).  alpha_out holds
 * n_layers doubles.  FIB_ERR_INVALID_ARG on bad kind, L out of [1, FIB_MAX_LAYERS],
 * L < 2 for a ramp, or a stride not coprime with L.                                   */
int fib_attn_schedule(int kind, int n_layers, int stride, double* alpha_out);

/* MASK-path distances of one layer ("Scaling": d_k = alpha f_k): the sorted distinct
 * values round_half_even(alpha * f) with W <= d <= N-1.  Writes min(count, cap) to out,
 * count to *n_out.  FIB_ERR_INVALID_ARG on null pointers, n_base < 0, W < 1, N < 1,
 * alpha not finite or <= 0.                                                           */
int fib_attn_mask_distances(const int32_t* base, int n_base, double alpha, int W, int N,
                            int32_t* out, int cap, int* n_out);

/* INTERP-path rungs of one layer ("Implementation": linear interpolation between the
 * bracketing rows): for each distinct f (ascending) with d = alpha*f, W-1 < d <= N-1:
 * f, lo = floor(d), w = (float)(d - lo).  Same size/error rules as above.               */
int fib_attn_interp_rungs(const int32_t* base, int n_base, double alpha, int W, int N,
                          int32_t* f_out, int32_t* lo_out, float* w_out, int cap,
                          int* n_out);

/* ------------------------------------------------------------------------- plan ----
 * Defines the attended set of every layer of a stack: "Attended set" (a dense local window
 * of W keys plus the Fibonacci offsets), "Scaling" (d_k = alpha_l f_k with one alpha per
 * layer), "Experimental variables" (the per-layer alpha of a schedule, or a learned one),
 * "Controls" (the power-of-two base) and "Implementation" (RoPE before the gather).
 * A plan fixes (base, per-layer alpha, W, N_max, D, mode, RoPE base) for a layer stack
 * and uploads the RoPE tables (built in binary64 on the host, stored float32) for
 * positions < N_max to the current device.  base_kind CUSTOM reads custom_base[n_custom]
 * (positive integers); otherwise custom_base is ignored.  alpha[n_layers] is copied.
 * Constraints: 1 <= W <= FIB_MAX_WINDOW, 1 <= N_max <= 1<<20, D == 64
 * (else FIB_ERR_UNSUPPORTED), every alpha finite and > 0, rope_base > 1.
 * Errors: FIB_ERR_INVALID_ARG, FIB_ERR_UNSUPPORTED, FIB_ERR_NOMEM, FIB_ERR_CUDA.        */
int fib_attn_plan_create(fib_attn_plan_t* out, int base_kind, const int32_t* custom_base,
                         int n_custom, const double* alpha, int n_layers, int W, int N_max,
                         int D, int mode, double rope_base);

/* Frees the plan and its device tables (synchronises the device first).  NULL is OK.
 * No counterpart in the paper.                                                        */
int fib_attn_plan_destroy(fib_attn_plan_t p);

/* Host copy of the MASK distances (mode MASK) or INTERP lo values (mode INTERP) that the
 * plan uses for `layer` at sequence length N (N <= N_max): "Scaling" (d_k = alpha_l f_k)
 * after the readings above.                                                            */
int fib_attn_plan_distances(fib_attn_plan_t p, int layer, int N, int32_t* out, int cap,
                            int* n_out);

/* ---------------------------------------------------------------------- forward ----
 * The layer's sparse attention: "Attended set" and "Scaling" give the keys each query
 * attends, "Implementation" the RoPE before the gather and the interpolated rows of a
 * non-integer distance, Key results 2 > "Efficiency" the two paths (MASK: integer distances
 * as a fused boolean mask; INTERP: the interpolated gather).
 * O = attention output (dtype of the inputs), lse = natural-log sum of exp(scores),
 * both for layer `layer` of the plan at sequence length N (1 <= N <= N_max).
 * q, k, v, o: [B, H, N, 64] device, dtype `dtype`.  lse: [B, H, N] float32 device, or
 * NULL to skip writing it.  alpha_dev (INTERP only): device float32 alpha[n_layers]
 * (a learned parameter; element `layer` is used, exactly as a float32) or NULL to use
 * the plan's binary64 alpha.  MASK ignores alpha_dev.  O must not alias q, k or v.
 * workspace: device scratch of at least fib_attn_fwd_workspace_size(p, B, H, N, dtype)
 * bytes, 256-byte aligned, caller-owned, not overlapping q, k, v or o; its contents on
 * entry are ignored and on return are unspecified.  bf16 with W <= 16 needs B*H*N*256
 * bytes: the keys rotated to their own positions and the values, both as float16, which
 * the tensor-core kernel reads instead of k and v.  Where the size is 0 (float32, or a
 * window wider than 16), workspace may be NULL.
 * Errors: FIB_ERR_INVALID_ARG (null/misaligned pointers, sizes, layer, a short or
 * misaligned workspace), FIB_ERR_CUDA.                                                  */
size_t fib_attn_fwd_workspace_size(fib_attn_plan_t p, int B, int H, int N, int dtype);
int fib_attn_fwd(fib_attn_plan_t p, int layer, int B, int H, int N, int dtype,
                 const void* q, const void* k, const void* v, void* o, float* lse,
                 const float* alpha_dev, void* workspace, size_t ws_bytes, void* stream);

/* Float16 range of the bf16 tensor-core path (bf16 with W <= 16; forward and backward):
 * its operands are float16, so every value it converts must satisfy |x| <= 65504: the
 * keys after RoPE, the values, the queries after RoPE times log2(e)/8 and, in the
 * backward, dO and dS = P (dO . v~ - Delta).  A query, key, value or dO beyond that (or not
 * finite) makes the call record FIB_ERR_RANGE in the plan's status word (read with
 * fib_attn_last_device_status); the outputs of that call are then unspecified and may be
 * infinite or NaN.  Values below 6.1e-5 in magnitude are held as float16 subnormals
 * (absolute spacing 6e-8).  Float32 inputs and bf16 with W > 16 take the CUDA-core
 * kernels, which compute in float32 and have no such limit.
 *
 * The two halves of the bf16 forward, for callers that reuse the prepared keys and values
 * (several query sets against one K/V) or time the halves apart.  fib_attn_fwd(...) ==
 * fib_attn_fwd_prepare_kv then fib_attn_fwd_attend on the same stream, bit for bit.
 * prepare_kv writes into workspace (sized by fib_attn_fwd_workspace_size) K rotated at each
 * row's own position ("Implementation": RoPE is applied before the rows are gathered)
 * and V, both as float16 [B, H, N, 64]; its layout inside the workspace is private to the
 * library.  attend reads q and a workspace that prepare_kv filled for the same plan, B, H
 * and N (not checked) and writes o and lse as fib_attn_fwd.  Both return
 * FIB_ERR_UNSUPPORTED where the workspace size is 0 (float32, or W > 16), else the
 * errors of fib_attn_fwd.                                                              */
int fib_attn_fwd_prepare_kv(fib_attn_plan_t p, int B, int H, int N, int dtype, const void* k,
                            const void* v, void* workspace, size_t ws_bytes, void* stream);
int fib_attn_fwd_attend(fib_attn_plan_t p, int layer, int B, int H, int N, int dtype,
                        const void* q, const void* workspace, size_t ws_bytes, void* o,
                        float* lse, const float* alpha_dev, void* stream);

/* ------------------------------------------------------------------ dense control ----
 * Dense causal attention with the same RoPE and scale: every query i attends every key
 * j <= i (Methodology > "Controls": a dense model of the same architecture as the upper
 * bound; Key results 3: dense attention at 4x the training length).  It equals fib_attn_fwd
 * of a plan whose window covers the sequence (W >= N), but runs the dense blocked kernel.
 * The plan supplies only its RoPE tables (N <= N_max) and status word; its layers, window
 * and rungs play no part.  bf16 only (FIB_ERR_UNSUPPORTED for float32); q, k, v, o, lse
 * and the errors as fib_attn_fwd; workspace: at least
 * fib_attn_dense_fwd_workspace_size(p, B, H, N, dtype) bytes (B*H*N*256 for bf16, the
 * rotated keys and the values as float16), 256-byte aligned, caller-owned.  The float16
 * range rule of the bf16 path applies.                                                  */
size_t fib_attn_dense_fwd_workspace_size(fib_attn_plan_t p, int B, int H, int N, int dtype);
int fib_attn_dense_fwd(fib_attn_plan_t p, int B, int H, int N, int dtype, const void* q,
                       const void* k, const void* v, void* o, float* lse, void* workspace,
                       size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------ decode ----
 * One new token per (b, h) against a KV cache (Key results 2, "Efficiency": inference
 * latency of the mask and the interpolated path).  The token sits at position pos of a
 * sequence of length N (0 <= pos < N <= N_max) and attends exactly what row pos of
 * fib_attn_fwd at length N attends (N matters for the power-of-two base only).
 * q: [B, H, 64] raw (unrotated) query; k_cache, v_cache: [B, H, N, 64] raw rows, of which
 * rows 0..pos are read; o: [B, H, 64]; lse: [B, H] float32 or NULL.  Dtype and alpha_dev
 * as fib_attn_fwd.  Errors as fib_attn_fwd, plus FIB_ERR_INVALID_ARG for pos outside
 * [0, N).                                                                              */
int fib_attn_decode(fib_attn_plan_t p, int layer, int B, int H, int N, int pos, int dtype,
                    const void* q, const void* k_cache, const void* v_cache, void* o, float* lse,
                    const float* alpha_dev, void* stream);

/* --------------------------------------------------------------------- backward ----
 * "Implementation": the interpolated rows make the output differentiable in alpha, and
 * "Experimental variables" > learned: alpha is then a trained per-layer parameter.
 * Gradients of l = sum(O * dO) for one layer, given the forward's o and lse.
 * dq, dk, dv: [B, H, N, 64] device (dtype of the inputs), fully written.
 * dalpha: device float32 scalar, written (not accumulated) with dl/dalpha_layer in
 * INTERP mode and 0 in MASK mode (static distances carry no alpha gradient).
 * workspace: device scratch of at least fib_attn_bwd_workspace_size(p, B, H, N) bytes,
 * 256-byte aligned, caller-owned; its contents on entry are ignored.  The size is the same
 * for both dtypes: for a plan with W <= 16 it is what the bf16 path needs (Q, K, V, dO
 * prepared once as float16 rows, B*H*N*512 bytes; Delta; the (P, dS) float pair of every
 * attended (query, key slot); the dalpha partials); the float32 path uses only its first
 * B*H*N*4 bytes and the partials.
 * Streams: on the bf16 tensor-core path with B*H >= 2, the second half of the (b, h) rows
 * runs on a stream the plan owns, forked from `stream` and joined back to it with events
 * before the call returns (so that work enqueued on `stream` afterwards, and a stream
 * capture of `stream`, see the whole backward); one plan's backward calls from several host
 * threads take turns to enqueue, and their device work must not overlap (the same stream,
 * or ordered by the caller).
 * Errors as fib_attn_fwd, plus FIB_ERR_INVALID_ARG for a short/misaligned workspace.  */
size_t fib_attn_bwd_workspace_size(fib_attn_plan_t p, int B, int H, int N);
int fib_attn_bwd(fib_attn_plan_t p, int layer, int B, int H, int N, int dtype,
                 const void* q, const void* k, const void* v, const void* o,
                 const float* lse, const void* dO, void* dq, void* dk, void* dv,
                 float* dalpha, const float* alpha_dev, void* workspace, size_t ws_bytes,
                 void* stream);

/* Backward from the forward's prepared rows.  K' (RoPE at each row's own position) and V'
 * as float16 rows are what the bf16 forward prepares in its workspace and what the bf16
 * backward needs of k and v ("Implementation": RoPE is applied before the rows are
 * gathered, in both passes); a training step that keeps that workspace from the layer's
 * forward (fib_attn_fwd or fib_attn_fwd_prepare_kv of the same plan, B, H, N and the same k
 * and v, not checked) hands it over here instead of k and v, and the backward prepares
 * only Q', dO' and Delta.  Results equal those of fib_attn_bwd on the same inputs up to the
 * float16 rounding of K' (the forward builds the RoPE factors of two rows in three by a
 * recurrence, the backward's own preparation reads them from the tables, so a K' element
 * can differ in its last bit); both are deterministic.  kv_prepared: that workspace, of
 * kv_bytes >= fib_attn_fwd_workspace_size(p, B, H, N, dtype), 256-byte aligned, read only.
 * Everything else as fib_attn_bwd, plus
 * FIB_ERR_UNSUPPORTED where the forward has no prepared rows (float32, or W > 16: call
 * fib_attn_bwd there) and FIB_ERR_INVALID_ARG for a short or misaligned kv_prepared or one
 * that is the backward workspace or an output.                                          */
int fib_attn_bwd_prepared(fib_attn_plan_t p, int layer, int B, int H, int N, int dtype,
                          const void* q, const void* kv_prepared, size_t kv_bytes, const void* o,
                          const float* lse, const void* dO, void* dq, void* dk, void* dv,
                          float* dalpha, const float* alpha_dev, void* workspace, size_t ws_bytes,
                          void* stream);

/* Backward without allocation.  The paper has no counterpart: this is an interface for
 * callers that cannot allocate device memory on the call path -- for example a plugin inside
 * a framework that owns the device heap, or a real-time loop that forbids allocation -- and
 * so cannot hand fib_attn_bwd a workspace.  Same arguments, results and errors as
 * fib_attn_bwd without workspace/ws_bytes (for bf16 within fib_attn_bwd's bound, not bit for
 * bit: this entry point always runs the CUDA-core kernels, which need no prepared rows): the
 * scratch is a fixed 8 MiB device array inside the library, held on every device that
 * loads it until the process exits.  A call whose CUDA-core scratch (4 bytes per
 * query-head plus 4 per 64-query tile) exceeds 8 MiB, i.e. B*H*N above about two million,
 * returns FIB_ERR_INVALID_ARG before any launch.  Every call looks up the array's device
 * address on the current device (cudaGetSymbolAddress, host-side work); the first call on a
 * device may also load the library's device code there, so make that first call before any
 * stream capture.  The address is not cached, so a call after a device reset still finds
 * the array.  Every call shares the array and it keeps the last call's contents (nothing
 * in it needs zeroing); calls whose kernels overlap on the GPU race on it.  Nothing is
 * allocated, by the library or through CUDA.                                              */
int fib_attn_bwd_noalloc(fib_attn_plan_t p, int layer, int B, int H, int N, int dtype,
                         const void* q, const void* k, const void* v, const void* o,
                         const float* lse, const void* dO, void* dq, void* dk, void* dv,
                         float* dalpha, const float* alpha_dev, void* stream);

/* ---------------------------------------------------------------- debug / status ----
 * The attended index sets ("Attended set"; INTERP: the two bracketing rows of
 * "Implementation") of queries [i_begin, i_end), produced by the same device
 * index code as the forward kernel.  out_dev: int32 [(i_end-i_begin), W + FIB_MAX_RUNGS]
 * device; slot s < W holds the window row i-s, slot W+r holds rung r's row (MASK: i-d;
 * INTERP: i-lo, whose partner row i-lo-1 carries weight w), -1 where not attended.
 * w_out_dev: float32 [FIB_MAX_RUNGS] device (INTERP weights; 0 for MASK) or NULL.
 * alpha_dev as fib_attn_fwd (INTERP: the device float32 alpha the forward would use, or
 * NULL for the plan's).  Errors: FIB_ERR_INVALID_ARG (layer, N, an empty or out-of-range
 * query range, misaligned pointers), FIB_ERR_CUDA.                                      */
int fib_attn_debug_indices(fib_attn_plan_t p, int layer, int N, int i_begin, int i_end,
                           int32_t* out_dev, float* w_out_dev, const float* alpha_dev,
                           void* stream);

/* Wait bound and test hooks of the plan's kernels (no counterpart in the paper: they
 * exist so that the error paths can be driven without any device fault).  Kernels that
 * stage rows with the bulk-copy engine wait on mbarriers; every such wait gives up after
 * wait_ns nanoseconds (default 1e9; accepted range [1e3, 6e10]), records FIB_ERR_TIMEOUT in
 * the status word, lets the copies already in flight land and returns without writing
 * output.  debug_flags: FIB_DEBUG_SKIP_COPY makes the bf16 tensor-core forward never
 * complete one of its staged copies (the values of the window block), which drives that
 * timeout path; FIB_DEBUG_CORRUPT_TABLE moves the first rung of the bf16 tensor-core
 * forward's host-built rung table to distance 0 (a row inside the window, so every address
 * stays inside the sequence), which its device-side table check rejects with
 * FIB_ERR_DEVICE_ASSERT before any rung row is read.  Host-only; takes effect on the next
 * launch.  FIB_ERR_INVALID_ARG on a null plan, an unknown flag or wait_ns out of range.   */
int fib_attn_plan_set_debug(fib_attn_plan_t p, int debug_flags, long long wait_ns);

/* Test hook (no counterpart in the paper): fills the shared memory of every SM of the current
 * device with the 32-bit `pattern` (one kernel taking each SM's whole shared memory), so that
 * a test can check that no kernel lets stale shared memory reach its outputs (a pattern of
 * 0x7fc00000 is a float NaN).  Enqueued on `stream`; allocates nothing.  FIB_ERR_CUDA on a
 * failed launch.                                                                       */
int fib_attn_debug_fill_shared(uint32_t pattern, void* stream);

/* Synchronises the plan's device, then returns and clears the device status word (no
 * counterpart in the paper): FIB_OK, FIB_ERR_TIMEOUT (a bounded wait gave up),
 * FIB_ERR_DEVICE_ASSERT (the tensor-core forward's check of its rung table: every rung
 * beyond the window and inside the sequence, in ascending order) or FIB_ERR_RANGE (a value
 * outside the float16 range, see fib_attn_fwd).  Where several calls recorded a code, the
 * last one written is returned.                                                        */
int fib_attn_last_device_status(fib_attn_plan_t p);

#ifdef __cplusplus
}
#endif
#endif /* FIB_ATTN_H */
