"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle on seeded inputs.

Tolerances:
  * index sets: bit-exact;
  * O: max-abs <= 1e-5 for float32 inputs; <= 1e-2 for bf16 inputs (float32 accumulation)
    against the oracle run on the same bf16-rounded values, plus the bf16 output's own
    rounding (at most half an ulp, bounded by 2^-8 |O|);
  * LSE (float32 output): 1e-5 (float32 inputs); 5e-3 for bf16 inputs: the tensor-core
    path rounds the RoPE-rotated Q' and K' to f16 (11-bit significand) for the window and
    every rung, so a 64-term score carries up to ~1e-3 of rounding error, which LSE
    inherits (the O bound above is the binding one);
  * dQ, dK, dV: relative L2 <= 2e-2;
  * dalpha (one scalar, a sum over batch rows and heads of contributions of both signs):
    |error| <= 2e-2 times the larger of |dalpha| and the root-sum-square of its per-(b, h)
    contributions, all from the oracle.  Where the heads' contributions cancel, |dalpha|
    measures the cancellation rather than the kernel (in one seeded case four contributions
    of 34e3, -19e3, -28e3 and 15e3 sum to 1.0e3, and rounding the forward's O to bf16 alone
    moves that sum by 0.8 %), so the bound takes the scale of the contributions.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from fibonacci_offset_sparse_gb300 import fib_attn as fa
from fibonacci_offset_sparse_gb300 import inputs

pytestmark = pytest.mark.gpu

F32_ATOL = 1e-5
BF16_ATOL = 1e-2
REL_L2 = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from fibonacci_offset_sparse_gb300 import build as b
    import os
    if not os.path.exists(b.LIB):
        b.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return fa.lib()


def _base_fn(kind):
    if kind == "fib":
        return lambda N: oracle.fibonacci_base()
    if kind == "pow2":
        return oracle.pow2_base
    return lambda N: list(kind)


def _plan(kind, alphas, W, N_max, mode):
    bk = {"fib": fa.FIB_BASE_FIBONACCI, "pow2": fa.FIB_BASE_POW2}.get(kind, fa.FIB_BASE_CUSTOM)
    custom = None if bk != fa.FIB_BASE_CUSTOM else list(kind)
    m = fa.FIB_MODE_MASK if mode == "mask" else fa.FIB_MODE_INTERP
    return fa.fib_attn_plan_create(bk, alphas, W, N_max, m, custom_base=custom)


_LOG = os.environ.get("FIB_PARITY_LOG")


def _record(kind, what, value):
    if _LOG:
        with open(_LOG, "a") as f:
            f.write(json.dumps({"check": kind, "case": what, "value": float(value)}) + "\n")


def _check_o(o_gpu, O_ref, dtype, what=""):
    og = o_gpu.detach().double().cpu().numpy()
    err = np.abs(og - O_ref)
    _record("o_maxabs_" + dtype, what, err.max())
    if dtype != "f32":
        _record("o_excess_over_rounding_" + dtype, what, (err - np.abs(O_ref) * 2.0 ** -8).max())
    if dtype == "f32":
        assert err.max() <= F32_ATOL, f"{what} max-abs {err.max():.3e}"
    else:
        bound = BF16_ATOL + np.abs(O_ref) * 2.0 ** -8
        assert np.all(err <= bound), f"{what} max-abs {err.max():.3e} (worst excess {(err - bound).max():.3e})"
    return err.max()


def _check_lse(lse_gpu, lse_ref, dtype, what=""):
    lg = lse_gpu.detach().double().cpu().numpy()
    tol = 1e-5 if dtype == "f32" else 5e-3
    err = np.abs(lg - lse_ref).max()
    _record("lse_maxabs_" + dtype, what, err)
    assert err <= tol, f"{what} lse max-abs {err:.3e}"


def _rel_l2(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def _oracle_bwd(qf, kf, vf, gf, alpha, base, W, mode):
    """The oracle's gradients, one (b, h) at a time (each head is independent): dq, dk, dv,
    dalpha (the sum over heads) and the root-sum-square of the per-head dalpha contributions."""
    B, H = qf.shape[:2]
    rq, rk, rv = np.zeros_like(qf), np.zeros_like(kf), np.zeros_like(vf)
    per = []
    for b in range(B):
        for h in range(H):
            sl = (slice(b, b + 1), slice(h, h + 1))
            gq, gk, gv, ga = oracle.attend_bwd(qf[sl], kf[sl], vf[sl], gf[sl], alpha, base, W, mode)
            rq[sl], rk[sl], rv[sl] = gq, gk, gv
            per.append(ga)
    return rq, rk, rv, float(sum(per)), float(np.sqrt(np.sum(np.square(per))))


def _check_dalpha(da, ra, rss, what):
    err = abs(float(da.item()) - ra)
    scale = max(abs(ra), rss)
    _record("bwd_rel_dalpha", what, err / max(scale, 1e-30))
    assert err <= REL_L2 * scale, f"{what} dalpha {da.item()} vs {ra} (per-head rss {rss:.4g})"


def _run_fwd(kind, alphas, W, B, H, N, dtype, mode, layers, config, alpha_dev=None, heads=None):
    """Forward of every listed layer at the full shape; the oracle on all heads, or on the
    head slice `heads` (a slice, or a function of the layer giving one)."""
    plan = _plan(kind, alphas, W, N, mode)
    adev = None if alpha_dev is None else torch.tensor(alpha_dev, dtype=torch.float32, device="cuda")
    for layer in layers:
        q, k, v = inputs.qkv(B, H, N, 64, config, layer, dtype)
        o, lse = fa.fib_attn_fwd(plan, layer, q.cuda(), k.cuda(), v.cuda(), alpha_dev=adev)
        torch.cuda.synchronize()
        assert fa.fib_attn_last_device_status(plan) == fa.FIB_OK
        a = alphas[layer] if alpha_dev is None else float(np.float32(alpha_dev[layer]))
        hs = slice(None) if heads is None else (heads(layer) if callable(heads) else heads)
        O_ref, lse_ref = oracle.attend(inputs.as_f64(q[:, hs]), inputs.as_f64(k[:, hs]),
                                       inputs.as_f64(v[:, hs]), a, _base_fn(kind)(N), W, mode)
        _check_o(o[:, hs], O_ref, dtype, f"layer {layer}")
        _check_lse(lse[:, hs], lse_ref, dtype, f"layer {layer}")
    plan.close()


# ------------------------------------------------------------------ the five workloads
def test_c0_fp32_mask_alpha1():
    """1 layer, B=1, H=1, N=256, fp32, W=8, Fibonacci, alpha=1 (mask path)."""
    _run_fwd("fib", [1.0], 8, 1, 1, 256, "f32", "mask", [0], 0)
    # the interpolated path at alpha = 1 reduces to the mask path
    _run_fwd("fib", [1.0], 8, 1, 1, 256, "f32", "interp", [0], 0)


def test_c1_linear_stack_bf16():
    """16 layers, B=8, H=8, N=1024, bf16, W=12, Fibonacci, linear schedule, mask path."""
    _run_fwd("fib", oracle.schedule("linear", 16), 12, 8, 8, 1024, "bf16", "mask", range(16), 1)


@pytest.mark.parametrize("kind", ["fib", "pow2"])
def test_c2_coprime_extrapolation_bf16(kind):
    """16 layers, B=2, H=8, N=4096, bf16, W=12, coprime schedule: every layer's forward at
    the full shape (each layer its own alpha and rung table, 8 to 11 rungs), O and LSE against
    the oracle on two of the eight heads of both batch rows, a different pair per layer, so
    that the 16 layers cover every head twice."""
    _run_fwd(kind, oracle.schedule("coprime", 16), 12, 2, 8, 4096, "bf16", "mask",
             range(16), 2 if kind == "fib" else 12, heads=lambda l: slice(2 * (l % 4), 2 * (l % 4) + 2))


@pytest.mark.parametrize("mode", ["mask", "interp"])
def test_c4_long_context_bf16(mode):
    """1 layer, B=1, H=8, N=131072, bf16, W=12, alpha=1.5; oracle on two heads."""
    _run_fwd("fib", [1.5], 12, 1, 8, 131072, "bf16", mode, [0], 4, heads=slice(2, 4))


def test_c3_learned_fwd_bwd_bf16():
    """16 layers, B=8, H=8, N=1024, bf16, W=10, alpha ~ U[0.9, 1.1] (device float32),
    interp forward + backward; layers sampled."""
    L, B, H, N, W = 16, 8, 8, 1024, 10
    alpha = inputs.learned_alpha(L, 3)
    plan = _plan("fib", [1.0] * L, W, N, "interp")
    adev = torch.tensor(alpha, dtype=torch.float32, device="cuda")
    for layer in (0, 5, 11):
        q, k, v = inputs.qkv(B, H, N, 64, 3, layer, "bf16")
        dO = inputs.upstream_grad(B, H, N, 64, 3, layer, "bf16")
        qc, kc, vc, dOc = q.cuda(), k.cuda(), v.cuda(), dO.cuda()
        o, lse = fa.fib_attn_fwd(plan, layer, qc, kc, vc, alpha_dev=adev)
        dq, dk, dv, da = fa.fib_attn_bwd(plan, layer, qc, kc, vc, o, lse, dOc, alpha_dev=adev)
        torch.cuda.synchronize()
        a = float(alpha[layer])
        qf, kf, vf, gf = (inputs.as_f64(x) for x in (q, k, v, dO))
        O_ref, lse_ref = oracle.attend(qf, kf, vf, a, oracle.fibonacci_base(), W, "interp")
        _check_o(o, O_ref, "bf16", f"layer {layer}")
        _check_lse(lse, lse_ref, "bf16")
        # the backward consumes the kernel's bf16 O; the oracle differentiates its own forward
        rq, rk, rv, ra, rss = _oracle_bwd(qf, kf, vf, gf, a, oracle.fibonacci_base(), W, "interp")
        for name, g, r in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
            e = _rel_l2(g.double().cpu().numpy(), r)
            _record("bwd_rel_l2_" + name, f"c3 layer {layer}", e)
            assert e <= REL_L2, f"layer {layer} {name} rel-L2 {e:.3e}"
        _check_dalpha(da, ra, rss, f"c3 layer {layer}")
    plan.close()


def test_c3_every_layer_fwd_bwd_bf16():
    """The learned-dilation training step of every one of the 16 layers (W=10, Fibonacci,
    alpha ~ U[0.9, 1.1] on the device, interp forward + backward), at N=1024 with B=2, H=2 so
    that the oracle's full backward (dalpha sums every head) stays cheap: O, LSE, dQ, dK, dV
    and dalpha of each layer against the oracle."""
    L, B, H, N, W = 16, 2, 2, 1024, 10
    alpha = inputs.learned_alpha(L, 3)
    plan = _plan("fib", [1.0] * L, W, N, "interp")
    adev = torch.tensor(alpha, dtype=torch.float32, device="cuda")
    for layer in range(L):
        q, k, v = inputs.qkv(B, H, N, 64, 31, layer, "bf16")
        dO = inputs.upstream_grad(B, H, N, 64, 31, layer, "bf16")
        qc, kc, vc, dOc = q.cuda(), k.cuda(), v.cuda(), dO.cuda()
        o, lse = fa.fib_attn_fwd(plan, layer, qc, kc, vc, alpha_dev=adev)
        dq, dk, dv, da = fa.fib_attn_bwd(plan, layer, qc, kc, vc, o, lse, dOc, alpha_dev=adev)
        torch.cuda.synchronize()
        assert fa.fib_attn_last_device_status(plan) == fa.FIB_OK
        a = float(alpha[layer])
        qf, kf, vf, gf = (inputs.as_f64(x) for x in (q, k, v, dO))
        O_ref, lse_ref = oracle.attend(qf, kf, vf, a, oracle.fibonacci_base(), W, "interp")
        _check_o(o, O_ref, "bf16", f"c3 sweep layer {layer}")
        _check_lse(lse, lse_ref, "bf16", f"c3 sweep layer {layer}")
        rq, rk, rv, ra, rss = _oracle_bwd(qf, kf, vf, gf, a, oracle.fibonacci_base(), W, "interp")
        for name, g, r in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
            e = _rel_l2(g.double().cpu().numpy(), r)
            _record("bwd_rel_l2_" + name, f"c3 sweep layer {layer}", e)
            assert e <= REL_L2, f"layer {layer} {name} rel-L2 {e:.3e}"
        _check_dalpha(da, ra, rss, f"c3 sweep layer {layer}")
    plan.close()


# ------------------------------------------------------------------ index sets (bit-exact)
def _check_indices(kind, alphas, W, N, mode, layers, alpha_dev=None, ranges=None):
    plan = _plan(kind, alphas, W, N, mode)
    adev = None if alpha_dev is None else torch.tensor(alpha_dev, dtype=torch.float32, device="cuda")
    for layer in layers:
        a = alphas[layer] if alpha_dev is None else float(np.float32(alpha_dev[layer]))
        ref = oracle.index_sets(_base_fn(kind)(N), a, W, N, mode)
        for (i0, i1) in (ranges or [(0, N)]):
            rows, w = fa.fib_attn_debug_indices(plan, layer, N, i0, i1, alpha_dev=adev)
            rows = rows.cpu().numpy()
            w = w.cpu().numpy()
            keys = oracle.virtual_keys(_base_fn(kind)(N), a, W, N, mode)
            nr = len(keys) - W
            for (_, _, wk, _), wg in zip(keys[W:], w[:nr]):
                assert wg == np.float32(wk)
            for i in range(i0, i1):
                got = [(int(x), float(w[s - W]) if s >= W else 0.0)
                       for s, x in enumerate(rows[i - i0]) if x >= 0]
                want = [(r, float(np.float32(ww))) for (r, ww) in ref[i]]
                assert got == want, (layer, i)
    plan.close()


def test_indices_c0_and_c1():
    _check_indices("fib", [1.0], 8, 256, "mask", [0])
    _check_indices("fib", oracle.schedule("linear", 16), 12, 1024, "mask", range(16))


@pytest.mark.parametrize("kind", ["fib", "pow2"])
def test_indices_c2(kind):
    _check_indices(kind, oracle.schedule("coprime", 16), 12, 4096, "mask", range(16),
                   ranges=[(0, 40), (1000, 1100), (4000, 4096)])


def test_indices_c3_device_alpha_and_c4():
    a = inputs.learned_alpha(16, 3)
    _check_indices("fib", [1.0] * 16, 10, 1024, "interp", range(16), alpha_dev=a)
    for mode in ("mask", "interp"):
        _check_indices("fib", [1.5], 12, 131072, mode, [0],
                       ranges=[(0, 64), (1470, 1500), (131000, 131072)])


# ------------------------------------------------------------------ edge cases, fp32
@pytest.mark.parametrize("mode", ["mask", "interp"])
@pytest.mark.parametrize("N,W,alpha,kind", [
    (1, 12, 1.0, "fib"),            # a single query
    (7, 12, 1.3, "fib"),            # N < W
    (65, 8, 0.5, "fib"),            # one full tile + a ragged tail of 1
    (200, 1, 1.5, "fib"),           # window of one (self only)
    (300, 64, 1.2345, "fib"),       # largest window
    (257, 6, 0.77, "pow2"),         # power-of-two base
    (150, 4, 1.0, (37,)),           # single-rung custom base
    (129, 12, 0.5 + 9 / 15, "fib"),  # alpha = binary64 1.1 (rounding canary)
])
def test_edge_cases_fp32(mode, N, W, alpha, kind):
    B, H = 2, 3
    plan = _plan(kind, [alpha], W, N, mode)
    q, k, v = inputs.qkv(B, H, N, 64, 100 + N, W, "f32")
    o, lse = fa.fib_attn_fwd(plan, 0, q.cuda(), k.cuda(), v.cuda())
    torch.cuda.synchronize()
    O_ref, lse_ref = oracle.attend(inputs.as_f64(q), inputs.as_f64(k), inputs.as_f64(v), alpha,
                                   _base_fn(kind)(N), W, mode)
    _check_o(o, O_ref, "f32")
    _check_lse(lse, lse_ref, "f32")
    plan.close()


@pytest.mark.parametrize("mode,alpha", [("interp", 1.2345), ("interp", 0.6789), ("interp", 1.0),
                                        ("mask", 0.5 + 4 / 15)])
@pytest.mark.parametrize("device_alpha", [False, True])
def test_backward_fp32(mode, alpha, device_alpha):
    B, H, N, W = 2, 2, 333, 8
    if device_alpha:
        alpha = float(np.float32(alpha))
    plan = _plan("fib", [alpha], W, N, mode)
    q, k, v = inputs.qkv(B, H, N, 64, 200, 0, "f32")
    dO = inputs.upstream_grad(B, H, N, 64, 200, 0, "f32")
    adev = torch.tensor([alpha], dtype=torch.float32, device="cuda") if device_alpha else None
    qc, kc, vc, dOc = q.cuda(), k.cuda(), v.cuda(), dO.cuda()
    o, lse = fa.fib_attn_fwd(plan, 0, qc, kc, vc, alpha_dev=adev)
    dq, dk, dv, da = fa.fib_attn_bwd(plan, 0, qc, kc, vc, o, lse, dOc, alpha_dev=adev)
    torch.cuda.synchronize()
    qf, kf, vf, gf = (inputs.as_f64(x) for x in (q, k, v, dO))
    rq, rk, rv, ra = oracle.attend_bwd(qf, kf, vf, gf, alpha, oracle.fibonacci_base(), W, mode)
    for name, g, r in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        e = _rel_l2(g.double().cpu().numpy(), r)
        assert e <= 1e-5, f"{name} rel-L2 {e:.3e}"
    if mode == "mask":
        assert float(da.item()) == 0.0
    else:
        assert abs(float(da.item()) - ra) <= 1e-4 * abs(ra) + 1e-4, (float(da.item()), ra)
    # deterministic: a second run gives identical bits
    dq2, dk2, dv2, da2 = fa.fib_attn_bwd(plan, 0, qc, kc, vc, o, lse, dOc, alpha_dev=adev)
    torch.cuda.synchronize()
    assert torch.equal(dq, dq2) and torch.equal(dk, dk2) and torch.equal(dv, dv2) and torch.equal(da, da2)
    plan.close()


@pytest.mark.parametrize("mode,alpha,W,N", [("mask", 0.5 + 4 / 15, 12, 1000), ("mask", 1.5, 16, 333),
                                             ("mask", 1.0, 1, 200), ("interp", 1.2345, 8, 1000),
                                             ("interp", 0.6789, 16, 333), ("interp", 1.0, 10, 517),
                                             ("interp", 1.5, 1, 130)])
@pytest.mark.parametrize("device_alpha", [False, True])
def test_backward_bf16_tensor_core(mode, alpha, W, N, device_alpha):
    """The bf16 backward (tensor-core path for W <= 16) against the oracle's gradients of its
    own forward: relative L2 of dQ, dK, dV and dalpha; ragged N (not a multiple of the 64-row
    tiles), windows 1..16, alpha = 1.0 (every interp weight 0: the partner-row term of
    dalpha), and a second run that must give identical bits."""
    B, H = 2, 2
    if device_alpha:
        alpha = float(np.float32(alpha))
    plan = _plan("fib", [alpha], W, N, mode)
    q, k, v = inputs.qkv(B, H, N, 64, 210, 0, "bf16")
    dO = inputs.upstream_grad(B, H, N, 64, 210, 0, "bf16")
    adev = torch.tensor([alpha], dtype=torch.float32, device="cuda") if device_alpha else None
    qc, kc, vc, dOc = q.cuda(), k.cuda(), v.cuda(), dO.cuda()
    o, lse = fa.fib_attn_fwd(plan, 0, qc, kc, vc, alpha_dev=adev)
    dq, dk, dv, da = fa.fib_attn_bwd(plan, 0, qc, kc, vc, o, lse, dOc, alpha_dev=adev)
    torch.cuda.synchronize()
    assert fa.fib_attn_last_device_status(plan) == fa.FIB_OK
    qf, kf, vf, gf = (inputs.as_f64(x) for x in (q, k, v, dO))
    rq, rk, rv, ra, rss = _oracle_bwd(qf, kf, vf, gf, alpha, oracle.fibonacci_base(), W, mode)
    what = f"{mode} alpha={alpha} W={W} N={N}"
    for name, g, r in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        e = _rel_l2(g.double().cpu().numpy(), r)
        _record("bwd_rel_l2_" + name, what, e)
        assert e <= REL_L2, f"{what} {name} rel-L2 {e:.3e}"
    if mode == "mask":
        assert float(da.item()) == 0.0
    else:
        _check_dalpha(da, ra, rss, what)
    dq2, dk2, dv2, da2 = fa.fib_attn_bwd(plan, 0, qc, kc, vc, o, lse, dOc, alpha_dev=adev)
    torch.cuda.synchronize()
    assert torch.equal(dq, dq2) and torch.equal(dk, dk2) and torch.equal(dv, dv2) and torch.equal(da, da2)
    plan.close()


@pytest.mark.parametrize("mode,alpha,W,N", [("mask", 0.9, 17, 333), ("interp", 1.2345, 17, 517),
                                             ("mask", 1.37, 24, 300), ("interp", 0.7771, 24, 401)])
def test_backward_bf16_cuda_core(mode, alpha, W, N):
    """bf16 with a window wider than 16 takes the CUDA-core forward and backward (float32
    arithmetic on the bf16 values): gradients against the oracle's, ragged N, and a second run
    with identical bits."""
    B, H = 2, 2
    plan = _plan("fib", [alpha], W, N, mode)
    q, k, v = inputs.qkv(B, H, N, 64, 220, W, "bf16")
    dO = inputs.upstream_grad(B, H, N, 64, 220, W, "bf16")
    qc, kc, vc, dOc = q.cuda(), k.cuda(), v.cuda(), dO.cuda()
    o, lse = fa.fib_attn_fwd(plan, 0, qc, kc, vc)
    dq, dk, dv, da = fa.fib_attn_bwd(plan, 0, qc, kc, vc, o, lse, dOc)
    torch.cuda.synchronize()
    qf, kf, vf, gf = (inputs.as_f64(x) for x in (q, k, v, dO))
    O_ref, _ = oracle.attend(qf, kf, vf, alpha, oracle.fibonacci_base(), W, mode)
    _check_o(o, O_ref, "bf16", f"cuda-core {mode} W={W}")
    rq, rk, rv, ra, rss = _oracle_bwd(qf, kf, vf, gf, alpha, oracle.fibonacci_base(), W, mode)
    what = f"cuda-core {mode} alpha={alpha} W={W} N={N}"
    for name, g, r in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        e = _rel_l2(g.double().cpu().numpy(), r)
        _record("bwd_rel_l2_" + name, what, e)
        assert e <= REL_L2, f"{what} {name} rel-L2 {e:.3e}"
    if mode == "mask":
        assert float(da.item()) == 0.0
    else:
        _check_dalpha(da, ra, rss, what)
    dq2, dk2, dv2, da2 = fa.fib_attn_bwd(plan, 0, qc, kc, vc, o, lse, dOc)
    torch.cuda.synchronize()
    assert torch.equal(dq, dq2) and torch.equal(dk, dk2) and torch.equal(dv, dv2) and torch.equal(da, da2)
    plan.close()


# ------------------------------------------------------------------ error paths on a GPU
def test_device_error_paths():
    plan = _plan("fib", [1.0, 1.0], 12, 256, "mask")
    lib = fa.lib()
    B, H, N = 1, 2, 128
    q = torch.zeros(B, H, N, 64, device="cuda")
    o = torch.empty_like(q)
    s = torch.cuda.current_stream().cuda_stream

    def fwd(layer=0, n=N, dtype=0, qp=None, op=None, lsep=None, wsp=None, ws_bytes=0):
        return lib.fib_attn_fwd(plan.handle, layer, B, H, n, dtype, qp or q.data_ptr(), q.data_ptr(),
                                q.data_ptr(), op or o.data_ptr(), lsep, None, wsp, ws_bytes, s)

    assert fwd() == fa.FIB_OK
    assert fwd(layer=2) == fa.FIB_ERR_INVALID_ARG            # layer out of range
    assert fwd(layer=-1) == fa.FIB_ERR_INVALID_ARG
    assert fwd(n=257) == fa.FIB_ERR_INVALID_ARG              # N > N_max
    assert fwd(n=0) == fa.FIB_ERR_INVALID_ARG
    assert fwd(dtype=5) == fa.FIB_ERR_INVALID_ARG
    assert fwd(qp=q.data_ptr() + 4) == fa.FIB_ERR_INVALID_ARG   # misaligned
    assert fwd(op=q.data_ptr()) == fa.FIB_ERR_INVALID_ARG       # o aliases q
    assert fwd(lsep=q.data_ptr() + 2) == fa.FIB_ERR_INVALID_ARG
    # bf16 needs the K'/V' workspace: null, short, misaligned or aliasing an input is refused
    assert fa.fib_attn_fwd_workspace_size(plan, B, H, N, torch.float32) == 0
    fneed = fa.fib_attn_fwd_workspace_size(plan, B, H, N, torch.bfloat16)
    assert fneed == B * H * N * 256
    fws = torch.empty(fneed + 256, dtype=torch.uint8, device="cuda")
    bf = fa.FIB_DTYPE_BF16
    assert fwd(dtype=bf) == fa.FIB_ERR_INVALID_ARG
    assert fwd(dtype=bf, wsp=fws.data_ptr(), ws_bytes=fneed - 1) == fa.FIB_ERR_INVALID_ARG
    assert fwd(dtype=bf, wsp=fws.data_ptr() + 16, ws_bytes=fneed) == fa.FIB_ERR_INVALID_ARG
    assert fwd(dtype=bf, wsp=q.data_ptr(), ws_bytes=fneed) == fa.FIB_ERR_INVALID_ARG
    assert fwd(dtype=bf, wsp=fws.data_ptr(), ws_bytes=fneed) == fa.FIB_OK
    ws_need = fa.fib_attn_bwd_workspace_size(plan, B, H, N)
    ws = torch.empty(ws_need, dtype=torch.uint8, device="cuda")
    lse = torch.empty(B, H, N, device="cuda")
    g = [torch.empty_like(q) for _ in range(3)]
    da = torch.empty(1, device="cuda")
    args = [plan.handle, 0, B, H, N, 0, q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(),
            lse.data_ptr(), q.data_ptr(), g[0].data_ptr(), g[1].data_ptr(), g[2].data_ptr(),
            da.data_ptr(), None, ws.data_ptr()]
    assert lib.fib_attn_bwd(*args, ws_need - 1, s) == fa.FIB_ERR_INVALID_ARG   # short workspace
    bad = list(args)
    bad[-1] = ws.data_ptr() + 16
    assert lib.fib_attn_bwd(*bad, ws_need, s) == fa.FIB_ERR_INVALID_ARG        # misaligned ws
    assert lib.fib_attn_bwd(*args, ws_need, s) == fa.FIB_OK
    assert fa.fib_attn_last_device_status(plan) == fa.FIB_OK
    plan.close()


# ------------------------------------------------------------------ edge cases, bf16
@pytest.mark.parametrize("mode", ["mask", "interp"])
@pytest.mark.parametrize("N,W,alpha,kind", [
    (1, 12, 1.0, "fib"),            # a single query
    (15, 12, 1.3, "fib"),           # less than one warp tile
    (65, 16, 0.5, "fib"),           # widest window on tensor cores; ragged tail of 1
    (77, 17, 0.9, "fib"),           # W = 17: CUDA-core kernel
    (200, 1, 1.5, "fib"),           # window of one
    (333, 8, 1.2345, "pow2"),
    (150, 4, 1.0, (37,)),
    (1000, 12, 1.4999, "fib"),      # rungs reaching across several 64-query tiles
    (300, 1, 1.37, tuple(range(1, 25))),  # 24 rungs within 33 rows: more than the near
                                          # block serves, the rest streamed
])
def test_edge_cases_bf16(mode, N, W, alpha, kind):
    B, H = 2, 3
    plan = _plan(kind, [alpha], W, N, mode)
    q, k, v = inputs.qkv(B, H, N, 64, 300 + N, W, "bf16")
    o, lse = fa.fib_attn_fwd(plan, 0, q.cuda(), k.cuda(), v.cuda())
    torch.cuda.synchronize()
    O_ref, lse_ref = oracle.attend(inputs.as_f64(q), inputs.as_f64(k), inputs.as_f64(v), alpha,
                                   _base_fn(kind)(N), W, mode)
    _check_o(o, O_ref, "bf16", f"edge N={N} W={W} {mode}")
    _check_lse(lse, lse_ref, "bf16")
    assert fa.fib_attn_last_device_status(plan) == fa.FIB_OK
    plan.close()


# ------------------------------------------------------------------ prepared halves
@pytest.mark.parametrize("mode", ["mask", "interp"])
def test_prepare_then_attend_equals_the_fused_call(mode):
    """fib_attn_fwd == fib_attn_fwd_prepare_kv + fib_attn_fwd_attend bit for bit, and one
    prepared K/V serves a second query set."""
    B, H, N, W = 2, 2, 1000, 12
    plan = _plan("fib", [0.8, 1.3], W, N, mode)
    q, k, v = (t.cuda() for t in inputs.qkv(B, H, N, 64, 7, 0, "bf16"))
    q2 = inputs.qkv(B, H, N, 64, 7, 1, "bf16")[0].cuda()
    o1, l1 = fa.fib_attn_fwd(plan, 1, q, k, v)
    ws = fa.fib_attn_fwd_prepare_kv(plan, k, v)
    assert ws.numel() == fa.fib_attn_fwd_workspace_size(plan, B, H, N, torch.bfloat16)
    o2, l2 = fa.fib_attn_fwd_attend(plan, 1, q, ws)
    o3, l3 = fa.fib_attn_fwd_attend(plan, 1, q2, ws)
    o4, l4 = fa.fib_attn_fwd(plan, 1, q2, k, v)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(o3, o4) and torch.equal(l3, l4)
    # float32 has no prepared path
    lib = fa.lib()
    qf = q.float()
    s = torch.cuda.current_stream().cuda_stream
    assert lib.fib_attn_fwd_prepare_kv(plan.handle, B, H, N, fa.FIB_DTYPE_F32, qf.data_ptr(), qf.data_ptr(),
                                       ws.data_ptr(), ws.numel(), s) == fa.FIB_ERR_UNSUPPORTED
    assert lib.fib_attn_fwd_attend(plan.handle, 1, B, H, N, fa.FIB_DTYPE_BF16, q.data_ptr(), ws.data_ptr(),
                                   ws.numel() - 1, o2.data_ptr(), None, None, s) == fa.FIB_ERR_INVALID_ARG
    assert lib.fib_attn_fwd_attend(plan.handle, 1, B, H, N, fa.FIB_DTYPE_BF16, q.data_ptr(), q.data_ptr(),
                                   ws.numel(), o2.data_ptr(), None, None, s) == fa.FIB_ERR_INVALID_ARG
    plan.close()


# ------------------------------------------------------------------ bounded waits
def test_starved_stage_times_out_and_context_survives():
    """The hook leaves one staged copy of every CTA (the values of its window block) out; each
    CTA's wait gives up after 2 ms, records FIB_ERR_TIMEOUT and exits.  The same context then
    runs a normal forward that matches the oracle."""
    B, H, N, W, alpha = 1, 2, 256, 12, 1.0
    plan = _plan("fib", [alpha], W, N, "mask")
    q, k, v = inputs.qkv(B, H, N, 64, 500, 0, "bf16")
    qc, kc, vc = q.cuda(), k.cuda(), v.cuda()
    assert fa.fib_attn_last_device_status(plan) == fa.FIB_OK
    fa.fib_attn_plan_set_debug(plan, True, 2_000_000)
    fa.fib_attn_fwd(plan, 0, qc, kc, vc)
    assert fa.fib_attn_last_device_status(plan) == fa.FIB_ERR_TIMEOUT
    assert fa.fib_attn_last_device_status(plan) == fa.FIB_OK  # reading clears it
    fa.fib_attn_plan_set_debug(plan, False, 1_000_000_000)
    o, lse = fa.fib_attn_fwd(plan, 0, qc, kc, vc)
    assert fa.fib_attn_last_device_status(plan) == fa.FIB_OK
    O_ref, lse_ref = oracle.attend(inputs.as_f64(q), inputs.as_f64(k), inputs.as_f64(v), alpha,
                                   oracle.fibonacci_base(), W, "mask")
    _check_o(o, O_ref, "bf16", "after timeout")
    with pytest.raises(fa.FibAttnError):
        fa.fib_attn_plan_set_debug(plan, False, 10)
    plan.close()


# ------------------------------------------------------------------ CUDA graph replay
def test_graph_replay_of_a_stack_with_varying_rung_counts():
    """Layers of the coprime stack keep 8 to 11 rungs, so their launches need different
    shared-memory sizes; a captured stack must replay every layer exactly as an eager call."""
    B, H, N, W = 1, 2, 4096, 12
    alphas = oracle.schedule("coprime", 16)
    plan = _plan("fib", alphas, W, N, "mask")
    xs = [tuple(t.cuda() for t in inputs.qkv(B, H, N, 64, 2, l, "bf16")) for l in range(16)]
    eager = [fa.fib_attn_fwd(plan, l, *xs[l])[0] for l in range(16)]
    outs = [torch.empty_like(x[0]) for x in xs]
    lses = [torch.empty(B, H, N, device="cuda") for _ in xs]
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for l in range(16):
            fa.fib_attn_fwd(plan, l, *xs[l], o=outs[l], lse=lses[l])
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    for l in range(16):
        assert torch.equal(outs[l], eager[l]), l
    assert fa.fib_attn_last_device_status(plan) == fa.FIB_OK
    plan.close()


# ------------------------------------------------------------------ device-side table check
@pytest.mark.parametrize("mode", ["mask", "interp"])
def test_corrupted_rung_table_is_rejected_on_the_device(mode):
    """The test hook moves the first rung of the tensor-core forward's table to distance 0
    (inside the window; every address it implies is still a row of the sequence).  The
    kernel's table check records FIB_ERR_DEVICE_ASSERT and returns before any rung row is
    read or any output written; the same context then runs a correct forward."""
    B, H, N, W, alpha = 1, 2, 256, 12, 1.2345
    plan = _plan("fib", [alpha], W, N, mode)
    q, k, v = inputs.qkv(B, H, N, 64, 510, 0, "bf16")
    qc, kc, vc = q.cuda(), k.cuda(), v.cuda()
    o = torch.full_like(qc, 7.0)
    lse = torch.full((B, H, N), 7.0, device="cuda")
    assert fa.fib_attn_last_device_status(plan) == fa.FIB_OK
    fa.fib_attn_plan_set_debug(plan, False, 1_000_000_000, corrupt_table=True)
    fa.fib_attn_fwd(plan, 0, qc, kc, vc, o=o, lse=lse)
    assert fa.fib_attn_last_device_status(plan) == fa.FIB_ERR_DEVICE_ASSERT
    assert bool((o == 7.0).all()) and bool((lse == 7.0).all())  # nothing was written
    fa.fib_attn_plan_set_debug(plan, False, 1_000_000_000)
    o, lse = fa.fib_attn_fwd(plan, 0, qc, kc, vc)
    assert fa.fib_attn_last_device_status(plan) == fa.FIB_OK
    O_ref, lse_ref = oracle.attend(inputs.as_f64(q), inputs.as_f64(k), inputs.as_f64(v), alpha,
                                   oracle.fibonacci_base(), W, mode)
    _check_o(o, O_ref, "bf16", "after table check")
    _check_lse(lse, lse_ref, "bf16", "after table check")
    assert fa.lib().fib_attn_plan_set_debug(plan.handle, 4, 1_000_000_000) == fa.FIB_ERR_INVALID_ARG  # unknown flag
    plan.close()


# ------------------------------------------------------------------ float16 range of the bf16 path
def test_values_near_the_float16_limit_match_the_oracle():
    """V scaled so that its largest magnitude is about 6e4 (inside float16's 65504): the
    forward still matches the oracle on the same bf16 values.  O is linear in V, so the
    absolute part of the bound scales with the factor; LSE does not depend on V."""
    B, H, N, W, alpha = 2, 2, 333, 12, 1.2345
    for mode in ("mask", "interp"):
        plan = _plan("fib", [alpha], W, N, mode)
        q, k, v = inputs.qkv(B, H, N, 64, 520, 0, "bf16")
        s = 6.0e4 / float(v.float().abs().max())
        v = (v.float() * s).to(torch.bfloat16)
        assert float(v.float().abs().max()) <= 65504.0
        o, lse = fa.fib_attn_fwd(plan, 0, q.cuda(), k.cuda(), v.cuda())
        torch.cuda.synchronize()
        assert fa.fib_attn_last_device_status(plan) == fa.FIB_OK
        O_ref, lse_ref = oracle.attend(inputs.as_f64(q), inputs.as_f64(k), inputs.as_f64(v), alpha,
                                       oracle.fibonacci_base(), W, mode)
        err = np.abs(o.double().cpu().numpy() - O_ref)
        bound = BF16_ATOL * s + np.abs(O_ref) * 2.0 ** -8
        assert np.all(err <= bound), (mode, float((err - bound).max()))
        _check_lse(lse, lse_ref, "bf16", f"near float16 limit {mode}")
        plan.close()


@pytest.mark.parametrize("which", ["q", "k", "v"])
def test_values_beyond_the_float16_limit_record_a_range_error(which):
    """One element of q, k or v set to 1e6 (a bf16 value beyond float16's range once rotated
    and scaled) makes the bf16 tensor-core forward and backward record FIB_ERR_RANGE; the
    same context then runs a correct forward on in-range values."""
    B, H, N, W, alpha = 1, 2, 200, 12, 1.0
    plan = _plan("fib", [alpha], W, N, "mask")
    q, k, v = inputs.qkv(B, H, N, 64, 530, 0, "bf16")
    dO = inputs.upstream_grad(B, H, N, 64, 530, 0, "bf16")
    big = {"q": q.clone(), "k": k.clone(), "v": v.clone()}
    big[which][0, 1, 100, 5] = 1.0e6
    xs = [big[n].cuda() for n in ("q", "k", "v")]
    o, lse = fa.fib_attn_fwd(plan, 0, *xs)
    assert fa.fib_attn_last_device_status(plan) == fa.FIB_ERR_RANGE
    fa.fib_attn_bwd(plan, 0, *xs, o, lse, dO.cuda())
    assert fa.fib_attn_last_device_status(plan) == fa.FIB_ERR_RANGE
    o, lse = fa.fib_attn_fwd(plan, 0, q.cuda(), k.cuda(), v.cuda())
    assert fa.fib_attn_last_device_status(plan) == fa.FIB_OK
    O_ref, _ = oracle.attend(inputs.as_f64(q), inputs.as_f64(k), inputs.as_f64(v), alpha,
                             oracle.fibonacci_base(), W, "mask")
    _check_o(o, O_ref, "bf16", "after range error")
    plan.close()


# ------------------------------------------------------------------ stale shared memory
@pytest.mark.parametrize("mode", ["mask", "interp"])
@pytest.mark.parametrize("pattern", [0x7FC00000, 0x7C007C00])  # a float32 NaN; float16 infinities
def test_stale_shared_memory_never_reaches_the_outputs(mode, pattern):
    """Every SM's shared memory is filled with a NaN / infinity pattern before each call, so
    that rows a kernel stages but does not copy (before position 0, after a ragged last row)
    hold it; the bf16 forward, backward and dense kernels must still match the oracle."""
    B, H, N, W, alpha = 2, 2, 333, 12, 1.2345
    plan = _plan("fib", [alpha], W, N, mode)
    q, k, v = inputs.qkv(B, H, N, 64, 540, 0, "bf16")
    dO = inputs.upstream_grad(B, H, N, 64, 540, 0, "bf16")
    qc, kc, vc, dOc = q.cuda(), k.cuda(), v.cuda(), dO.cuda()
    fa.fib_attn_debug_fill_shared(pattern)
    o, lse = fa.fib_attn_fwd(plan, 0, qc, kc, vc)
    fa.fib_attn_debug_fill_shared(pattern)
    dq, dk, dv, da = fa.fib_attn_bwd(plan, 0, qc, kc, vc, o, lse, dOc)
    torch.cuda.synchronize()
    assert fa.fib_attn_last_device_status(plan) == fa.FIB_OK
    qf, kf, vf, gf = (inputs.as_f64(x) for x in (q, k, v, dO))
    O_ref, lse_ref = oracle.attend(qf, kf, vf, alpha, oracle.fibonacci_base(), W, mode)
    _check_o(o, O_ref, "bf16", f"stale smem {mode}")
    _check_lse(lse, lse_ref, "bf16", f"stale smem {mode}")
    rq, rk, rv, ra, rss = _oracle_bwd(qf, kf, vf, gf, alpha, oracle.fibonacci_base(), W, mode)
    for name, g, r in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        e = _rel_l2(g.double().cpu().numpy(), r)
        assert e <= REL_L2, f"stale smem {mode} {name} rel-L2 {e:.3e}"
    if mode == "interp":
        _check_dalpha(da, ra, rss, f"stale smem {mode}")
    fa.fib_attn_debug_fill_shared(pattern)
    od, lsed = fa.fib_attn_dense_fwd(plan, qc, kc, vc)
    torch.cuda.synchronize()
    Od_ref, lsed_ref = oracle.attend(qf, kf, vf, 1.0, oracle.fibonacci_base(), N, "mask")
    _check_o(od, Od_ref, "bf16", "stale smem dense")
    _check_lse(lsed, lsed_ref, "bf16", "stale smem dense")
    plan.close()
