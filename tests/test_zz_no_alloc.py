"""The allocation-free backward entry point against the ordinary one.

fib_attn_bwd_noalloc serves callers that cannot allocate device memory on the call path
(a plugin inside a framework that owns the device heap, a real-time loop that forbids
allocation): it takes no workspace and uses the library's fixed scratch array instead.
This file is collected last, so a run that stops at its first failure has already run every
other test; it also passes on its own in a fresh process.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from fibonacci_offset_sparse_gb300 import fib_attn as fa
from fibonacci_offset_sparse_gb300 import inputs

pytestmark = pytest.mark.gpu


def _rel_l2(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from fibonacci_offset_sparse_gb300 import build as b
    if not os.path.exists(b.LIB):
        b.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return fa.lib()


@pytest.mark.parametrize("dtype,mode,alpha", [("f32", "interp", 1.2345), ("bf16", "interp", 0.9871),
                                              ("f32", "mask", 0.5 + 4 / 15)])
def test_noalloc_backward_matches_workspace_backward_twice(dtype, mode, alpha):
    B, H, N, W = 2, 3, 333, 8
    m = fa.FIB_MODE_MASK if mode == "mask" else fa.FIB_MODE_INTERP
    plan = fa.fib_attn_plan_create(fa.FIB_BASE_FIBONACCI, [alpha, alpha], W, N, m)
    # the tolerances of the other backward tests: fp32 rel-L2 1e-5, bf16 rel-L2 2e-2.  For
    # bf16 the two entry points run different kernels (the ordinary one the tensor-core path
    # with its prepared float16 rows, the allocation-free one the CUDA-core path, which needs
    # no such scratch), so they agree to the bf16 bound, not bit for bit.
    tol = 1e-5 if dtype == "f32" else 2e-2
    for call in range(2):  # two calls in a row: the second starts from the first one's scratch
        q, k, v = (t.cuda() for t in inputs.qkv(B, H, N, 64, 700 + call, call, dtype))
        dO = inputs.upstream_grad(B, H, N, 64, 700 + call, call, dtype).cuda()
        o, lse = fa.fib_attn_fwd(plan, call, q, k, v)
        rq, rk, rv, ra = fa.fib_attn_bwd(plan, call, q, k, v, o, lse, dO)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
        da = torch.empty(1, dtype=torch.float32, device="cuda")
        rc = fa.lib().fib_attn_bwd_noalloc(
            plan.handle, call, B, H, N, fa._DT[q.dtype], q.data_ptr(), k.data_ptr(), v.data_ptr(),
            o.data_ptr(), lse.data_ptr(), dO.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
            da.data_ptr(), None, torch.cuda.current_stream().cuda_stream)
        assert rc == fa.FIB_OK, fa.error_string(rc)
        torch.cuda.synchronize()
        for g, r in ((dq, rq), (dk, rk), (dv, rv)):
            assert _rel_l2(g, r) <= tol
        if mode == "mask":
            assert float(da.item()) == 0.0 == float(ra.item())
        else:
            rel = 1e-4 if dtype == "f32" else 2e-2
            assert abs(float(da.item()) - float(ra.item())) <= rel * abs(float(ra.item())) + 1e-4
    plan.close()


def _noalloc(plan, layer, q, k, v, o, lse, dO):
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    da = torch.empty(1, dtype=torch.float32, device="cuda")
    fa.fib_attn_bwd_noalloc(plan, layer, q, k, v, o, lse, dO, dq, dk, dv, da)
    return dq, dk, dv, da


@pytest.mark.parametrize("dtype,mode,alpha,W,N", [("bf16", "interp", 1.2345, 8, 333), ("bf16", "mask", 0.9, 12, 300),
                                                  ("f32", "interp", 0.7771, 8, 257), ("bf16", "interp", 1.1, 24, 401)])
def test_noalloc_backward_matches_the_oracle(dtype, mode, alpha, W, N):
    """The allocation-free backward checked directly against the float64 oracle's gradients
    of its own forward (relative L2 <= 2e-2 for bf16 inputs, 1e-5 for float32)."""
    B, H = 2, 2
    m = fa.FIB_MODE_MASK if mode == "mask" else fa.FIB_MODE_INTERP
    plan = fa.fib_attn_plan_create(fa.FIB_BASE_FIBONACCI, [alpha], W, N, m)
    q, k, v = inputs.qkv(B, H, N, 64, 710, W, dtype)
    dO = inputs.upstream_grad(B, H, N, 64, 710, W, dtype)
    qc, kc, vc, gc = q.cuda(), k.cuda(), v.cuda(), dO.cuda()
    o, lse = fa.fib_attn_fwd(plan, 0, qc, kc, vc)
    dq, dk, dv, da = _noalloc(plan, 0, qc, kc, vc, o, lse, gc)
    torch.cuda.synchronize()
    qf, kf, vf, gf = (inputs.as_f64(x) for x in (q, k, v, dO))
    rq, rk, rv, ra = oracle.attend_bwd(qf, kf, vf, gf, alpha, oracle.fibonacci_base(), W, mode)
    tol = 1e-5 if dtype == "f32" else 2e-2
    for g, r in ((dq, rq), (dk, rk), (dv, rv)):
        g = g.double().cpu().numpy()
        assert np.linalg.norm(g - r) <= tol * np.linalg.norm(r)
    if mode == "mask":
        assert float(da.item()) == 0.0
    else:
        assert abs(float(da.item()) - ra) <= (1e-4 if dtype == "f32" else 2e-2) * abs(ra)
    plan.close()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_noalloc_backward_is_bit_identical_where_both_run_the_cuda_core_kernels(dtype):
    """With a window wider than 16 both entry points run the same CUDA-core kernels (only the
    scratch's address differs), so their gradients agree bit for bit, twice in a row."""
    B, H, N, W, alpha = 2, 3, 300, 20, 1.2345
    plan = fa.fib_attn_plan_create(fa.FIB_BASE_FIBONACCI, [alpha], W, N, fa.FIB_MODE_INTERP)
    for call in range(2):
        q, k, v = (t.cuda() for t in inputs.qkv(B, H, N, 64, 720 + call, 0, dtype))
        dO = inputs.upstream_grad(B, H, N, 64, 720 + call, 0, dtype).cuda()
        o, lse = fa.fib_attn_fwd(plan, 0, q, k, v)
        ref = fa.fib_attn_bwd(plan, 0, q, k, v, o, lse, dO)
        got = _noalloc(plan, 0, q, k, v, o, lse, dO)
        torch.cuda.synchronize()
        for g, r in zip(got, ref):
            assert torch.equal(g, r)
    plan.close()


def test_noalloc_backward_rejects_oversize_before_launching():
    plan = fa.fib_attn_plan_create(fa.FIB_BASE_FIBONACCI, [1.0], 8, 1 << 20, fa.FIB_MODE_MASK)
    x = torch.zeros(128, dtype=torch.uint8, device="cuda")  # never touched: rejected first
    p = x.data_ptr()
    B, H, N = 4, 8, 1 << 20  # 32M rows: far beyond the fixed scratch
    assert fa.fib_attn_bwd_workspace_size(plan, B, H, N) > 8 << 20
    # inputs may alias one another; outputs are distinct and aligned, so only the size fails
    rc = fa.lib().fib_attn_bwd_noalloc(plan.handle, 0, B, H, N, fa.FIB_DTYPE_F32, p, p, p, p, p + 64, p,
                                       p + 16, p + 32, p + 48, p + 80, None, None)
    assert rc == fa.FIB_ERR_INVALID_ARG
    plan.close()
