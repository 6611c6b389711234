"""fib_attn_bwd_prepared: the backward from the forward's prepared K'/V' rows.

The forward's workspace holds K' = RoPE(k) at each row's own position and V' as float16
rows, what the bf16 backward otherwise prepares from k and v.  The forward builds the RoPE
factors of two rows in three by a recurrence and the backward's own preparation reads them
from the tables, so a K' element can differ in its last float16 bit: the prepared backward
must match fib_attn_bwd to within that rounding (relative L2 <= 2e-3 for dQ, dK, dV and
dalpha), be deterministic, and match the float64 oracle with the parity tests' bounds,
whether fib_attn_fwd or fib_attn_fwd_prepare_kv filled the workspace, with the (b, h) rows
unsplit (B*H = 1) or split in two halves.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from fibonacci_offset_sparse_gb300 import fib_attn as fa
from fibonacci_offset_sparse_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from fibonacci_offset_sparse_gb300 import build as b
    if not os.path.exists(b.LIB):
        b.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return fa.lib()


def _plan(mode, alpha, W, N):
    m = fa.FIB_MODE_MASK if mode == "mask" else fa.FIB_MODE_INTERP
    return fa.fib_attn_plan_create(fa.FIB_BASE_FIBONACCI, [alpha], W, N, m)


@pytest.mark.parametrize("mode,B,H,N,W,device_alpha", [("interp", 2, 3, 700, 12, True), ("interp", 1, 1, 333, 10, False),
                                                       ("mask", 2, 2, 1000, 12, False), ("mask", 1, 3, 129, 16, False)])
@pytest.mark.parametrize("filled_by", ["fwd", "prepare_kv"])
def test_prepared_backward_matches_the_backward(mode, B, H, N, W, device_alpha, filled_by):
    alpha = float(np.float32(1.2345))
    plan = _plan(mode, alpha, W, N)
    adev = torch.tensor([alpha], dtype=torch.float32, device="cuda") if device_alpha else None
    q, k, v = (t.cuda() for t in inputs.qkv(B, H, N, 64, 750, W, "bf16"))
    dO = inputs.upstream_grad(B, H, N, 64, 750, W, "bf16").cuda()
    kv = torch.empty(fa.fib_attn_fwd_workspace_size(plan, B, H, N, torch.bfloat16), dtype=torch.uint8, device="cuda")
    o, lse = fa.fib_attn_fwd(plan, 0, q, k, v, alpha_dev=adev, workspace=kv)
    if filled_by == "prepare_kv":  # a second filling of a fresh buffer by the split entry point
        kv = torch.full_like(kv, 0x7b)
        fa.fib_attn_fwd_prepare_kv(plan, k, v, workspace=kv)
    ref = fa.fib_attn_bwd(plan, 0, q, k, v, o, lse, dO, alpha_dev=adev)
    got = fa.fib_attn_bwd_prepared(plan, 0, q, kv, o, lse, dO, alpha_dev=adev)
    again = fa.fib_attn_bwd_prepared(plan, 0, q, kv, o, lse, dO, alpha_dev=adev)
    torch.cuda.synchronize()
    assert fa.fib_attn_last_device_status(plan) == fa.FIB_OK
    for g, h in zip(got, again):
        assert torch.equal(g, h)
    for g, r in zip(got[:3], ref[:3]):
        g, r = g.double(), r.double()
        assert float(torch.linalg.norm(g - r)) <= 2e-3 * float(torch.linalg.norm(r))
    if mode == "mask":
        assert float(got[3].item()) == 0.0
    else:
        assert abs(float(got[3].item()) - float(ref[3].item())) <= 2e-3 * abs(float(ref[3].item())) + 1e-3
    plan.close()


def test_prepared_backward_matches_the_oracle():
    """One interp case against the float64 oracle directly (relative L2 <= 2e-2 for dQ, dK,
    dV; dalpha within 2e-2 of the larger of |dalpha| and its per-head root-sum-square)."""
    B, H, N, W, alpha = 2, 2, 517, 12, 0.9871
    plan = _plan("interp", alpha, W, N)
    q, k, v = inputs.qkv(B, H, N, 64, 760, 0, "bf16")
    dO = inputs.upstream_grad(B, H, N, 64, 760, 0, "bf16")
    qc, kc, vc, gc = q.cuda(), k.cuda(), v.cuda(), dO.cuda()
    kv = torch.empty(fa.fib_attn_fwd_workspace_size(plan, B, H, N, torch.bfloat16), dtype=torch.uint8, device="cuda")
    o, lse = fa.fib_attn_fwd(plan, 0, qc, kc, vc, workspace=kv)
    dq, dk, dv, da = fa.fib_attn_bwd_prepared(plan, 0, qc, kv, o, lse, gc)
    torch.cuda.synchronize()
    qf, kf, vf, gf = (inputs.as_f64(x) for x in (q, k, v, dO))
    rq, rk, rv = np.zeros_like(qf), np.zeros_like(kf), np.zeros_like(vf)
    per = []
    for b in range(B):
        for h in range(H):
            sl = (slice(b, b + 1), slice(h, h + 1))
            gq, gk, gv, ga = oracle.attend_bwd(qf[sl], kf[sl], vf[sl], gf[sl], alpha, oracle.fibonacci_base(), W, "interp")
            rq[sl], rk[sl], rv[sl] = gq, gk, gv
            per.append(ga)
    for g, r in ((dq, rq), (dk, rk), (dv, rv)):
        assert np.linalg.norm(g.double().cpu().numpy() - r) <= 2e-2 * np.linalg.norm(r)
    ra = float(sum(per))
    assert abs(float(da.item()) - ra) <= 2e-2 * max(abs(ra), float(np.sqrt(np.sum(np.square(per)))))
    plan.close()


def test_prepared_backward_rejects_what_it_cannot_serve():
    B, H, N = 1, 2, 256
    lib = fa.lib()
    x = torch.zeros(B, H, N, 64, dtype=torch.bfloat16, device="cuda")
    outs = [torch.empty_like(x) for _ in range(3)]
    lse = torch.zeros(B, H, N, device="cuda")
    da = torch.empty(1, device="cuda")
    plan = _plan("interp", 1.1, 12, N)
    ws = torch.empty(fa.fib_attn_bwd_workspace_size(plan, B, H, N), dtype=torch.uint8, device="cuda")
    need = fa.fib_attn_fwd_workspace_size(plan, B, H, N, torch.bfloat16)
    kv = torch.zeros(need, dtype=torch.uint8, device="cuda")

    def call(plan_, dtype, kv_ptr, kv_bytes, ws_ptr=ws.data_ptr()):
        return lib.fib_attn_bwd_prepared(plan_.handle, 0, B, H, N, dtype, x.data_ptr(), kv_ptr, kv_bytes,
                                         x.data_ptr(), lse.data_ptr(), x.data_ptr(), outs[0].data_ptr(),
                                         outs[1].data_ptr(), outs[2].data_ptr(), da.data_ptr(), None, ws_ptr,
                                         ws.numel(), None)
    assert call(plan, fa.FIB_DTYPE_F32, kv.data_ptr(), need) == fa.FIB_ERR_UNSUPPORTED  # no prepared rows
    assert call(plan, fa.FIB_DTYPE_BF16, kv.data_ptr(), need - 16) == fa.FIB_ERR_INVALID_ARG  # short
    assert call(plan, fa.FIB_DTYPE_BF16, None, need) == fa.FIB_ERR_INVALID_ARG
    assert call(plan, fa.FIB_DTYPE_BF16, ws.data_ptr(), need) == fa.FIB_ERR_INVALID_ARG  # the workspace itself
    plan.close()
    wide = _plan("interp", 1.1, 20, N)  # a window beyond 16: the forward prepares nothing
    assert fa.fib_attn_fwd_workspace_size(wide, B, H, N, torch.bfloat16) == 0
    assert call(wide, fa.FIB_DTYPE_BF16, kv.data_ptr(), need) == fa.FIB_ERR_UNSUPPORTED
    wide.close()
    torch.cuda.synchronize()
