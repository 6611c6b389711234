"""The torch.autograd wrapper and the synthetic retrieval probe of learned alpha, on a GPU."""
import os

import numpy as np
import pytest
import torch

from fibonacci_offset_sparse_gb300 import fib_attn as fa
from fibonacci_offset_sparse_gb300 import inputs, probe
from fibonacci_offset_sparse_gb300.autograd import fib_attention

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from fibonacci_offset_sparse_gb300 import build as b
    if not os.path.exists(b.LIB):
        b.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return fa.lib()


@pytest.mark.parametrize("dtype,W", [("f32", 8), ("bf16", 8), ("bf16", 20)])
def test_autograd_is_the_library_forward_and_backward(dtype, W):
    """The Function's outputs and gradients are the library calls' bit for bit: from the kept
    K'/V' workspace where the forward prepares one (bf16, W <= 16), else from k and v."""
    B, H, N, L = 2, 2, 300, 3
    plan = fa.fib_attn_plan_create(fa.FIB_BASE_FIBONACCI, [1.0] * L, W, N, fa.FIB_MODE_INTERP)
    alpha = torch.tensor([0.9, 1.2345, 1.1], dtype=torch.float32, device="cuda", requires_grad=True)
    q, k, v = (t.cuda().requires_grad_(True) for t in inputs.qkv(B, H, N, 64, 300, 1, dtype))
    g = inputs.upstream_grad(B, H, N, 64, 300, 1, dtype).cuda()
    o = fib_attention(plan, 1, q, k, v, alpha)
    o.backward(g)
    # the Function keeps the forward's prepared K'/V' where there are any (bf16) and starts
    # the backward from them
    need = fa.fib_attn_fwd_workspace_size(plan, B, H, N, q.dtype)
    kv = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")
    o2, lse2 = fa.fib_attn_fwd(plan, 1, q.detach(), k.detach(), v.detach(), alpha_dev=alpha.detach(),
                               workspace=kv if need else None)
    if need:
        dq, dk, dv, da = fa.fib_attn_bwd_prepared(plan, 1, q.detach(), kv, o2, lse2, g, alpha_dev=alpha.detach())
    else:
        dq, dk, dv, da = fa.fib_attn_bwd(plan, 1, q.detach(), k.detach(), v.detach(), o2, lse2, g,
                                         alpha_dev=alpha.detach())
    assert torch.equal(o, o2)
    assert torch.equal(q.grad, dq) and torch.equal(k.grad, dk) and torch.equal(v.grad, dv)
    assert float(alpha.grad[1]) == float(da[0]) and float(alpha.grad[0]) == 0.0 == float(alpha.grad[2])
    plan.close()


def test_dalpha_is_the_derivative_of_the_library_forward():
    """d(sum O.G)/dalpha from the backward against central differences of the float32
    forward.  h = 2^-12 keeps every alpha*f (f <= 299) off the integers within +-h f: the
    nearest is 34 alpha = 41.973, 0.027 below 42, where the rows would change and the
    derivative jumps."""
    B, H, N, W = 2, 2, 300, 8
    plan = fa.fib_attn_plan_create(fa.FIB_BASE_FIBONACCI, [1.0], W, N, fa.FIB_MODE_INTERP)
    q, k, v = (t.cuda() for t in inputs.qkv(B, H, N, 64, 301, 0, "f32"))
    g = inputs.upstream_grad(B, H, N, 64, 301, 0, "f32").cuda()
    a0 = 1.2345
    alpha = torch.tensor([a0], dtype=torch.float32, device="cuda", requires_grad=True)
    (fib_attention(plan, 0, q, k, v, alpha) * g).sum().backward()
    h = 2.0 ** -12

    def loss(a):
        at = torch.tensor([a], dtype=torch.float32, device="cuda")
        o, _ = fa.fib_attn_fwd(plan, 0, q, k, v, alpha_dev=at)
        return float((o.double() * g.double()).sum())

    fd = (loss(a0 + h) - loss(a0 - h)) / (2 * h)
    got = float(alpha.grad[0])
    assert abs(got - fd) <= 2e-3 * abs(fd) + 1e-3, (got, fd)
    plan.close()


def test_probe_retrieves_only_through_a_rung_on_the_target():
    """The probe's task at alpha = 1: a target distance on the rung lattice (34) is retrieved
    (loss near 0), one that no rung reaches (30) is not (loss near that of an average of
    random rows); a few descent steps keep everything finite and alpha inside (0.5, 1.5)."""
    on = probe.run(34, steps=5, lr=1e-3, B=2, H=2, N=256, record_every=1)
    off = probe.run(30, steps=5, lr=1e-3, B=2, H=2, N=256, record_every=1)
    assert on["loss"][0] < 0.05 < 0.5 < off["loss"][0]
    for r in (on, off):
        assert np.isfinite(r["loss"]).all() and np.isfinite(r["dalpha"]).all()
        assert all(0.5 < a < 1.5 for a in r["alpha"])
