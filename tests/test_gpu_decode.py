"""Single-token decode against a KV cache: row pos of the forward, from the oracle."""
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


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("mode,alpha,kind,W,N", [("mask", 1.5, "fib", 12, 2000), ("interp", 1.2345, "fib", 10, 1500),
                                                 ("mask", 0.77, "pow2", 8, 1024), ("interp", 1.0, "fib", 12, 300)])
def test_decode_equals_forward_row(dtype, mode, alpha, kind, W, N):
    B, H = 2, 3
    m = fa.FIB_MODE_MASK if mode == "mask" else fa.FIB_MODE_INTERP
    bk = fa.FIB_BASE_FIBONACCI if kind == "fib" else fa.FIB_BASE_POW2
    plan = fa.fib_attn_plan_create(bk, [alpha], W, N, m)
    q, k, v = inputs.qkv(B, H, N, 64, 800, W, dtype)
    kc, vc = k.cuda(), v.cuda()
    base = oracle.fibonacci_base() if kind == "fib" else oracle.pow2_base(N)
    O_ref, lse_ref = oracle.attend(inputs.as_f64(q), inputs.as_f64(k), inputs.as_f64(v), alpha, base, W, mode)
    tol = 1e-5 if dtype == "f32" else 1e-2
    for pos in sorted({p for p in (0, 1, W - 1, W, 377, N // 2, N - 1) if p < N}):
        o, lse = fa.fib_attn_decode(plan, 0, pos, q[:, :, pos].contiguous().cuda(), kc, vc)
        torch.cuda.synchronize()
        ref = O_ref[:, :, pos]
        err = np.abs(o.double().cpu().numpy() - ref)
        bound = tol + (0 if dtype == "f32" else np.abs(ref) * 2.0 ** -8)
        assert np.all(err <= bound), (pos, err.max())
        assert np.abs(lse.double().cpu().numpy() - lse_ref[:, :, pos]).max() <= (1e-5 if dtype == "f32" else 1e-3)
    with pytest.raises(fa.FibAttnError):
        fa.fib_attn_decode(plan, 0, N, q[:, :, 0].contiguous().cuda(), kc, vc)
    plan.close()
