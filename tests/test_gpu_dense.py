"""GPU parity of the dense causal control (fib_attn_dense_fwd) against the float64 oracle.

The oracle's sparse attention with a window covering the whole sequence (W >= N) is dense
causal attention with the same RoPE (pinned on the CPU by
test_oracle.py::test_window_covering_sequence_is_dense_causal), so it is the reference here.
Tolerances as the other bf16 forward checks: O max-abs <= 1e-2 plus the bf16 output's own
rounding, LSE <= 5e-3.
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


@pytest.mark.parametrize("B,H,N", [(1, 1, 1), (1, 2, 63), (2, 1, 64), (1, 3, 65), (2, 2, 333), (1, 2, 2048)])
def test_dense_causal_matches_the_oracle(B, H, N):
    plan = fa.fib_attn_plan_create(fa.FIB_BASE_FIBONACCI, [1.0], 1, N, fa.FIB_MODE_MASK)
    q, k, v = inputs.qkv(B, H, N, 64, 800, N, "bf16")
    o, lse = fa.fib_attn_dense_fwd(plan, q.cuda(), k.cuda(), v.cuda())
    torch.cuda.synchronize()
    assert fa.fib_attn_last_device_status(plan) == fa.FIB_OK
    O_ref, lse_ref = oracle.attend(inputs.as_f64(q), inputs.as_f64(k), inputs.as_f64(v), 1.0,
                                   oracle.fibonacci_base(), N, "mask")
    err = np.abs(o.double().cpu().numpy() - O_ref)
    bound = 1e-2 + np.abs(O_ref) * 2.0 ** -8
    assert np.all(err <= bound), float((err - bound).max())
    assert np.abs(lse.double().cpu().numpy() - lse_ref).max() <= 5e-3
    plan.close()


def test_dense_causal_refuses_float32_and_short_workspaces():
    N = 128
    plan = fa.fib_attn_plan_create(fa.FIB_BASE_FIBONACCI, [1.0], 1, N, fa.FIB_MODE_MASK)
    q = torch.zeros(1, 1, N, 64, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    lib = fa.lib()
    assert lib.fib_attn_dense_fwd_workspace_size(plan.handle, 1, 1, N, fa.FIB_DTYPE_F32) == 0
    need = lib.fib_attn_dense_fwd_workspace_size(plan.handle, 1, 1, N, fa.FIB_DTYPE_BF16)
    assert need == N * 256
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    o = torch.empty_like(q)
    assert lib.fib_attn_dense_fwd(plan.handle, 1, 1, N, fa.FIB_DTYPE_F32, q.data_ptr(), q.data_ptr(), q.data_ptr(),
                                  o.data_ptr(), None, ws.data_ptr(), need, s) == fa.FIB_ERR_UNSUPPORTED
    qb, ob = q.bfloat16(), o.bfloat16()
    assert lib.fib_attn_dense_fwd(plan.handle, 1, 1, N, fa.FIB_DTYPE_BF16, qb.data_ptr(), qb.data_ptr(),
                                  qb.data_ptr(), ob.data_ptr(), None, ws.data_ptr(), need - 1, s) == fa.FIB_ERR_INVALID_ARG
    assert lib.fib_attn_dense_fwd(plan.handle, 1, 1, N + 1, fa.FIB_DTYPE_BF16, qb.data_ptr(), qb.data_ptr(),
                                  qb.data_ptr(), ob.data_ptr(), None, ws.data_ptr(), need, s) == fa.FIB_ERR_INVALID_ARG
    plan.close()
