"""The bf16 backward's two halves: with B*H >= 2 the (b, h) rows are split in two and the
second half runs on the plan's own stream, forked from the caller's stream and joined back to
it with events.  These tests check that the split is invisible to the caller: an odd split
and the unsplit single-(b, h) call match the oracle, the results are ordered on the caller's
stream, and a CUDA graph captured on the caller's stream replays the whole backward.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from fibonacci_offset_sparse_gb300 import fib_attn as fa
from fibonacci_offset_sparse_gb300 import inputs

pytestmark = pytest.mark.gpu

REL_L2 = 2e-2  # the bf16 backward bound of the parity tests


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from fibonacci_offset_sparse_gb300 import build as b
    if not os.path.exists(b.LIB):
        b.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return fa.lib()


def _plan(alpha, W, N, mode):
    m = fa.FIB_MODE_MASK if mode == "mask" else fa.FIB_MODE_INTERP
    return fa.fib_attn_plan_create(fa.FIB_BASE_FIBONACCI, [alpha], W, N, m)


@pytest.mark.parametrize("B,H,mode", [(1, 1, "interp"), (1, 1, "mask"), (1, 3, "interp"), (3, 1, "mask")])
def test_unsplit_and_odd_split_match_the_oracle(B, H, mode):
    """B*H = 1 runs unsplit; B*H = 3 splits 1 + 2.  dQ, dK, dV within relative L2 2e-2 of
    the oracle per (b, h); dalpha within 2e-2 of the larger of |dalpha| and the
    root-sum-square of its per-(b, h) contributions (interp), exactly 0 (mask)."""
    N, W, alpha = 517, 12, 1.2345
    plan = _plan(alpha, W, N, mode)
    q, k, v = inputs.qkv(B, H, N, 64, 730, B * H, "bf16")
    dO = inputs.upstream_grad(B, H, N, 64, 730, B * H, "bf16")
    qc, kc, vc, gc = q.cuda(), k.cuda(), v.cuda(), dO.cuda()
    o, lse = fa.fib_attn_fwd(plan, 0, qc, kc, vc)
    dq, dk, dv, da = fa.fib_attn_bwd(plan, 0, qc, kc, vc, o, lse, gc)
    torch.cuda.synchronize()
    assert fa.fib_attn_last_device_status(plan) == fa.FIB_OK
    qf, kf, vf, gf = (inputs.as_f64(x) for x in (q, k, v, dO))
    per = []
    for b in range(B):
        for h in range(H):
            sl = (slice(b, b + 1), slice(h, h + 1))
            rq, rk, rv, ra = oracle.attend_bwd(qf[sl], kf[sl], vf[sl], gf[sl], alpha, oracle.fibonacci_base(), W, mode)
            for g, r in ((dq, rq), (dk, rk), (dv, rv)):
                g = g[sl].double().cpu().numpy()
                assert np.linalg.norm(g - r) <= REL_L2 * np.linalg.norm(r)
            per.append(ra)
    if mode == "mask":
        assert float(da.item()) == 0.0
    else:
        ref = float(sum(per))
        scale = max(abs(ref), float(np.sqrt(np.sum(np.square(per)))))
        assert abs(float(da.item()) - ref) <= REL_L2 * scale
    plan.close()


def _case():
    B, H, N, W, alpha = 2, 3, 700, 12, 0.9871
    plan = _plan(alpha, W, N, "interp")
    q, k, v = (t.cuda() for t in inputs.qkv(B, H, N, 64, 740, 0, "bf16"))
    dO = inputs.upstream_grad(B, H, N, 64, 740, 0, "bf16").cuda()
    adev = torch.tensor([alpha], dtype=torch.float32, device="cuda")
    o, lse = fa.fib_attn_fwd(plan, 0, q, k, v, alpha_dev=adev)
    return plan, (q, k, v, o, lse, dO), adev


def test_results_are_ordered_on_the_callers_stream():
    """On a side stream: outputs poisoned with NaN, the backward, then copies of its outputs
    enqueued at once on the same stream; the copies equal the eager results bit for bit."""
    plan, (q, k, v, o, lse, dO), adev = _case()
    ref = fa.fib_attn_bwd(plan, 0, q, k, v, o, lse, dO, alpha_dev=adev)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        outs = [torch.full_like(q, float("nan")) for _ in range(3)]
        da = torch.full((1,), float("nan"), dtype=torch.float32, device="cuda")
        fa.fib_attn_bwd(plan, 0, q, k, v, o, lse, dO, *outs, dalpha=da, alpha_dev=adev)
        copies = [x.clone() for x in outs + [da]]
    torch.cuda.synchronize()
    for c, r in zip(copies, ref):
        assert torch.equal(c, r)
    plan.close()


@pytest.mark.parametrize("entry", ["bwd", "bwd_prepared"])
def test_graph_replay_equals_the_eager_backward(entry):
    """The backward (from k and v, or from the forward's prepared K'/V') captured in a CUDA
    graph on the caller's stream (the side stream joins the capture through the fork event)
    and replayed twice gives the eager result bit for bit."""
    plan, (q, k, v, o, lse, dO), adev = _case()
    kv = torch.empty(fa.fib_attn_fwd_workspace_size(plan, *q.shape[:3], q.dtype), dtype=torch.uint8, device="cuda")
    fa.fib_attn_fwd_prepare_kv(plan, k, v, workspace=kv)

    def run(*out, **kw):
        if entry == "bwd":
            return fa.fib_attn_bwd(plan, 0, q, k, v, o, lse, dO, *out, alpha_dev=adev, **kw)
        return fa.fib_attn_bwd_prepared(plan, 0, q, kv, o, lse, dO, *out, alpha_dev=adev, **kw)
    ref = run()
    torch.cuda.synchronize()
    outs = [torch.empty_like(q) for _ in range(3)]
    da = torch.empty(1, dtype=torch.float32, device="cuda")
    ws = torch.empty(fa.fib_attn_bwd_workspace_size(plan, *q.shape[:3]), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # one eager call on the capture stream first (as torch advises)
        run(*outs, dalpha=da, workspace=ws)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        run(*outs, dalpha=da, workspace=ws)
    for _ in range(2):
        for x in outs + [da]:
            x.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        for x, r in zip(outs + [da], ref):
            assert torch.equal(x, r)
    assert fa.fib_attn_last_device_status(plan) == fa.FIB_OK
    plan.close()


def test_two_plans_run_their_backwards_concurrently():
    """Two plans (each with its own side stream) on two caller streams at once: every result
    equals the same call made alone, bit for bit."""
    cases = []
    for i, (alpha, mode) in enumerate(((0.9871, "interp"), (1.3, "mask"))):
        plan = _plan(alpha, 12, 640, mode)
        q, k, v = (t.cuda() for t in inputs.qkv(2, 2, 640, 64, 770 + i, 0, "bf16"))
        dO = inputs.upstream_grad(2, 2, 640, 64, 770 + i, 0, "bf16").cuda()
        o, lse = fa.fib_attn_fwd(plan, 0, q, k, v)
        ref = fa.fib_attn_bwd(plan, 0, q, k, v, o, lse, dO)
        cases.append((plan, (q, k, v, o, lse, dO), ref))
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    got = []
    for s, (plan, args, _) in zip(streams, cases):
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            got.append(fa.fib_attn_bwd(plan, 0, *args))
    torch.cuda.synchronize()
    for g, (plan, _, ref) in zip(got, cases):
        for x, r in zip(g, ref):
            assert torch.equal(x, r)
        assert fa.fib_attn_last_device_status(plan) == fa.FIB_OK
        plan.close()
