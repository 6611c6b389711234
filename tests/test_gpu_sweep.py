"""Seeded random sweep of the forward, the backward and decode against the float64 oracle.

The hand-picked parity cases pin the configurations the pages measure and the known edge
cases; this sweep draws 96 more cases from one fixed seed, over lengths 1..2500 (log-uniform,
mostly ragged against the 64-row tiles), windows 1..16 (bf16 tensor-core path), 17..24 (bf16
CUDA-core backward) and 1..40 (float32), alpha in [0.5, 1.5], the Fibonacci and the
power-of-two bases, both modes, one to six (b, h) rows (B*H = 1 runs the backward unsplit), and
alpha from the plan or from the device.  Tolerances are those of the parity tests, with an
absolute floor for gradients whose reference is (near) zero, e.g. N = 1 where dS vanishes:
  * O: max-abs <= 1e-2 beyond the bf16 output's own rounding (2^-8 |O|), 1e-5 float32;
  * LSE: 5e-3 (bf16), 1e-5 (float32); decode (one row, pos drawn per case): O as above,
    LSE 1e-3 (bf16: the decode kernel computes in float32 from the bf16 values), 1e-5;
  * dQ, dK, dV: ||g - r|| <= 2e-2 ||r|| + 1e-3 sqrt(n) (bf16), 1e-5 ||r|| + 1e-7 sqrt(n);
  * dalpha: within 2e-2 (1e-4 float32) of the larger of |dalpha| and the root-sum-square
    of its per-(b, h) contributions, plus 1e-4; exactly 0 in mask mode.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from fibonacci_offset_sparse_gb300 import fib_attn as fa
from fibonacci_offset_sparse_gb300 import inputs

pytestmark = pytest.mark.gpu


def _cases(n):
    rng = np.random.default_rng(20261203)
    out = []
    for i in range(n):
        mode = ("mask", "interp")[int(rng.integers(0, 2))]
        kind = rng.random()
        dtype = "f32" if kind < 0.25 else "bf16"
        if dtype == "f32":
            W = int(rng.integers(1, 41))
        elif kind < 0.4:
            W = int(rng.integers(17, 25))  # bf16 beyond the tensor-core window
        else:
            W = int(rng.integers(1, 17))
        N = max(1, int(np.exp(rng.uniform(0.0, np.log(2500.0)))))
        B, H = int(rng.integers(1, 3)), int(rng.integers(1, 4))
        alpha = float(np.float32(rng.uniform(0.5, 1.5)))
        base = "fib" if rng.random() < 0.7 else "pow2"
        dev_alpha = mode == "interp" and bool(rng.random() < 0.5)
        out.append((i, mode, dtype, W, N, B, H, alpha, base, dev_alpha))
    return out


CASES = _cases(96)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from fibonacci_offset_sparse_gb300 import build as b
    if not os.path.exists(b.LIB):
        b.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return fa.lib()


@pytest.mark.parametrize("case", CASES, ids=[f"c{c[0]}-{c[1]}-{c[2]}-W{c[3]}-N{c[4]}-BH{c[5] * c[6]}-{c[8]}"
                                            + ("-dev" if c[9] else "") for c in CASES])
def test_random_case_forward_and_backward_match_the_oracle(case):
    i, mode, dtype, W, N, B, H, alpha, base, dev_alpha = case
    bk = fa.FIB_BASE_FIBONACCI if base == "fib" else fa.FIB_BASE_POW2
    m = fa.FIB_MODE_MASK if mode == "mask" else fa.FIB_MODE_INTERP
    plan = fa.fib_attn_plan_create(bk, [alpha], W, N, m)
    adev = torch.tensor([alpha], dtype=torch.float32, device="cuda") if dev_alpha else None
    q, k, v = inputs.qkv(B, H, N, 64, 800 + i, 0, dtype)
    dO = inputs.upstream_grad(B, H, N, 64, 800 + i, 0, dtype)
    qc, kc, vc, gc = q.cuda(), k.cuda(), v.cuda(), dO.cuda()
    o, lse = fa.fib_attn_fwd(plan, 0, qc, kc, vc, alpha_dev=adev)
    dq, dk, dv, da = fa.fib_attn_bwd(plan, 0, qc, kc, vc, o, lse, gc, alpha_dev=adev)
    pos = (7919 * i) % N  # one decode step against the whole cache: row pos of the forward
    od, lsed = fa.fib_attn_decode(plan, 0, pos, qc[:, :, pos].contiguous(), kc, vc, alpha_dev=adev)
    torch.cuda.synchronize()
    assert fa.fib_attn_last_device_status(plan) == fa.FIB_OK
    plan.close()

    ob = oracle.fibonacci_base() if base == "fib" else oracle.pow2_base(N)
    qf, kf, vf, gf = (inputs.as_f64(x) for x in (q, k, v, dO))
    O_ref, lse_ref = oracle.attend(qf, kf, vf, alpha, ob, W, mode)
    bf = dtype == "bf16"
    o_err = np.abs(o.double().cpu().numpy() - O_ref) - (2.0 ** -8 * np.abs(O_ref) if bf else 0.0)
    assert o_err.max() <= (1e-2 if bf else 1e-5)
    assert np.abs(lse.double().cpu().numpy() - lse_ref).max() <= (5e-3 if bf else 1e-5)
    d_err = np.abs(od.double().cpu().numpy() - O_ref[:, :, pos]) - (2.0 ** -8 * np.abs(O_ref[:, :, pos]) if bf else 0.0)
    assert d_err.max() <= (1e-2 if bf else 1e-5)
    assert np.abs(lsed.double().cpu().numpy() - lse_ref[:, :, pos]).max() <= (1e-3 if bf else 1e-5)

    rq, rk, rv = np.zeros_like(qf), np.zeros_like(kf), np.zeros_like(vf)
    per = []
    for b in range(B):
        for h in range(H):
            sl = (slice(b, b + 1), slice(h, h + 1))
            gq, gk, gv, ga = oracle.attend_bwd(qf[sl], kf[sl], vf[sl], gf[sl], alpha, ob, W, mode)
            rq[sl], rk[sl], rv[sl] = gq, gk, gv
            per.append(ga)
    rel, floor = (2e-2, 1e-3) if bf else (1e-5, 1e-7)
    for name, g, r in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        e = np.linalg.norm(g.double().cpu().numpy() - r)
        assert e <= rel * np.linalg.norm(r) + floor * np.sqrt(r.size), name
    if mode == "mask":
        assert float(da.item()) == 0.0
    else:
        ra = float(sum(per))
        scale = max(abs(ra), float(np.sqrt(np.sum(np.square(per)))))
        assert abs(float(da.item()) - ra) <= (2e-2 if bf else 1e-4) * scale + 1e-4
