"""CPU-only checks of the native library: it builds/loads, exports every symbol declared in
include/*.h, and its host planner agrees exactly with the oracle.  No device calls."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from fibonacci_offset_sparse_gb300 import fib_attn as fa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built_lib():
    from fibonacci_offset_sparse_gb300 import build as b
    srcs = [os.path.join(b.CSRC, s) for s in os.listdir(b.CSRC)] + [os.path.join(ROOT, "include", "fib_attn.h")]
    if not os.path.exists(b.LIB) or os.path.getmtime(b.LIB) < max(os.path.getmtime(s) for s in srcs):
        b.build()
    return fa.lib()


def _declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"\b(fib_attn_\w+)\s*\(", text)
    return sorted(set(names))


def test_library_exports_every_declared_symbol(built_lib):
    declared = _declared_functions()
    assert len(declared) >= 13
    for name in declared:
        assert hasattr(built_lib, name), name
    assert sorted(fa.EXPORTS) == declared


def test_error_strings():
    for code in range(8):
        assert fa.error_string(code)
    assert fa.error_string(99) == "unknown status"


def test_bases_match_oracle():
    assert fa.fib_attn_base(fa.FIB_BASE_FIBONACCI) == oracle.fibonacci_base()
    for N in (2, 3, 4, 1000, 1024, 1025, 4096, 131072):
        assert fa.fib_attn_base(fa.FIB_BASE_POW2, N) == oracle.pow2_base(N)


@pytest.mark.parametrize("kind,name", [(fa.FIB_SCHED_FIXED, "fixed"), (fa.FIB_SCHED_LINEAR, "linear"),
                                       (fa.FIB_SCHED_COPRIME, "coprime")])
@pytest.mark.parametrize("L", [2, 3, 16, 33])
def test_schedules_match_oracle_bit_exact(kind, name, L):
    if name == "coprime" and np.gcd(7, L) != 1:
        with pytest.raises(fa.FibAttnError):
            fa.fib_attn_schedule(kind, L, 7)
        return
    got = fa.fib_attn_schedule(kind, L, 7)
    want = oracle.schedule(name, L, 7)
    assert got == want  # bit-exact binary64


def _alphas():
    out = oracle.schedule("linear", 16) + oracle.schedule("coprime", 16)
    out += list(np.random.default_rng(5).uniform(0.5, 1.5, 40)) + [0.5, 1.0, 1.5, 1.1, 0.7]
    return out


@pytest.mark.parametrize("W,N", [(12, 1024), (12, 4096), (8, 256), (10, 1024), (12, 131072), (1, 50),
                                 (64, 100)])
def test_mask_distances_match_oracle(W, N):
    for base in (oracle.fibonacci_base(), oracle.pow2_base(N), [3, 7, 7, 100]):
        for a in _alphas():
            assert fa.fib_attn_mask_distances(base, a, W, N) == oracle.mask_distances(base, a, W, N)


@pytest.mark.parametrize("W,N", [(10, 1024), (12, 131072), (8, 256), (1, 40)])
def test_interp_rungs_match_oracle(W, N):
    for base in (oracle.fibonacci_base(), oracle.pow2_base(N), [5, 5, 9]):
        for a in _alphas() + list(np.random.default_rng(6).uniform(0.9, 1.1, 20).astype(np.float32)):
            got = fa.fib_attn_interp_rungs(base, float(a), W, N)
            want = oracle.interp_rungs(base, float(a), W, N)
            assert [(f, lo) for f, lo, _ in got] == [(f, lo) for f, lo, _ in want]
            for (_, _, w1), (_, _, w2) in zip(got, want):
                assert w1 == np.float32(w2)  # float32 rounding of the same binary64 w


def test_host_error_paths():
    lib = fa.lib()
    n = ctypes.c_int(0)
    assert lib.fib_attn_base(7, 10, None, 0, ctypes.byref(n)) == fa.FIB_ERR_INVALID_ARG
    assert lib.fib_attn_base(fa.FIB_BASE_POW2, 1, None, 0, ctypes.byref(n)) == fa.FIB_ERR_INVALID_ARG
    assert lib.fib_attn_base(fa.FIB_BASE_FIBONACCI, 10, None, 0, None) == fa.FIB_ERR_INVALID_ARG
    out = (ctypes.c_double * 4)()
    assert lib.fib_attn_schedule(fa.FIB_SCHED_LINEAR, 1, 7, out) == fa.FIB_ERR_INVALID_ARG
    assert lib.fib_attn_schedule(fa.FIB_SCHED_COPRIME, 14, 7, out) == fa.FIB_ERR_INVALID_ARG
    assert lib.fib_attn_schedule(9, 4, 7, out) == fa.FIB_ERR_INVALID_ARG
    assert lib.fib_attn_schedule(fa.FIB_SCHED_FIXED, 0, 7, out) == fa.FIB_ERR_INVALID_ARG
    b = (ctypes.c_int32 * 2)(1, 2)
    d = (ctypes.c_int32 * 4)()
    for alpha, W, N in ((0.0, 4, 10), (float("nan"), 4, 10), (1.0, 0, 10), (1.0, 4, 0)):
        assert lib.fib_attn_mask_distances(b, 2, alpha, W, N, d, 4, ctypes.byref(n)) == fa.FIB_ERR_INVALID_ARG
    bad = (ctypes.c_int32 * 2)(0, 2)
    assert lib.fib_attn_mask_distances(bad, 2, 1.0, 1, 10, d, 4, ctypes.byref(n)) == fa.FIB_ERR_INVALID_ARG
    # a short output buffer is filled up to cap and the full count reported
    base = (ctypes.c_int32 * 15)(*oracle.fibonacci_base())
    assert lib.fib_attn_mask_distances(base, 15, 1.0, 1, 5000, d, 4, ctypes.byref(n)) == fa.FIB_OK
    assert n.value == 15 and list(d) == [1, 2, 3, 5]


def test_plan_create_rejects_bad_arguments_before_any_device_call():
    lib = fa.lib()
    h = ctypes.c_void_p()
    a = (ctypes.c_double * 2)(1.0, 1.0)
    args = dict(kind=0, cb=None, nc=0, a=a, L=2, W=12, N=1024, D=64, mode=0, rb=10000.0)

    def call(**kw):
        x = dict(args, **kw)
        return lib.fib_attn_plan_create(ctypes.byref(h), x["kind"], x["cb"], x["nc"], x["a"], x["L"],
                                        x["W"], x["N"], x["D"], x["mode"], x["rb"])

    assert call(D=128) == fa.FIB_ERR_UNSUPPORTED
    assert call(W=0) == fa.FIB_ERR_INVALID_ARG
    assert call(W=65) == fa.FIB_ERR_INVALID_ARG
    assert call(N=0) == fa.FIB_ERR_INVALID_ARG
    assert call(mode=2) == fa.FIB_ERR_INVALID_ARG
    assert call(kind=2) == fa.FIB_ERR_INVALID_ARG            # custom without a list
    assert call(rb=1.0) == fa.FIB_ERR_INVALID_ARG
    assert call(a=(ctypes.c_double * 2)(1.0, -1.0)) == fa.FIB_ERR_INVALID_ARG
    assert lib.fib_attn_plan_create(None, 0, None, 0, a, 2, 12, 1024, 64, 0, 10000.0) == fa.FIB_ERR_INVALID_ARG
    assert lib.fib_attn_plan_destroy(None) == fa.FIB_OK
    assert lib.fib_attn_fwd(None, 0, 1, 1, 1, 0, None, None, None, None, None, None, None, 0,
                            None) == fa.FIB_ERR_INVALID_ARG
    assert lib.fib_attn_fwd_workspace_size(None, 1, 1, 1, fa.FIB_DTYPE_BF16) == 0
    assert lib.fib_attn_last_device_status(None) == fa.FIB_ERR_INVALID_ARG
    assert lib.fib_attn_bwd_workspace_size(None, 1, 1, 1) == 0
