"""Pins of the float64 oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: values the pages print
(tests/golden/), closed forms, brute force on tiny inputs, a library routine in a special
case (torch scaled-dot-product attention), an independent autograd formulation, and
central finite differences.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from fibonacci_offset_sparse_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _kv(path):
    out = {}
    for line in open(os.path.join(GOLDEN, path)):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        k, v = line.split(":", 1)
        out[k.strip()] = v.split()
    return out


def _rhe_exact(alpha, f):
    """Round-half-even, in rational arithmetic, of the binary64 product alpha (x) f
    (Python's Fraction -> float conversion rounds the exact product to nearest, ties
    to even, as an IEEE multiply does)."""
    x = Fraction(float(Fraction(float(alpha)) * int(f)))
    fl = x.numerator // x.denominator
    rem = x - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        return fl + 1
    return fl


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


# ----------------------------------------------------------------------------- bases
def test_fibonacci_base_matches_pages():
    g = _kv("fibonacci_base.txt")
    fib = oracle.fibonacci_base()
    assert fib[:4] == [int(x) for x in g["first"]]
    assert fib[-1] == int(g["last"][0])
    assert len(fib) == 15
    for a, b, c in zip(fib, fib[1:], fib[2:]):
        assert c == a + b
    assert len(set(fib)) == len(fib)


def test_pow2_base_offsets_at_eval_length():
    g = _kv("pow2_eval4096.txt")
    n_eval, n_train = int(g["N_eval"][0]), int(g["N_train"][0])
    b_eval, b_train = oracle.pow2_base(n_eval), oracle.pow2_base(n_train)
    for x in g["present_at_eval"]:
        assert int(x) in b_eval and int(x) not in b_train
    assert all(b < n_eval for b in b_eval) and all(2 * b == c for b, c in zip(b_eval, b_eval[1:]))
    assert b_eval[0] == 1


# ----------------------------------------------------------------------------- schedules
def test_schedules_match_pages():
    g = _kv("schedules.txt")
    L = int(g["layers"][0])
    lin = oracle.schedule("linear", L)
    assert lin[0] == float(g["linear_layer0"][0]) and lin[-1] == float(g["linear_layer15"][0])
    steps = np.diff(lin)
    assert np.allclose(steps, steps[0], rtol=0, atol=1e-12)      # a linear ramp
    assert min(lin) >= float(g["alpha_min"][0]) and max(lin) <= float(g["alpha_max"][0])
    assert oracle.schedule("fixed", L) == [float(g["fixed"][0])] * L
    cop = oracle.schedule("coprime", L, int(g["coprime_stride"][0]))
    assert sorted(cop) == sorted(lin)                             # same multiset, exactly
    # each layer l takes the ramp value of layer 7 l mod L
    for l in range(L):
        assert cop[l] == lin[(7 * l) % L]
    # the stride spreads adjacent layers apart: every adjacent jump is larger than the ramp's
    assert min(abs(np.diff(cop))) > max(abs(steps)) * 5


# ----------------------------------------------------------------------------- distances
def test_rounding_cases_by_hand():
    for line in open(os.path.join(GOLDEN, "rounding_cases.txt")):
        if line.startswith("#") or not line.strip():
            continue
        a, f, d = line.split()[:3]
        assert oracle.round_half_even(float(a) * int(f)) == int(d), line
        assert _rhe_exact(float(a), int(f)) == int(d), line


@pytest.mark.parametrize("sched,L,N,base", [
    ("linear", 16, 1024, "fib"), ("coprime", 16, 4096, "fib"), ("coprime", 16, 4096, "pow2"),
    ("fixed", 1, 256, "fib")])
def test_mask_distances_vs_exact_rational(sched, L, N, base):
    W = 12
    for a in oracle.schedule(sched, L):
        b = oracle.fibonacci_base() if base == "fib" else oracle.pow2_base(N)
        want = sorted({_rhe_exact(a, f) for f in b} & set(range(W, N)))
        assert oracle.mask_distances(b, a, W, N) == want


def _brute_mask_sets(base, alpha, W, N):
    ds = {_rhe_exact(alpha, f) for f in base}
    return [sorted(j for j in range(i + 1) if (i - j) < W or (i - j) in ds) for i in range(N)]


@pytest.mark.parametrize("alpha,W,N", [(1.0, 8, 256), (0.5, 12, 300), (1.5, 12, 1500),
                                       (1.1, 6, 200), (0.5 + 13 / 15, 10, 700), (1.0, 1, 40)])
def test_mask_index_sets_bruteforce(alpha, W, N):
    base = oracle.fibonacci_base()
    got = oracle.index_sets(base, alpha, W, N, oracle.MODE_MASK)
    want = _brute_mask_sets(base, alpha, W, N)
    for i in range(N):
        rows = [r for (r, w) in got[i]]
        assert all(w == 0.0 for (r, w) in got[i])
        assert len(rows) == len(set(rows)), i            # a set: no key twice
        assert sorted(rows) == want[i], i


@pytest.mark.parametrize("alpha,W,N", [(1.23, 8, 400), (0.61, 12, 300), (1.0, 10, 200),
                                       (1.4999, 12, 1500)])
def test_interp_index_sets_bruteforce(alpha, W, N):
    base = oracle.fibonacci_base()
    got = oracle.index_sets(base, alpha, W, N, oracle.MODE_INTERP)
    for i in range(N):
        want = [(i - t, 0.0) for t in range(W) if t <= i]
        for f in base:
            d = Fraction(float(alpha)) * f  # exact product of the binary64 alpha
            if d > W - 1 and d <= i:
                lo = d.numerator // d.denominator
                want.append((i - lo, float(d - lo)))
        assert len(got[i]) == len(want)
        for (r, w), (r2, w2) in zip(got[i], want):
            assert r == r2 and abs(w - w2) < 1e-12
            if w > 0:
                assert r - 1 >= 0                      # both bracketing rows exist


# ----------------------------------------------------------------------------- RoPE
def _rope_complex(x, rope_base=10000.0):
    """Textbook complex form: pair (x_m, x_{m+D/2}) as x_m + i x_{m+D/2}, times
    exp(i p rope_base^(-2m/D))."""
    N, D = x.shape[-2], x.shape[-1]
    z = x[..., : D // 2] + 1j * x[..., D // 2:]
    p = np.arange(N)[:, None]
    m = np.arange(D // 2)[None, :]
    z = z * np.exp(1j * p * rope_base ** (-2.0 * m / D))
    return np.concatenate([z.real, z.imag], axis=-1)


def test_rope_closed_forms():
    # D = 2: the single frequency is 1 rad per position; (1, 0) at p -> (cos p, sin p)
    x = np.zeros((5, 2))
    x[:, 0] = 1.0
    y = oracle.rope(x)
    p = np.arange(5)
    assert np.allclose(y[:, 0], np.cos(p), atol=1e-15) and np.allclose(y[:, 1], np.sin(p), atol=1e-15)
    x = _rand((2, 3, 37, 64), 1)
    assert np.allclose(oracle.rope(x), _rope_complex(x), rtol=0, atol=1e-12)
    assert np.allclose(oracle.rope(x)[..., 0, :], x[..., 0, :], atol=0)       # identity at p = 0
    assert np.allclose(np.linalg.norm(oracle.rope(x), axis=-1), np.linalg.norm(x, axis=-1))
    assert np.allclose(oracle.rope(oracle.rope(x), inverse=True), x, atol=1e-12)


def test_rope_relative_position():
    q, k = _rand((1, 64), 2), _rand((1, 64), 3)
    N = 300
    qs, ks = np.repeat(q, N, 0), np.repeat(k, N, 0)
    qr, kr = oracle.rope(qs), oracle.rope(ks)
    for delta in (0, 1, 13, 144):
        dots = [qr[i] @ kr[i - delta] for i in range(delta, N)]
        assert np.allclose(dots, dots[0], rtol=0, atol=1e-10)


# ----------------------------------------------------------------------------- forward
def test_window_covering_sequence_is_dense_causal():
    B, H, N, D = 2, 2, 48, 64
    q, k, v = (_rand((B, H, N, D), s) for s in (4, 5, 6))
    for mode in (oracle.MODE_MASK, oracle.MODE_INTERP):
        O, lse = oracle.attend(q, k, v, 1.3, oracle.fibonacci_base(), W=N, mode=mode)
        qt, kt = torch.from_numpy(_rope_complex(q)), torch.from_numpy(_rope_complex(k))
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, torch.from_numpy(v),
                                                               is_causal=True)
        assert np.allclose(O, ref.numpy(), rtol=0, atol=1e-12)
        s = (qt @ kt.transpose(-1, -2) / math.sqrt(D)).numpy()
        s = np.where(np.tril(np.ones((N, N), bool)), s, -np.inf)
        assert np.allclose(lse, np.logaddexp.reduce(s, axis=-1), atol=1e-12)


def _dense_masked(q, k, v, allowed):
    """Dense softmax attention with an explicit boolean mask, float64 (textbook)."""
    D = q.shape[-1]
    qr, kr = _rope_complex(q), _rope_complex(k)
    s = np.einsum("bhid,bhjd->bhij", qr, kr) / math.sqrt(D)
    s = np.where(allowed, s, -np.inf)
    m = s.max(-1, keepdims=True)
    e = np.exp(s - m)
    lse = (m + np.log(e.sum(-1, keepdims=True)))[..., 0]
    return np.einsum("bhij,bhjd->bhid", e / e.sum(-1, keepdims=True), v), lse


@pytest.mark.parametrize("W,N", [(8, 256), (12, 130), (3, 64)])
def test_alpha_one_interp_equals_mask_equals_dense_masked(W, N):
    B, H, D = 1, 2, 64
    q, k, v = (_rand((B, H, N, D), s) for s in (7, 8, 9))
    base = oracle.fibonacci_base()
    for _, lo, w, _f in oracle.virtual_keys(base, 1.0, W, N, oracle.MODE_INTERP):
        assert w == 0.0
    Om, lm = oracle.attend(q, k, v, 1.0, base, W, oracle.MODE_MASK)
    Oi, li = oracle.attend(q, k, v, 1.0, base, W, oracle.MODE_INTERP)
    assert np.allclose(Om, Oi, rtol=0, atol=1e-13) and np.allclose(lm, li, atol=1e-13)
    sets = _brute_mask_sets(base, 1.0, W, N)
    allowed = np.zeros((N, N), bool)
    for i, js in enumerate(sets):
        allowed[i, js] = True
    Od, ld = _dense_masked(q, k, v, allowed)
    assert np.allclose(Om, Od, rtol=0, atol=1e-12) and np.allclose(lm, ld, atol=1e-12)


def _bruteforce_attend(q, k, v, alpha, base, W, mode):
    """Per-query pure-python statement of the attended set and the softmax, float64."""
    N, D = q.shape[-2], q.shape[-1]
    qr, kr = _rope_complex(q), _rope_complex(k)
    O = np.zeros_like(q)
    lse = np.zeros(q.shape[:-1])
    for b in range(q.shape[0]):
        for h in range(q.shape[1]):
            for i in range(N):
                keys, vals = [], []
                for t in range(min(W, i + 1)):
                    keys.append(kr[b, h, i - t])
                    vals.append(v[b, h, i - t])
                if mode == "mask":
                    ds = sorted({_rhe_exact(alpha, f) for f in base})
                    for d in ds:
                        if d >= W and d <= i:
                            keys.append(kr[b, h, i - d])
                            vals.append(v[b, h, i - d])
                else:
                    for f in sorted(set(base)):
                        d = float(alpha) * f
                        if d > W - 1 and d <= i:
                            lo = math.floor(d)
                            w = d - lo
                            j = i - lo
                            kk = (1 - w) * kr[b, h, j] + (w * kr[b, h, j - 1] if w else 0)
                            vv = (1 - w) * v[b, h, j] + (w * v[b, h, j - 1] if w else 0)
                            keys.append(kk)
                            vals.append(vv)
                s = np.array([qr[b, h, i] @ kk for kk in keys]) / math.sqrt(D)
                m = s.max()
                e = np.exp(s - m)
                lse[b, h, i] = m + math.log(e.sum())
                O[b, h, i] = (e[:, None] * np.array(vals)).sum(0) / e.sum()
    return O, lse


@pytest.mark.parametrize("mode,alpha,W,N", [("interp", 1.2345, 8, 120), ("interp", 0.6180, 4, 90),
                                            ("mask", 0.5 + 4 / 15, 12, 150), ("mask", 1.5, 6, 60)])
def test_forward_bruteforce_tiny(mode, alpha, W, N):
    B, H, D = 1, 2, 16
    q, k, v = (_rand((B, H, N, D), s) for s in (10, 11, 12))
    base = oracle.fibonacci_base()
    O, lse = oracle.attend(q, k, v, alpha, base, W, mode)
    O2, lse2 = _bruteforce_attend(q, k, v, alpha, base, W, mode)
    assert np.allclose(O, O2, rtol=0, atol=1e-12) and np.allclose(lse, lse2, rtol=0, atol=1e-12)


def test_first_query_closed_form():
    q, k, v = (_rand((2, 3, 50, 64), s) for s in (13, 14, 15))
    for mode, a in (("mask", 1.0), ("interp", 1.37)):
        O, lse = oracle.attend(q, k, v, a, oracle.fibonacci_base(), 12, mode)
        assert np.array_equal(O[..., 0, :], v[..., 0, :]) or np.allclose(O[..., 0, :], v[..., 0, :], atol=1e-15)
        assert np.allclose(lse[..., 0], (q[..., 0, :] * k[..., 0, :]).sum(-1) / 8.0, atol=1e-13)


@pytest.mark.parametrize("mode,alpha", [("interp", 1.31), ("interp", 0.77), ("mask", 0.9)])
def test_zero_keys_give_mean_of_attended_values(mode, alpha):
    """With k = 0 every score is 0: O(i) is the plain mean of the attended value rows,
    each interpolated row weighted (1-w, w) between its two source rows; LSE = log count."""
    B, H, N, D, W = 1, 1, 200, 64, 8
    v = _rand((B, H, N, D), 16)
    q = _rand((B, H, N, D), 17)
    k = np.zeros_like(q)
    base = oracle.fibonacci_base()
    O, lse = oracle.attend(q, k, v, alpha, base, W, mode)
    for i in (0, 5, 7, 8, 40, 99, 199):
        rows = oracle.index_sets(base, alpha, W, N, mode)[i]
        acc = np.zeros(D)
        for (r, w) in rows:
            acc += (1 - w) * v[0, 0, r] + (w * v[0, 0, r - 1] if w else 0)
        assert np.allclose(O[0, 0, i], acc / len(rows), atol=1e-13)
        assert abs(lse[0, 0, i] - math.log(len(rows))) < 1e-13


# ----------------------------------------------------------------------------- backward
def _torch_attend(q, k, v, alpha, base, W, mode):
    """Autograd formulation: alpha is a tensor, d = alpha f, lo = floor(d) (no gradient),
    w = d - lo; each query gathers its virtual keys by index."""
    N, D = q.shape[-2], q.shape[-1]
    pos = torch.arange(N, dtype=torch.float64)
    half = D // 2
    ang = pos[:, None] * (10000.0 ** (-2.0 * torch.arange(half, dtype=torch.float64) / D))[None, :]
    c, s = torch.cos(ang), torch.sin(ang)

    def rot(x):
        return torch.cat([x[..., :half] * c - x[..., half:] * s, x[..., half:] * c + x[..., :half] * s], -1)

    qr, kr = rot(q), rot(k)
    ar = torch.arange(N)
    scores, vals = [], []
    for t in range(W):
        idx = (ar - t).clamp(min=0)
        ok = ar >= t
        scores.append(torch.where(ok, (qr * kr[..., idx, :]).sum(-1), torch.tensor(-math.inf, dtype=torch.float64)))
        vals.append(v[..., idx, :])
    seen = set()
    for f in sorted(set(base)):
        d = alpha * f
        if mode == "mask":
            dd = _rhe_exact(float(alpha), f)
            if not (dd >= W and dd <= N - 1) or dd in seen:
                continue
            seen.add(dd)
            lo, w = dd, alpha * 0.0
            valid = ar >= dd
        else:
            if not (float(d) > W - 1 and float(d) <= N - 1):
                continue
            lo = math.floor(float(d))
            w = d - lo
            valid = pos >= d.detach()
        i0 = (ar - lo).clamp(min=0)
        # where the second bracketing row does not exist (only at w == 0) use the first
        # row in its place, so that its derivative term vanishes
        i1 = torch.where(ar - lo - 1 >= 0, ar - lo - 1, i0)
        kk = (1 - w) * kr[..., i0, :] + w * kr[..., i1, :]
        vv = (1 - w) * v[..., i0, :] + w * v[..., i1, :]
        scores.append(torch.where(valid, (qr * kk).sum(-1), torch.tensor(-math.inf, dtype=torch.float64)))
        vals.append(vv)
    S = torch.stack(scores, -1) / math.sqrt(D)
    P = torch.softmax(S, -1)
    return (P[..., None] * torch.stack(vals, -2)).sum(-2)


@pytest.mark.parametrize("mode,alpha,W,N", [("interp", 1.2345, 8, 160), ("interp", 0.7071, 12, 200),
                                            ("interp", 1.0, 10, 120), ("mask", 0.5 + 4 / 15, 12, 150)])
def test_backward_vs_autograd(mode, alpha, W, N):
    B, H, D = 2, 2, 64
    q, k, v, dO = (_rand((B, H, N, D), s) for s in (20, 21, 22, 23))
    base = oracle.fibonacci_base()
    dq, dk, dv, da = oracle.attend_bwd(q, k, v, dO, alpha, base, W, mode)
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    ta = torch.tensor(alpha, dtype=torch.float64, requires_grad=True)
    O = _torch_attend(tq, tk, tv, ta, base, W, mode)
    On, _ = oracle.attend(q, k, v, alpha, base, W, mode)
    assert np.allclose(O.detach().numpy(), On, atol=1e-12)
    (O * torch.from_numpy(dO)).sum().backward()
    assert np.allclose(dq, tq.grad.numpy(), atol=1e-11)
    assert np.allclose(dk, tk.grad.numpy(), atol=1e-11)
    assert np.allclose(dv, tv.grad.numpy(), atol=1e-11)
    if mode == "interp":
        g = float(ta.grad)
        assert abs(da - g) <= 1e-9 * max(1.0, abs(g))
    else:
        assert da == 0.0


def _far_from_kinks(alpha, base, W, N, eps=1e-3):
    for f in base:
        d = alpha * f
        if abs(d - round(d)) < eps or abs(d - (W - 1)) < eps:
            return False
    return True


@pytest.mark.parametrize("alpha,W,N", [(1.2345, 8, 300), (0.8123, 12, 400), (1.4321, 6, 512)])
def test_dalpha_central_differences(alpha, W, N):
    B, H, D = 2, 1, 64
    base = oracle.fibonacci_base()
    assert _far_from_kinks(alpha, base, W, N)
    q, k, v, dO = (_rand((B, H, N, D), s) for s in (30, 31, 32, 33))
    _, _, _, da = oracle.attend_bwd(q, k, v, dO, alpha, base, W, "interp")
    h = 1e-6

    def loss(a):
        return float((oracle.attend(q, k, v, a, base, W, "interp")[0] * dO).sum())

    fd = (loss(alpha + h) - loss(alpha - h)) / (2 * h)
    assert abs(da - fd) <= 1e-5 * abs(fd)


def test_dqkv_central_differences():
    B, H, N, D, W, alpha = 1, 2, 96, 64, 8, 1.2345
    base = oracle.fibonacci_base()
    q, k, v, dO = (_rand((B, H, N, D), s) for s in (40, 41, 42, 43))
    grads = oracle.attend_bwd(q, k, v, dO, alpha, base, W, "interp")[:3]
    rng = np.random.default_rng(44)
    h = 1e-6
    for which, g in zip(range(3), grads):
        for _ in range(6):
            idx = (0, rng.integers(H), rng.integers(N), rng.integers(D))
            args = [q.copy(), k.copy(), v.copy()]
            args[which][idx] += h
            lp = float((oracle.attend(*args, alpha, base, W, "interp")[0] * dO).sum())
            args[which][idx] -= 2 * h
            lm = float((oracle.attend(*args, alpha, base, W, "interp")[0] * dO).sum())
            fd = (lp - lm) / (2 * h)
            assert abs(g[idx] - fd) <= 1e-6 + 1e-5 * abs(fd)


def test_learned_alpha_inputs_are_float32_values():
    a = inputs.learned_alpha(16, 3)
    assert np.all((a >= 0.9) & (a <= 1.1))
    assert np.array_equal(a, a.astype(np.float32).astype(np.float64))
