"""Plain float64 CPU oracle for Depth-Staggered Fibonacci Spacing sparse attention.

TEST INFRASTRUCTURE ONLY.  This module is the slow, obviously-correct statement of
what the attention computes.  Only the test-suite, the smoke check and the CPU-baseline
leg of the benchmark may import it; the product library never calls it, and it shares
no code, tables or constants with the CUDA path.

Source: "Depth-Staggered Fibonacci Spacing for Sparse Attention: Static Schedules Beat
Learned Dilation and Extrapolate Where Dense Attention Fails" (gist.science technical
summary, Korean and Spanish editions), section "Methodology":
  * "Attended set": each query at position i attends to a dense local window of size W
    plus a sparse offset set built from the Fibonacci list fib = [1, 2, 3, 5, ..., 987].
  * "Scaling": every offset f_k is scaled by a per-layer scalar alpha into the target
    distance d_k = alpha * f_k, with alpha restricted to [0.5, 1.5].
  * "Implementation": non-integer offsets are served by linear interpolation between the
    two bracketing key/value rows, so that alpha receives a gradient; rotary position
    embedding (RoPE) is applied before the rows are gathered.
  * "Experimental variables": fixed (alpha = 1), learned (free per-layer parameter,
    initialised at alpha = 1), staggered linear (0.5 at layer 0 to 1.5 at layer 15),
    staggered coprime (the linear multiset reassigned by l -> 7 l mod L).
  * "Controls": a reach-matched power-of-two ("log-sparse") base.
  * Section "Key results" 2, "Efficiency": static (integer) schedules take a fused
    boolean-mask path, non-integer ones an interpolated gather.

Readings taken where the pages are silent (each one is restated where it is used):
  R1  the window of size W holds distances 0..W-1, i.e. it includes the query itself;
  R2  the attended set is a set: mask-mode rungs are kept iff d >= W (integer d) and
      deduplicated; interp-mode rungs are kept iff d > W-1;
  R3  a static non-integer distance alpha*f is rounded half-to-even, applied to the
      binary64 product of the binary64 alpha and the integer f;
  R4  a rung is attended by query i iff its (real) distance d <= i: no padding, no clamp;
  R5  the softmax scale is 1/sqrt(D);
  R6  RoPE pairs dimension m with m + D/2 ("rotate half"), positions 0..N-1, angle
      p * base^(-2m/D), base 10000, no scaling;
  R7  K is rotated at its own integer position, then blended; V is never rotated;
  R8  dalpha at an integer distance is the right derivative (lo held fixed, dw/dalpha = f);
      where the second bracketing row i-lo-1 does not exist (i == lo, w == 0) that
      derivative term is taken as zero;
  R9  the learned theta -> alpha map lies outside the attention op: the op returns
      dL/dalpha;
  R10 the coprime schedule is alpha_cop[l] = alpha_lin[(7 l) mod L];
  R11 the power-of-two base is {2^k : 2^k < N};
  R12 alpha is one scalar per layer, shared by every batch row and head.

All arrays are float64 numpy arrays of layout [B, H, N, D] (LSE: [B, H, N]).
"""
from __future__ import annotations

import math

import numpy as np

MODE_MASK = "mask"
MODE_INTERP = "interp"


# --------------------------------------------------------------------------------------
# Base lists and schedules ("Attended set", "Controls", "Experimental variables")
# --------------------------------------------------------------------------------------
def fibonacci_base(limit: int = 987) -> list[int]:
    """Fibonacci numbers 1, 2, 3, 5, ... up to `limit`, the repeated leading 1 dropped.

    Follows "Attended set": fib = [1, 2, 3, 5, ..., 987].
    """
    out = [1, 2]
    while out[-1] + out[-2] <= limit:
        out.append(out[-1] + out[-2])
    return [f for f in out if f <= limit]


def pow2_base(n: int) -> list[int]:
    """Reach-matched power-of-two control base, read as {2^k : 2^k < n} (reading R11).

    Follows "Controls" (log-sparse base) and "Base sensitivity" (offsets 1024 and 2048
    appear at evaluation length 4096).
    """
    out = []
    p = 1
    while p < n:
        out.append(p)
        p *= 2
    return out


def schedule(kind: str, n_layers: int, stride: int = 7) -> list[float]:
    """Per-layer alpha for the four schedules of "Experimental variables".

    fixed:   alpha = 1 for every layer.
    linear:  a ramp from 0.5 at layer 0 to 1.5 at the last layer, 0.5 + l/(L-1) in binary64.
    coprime: the linear multiset reassigned by the coprime stride, alpha_lin[(stride*l) mod L]
             (reading R10).
    The learned schedule is caller-supplied (reading R9).
    """
    L = int(n_layers)
    if L < 1:
        raise ValueError("n_layers must be >= 1")
    if kind == "fixed":
        return [1.0] * L
    if kind in ("linear", "coprime"):
        if L < 2:
            raise ValueError("a ramp needs at least two layers")
        lin = [0.5 + l / float(L - 1) for l in range(L)]
        if kind == "linear":
            return lin
        if math.gcd(stride, L) != 1:
            raise ValueError("stride must be coprime with the layer count")
        return [lin[(stride * l) % L] for l in range(L)]
    raise ValueError(f"unknown schedule {kind!r}")


def round_half_even(x: float) -> int:
    """Round-half-to-even of a binary64 value (reading R3)."""
    return int(np.round(np.float64(x)))


def mask_distances(base, alpha: float, W: int, N: int) -> list[int]:
    """Static ("boolean mask") rung distances of one layer.

    d = round_half_even(alpha (x) f) for every f in the base (reading R3); keep d >= W (the
    window already holds 0..W-1, readings R1-R2) and d <= N-1 (a larger distance is never
    causal at length N); sorted, duplicates removed.  Follows "Scaling": d_k = alpha f_k.
    """
    ds = set()
    for f in base:
        d = round_half_even(np.float64(alpha) * np.float64(f))
        if W <= d <= N - 1:
            ds.add(d)
    return sorted(ds)


def interp_rungs(base, alpha: float, W: int, N: int):
    """Interpolated rungs of one layer: list of (f, lo, w) with d = alpha*f.

    Keep a rung iff d > W-1 (so that neither bracketing row falls inside the window
    except at integer d, reading R2) and d <= N-1 (else never causal).  lo = floor(d),
    w = d - lo; the virtual key is (1-w) row(i-lo) + w row(i-lo-1) ("Implementation").
    Duplicated base entries give one rung.
    """
    out = []
    for f in sorted(set(int(x) for x in base)):
        d = np.float64(alpha) * np.float64(f)
        if d > W - 1 and d <= N - 1:
            lo = math.floor(d)
            out.append((int(f), int(lo), float(d - lo)))
    return out


# --------------------------------------------------------------------------------------
# RoPE (reading R6), applied before the gather ("Implementation")
# --------------------------------------------------------------------------------------
def rope_angles(n: int, D: int, rope_base: float = 10000.0) -> np.ndarray:
    """angle[p, m] = p * rope_base^(-2m/D) for p < n, m < D/2 (float64)."""
    m = np.arange(D // 2, dtype=np.float64)
    theta = rope_base ** (-2.0 * m / D)
    p = np.arange(n, dtype=np.float64)
    return p[:, None] * theta[None, :]


def rope(x: np.ndarray, rope_base: float = 10000.0, inverse: bool = False) -> np.ndarray:
    """Rotate-half RoPE of x[..., N, D] at positions 0..N-1; inverse=True rotates back."""
    N, D = x.shape[-2], x.shape[-1]
    ang = rope_angles(N, D, rope_base)
    c, s = np.cos(ang), np.sin(ang)
    if inverse:
        s = -s
    x1, x2 = x[..., : D // 2], x[..., D // 2:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


# --------------------------------------------------------------------------------------
# The attended set, as a list of virtual keys per layer
# --------------------------------------------------------------------------------------
def virtual_keys(base, alpha: float, W: int, N: int, mode: str):
    """Virtual keys shared by every query of a layer.

    Each entry is (dist, lo, w, f): query i reads (1-w) row(i-lo) + w row(i-lo-1) when
    dist <= i (reading R4).  Window keys: dist = lo = t for t < W, w = 0, f = 0.
    Mask rungs: dist = lo = d, w = 0, f = 0.  Interp rungs: dist = alpha*f, lo, w, f.
    """
    keys = [(float(t), t, 0.0, 0) for t in range(W)]
    if mode == MODE_MASK:
        keys += [(float(d), d, 0.0, 0) for d in mask_distances(base, alpha, W, N)]
    elif mode == MODE_INTERP:
        keys += [(float(np.float64(alpha) * np.float64(f)), lo, w, f)
                 for (f, lo, w) in interp_rungs(base, alpha, W, N)]
    else:
        raise ValueError(mode)
    return keys


def index_sets(base, alpha: float, W: int, N: int, mode: str):
    """Per query i the attended rows: a list of (row_lo, w) in virtual-key order.

    row_lo = i - lo; the second row (row_lo - 1) carries weight w, the first 1 - w.
    """
    keys = virtual_keys(base, alpha, W, N, mode)
    out = []
    for i in range(N):
        out.append([(i - lo, w) for (dist, lo, w, f) in keys if dist <= i])
    return out


def _shift(x: np.ndarray, s: int) -> np.ndarray:
    """y[..., i, :] = x[..., i - s, :] where 0 <= i - s < N, else 0."""
    y = np.zeros_like(x)
    N = x.shape[-2]
    if s >= 0:
        if s < N:
            y[..., s:, :] = x[..., : N - s, :]
    else:
        if -s < N:
            y[..., : N + s, :] = x[..., -s:, :]
    return y


def _gather(rows: np.ndarray, lo: int, w: float) -> np.ndarray:
    """Blend (1-w) rows[i-lo] + w rows[i-lo-1] for every i (out-of-range rows read as 0)."""
    g = (1.0 - w) * _shift(rows, lo)
    if w != 0.0:
        g = g + w * _shift(rows, lo + 1)
    return g


# --------------------------------------------------------------------------------------
# Forward
# --------------------------------------------------------------------------------------
def attend(q, k, v, alpha: float, base, W: int, mode: str = MODE_MASK,
           rope_base: float = 10000.0):
    """One layer of the sparse attention, float64.  Returns (O [B,H,N,D], LSE [B,H,N]).

    Steps ("Attended set", "Scaling", "Implementation"):
      1. q' = rope(q), k' = rope(k) at positions 0..N-1; v is not rotated.
      2. for every virtual key c of the layer, the blended key/value row and the score
         s_c(i) = q'_i . k~_c(i) / sqrt(D), valid iff dist_c <= i.
      3. LSE(i) = log sum_c exp s_c(i) (max-stabilised); O(i) = sum_c exp(s_c - LSE) v~_c.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    N, D = q.shape[-2], q.shape[-1]
    qr, kr = rope(q, rope_base), rope(k, rope_base)
    keys = virtual_keys(base, alpha, W, N, mode)
    pos = np.arange(N, dtype=np.float64)
    scale = 1.0 / math.sqrt(D)
    S = np.full(q.shape[:-1] + (len(keys),), -np.inf)
    for c, (dist, lo, w, f) in enumerate(keys):
        kt = _gather(kr, lo, w)
        s = np.einsum("...nd,...nd->...n", qr, kt) * scale
        S[..., c] = np.where(pos >= dist, s, -np.inf)
    m = S.max(axis=-1)
    lse = m + np.log(np.exp(S - m[..., None]).sum(axis=-1))
    O = np.zeros_like(q)
    for c, (dist, lo, w, f) in enumerate(keys):
        p = np.exp(S[..., c] - lse)
        O += p[..., None] * _gather(v, lo, w)
    return O, lse


# --------------------------------------------------------------------------------------
# Backward for the loss l = sum(O * dO)
# --------------------------------------------------------------------------------------
def attend_bwd(q, k, v, dO, alpha: float, base, W: int, mode: str = MODE_INTERP,
               rope_base: float = 10000.0):
    """Gradients (dq, dk, dv, dalpha) of l = sum(O * dO), float64.

    Standard softmax backward on the virtual keys: P = exp(s - LSE), dP = dO . v~,
    Delta = sum_c P dP (= dO . O), dS = P (dP - Delta).  dq' = sum_c dS k~ / sqrt(D);
    each blended key/value row scatters its gradient back to its two source rows with
    weights (1-w) and w; dq, dk are rotated back by the inverse RoPE.  dalpha follows
    "Implementation" (interpolation gives alpha a gradient): for an interp rung with
    d = alpha f, dw/dalpha = f with lo held fixed (reading R8), so
      dalpha = sum_{i,c} f_c [dS (q'_i . (k'[i-lo-1] - k'[i-lo])) / sqrt(D)
                              + P dO_i . (v[i-lo-1] - v[i-lo])]
    summed over batch rows and heads (reading R12).  Mask mode has no dalpha (0).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    dO = np.asarray(dO, dtype=np.float64)
    N, D = q.shape[-2], q.shape[-1]
    qr, kr = rope(q, rope_base), rope(k, rope_base)
    O, lse = attend(q, k, v, alpha, base, W, mode, rope_base)
    keys = virtual_keys(base, alpha, W, N, mode)
    pos = np.arange(N, dtype=np.float64)
    scale = 1.0 / math.sqrt(D)
    delta = np.einsum("...nd,...nd->...n", dO, O)
    dqr = np.zeros_like(q)
    dkr = np.zeros_like(k)
    dv = np.zeros_like(v)
    dalpha = 0.0
    for (dist, lo, w, f) in keys:
        valid = pos >= dist
        kt, vt = _gather(kr, lo, w), _gather(v, lo, w)
        s = np.einsum("...nd,...nd->...n", qr, kt) * scale
        p = np.where(valid, np.exp(np.where(valid, s, 0.0) - lse), 0.0)
        dp = np.einsum("...nd,...nd->...n", dO, vt)
        ds = p * (dp - delta)
        dqr += (ds * scale)[..., None] * kt
        gk = (ds * scale)[..., None] * qr          # gradient w.r.t. the blended key row
        gv = p[..., None] * dO                     # gradient w.r.t. the blended value row
        # row i-lo gets (1-w) of it, row i-lo-1 gets w of it
        dkr += (1.0 - w) * _shift(gk, -lo)
        dv += (1.0 - w) * _shift(gv, -lo)
        if w != 0.0:
            dkr += w * _shift(gk, -(lo + 1))
            dv += w * _shift(gv, -(lo + 1))
        if mode == MODE_INTERP and f != 0:
            # rows i-lo-1 exist iff i >= lo+1; where they do not the term is zero (R8)
            has2 = valid & (pos >= lo + 1)
            term = _dw_term(ds * scale, p, qr, dO,
                            _shift(kr, lo + 1) - _shift(kr, lo),
                            _shift(v, lo + 1) - _shift(v, lo))
            dalpha += f * float(np.where(has2, term, 0.0).sum())
    dq = rope(dqr, rope_base, inverse=True)
    dk = rope(dkr, rope_base, inverse=True)
    return dq, dk, dv, dalpha


def _dw_term(ds_scaled, p, qr, dO, dk_rows, dv_rows):
    """dl/dw of one rung per query: the blended key moves along k'[i-lo-1] - k'[i-lo]
    (through the score) and the blended value along v[i-lo-1] - v[i-lo]."""
    return ds_scaled * np.einsum("...nd,...nd->...n", qr, dk_rows) \
        + p * np.einsum("...nd,...nd->...n", dO, dv_rows)
