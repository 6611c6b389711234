"""Plant plausible mistakes in the oracle (on the CPU) and check that a pin catches each.

Each case monkeypatches one oracle helper with a wrong variant, runs one of the pins in
test_oracle.py and expects it to fail.
"""
import numpy as np
import pytest

import oracle
from oracle import fib_oracle as fo
from tests import test_oracle as pins


def _swapped_gather(rows, lo, w):
    g = w * fo._shift(rows, lo)
    if w != 0.0:
        g = g + (1.0 - w) * fo._shift(rows, lo + 1)
    return g


def _rope_wrong_sign(x, rope_base=10000.0, inverse=False):
    return fo.__dict__["_orig_rope"](x, rope_base, not inverse)


def _rope_interleaved(x, rope_base=10000.0, inverse=False):
    D = x.shape[-1]
    perm = np.arange(D).reshape(2, D // 2).T.reshape(-1)  # pairs (0,1),(2,3),...
    y = fo.__dict__["_orig_rope"](x[..., perm], rope_base, inverse)
    out = np.empty_like(y)
    out[..., perm] = y
    return out


def _window_too_wide(base, alpha, W, N, mode):
    return fo.__dict__["_orig_vk"](base, alpha, W + 1, N, mode)


def _keep_rule_shifted(base, alpha, W, N):
    return [(f, lo, w) for (f, lo, w) in fo.__dict__["_orig_ir"](base, alpha, W, N)
            if np.float64(alpha) * f >= W]


def _round_half_up(x):
    return int(np.floor(np.float64(x) + 0.5))


MUTATIONS = {
    "blend weights swapped": ("_gather", _swapped_gather,
                              lambda: pins.test_forward_bruteforce_tiny("interp", 1.2345, 8, 120)),
    "rope sign flipped": ("rope", _rope_wrong_sign, pins.test_rope_closed_forms),
    "rope pairs interleaved": ("rope", _rope_interleaved, pins.test_rope_closed_forms),
    "window one too wide": ("virtual_keys", _window_too_wide,
                            lambda: pins.test_mask_index_sets_bruteforce(0.5, 12, 300)),
    "interp keep rule d >= W": ("interp_rungs", _keep_rule_shifted,
                                lambda: pins.test_interp_index_sets_bruteforce(1.4999, 12, 1500)),
    "round half up": ("round_half_even", _round_half_up, pins.test_rounding_cases_by_hand),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pin_catches_mutation(name, monkeypatch):
    attr, fn, pin = MUTATIONS[name]
    monkeypatch.setitem(fo.__dict__, "_orig_rope", fo.rope)
    monkeypatch.setitem(fo.__dict__, "_orig_vk", fo.virtual_keys)
    monkeypatch.setitem(fo.__dict__, "_orig_ir", fo.interp_rungs)
    monkeypatch.setattr(fo, attr, fn)
    if hasattr(oracle, attr):
        monkeypatch.setattr(oracle, attr, fn)
    with pytest.raises(AssertionError):
        pin()


def _dw_term_no_value(ds_scaled, p, qr, dO, dk_rows, dv_rows):
    return ds_scaled * np.einsum("...nd,...nd->...n", qr, dk_rows)


def _dw_term_sign(ds_scaled, p, qr, dO, dk_rows, dv_rows):
    return -fo.__dict__["_orig_dw"](ds_scaled, p, qr, dO, dk_rows, dv_rows)


@pytest.mark.parametrize("fn", [_dw_term_no_value, _dw_term_sign])
def test_dalpha_mutations_are_caught(fn, monkeypatch):
    monkeypatch.setitem(fo.__dict__, "_orig_dw", fo._dw_term)
    monkeypatch.setattr(fo, "_dw_term", fn)
    with pytest.raises(AssertionError):
        pins.test_backward_vs_autograd("interp", 1.2345, 8, 160)
    with pytest.raises(AssertionError):
        pins.test_dalpha_central_differences(1.2345, 8, 300)
