"""Pins of the fp64 RMSNorm oracle and of the emulator's rsqrt / RMSNorm.

The oracle is checked against exact rational arithmetic (tiny rows), the
closed form of a constant row, exact scale invariance (eps = 0, power-of-two
scales), the unit mean square of a normalised row, and the fp32-then-bf16
residual boundary written out by hand; planted mistakes each fail a pin.
The emulator's rsqrt is swept over 2^-40..2^40 against fp64, and its
RMSNorm agrees with the oracle within one bf16 rounding.
"""
import importlib.util
import math
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np
import pytest

from invariant_selected_token_gb300 import workloads as WL
from oracle import emulator as E
from oracle import rmsnorm as R


def _bits(x):
    return WL.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def pin_brute_force(M):
    getcontext().prec = 40
    rng = np.random.default_rng(1)
    for H in (1, 3, 8):
        x = _bits(rng.standard_normal((2, H)))
        g = _bits(rng.standard_normal(H))
        eps = 1e-3
        y, _ = M.rmsnorm(x, g, eps)
        xd = WL.bf16_bits_to_f32(x).astype(np.float64)
        gd = WL.bf16_bits_to_f32(g).astype(np.float64)
        for t in range(2):
            ms = sum(Fraction(float(v)) ** 2 for v in xd[t]) / H + Fraction(eps)
            inv = 1 / (Decimal(ms.numerator) / Decimal(ms.denominator)).sqrt()
            for i in range(H):
                want = float(Decimal(float(xd[t, i])) * inv * Decimal(float(gd[i])))
                assert abs(y[t, i] - want) <= 1e-14 * max(1.0, abs(want)), (H, t, i)


def pin_constant_row(M):
    H = 64
    for c in (0.5, -3.0, 100.0):
        x = _bits(np.full((1, H), c))
        g = _bits(np.linspace(-2, 2, H))
        eps = 1e-6
        y, _ = M.rmsnorm(x, g, eps)
        want = WL.bf16_bits_to_f32(g).astype(np.float64) * (c / math.sqrt(c * c + eps))
        assert np.all(np.abs(y[0] - want) <= 1e-12 * np.maximum(1, np.abs(want)))


def pin_scale_invariance(M):
    rng = np.random.default_rng(2)
    x = _bits(rng.standard_normal((3, 128)))
    g = _bits(rng.standard_normal(128))
    y0, _ = M.rmsnorm(x, g, 0.0)
    for k in (-3, 5):
        xs = _bits(WL.bf16_bits_to_f32(x) * np.float32(2.0 ** k))
        y1, _ = M.rmsnorm(xs, g, 0.0)
        assert np.all(np.abs(y1 - y0) <= 1e-15 * np.maximum(1, np.abs(y0)))


def pin_unit_mean_square(M):
    rng = np.random.default_rng(3)
    x = _bits(rng.standard_normal((4, 256)) * 7)
    ones = _bits(np.ones(256))
    y, _ = M.rmsnorm(x, ones, 0.0)
    assert np.all(np.abs((y * y).mean(axis=1) - 1.0) <= 1e-13)


def pin_residual_boundary(M):
    # 1 + 2^-8 is exact in fp32 and a tie in bf16 (7 fraction bits): ties to even -> 1
    # 1 + 3*2^-8 rounds up to 1 + 2^-6 (nearest); 256 + 1 -> 256 (tie, even); -2 + 0.75 = -1.25
    x = _bits(np.array([[1.0, 1.0, 256.0, -2.0]]))
    r = _bits(np.array([[2.0 ** -8, 3 * 2.0 ** -8, 1.0, 0.75]]))
    got = WL.bf16_bits_to_f32(M.residual_add(x, r))
    assert got.tolist() == [[1.0, 1.0 + 2.0 ** -6, 256.0, -1.25]]
    g = _bits(np.ones(4))
    y, xr = M.rmsnorm(x, g, 1e-6, r)
    assert np.array_equal(xr, M.residual_add(x, r))


PINS = [pin_brute_force, pin_constant_row, pin_scale_invariance, pin_unit_mean_square,
        pin_residual_boundary]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_rmsnorm_oracle_pin(pin):
    pin(R)


def _copy():
    spec = importlib.util.spec_from_file_location("rmsnorm_mutant", R.__file__)
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def _mut_no_eps(m):
    orig = m.rmsnorm
    m.rmsnorm = lambda x, g, eps, r=None: orig(x, g, 0.0, r)


def _mut_sum_not_mean(m):
    def rmsnorm(x_bits, gamma_bits, eps, residual_bits=None):
        xr = x_bits if residual_bits is None else m.residual_add(x_bits, residual_bits)
        x = m.decode_bf16(xr)
        g = m.decode_bf16(gamma_bits)
        y = x / np.sqrt((x * x).sum(axis=1) + eps)[:, None] * g[None, :]
        return y, xr
    m.rmsnorm = rmsnorm


def _mut_gamma_reversed(m):
    orig = m.rmsnorm
    m.rmsnorm = lambda x, g, eps, r=None: orig(x, np.ascontiguousarray(g[::-1]), eps, r)


def _mut_residual_truncated(m):
    def residual_add(x_bits, r_bits):
        xs = (np.asarray(x_bits, np.uint16).astype(np.uint32) << 16).view(np.float32)
        rs = (np.asarray(r_bits, np.uint16).astype(np.uint32) << 16).view(np.float32)
        return ((xs + rs).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    m.residual_add = residual_add


@pytest.mark.parametrize("mutate", [_mut_no_eps, _mut_sum_not_mean, _mut_gamma_reversed,
                                    _mut_residual_truncated], ids=lambda f: f.__name__)
def test_rmsnorm_planted_mistake_is_caught(mutate):
    m = _copy()
    mutate(m)
    caught = 0
    for pin in PINS:
        try:
            pin(m)
        except Exception:
            caught += 1
    assert caught > 0


def test_emulator_rsqrt_sweep():
    max_ulp, worst, count = E.rsqrt_sweep(2.0 ** -40, 2.0 ** 40)
    assert count == 80 * (1 << 23) + 1
    assert max_ulp < 1.0, (max_ulp, worst)
    assert E.rsqrt(1.0) == 1.0 and E.rsqrt(4.0) == 0.5 and E.rsqrt(0.25) == 2.0


@pytest.mark.parametrize("T,H,res", [(7, 64, False), (5, 4096, True), (3, 2560, True), (2, 96, False)])
def test_emulator_rmsnorm_vs_oracle(T, H, res):
    rng = np.random.default_rng(H)
    x = _bits(rng.standard_normal((T, H)) * 3)
    r = _bits(rng.standard_normal((T, H))) if res else None
    g = _bits(1 + 0.1 * rng.standard_normal(H))
    y_bits, xr = E.rmsnorm(x, g, 1e-6, r)
    y_ref, xr_ref = R.rmsnorm(x, g, 1e-6, r)
    if res:
        assert np.array_equal(xr, xr_ref)
    y = WL.bf16_bits_to_f32(y_bits).astype(np.float64)
    # within one bf16 ulp (2^-7 relative) of the fp64 value
    assert np.all(np.abs(y - y_ref) <= 2.0 ** -7 * np.abs(y_ref) + 1e-30)
