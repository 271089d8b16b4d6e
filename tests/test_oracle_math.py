"""Pins of the oracle's scalar arithmetic against mathematics.

lse(a,b) = log(e^a + e^b) = max + F(|a-b|) with F(d) = log(1 + e^-d) ("GPU CTC
Prefix Beam Search Decoder", section 3, the logsumexp definition).  F is a
piecewise degree-5 Taylor polynomial; its coefficients are checked against
Taylor coefficients computed to 40 digits by mpmath, F against numpy's float64
log1p(exp(-d)), and lse against float64 logaddexp.
"""
import functools
import math

import numpy as np
import pytest

NEG = np.float32(np.finfo(np.float32).min)


def ulp_err(got, exact):
    got = np.asarray(got, np.float64)
    exact = np.asarray(exact, np.float64)
    sp = np.spacing(np.abs(exact).astype(np.float32)).astype(np.float64)
    return np.abs(got - exact) / np.maximum(sp, np.finfo(np.float32).tiny)


@functools.lru_cache(maxsize=1)
def exact_coefficients():
    """F^(n)(k/4 + 1/8) / n! for k < 96, n <= 5, to 40 digits, rounded once to float32."""
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 40
    f = lambda x: mpmath.log1p(mpmath.exp(-x))
    out = np.empty((96, 6), np.float32)
    for k in range(96):
        d0 = mpmath.mpf(k) / 4 + mpmath.mpf(1) / 8
        for n, c in enumerate(mpmath.taylor(f, d0, 5)):
            out[k, n] = np.float32(float(c))  # float(c): nearest double; then nearest float
    return out


def test_F_coefficients_are_rounded_taylor_coefficients(oracle):
    got = oracle.F_coefficients()
    want = exact_coefficients()
    assert np.array_equal(got.view(np.int32), want.view(np.int32)), np.argwhere(got != want)[:5]


def test_F_matches_log1p_exp_within_2ulp(oracle):
    d = np.linspace(0.0, 24.0, 2_000_001).astype(np.float32)
    rng = np.random.default_rng(1)
    d = np.concatenate([d, rng.uniform(0.0, 24.0, 500_000).astype(np.float32),
                        np.float32(2.0) ** -np.arange(1, 140, dtype=np.float32)])
    d = d[d < 24.0]
    err = ulp_err(oracle.F(d), np.log1p(np.exp(-d.astype(np.float64))))
    assert err.max() <= 2.0, err.max()


def test_F_special_values(oracle):
    assert abs(float(oracle.F(np.float32(0.0))[()]) - math.log(2.0)) < 1e-7
    for d in (24.0, 30.0, 1e30, float(np.finfo(np.float32).max), float("inf"), float("nan")):
        assert oracle.F(np.float32(d))[()] == 0.0
    # positive (so lse >= max) and decreasing across every segment boundary
    d = np.linspace(0.0, 23.999, 200_001).astype(np.float32)
    f = oracle.F(d)
    assert (f > 0).all() and (np.diff(f.astype(np.float64)) <= 0).all()


def test_lse_matches_logaddexp(oracle):
    rng = np.random.default_rng(3)
    a = (-rng.exponential(50.0, 400_000)).astype(np.float32)
    b = (a - rng.exponential(5.0, 400_000)).astype(np.float32)
    got = oracle.lse(a, b)
    exact = np.logaddexp(a.astype(np.float64), b.astype(np.float64))
    # Absolute bound (near a result of 0 the final addition cancels, so no
    # relative bound can hold): one rounding of max + F(.), two ulps of F,
    # F's cut at d = 24 (F(24) < 4e-11), and the half-ulp rounding of
    # d = |a - b| propagated through |F'(d)| = e/(1+e).
    err = np.abs(got.astype(np.float64) - exact)
    d = np.abs(a.astype(np.float64) - b.astype(np.float64))
    e = np.exp(-d)
    sp = lambda v: np.spacing(np.abs(v).astype(np.float32)).astype(np.float64)
    tol = sp(exact) + 2.0 * sp(np.log1p(e)) + math.log1p(math.exp(-24.0)) + 0.5 * sp(d) * e / (1.0 + e)
    assert (err <= tol).all(), (err / tol).max()


def test_lse_identities(oracle):
    rng = np.random.default_rng(4)
    a = (-rng.exponential(100.0, 100_000)).astype(np.float32)
    b = (-rng.exponential(100.0, 100_000)).astype(np.float32)
    # symmetric bit for bit
    assert np.array_equal(oracle.lse(a, b).view(np.int32), oracle.lse(b, a).view(np.int32))
    # NEG is the identity, exactly
    assert np.array_equal(oracle.lse(a, np.full_like(a, NEG)).view(np.int32), a.view(np.int32))
    assert oracle.lse(NEG, NEG)[()] == NEG
    # lse(x, x) = x + ln 2
    x = a[:1000]
    assert np.allclose(oracle.lse(x, x), x.astype(np.float64) + math.log(2.0), rtol=0, atol=1e-4)
    # monotone in each argument
    assert (oracle.lse(a, b) >= np.maximum(a, b)).all()


def test_add_clamps_at_neg(oracle):
    assert oracle.add(NEG, NEG)[()] == NEG
    assert oracle.add(np.float32(-1.0), NEG)[()] == NEG
    assert oracle.add(np.float32(-1.5), np.float32(-2.25))[()] == np.float32(-3.75)


@pytest.mark.parametrize("thr", [0.98, 0.999, 0.5, 1e-3])
def test_log_threshold_is_float_of_double_log(oracle, thr):
    assert oracle.log_threshold(thr) == np.float32(math.log(np.float64(np.float32(thr))))
