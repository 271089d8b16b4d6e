"""Pins of the oracle's scalar arithmetic against mathematics (float64).

E(x) = exp(x), L(x) = log(1+x) and lse(a,b) = log(e^a + e^b) are the
definitions ("GPU CTC Prefix Beam Search Decoder", section 3, the logsumexp
definition); numpy's float64 exp/log1p/logaddexp stand in for the exact values.
"""
import math

import numpy as np
import pytest

NEG = np.float32(np.finfo(np.float32).min)


def ulp_err(got, exact):
    got = np.asarray(got, np.float64)
    exact = np.asarray(exact, np.float64)
    sp = np.spacing(np.abs(exact).astype(np.float32)).astype(np.float64)
    return np.abs(got - exact) / np.maximum(sp, np.finfo(np.float32).tiny)


def test_E_matches_exp_within_2ulp(oracle):
    x = np.linspace(-87.0, 0.0, 1_000_003).astype(np.float32)
    rng = np.random.default_rng(1)
    x = np.concatenate([x, -rng.exponential(3.0, 200_000).astype(np.float32)])
    x = x[x >= -87.0]
    err = ulp_err(oracle.E(x), np.exp(x.astype(np.float64)))
    assert err.max() <= 2.0, err.max()


def test_E_special_values(oracle):
    assert oracle.E(np.float32(0.0))[()] == 1.0
    assert oracle.E(np.float32(-0.0))[()] == 1.0
    assert oracle.E(np.float32(-87.5))[()] == 0.0
    assert oracle.E(NEG)[()] == 0.0
    assert oracle.E(np.float32(np.nan))[()] == 0.0
    # every nonzero result is a normal float
    x = np.linspace(-87.0, -80.0, 10001).astype(np.float32)
    e = oracle.E(x)
    assert (e >= np.finfo(np.float32).tiny).all()


def test_L_matches_log1p_within_2ulp(oracle):
    x = np.linspace(0.0, 1.0, 1_000_001).astype(np.float32)
    rng = np.random.default_rng(2)
    x = np.concatenate([x, rng.random(200_000).astype(np.float32),
                        np.float32(2.0) ** -np.arange(1, 140, dtype=np.float32)])
    got = oracle.L(x)
    err = ulp_err(got, np.log1p(x.astype(np.float64)))
    assert err.max() <= 2.0, err.max()
    assert oracle.L(np.float32(0.0))[()] == 0.0
    assert abs(float(oracle.L(np.float32(1.0))[()]) - math.log(2.0)) < 1e-7


def test_lse_matches_logaddexp(oracle):
    rng = np.random.default_rng(3)
    a = (-rng.exponential(50.0, 400_000)).astype(np.float32)
    b = (a - rng.exponential(5.0, 400_000)).astype(np.float32)
    got = oracle.lse(a, b)
    exact = np.logaddexp(a.astype(np.float64), b.astype(np.float64))
    # Absolute bound (near a result of 0 the final addition cancels, so no
    # relative bound can hold): one rounding of max + L(.), two ulps of L,
    # two ulps of E propagated through 1/(1+e), and the half-ulp rounding of
    # d = |a - b| propagated through e/(1+e).
    err = np.abs(got.astype(np.float64) - exact)
    d = np.abs(a.astype(np.float64) - b.astype(np.float64))
    e = np.exp(-d)
    sp = lambda v: np.spacing(np.abs(v).astype(np.float32)).astype(np.float64)
    tol = (sp(exact) + 2.0 * sp(np.log1p(e)) + 2.0 * sp(e) / (1.0 + e)
           + 0.5 * sp(d) * e / (1.0 + e))
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
