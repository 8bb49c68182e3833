"""Pins for reverse water-filling, the integer bit allocation and step sizes."""
import itertools
import os

import numpy as np
import pytest
from scipy import integrate, optimize

import oracle


@pytest.mark.parametrize("decay,total", [(0.9, 2.75 * 128), (0.95, 2.0 * 128), (0.7, 40.0)])
def test_waterfill_closed_form(decay, total):
    lam = decay ** np.arange(128)
    th, R, D = oracle.waterfill_theta(lam, total)
    # rates sum to the budget, R_j = max(0, 1/2 log2(lam/theta)), D_j = min(theta, lam)
    assert abs(R.sum() - total) < 1e-12 * total
    assert np.allclose(R, np.maximum(0, 0.5 * np.log2(lam / th)), atol=1e-13)
    assert np.allclose(D, np.minimum(th, lam))
    # independent root finding of the same condition (scipy brentq on log theta)
    f = lambda lt: np.maximum(0, 0.5 * np.log2(lam / 2.0 ** lt)).sum() - total
    lt = optimize.brentq(f, np.log2(lam.min()) - 2 * total, np.log2(lam.max()), xtol=1e-14)
    assert abs(np.log2(th) - lt) < 1e-9


def _brute(lam, B):
    best, arg = None, None
    for b in itertools.product(range(9), repeat=len(lam)):
        if sum(b) != B:
            continue
        v = sum(l * 4.0 ** -bb for l, bb in zip(lam, b))
        if best is None or v < best - 1e-15:
            best, arg = v, b
    return best, arg


@pytest.mark.parametrize("seed", range(6))
def test_integer_allocation_is_exhaustive_optimum(seed):
    rng = np.random.default_rng(seed)
    d = 4 if seed < 3 else 5
    lam = np.sort(rng.exponential(size=d))[::-1]
    B = int(rng.integers(1, 8 * d))
    bits, margin = oracle.allocate_bits(lam, B)
    best, arg = _brute(lam, B)
    assert bits.sum() == B
    assert abs(sum(l * 4.0 ** -b for l, b in zip(lam, bits)) - best) <= 1e-14 * best
    if margin > 1e-9:
        assert tuple(bits) == arg


def test_allocation_properties():
    lam = 0.95 ** np.arange(128)
    bits, _ = oracle.allocate_bits(lam, 352)
    assert bits.sum() == 352 and bits.min() >= 0 and bits.max() <= 8
    assert np.all(np.diff(bits) <= 0)          # non-increasing with the eigenvalue
    # equal eigenvalues: widths differ by at most one and extras go to the lowest j
    b, _ = oracle.allocate_bits(np.ones(10), 23)
    assert list(b) == [3, 3, 3, 2, 2, 2, 2, 2, 2, 2]
    # the whole budget at 8 bits each, and zero budget
    assert list(oracle.allocate_bits(np.ones(4), 32)[0]) == [8] * 4
    assert list(oracle.allocate_bits(np.ones(4), 0)[0]) == [0] * 4
    with pytest.raises(ValueError):
        oracle.allocate_bits(np.ones(4), 33)


def test_integer_allocation_tracks_continuous_waterfill():
    """Integer widths stay within one bit of the continuous rates."""
    lam = 0.93 ** np.arange(128)
    th, R, _ = oracle.waterfill_theta(lam, 352)
    bits, _ = oracle.allocate_bits(lam, 352)
    assert np.all(np.abs(bits - R) <= 1.0 + 1e-9)


def test_step_table_against_max_1960(golden_dir):
    rows = [l.split() for l in open(os.path.join(golden_dir, "max1960_uniform_steps.txt"))
            if l.strip() and not l.startswith("#")]
    for b, n, step in rows:
        s = oracle.gauss_uniform_step(int(b))
        digits = len(step.split(".")[1])
        assert abs(s - float(step)) <= 0.6 * 10.0 ** -digits, (b, s, step)
    # b = 1 has a closed form: the levels are +-E|x| = +-sqrt(2/pi)
    assert abs(oracle.gauss_uniform_step(1) - 2 * np.sqrt(2 / np.pi)) < 1e-13


@pytest.mark.parametrize("b", [1, 2, 3, 4, 6, 8])
def test_step_minimizes_mse_and_mse_matches_integral(b):
    s = oracle.gauss_uniform_step(b)
    m = oracle.gauss_uniform_mse(b, s)
    assert m < oracle.gauss_uniform_mse(b, s * (1 + 1e-4))
    assert m < oracle.gauss_uniform_mse(b, s * (1 - 1e-4))
    # the closed-form MSE against adaptive quadrature of (x - Q(x))^2 phi(x)
    N = 2 ** b
    Qx = lambda x: (np.clip(np.floor(x / s + N / 2), 0, N - 1) - (N - 1) / 2) * s
    phi = lambda x: np.exp(-x * x / 2) / np.sqrt(2 * np.pi)
    pts = [(k - N / 2) * s for k in range(1, N)]
    quad = integrate.quad(lambda x: (x - Qx(x)) ** 2 * phi(x), -12, 12, points=pts, limit=2000)[0]
    assert abs(quad - m) < 1e-9 * max(m, 1e-6) + 1e-12


def test_step_mse_monte_carlo():
    rng = np.random.default_rng(7)
    x = rng.standard_normal(1_000_000)
    for b in (1, 2, 3, 5):
        s = oracle.gauss_uniform_step(b)
        bits = np.full(1, b)
        N = 2 ** b
        u = np.clip(np.rint(x / s + (N - 1) / 2), 0, N - 1)
        err = np.mean((x - (u - (N - 1) / 2) * s) ** 2)
        assert abs(err / oracle.gauss_uniform_mse(b, s) - 1) < 0.01
    del bits
