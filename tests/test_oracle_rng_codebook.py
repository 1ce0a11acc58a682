"""Pins for the oracle's random streams and Lloyd-Max codebooks (CPU only)."""

import math
import os

import numpy as np
import pytest
from scipy import integrate, stats

from oracle import gaussian_stream, lloyd_max_gaussian, splitmix64_stream

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def test_splitmix64_published_vector():
    # stream 0 with seed 0 is the sequential generator started from state 0
    want = [int(x[0], 16) for x in _golden_lines("splitmix64_seed0.txt")]
    got = [int(v) for v in splitmix64_stream(0, 0, 4)]
    assert got == want


def test_splitmix64_counter_offset():
    # drawing from `start` continues the same stream
    a = splitmix64_stream(7, 3, 10)
    b = splitmix64_stream(7, 3, 6, start=4)
    assert np.array_equal(a[4:], b)


def test_gaussian_stream_is_standard_normal():
    g = gaussian_stream(12345, 1, 200000)
    assert abs(g.mean()) < 5 * (1 / math.sqrt(g.size))
    assert abs(g.var() - 1.0) < 5 * math.sqrt(2.0 / g.size)
    assert abs(stats.kurtosis(g, fisher=False) - 3.0) < 5 * math.sqrt(24.0 / g.size)
    assert stats.kstest(g, "norm").pvalue > 1e-4
    # streams 1 and 2 are uncorrelated
    h = gaussian_stream(12345, 2, 200000)
    assert abs(np.corrcoef(g, h)[0, 1]) < 5 / math.sqrt(g.size)


def test_codebook_one_bit_closed_form():
    cb = lloyd_max_gaussian(1)
    c = math.sqrt(2.0 / math.pi)
    assert np.allclose(cb.centroids, [-c, c], atol=1e-15)
    assert cb.boundaries.tolist() == [0.0]
    assert abs(cb.mse() - (1.0 - 2.0 / math.pi)) < 1e-15


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_codebook_matches_max_table(bits):
    rows = {(int(r[0]), r[1]): [float(x) for x in r[2:]] for r in _golden_lines("max1960_gaussian.txt")}
    cb = lloyd_max_gaussian(bits)
    n = 1 << bits
    h = n // 2
    # 4-significant-digit table; the 16-level row carries rounding up to 1e-4 in the 4th digit
    tol = 1.5e-4 if bits < 4 else 2.5e-4
    assert np.allclose(cb.centroids[h:], rows[(n, "outputs")], atol=tol, rtol=6e-4)
    assert np.allclose(cb.boundaries[h:], rows[(n, "thresholds")], atol=tol, rtol=6e-4)
    assert cb.boundaries[h - 1] == 0.0
    assert np.array_equal(cb.centroids, -cb.centroids[::-1])


@pytest.mark.parametrize("bits", [1, 2, 3, 4, 5])
def test_codebook_lloyd_conditions_by_quadrature(bits):
    """Independent check: conditional means by numerical integration, nearest-neighbour boundaries."""
    cb = lloyd_max_gaussian(bits)
    t = np.concatenate([[-np.inf], cb.boundaries, [np.inf]])
    for k, c in enumerate(cb.centroids):
        mass = integrate.quad(stats.norm.pdf, t[k], t[k + 1], epsabs=1e-15, epsrel=1e-13)[0]
        mom = integrate.quad(lambda z: z * stats.norm.pdf(z), t[k], t[k + 1], epsabs=1e-15, epsrel=1e-13)[0]
        assert abs(mom / mass - c) < 1e-9
    assert np.allclose(cb.boundaries, 0.5 * (cb.centroids[:-1] + cb.centroids[1:]), atol=0, rtol=0)
    mse_q = sum(integrate.quad(lambda z: (z - c) ** 2 * stats.norm.pdf(z), t[k], t[k + 1],
                               epsabs=1e-15, epsrel=1e-13)[0] for k, c in enumerate(cb.centroids))
    assert abs(mse_q - cb.mse()) < 1e-12


def test_codebook_mse_ladder_and_bounds():
    """About 4x less distortion per extra bit, between 4**-b and (sqrt(3) pi / 2) 4**-b."""
    d = [lloyd_max_gaussian(b).mse() for b in range(1, 5)]
    assert np.allclose(d, [0.363380, 0.117482, 0.034548, 0.009501], atol=2e-6)
    for b, v in enumerate(d, start=1):
        assert 4.0 ** -b <= v <= math.sqrt(3) * math.pi / 2 * 4.0 ** -b
    ratios = [d[i] / d[i + 1] for i in range(3)]
    assert all(3.0 < r < 4.0 for r in ratios) and ratios == sorted(ratios)
