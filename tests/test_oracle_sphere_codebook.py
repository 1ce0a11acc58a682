"""Pins for the oracle's Lloyd-Max codebook fitted to the exact density of a
rotated coordinate (CPU only).

[P4] riverfrot.github.io "TurboQuant란 무엇이며…", §4.2: after the random
rotation every coordinate follows a Beta distribution that approaches the
Gaussian at high d.  In unit-variance units u = sqrt(d) z, z a coordinate of a
uniform point on the unit sphere of R^d, the density is
f(u) = Gamma(d/2) / (sqrt(pi d) Gamma((d-1)/2)) (1 - u^2/d)^((d-3)/2) on |u| < sqrt(d).
The pins below integrate that density directly (scipy quad), independently of
the closed-form tail and moment the oracle iterates with.
"""

import math

import numpy as np
import pytest
from scipy import integrate

from oracle import lloyd_max_gaussian, lloyd_max_sphere


def _density(d):
    c = math.exp(math.lgamma(d / 2.0) - math.lgamma((d - 1) / 2.0)) / math.sqrt(math.pi * d)
    return lambda u: c * (1.0 - u * u / d) ** ((d - 3) / 2.0)


def _cells(book, d):
    t = [-math.sqrt(d)] + list(book.boundaries) + [math.sqrt(d)]
    return [(t[k], t[k + 1]) for k in range(len(book.centroids))]


@pytest.mark.parametrize("d", [16, 128, 1000])
def test_density_is_normalised_with_unit_variance(d):
    f, r = _density(d), math.sqrt(d)
    assert integrate.quad(f, -r, r, epsabs=1e-14)[0] == pytest.approx(1.0, abs=1e-10)
    assert integrate.quad(lambda u: u * u * f(u), -r, r, epsabs=1e-14)[0] == pytest.approx(1.0, abs=1e-10)


@pytest.mark.parametrize("d", [16, 128, 1000])
def test_one_bit_closed_form(d):
    """1 bit: boundary 0, centroids +-E|U| = +-sqrt(d) Gamma(d/2) / (sqrt(pi) Gamma((d+1)/2))."""
    book = lloyd_max_sphere(1, d)
    want = math.sqrt(d) * math.exp(math.lgamma(d / 2.0) - math.lgamma((d + 1) / 2.0)) / math.sqrt(math.pi)
    assert book.boundaries[0] == 0.0
    assert book.centroids[1] == pytest.approx(want, rel=1e-12)      # lgamma rounding at large d
    assert book.centroids[0] == -book.centroids[1]


@pytest.mark.parametrize("bits,d", [(2, 128), (3, 128), (4, 128), (3, 4), (4, 5), (4, 9)])
def test_lloyd_conditions_by_quadrature(bits, d):
    """Each centroid is the conditional mean of its cell under f, each boundary the midpoint of its neighbours.
    Small d (support |u| < sqrt(d) shorter than the Gaussian's bulk) included: every cell must keep mass."""
    book, f = lloyd_max_sphere(bits, d), _density(d)
    assert np.all(np.isfinite(book.centroids)) and np.all(np.abs(book.centroids) < math.sqrt(d))
    for (a, b), c in zip(_cells(book, d), book.centroids):
        p0 = integrate.quad(f, a, b, epsabs=1e-15, epsrel=1e-13)[0]
        m1 = integrate.quad(lambda u: u * f(u), a, b, epsabs=1e-15, epsrel=1e-13)[0]
        assert m1 / p0 == pytest.approx(c, abs=1e-9)
    mid = 0.5 * (book.centroids[:-1] + book.centroids[1:])
    assert np.max(np.abs(mid - book.boundaries)) < 1e-15
    assert np.all(np.diff(book.centroids) > 0)


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_optimal_for_its_density(bits):
    """Under the rotated-coordinate density the fitted codebook distorts less than the Gaussian one
    (Lloyd-Max optimality), by a margin that is O(1/d)."""
    d = 128
    f = _density(d)

    def distortion(book):
        total = 0.0
        for (a, b), c in zip(_cells(book, d), book.centroids):
            total += integrate.quad(lambda u: (u - c) ** 2 * f(u), a, b, epsabs=1e-15, epsrel=1e-13)[0]
        return total

    ds, dg = distortion(lloyd_max_sphere(bits, d)), distortion(lloyd_max_gaussian(bits))
    assert ds < dg
    assert (dg - ds) / ds < 0.05


def test_gaussian_limit():
    """The density tends to N(0,1) as d grows, and so does the codebook, at a rate of about 1/d."""
    g = lloyd_max_gaussian(3).centroids
    gaps = [np.max(np.abs(lloyd_max_sphere(3, d).centroids - g)) for d in (128, 1280, 12800)]
    assert gaps[0] > gaps[1] > gaps[2]
    assert gaps[2] < 3e-4
    assert gaps[0] / gaps[1] == pytest.approx(10.0, rel=0.1)
    assert gaps[1] / gaps[2] == pytest.approx(10.0, rel=0.1)
