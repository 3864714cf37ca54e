"""Pins of the oracle's TurboQuant pieces: SplitMix64, FWHT, rotation,
norms, the Beta Lloyd-Max codebook and the rotated scalar code (no GPU)."""
import math

import numpy as np
import pytest
import scipy.integrate
import scipy.linalg
import scipy.special

from oracle import turboquant as tq
from tests.conftest import read_golden


def test_splitmix64_published_vectors():
    for row in read_golden("splitmix64_vectors.txt"):
        seed, outs = int(row[0]), [int(x) for x in row[1:]]
        assert tq.splitmix64(seed, len(outs)) == outs


def test_signs_deterministic_and_seeded():
    a, b, c = tq.signs(42, 128), tq.signs(42, 128), tq.signs(43, 128)
    assert np.array_equal(a, b) and not np.array_equal(a, c)
    assert set(np.unique(a)) <= {-1.0, 1.0}
    assert 30 < np.sum(a > 0) < 98


@pytest.mark.parametrize("d", [8, 64, 128])
def test_fwht_matches_sylvester_hadamard(d):
    """FWHT equals the Sylvester Hadamard matrix product (library routine)
    exactly on small integers, and FWHT(e_j)_i = (-1)^popcount(i & j)."""
    rng = np.random.default_rng(d)
    x = rng.integers(-8, 9, size=(5, d)).astype(np.float32)
    H = scipy.linalg.hadamard(d).astype(np.float64)
    assert np.array_equal(tq.fwht(x).astype(np.float64), x.astype(np.float64) @ H.T)
    for j in (0, 1, d // 2 + 3, d - 1):
        e = np.zeros(d, np.float32)
        e[j] = 1
        want = np.array([(-1) ** bin(i & j).count("1") for i in range(d)], np.float32)
        assert np.array_equal(tq.fwht(e), want)


def test_fwht_self_inverse_up_to_d():
    x = np.random.default_rng(1).integers(-100, 100, size=(3, 128)).astype(np.float32)
    assert np.array_equal(tq.fwht(tq.fwht(x)), 128 * x)


def test_rotation_orthogonal_and_inverse():
    """R R^T = I (Foundry spec, unit test 2) and unrotate inverts rotate."""
    d = 128
    sgn = tq.signs(7, d)
    R = tq.rotate(np.eye(d, dtype=np.float32), sgn).T       # columns R e_j
    assert np.max(np.abs(R @ R.T - np.eye(d))) < 1e-6
    x = np.random.default_rng(2).standard_normal((4, d)).astype(np.float32)
    assert np.max(np.abs(tq.unrotate(tq.rotate(x, sgn), sgn) - x)) < 1e-5
    assert np.allclose(np.linalg.norm(tq.rotate(x, sgn), axis=1), np.linalg.norm(x, axis=1), rtol=1e-6)
    # As-built order: signs first, then the Hadamard transform.
    H = scipy.linalg.hadamard(d) / math.sqrt(d)
    assert np.allclose(R, H @ np.diag(sgn), atol=1e-7)


def test_tree_sum_fixed_order():
    a = np.array([1e8, 1.0, -1e8, 1.0], np.float32)
    # stride 2 first: (1e8 + -1e8) + (1 + 1) = 2; left-to-right would give 1.
    assert tq.tree_sum(a) == np.float32(2.0)


# ------------------------------------------------------------------ codebook

@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_codebook_uniform_closed_form(bits):
    """Beta(1, 1) is uniform: Lloyd-Max levels are (2i+1)/(2L), boundaries i/L."""
    b, c, _ = tq.lloyd_max_beta(1.0, bits)
    L = 1 << bits
    assert np.allclose(b, np.arange(1, L) / L, atol=1e-12)
    assert np.allclose(c, (2 * np.arange(L) + 1) / (2 * L), atol=1e-12)


@pytest.mark.parametrize("a", [32.0, 64.0])
def test_codebook_one_bit_closed_form(a):
    """1 bit: boundary 1/2, centroids 1/2 -+ 4^-a / (a B(a, a)), from
    d/dx[x^a (1-x)^a] = a x^(a-1) (1-x)^(a-1) (1 - 2x)."""
    b, c, _ = tq.lloyd_max_beta(a, 1)
    off = 4.0 ** (-a) / (a * scipy.special.beta(a, a))
    assert abs(b[0] - 0.5) < 1e-15
    assert np.allclose(c, [0.5 - off, 0.5 + off], atol=1e-13)


@pytest.mark.parametrize("d,bits", [(64, 2), (128, 2), (128, 3), (64, 3), (128, 4), (64, 4)])
def test_codebook_lloyd_conditions_by_quadrature(d, bits):
    """Centroid condition (checked with adaptive quadrature of the density, a
    different routine than the oracle's incomplete beta) and midpoint
    condition; symmetry b_i = 1 - b_(L-i)."""
    a = d / 2
    b, c, _ = tq.lloyd_max_beta(a, bits)
    logB = scipy.special.betaln(a, a)
    f = lambda x: math.exp((a - 1) * (math.log(x) + math.log1p(-x)) - logB)
    edges = np.concatenate([[0.0], b, [1.0]])
    for i in range(len(c)):
        lo, hi = edges[i], edges[i + 1]
        pts = [0.5] if lo < 0.5 < hi else None
        m0 = scipy.integrate.quad(f, lo, hi, epsabs=0, epsrel=1e-13, limit=200, points=pts)[0]
        m1 = scipy.integrate.quad(lambda x: x * f(x), lo, hi, epsabs=0, epsrel=1e-13, limit=200, points=pts)[0]
        assert abs(m1 / m0 - c[i]) < 1e-9
    assert np.allclose(b, 0.5 * (c[:-1] + c[1:]), atol=1e-13)
    assert np.allclose(b, 1.0 - b[::-1], atol=1e-12)


@pytest.mark.parametrize("levels_row", [1, 2, 3])
def test_codebook_near_gaussian_lloyd_max(levels_row):
    """For d = 128 the Beta(64, 64) code sits at the Gaussian Lloyd-Max levels
    scaled by its sigma (tests/golden/gaussian_lloyd_max.txt)."""
    row = read_golden("gaussian_lloyd_max.txt")[levels_row]
    L = int(row[0])
    pos = np.array([float(x) for x in row[1:-1]])
    a = 64.0
    sigma = math.sqrt(a * a / ((2 * a) ** 2 * (2 * a + 1)))
    _, c, _ = tq.lloyd_max_beta(a, int(math.log2(L)))
    got = (c[L // 2:] - 0.5) / sigma
    assert np.allclose(got, pos, rtol=0.02)


def test_codebook_float32_middle_boundary_is_half():
    for d in (64, 128):
        for bits in (2, 3, 4):
            b, _ = tq.codebook(d, bits)
            assert b.dtype == np.float32 and b[len(b) // 2] == np.float32(0.5)


# ------------------------------------------------------------------ quantiser

def test_zero_vector():
    d = 128
    sgn = tq.signs(1, d)
    bnd, cen = tq.codebook(d, 4)
    codes, n = tq.quantize(np.zeros((2, d), np.float32), sgn, bnd)
    assert np.all(n == 0)
    assert np.all(tq.dequantize(codes, n, sgn, cen) == 0)


@pytest.mark.parametrize("bits,row", [(2, 1), (3, 2), (4, 3)])
def test_roundtrip_mse_matches_lloyd_max_distortion(bits, row):
    """Relative round-trip MSE of random Gaussian vectors equals the Gaussian
    Lloyd-Max distortion per coordinate (Foundry unit test 1: roundtrip MSE
    per bit width; values in tests/golden/gaussian_lloyd_max.txt)."""
    d = 128
    mse_ref = float(read_golden("gaussian_lloyd_max.txt")[row][-1])
    sgn = tq.signs(3, d)
    bnd, cen = tq.codebook(d, bits)
    x = np.random.default_rng(bits).standard_normal((4000, d)).astype(np.float32)
    codes, n = tq.quantize(x, sgn, bnd)
    xh = tq.dequantize(codes, n, sgn, cen)
    rel = np.mean(np.sum((x - xh) ** 2, 1) / np.sum(x * x, 1))
    assert abs(rel / mse_ref - 1) < 0.05


def test_code_counts_boundaries_ties_up():
    """code = #{i : w >= b_i}: a coordinate exactly on a boundary goes up."""
    bnd = np.array([0.25, 0.5, 0.75], np.float32)
    w = np.array([0.0, 0.25, 0.3, 0.5, 0.75, 1.0], np.float32)
    assert list((w[:, None] >= bnd).sum(-1)) == [0, 1, 1, 2, 3, 3]


def test_dot_product_preserved():
    """Foundry unit test 3: dot(q, k) close to dot(q, k_hat) at 4 bits."""
    d = 128
    sgn = tq.signs(5, d)
    bnd, cen = tq.codebook(d, 4)
    rng = np.random.default_rng(9)
    q = rng.standard_normal((500, d)).astype(np.float32)
    k = rng.standard_normal((500, d)).astype(np.float32)
    kh = tq.dequantize(*tq.quantize(k, sgn, bnd), sgn, cen)
    err = np.abs(np.sum(q * k, 1) - np.sum(q * kh, 1))
    assert np.median(err / (np.linalg.norm(q, axis=1) * np.linalg.norm(k, axis=1))) < 0.02


def test_rotated_domain_dot_equals_original():
    """dot(q, R^T y_hat) = dot(R q, y_hat) (Foundry spec, fused dequant-dot)."""
    d = 128
    sgn = tq.signs(5, d)
    bnd, cen = tq.codebook(d, 4)
    rng = np.random.default_rng(10)
    q = rng.standard_normal((50, d)).astype(np.float32)
    k = rng.standard_normal((50, d)).astype(np.float32)
    codes, n = tq.quantize(k, sgn, bnd)
    yh = tq.dequantize_rotated(codes, n, cen)
    a = np.sum(q.astype(np.float64) * tq.unrotate(yh, sgn), 1)
    b = np.sum(tq.rotate(q, sgn).astype(np.float64) * yh, 1)
    assert np.allclose(a, b, rtol=1e-5, atol=1e-4)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("bits", [2, 3, 4])
def test_codebook_boundaries_farther_apart_than_guess_cells(d, bits):
    """The quantiser's code search guesses from cells of width 1/256 in w and
    falls back to a binary search only where a cell holds two boundaries;
    the Beta codebooks of every supported width and head_dim keep their
    boundaries more than a cell apart, so the guess path is the one taken."""
    bnd, _ = tq.codebook(d, bits)
    assert np.all(np.diff(bnd.astype(np.float64)) > 1.0 / 256)
