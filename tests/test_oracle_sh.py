"""Pins of the oracle's real spherical-harmonic basis (Kopanas, Step 3: 16 coefficients
per channel, colour = sum_k Y_k(d) s_k)."""

import numpy as np
from scipy.special import sph_harm_y

import oracle


def _dirs(n, seed=0):
    d = np.random.default_rng(seed).standard_normal((n, 3))
    return d / np.linalg.norm(d, axis=1, keepdims=True)


def test_basis_matches_scipy_real_harmonics():
    """Real SH from scipy's complex Y_l^m: m > 0 -> sqrt2 (-1)^m Re Y_l^m, m < 0 ->
    sqrt2 (-1)^m Im Y_l^|m|; the (-1)^m removes the Condon-Shortley phase."""
    d = _dirs(500)
    Y, _ = oracle.sh_basis(d)
    theta, phi = np.arccos(d[:, 2]), np.arctan2(d[:, 1], d[:, 0])
    k = 0
    for l in range(4):
        for m in range(-l, l + 1):
            if m == 0:
                ref = sph_harm_y(l, 0, theta, phi).real
            elif m > 0:
                ref = np.sqrt(2) * (-1) ** m * sph_harm_y(l, m, theta, phi).real
            else:
                ref = np.sqrt(2) * (-1) ** m * sph_harm_y(l, -m, theta, phi).imag
            np.testing.assert_allclose(Y[:, k], ref, atol=1e-13)
            k += 1


def test_basis_orthonormal_by_quadrature():
    # Gauss-Legendre in cos(theta) x uniform phi integrates degree <= 6 products exactly
    x, w = np.polynomial.legendre.leggauss(8)
    phi = np.arange(16) * (2 * np.pi / 16)
    ct, ph = np.meshgrid(x, phi, indexing="ij")
    st = np.sqrt(1 - ct ** 2)
    d = np.stack([st * np.cos(ph), st * np.sin(ph), ct], -1).reshape(-1, 3)
    wt = (w[:, None] * np.full(16, 2 * np.pi / 16)[None, :]).reshape(-1)
    Y, _ = oracle.sh_basis(d)
    G = (Y * wt[:, None]).T @ Y
    np.testing.assert_allclose(G, np.eye(16), atol=1e-12)


def test_basis_gradient_tangential_part_matches_finite_differences():
    d = _dirs(50, 1)
    _, dY = oracle.sh_basis(d)
    h = 1e-6
    for i in range(len(d)):
        # two tangent directions at d
        t1 = np.cross(d[i], [1.0, 0.3, -0.2])
        t1 /= np.linalg.norm(t1)
        t2 = np.cross(d[i], t1)
        for t in (t1, t2):
            dp = d[i] * np.cos(h) + t * np.sin(h)
            dm = d[i] * np.cos(h) - t * np.sin(h)
            fd = (oracle.sh_basis(dp[None])[0][0] - oracle.sh_basis(dm[None])[0][0]) / (2 * h)
            np.testing.assert_allclose(dY[i] @ t, fd, atol=1e-7)
