"""Pins of the oracle's L1 + SSIM training loss and its gradient.

The loss is the usual 3DGS objective (1 - lambda) mean|x - y| + lambda (1 - mean SSIM)
with the structural similarity of Wang et al. (2004) over an 11 x 11 Gaussian window
(sigma 1.5) and zero outside the image.  The pins below do not retype the oracle's
formulas: they check it against closed forms of special inputs, against a library
blur (scipy's truncated Gaussian filter) for the window, and its gradient against
central differences of its own loss.
"""

import numpy as np
import pytest
from scipy.ndimage import gaussian_filter, gaussian_filter1d

import oracle

SIG = oracle.SSIM_SIGMA
TRUNC = 5.0 / SIG  # scipy's radius int(truncate * sigma + 0.5) = 5: 11 taps


def _mass(n):
    """Weight of the normalised 11-tap window that falls inside [0, n) at each position."""
    return gaussian_filter1d(np.ones(n), SIG, mode="constant", cval=0.0, truncate=TRUNC)


def _blur(a):
    """The windowed mean with zero outside, per channel, from scipy."""
    return gaussian_filter(a, (SIG, SIG, 0), mode="constant", cval=0.0, truncate=TRUNC)


def test_identical_images():
    rng = np.random.default_rng(1)
    x = rng.random((13, 17, 3), dtype=np.float32)
    L = oracle.loss_l1_ssim(x, x, want_map=True)
    assert L.loss == 0.0 and L.l1 == 0.0
    np.testing.assert_allclose(L.ssim_map, 1.0, rtol=0, atol=1e-14)
    # SSIM is at its maximum and |x - y| at its kink: the gradient is zero
    assert np.abs(L.dL_dimg).max() < 1e-15


def test_constant_images_closed_form_with_borders():
    # x = a, y = b everywhere: with m the window mass inside the image,
    # mu = a m, e_xx = a^2 m, var = a^2 m (1 - m), cov = a b m (1 - m)
    H, W = 14, 19
    a = np.array([0.3, 0.8, 0.55])
    b = np.array([0.6, 0.1, 0.55])
    x = np.broadcast_to(a, (H, W, 3)).astype(np.float32)
    y = np.broadcast_to(b, (H, W, 3)).astype(np.float32)
    a = x[0, 0].astype(np.float64)
    b = y[0, 0].astype(np.float64)
    c1, c2 = oracle.SSIM_C1, oracle.SSIM_C2
    m = (_mass(H)[:, None] * _mass(W)[None, :])[..., None]
    num = (2 * a * b * m * m + c1) * (2 * a * b * m * (1 - m) + c2)
    den = ((a * a + b * b) * m * m + c1) * ((a * a + b * b) * m * (1 - m) + c2)
    L = oracle.loss_l1_ssim(x, y, want_map=True)
    np.testing.assert_allclose(L.ssim_map, num / den, rtol=1e-12, atol=0)
    # the interior reduces to the luminance term alone
    inner = L.ssim_map[5:-5, 5:-5]
    np.testing.assert_allclose(inner, np.broadcast_to((2 * a * b + c1) / (a * a + b * b + c1),
                                                      inner.shape), rtol=1e-12)


@pytest.mark.parametrize("alpha", [0.5, 1.7, -0.8])
def test_scaled_image_without_constants(alpha):
    # y = alpha x and c1 = c2 = 0: mu_y = alpha mu_x, var_y = alpha^2 var_x and
    # cov = alpha var_x at every pixel (the zero outside scales too), so
    # SSIM = (2 alpha / (1 + alpha^2))^2 everywhere, whatever x is
    rng = np.random.default_rng(2)
    x = (0.2 + 0.8 * rng.random((12, 15, 3))).astype(np.float32)
    y = (np.float64(alpha) * x.astype(np.float64)).astype(np.float32)
    L = oracle.loss_l1_ssim(x, y, c1=0.0, c2=0.0, want_map=True)
    # y is alpha x rounded to float32; the closed form holds to that rounding
    want = (2 * alpha / (1 + alpha * alpha)) ** 2
    np.testing.assert_allclose(L.ssim_map, want, rtol=2e-5)


def test_affine_image_interior_closed_form():
    # y = alpha x + beta, c1 = c2 = 0, pixels whose window lies inside the image:
    # SSIM = 2 mu_x mu_y / (mu_x^2 + mu_y^2) * 2 alpha / (1 + alpha^2), mu_y = alpha mu_x + beta
    rng = np.random.default_rng(3)
    alpha, beta = 0.7, 0.25
    x = (0.2 + 0.8 * rng.random((20, 22, 3))).astype(np.float32)
    y = (alpha * x.astype(np.float64) + beta).astype(np.float32)
    yd = y.astype(np.float64)
    L = oracle.loss_l1_ssim(x, y, c1=0.0, c2=0.0, want_map=True)
    mx = _blur(x.astype(np.float64))
    my = _blur(yd)
    want = 2 * mx * my / (mx * mx + my * my) * (2 * alpha / (1 + alpha * alpha))
    np.testing.assert_allclose(L.ssim_map[5:-5, 5:-5], want[5:-5, 5:-5], rtol=2e-5)


def test_ssim_map_against_library_blur():
    # the windowed moments against scipy's filter (a library routine for w *),
    # assembled into SSIM; constants at their usual values
    rng = np.random.default_rng(4)
    x = rng.random((16, 21, 3), dtype=np.float32)
    y = np.clip(x + 0.2 * rng.standard_normal(x.shape), 0, 1).astype(np.float32)
    xd, yd = x.astype(np.float64), y.astype(np.float64)
    mx, my = _blur(xd), _blur(yd)
    vx = _blur(xd * xd) - mx * mx
    vy = _blur(yd * yd) - my * my
    cv = _blur(xd * yd) - mx * my
    c1, c2 = oracle.SSIM_C1, oracle.SSIM_C2
    want = (2 * mx * my + c1) * (2 * cv + c2) / ((mx * mx + my * my + c1) * (vx + vy + c2))
    L = oracle.loss_l1_ssim(x, y, want_map=True)
    np.testing.assert_allclose(L.ssim_map, want, rtol=1e-10, atol=1e-12)
    # symmetric in its two images
    Ls = oracle.loss_l1_ssim(y, x, want_map=True)
    np.testing.assert_allclose(Ls.ssim_map, L.ssim_map, rtol=1e-13, atol=1e-15)
    assert L.ssim_map.max() <= 1.0 + 1e-12


def test_l1_term_alone():
    rng = np.random.default_rng(5)
    x = rng.random((9, 10, 3), dtype=np.float32)
    y = rng.random((9, 10, 3), dtype=np.float32)
    y[0, 0, 0] = x[0, 0, 0]  # an exact tie takes derivative 0
    L = oracle.loss_l1_ssim(x, y, lam=0.0)
    d = x.astype(np.float64) - y.astype(np.float64)
    assert L.loss == pytest.approx(np.abs(d).mean(), rel=1e-14)
    np.testing.assert_array_equal(L.dL_dimg, np.sign(d) / d.size)


def test_mixture_of_terms():
    rng = np.random.default_rng(6)
    x = rng.random((11, 12, 3), dtype=np.float32)
    y = rng.random((11, 12, 3), dtype=np.float32)
    L = oracle.loss_l1_ssim(x, y, lam=0.3)
    assert L.loss == pytest.approx(0.7 * L.l1 + 0.3 * (1 - L.ssim), rel=1e-14)


@pytest.mark.parametrize("shape,lam", [((9, 11), 0.2), ((14, 13), 1.0)])
def test_gradient_central_differences(shape, lam):
    # every element of an image smaller than or near the window, so border and
    # interior pixels both enter; |x - y| stays above the step to avoid the kink
    rng = np.random.default_rng(7)
    H, W = shape
    x = (0.1 + 0.8 * rng.random((H, W, 3))).astype(np.float32)
    off = (0.02 + 0.1 * rng.random(x.shape)) * rng.choice([-1.0, 1.0], x.shape)
    y = (x.astype(np.float64) + off).astype(np.float32)
    g = oracle.loss_l1_ssim(x, y, lam=lam).dL_dimg
    h = np.float32(2.0 ** -10)
    fd = np.empty_like(g)
    for idx in np.ndindex(x.shape):
        xp = x.copy()
        xm = x.copy()
        xp[idx] += h
        xm[idx] -= h
        step = np.float64(xp[idx]) - np.float64(xm[idx])
        fd[idx] = (oracle.loss_l1_ssim(xp, y, lam=lam).loss
                   - oracle.loss_l1_ssim(xm, y, lam=lam).loss) / step
    scale = np.abs(g).max()
    np.testing.assert_allclose(g, fd, rtol=0, atol=2e-5 * scale)
    assert scale > 0
