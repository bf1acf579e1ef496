"""The L1 + SSIM loss kernel (gs_loss_l1_ssim) against the oracle.

Tolerances (fp32 kernel, fp64 oracle).  The SSIM's variances are differences of
windowed moments, var = E[x^2] - mu^2: with values in [0, 1] each carries an absolute
rounding error of a few units of u = 2^-24 (E[x^2] <= 1), and B2 = var_x + var_y + c2
is at least c2 = 0.03^2, so SSIM and its derivatives carry a relative error up to
eps = 8 u / c2 = 5.3e-4, reached where both images are flat over the window.  The
gradient is compared element by element against the oracle's magnitude of its terms
(the same sums over absolute values): |gpu - ref| <= eps mag + 1e-6 max(mag).  Where
an image is flat the error repeats at every pixel instead of averaging out, so the
mean SSIM is held to the same bound, |gpu - ref| <= eps (|SSIM| <= 1), the loss to
lambda eps, and the mean |x - y|, a plain fp32 sum, to 1e-6 relative.
"""

import numpy as np
import pytest

import oracle
import synthetic_scenes as ss

pytestmark = pytest.mark.gpu

EPS = 8 * 2.0 ** -24 / 0.03 ** 2  # 5.3e-4
G_RTOL = EPS
G_ATOL = 1e-6


def _gpu_loss(x, y, settings=None):
    import torch

    import differentiable_gaussian_splatting_gb300 as gs

    H, W = x.shape[:2]
    xi = torch.from_numpy(np.ascontiguousarray(x)).cuda()
    yi = torch.from_numpy(np.ascontiguousarray(y)).cuda()
    d = torch.full_like(xi, float("nan"))
    out = torch.zeros(4, dtype=torch.float32, device="cuda")
    ws = torch.empty(gs.gs_loss_workspace_bytes(W, H), dtype=torch.uint8, device="cuda")
    gs.gs_loss_l1_ssim(W, H, xi, yi, d, out, ws, settings)
    torch.cuda.synchronize()
    return d.cpu().numpy(), out[:3].cpu().numpy().astype(np.float64)


def _compare(x, y, lam=0.2):
    import differentiable_gaussian_splatting_gb300 as gs

    s = gs.LossSettings.default()
    s.lambda_ = lam
    g, out = _gpu_loss(x, y, s)
    ref = oracle.loss_l1_ssim(x, y, lam=lam, want_map=True)
    assert np.isfinite(g).all()
    tol = (lam * EPS + 1e-6 * ref.l1, 1e-6 * ref.l1 + 1e-7, EPS)
    for k, want in enumerate((ref.loss, ref.l1, ref.ssim)):
        assert abs(out[k] - want) <= tol[k], (k, out[k], want)
    err = np.abs(g - ref.dL_dimg)
    bound = G_RTOL * ref.mag + G_ATOL * ref.mag.max()
    worst = np.unravel_index(np.argmax(err / bound), err.shape)
    assert (err <= bound).all(), (worst, g[worst], ref.dL_dimg[worst], ref.mag[worst])
    return g, ref


@pytest.mark.parametrize("H,W,seed", [(1, 1, 0), (5, 7, 1), (11, 11, 2), (37, 70, 3),
                                      (64, 96, 4), (100, 130, 5), (33, 129, 6)])
def test_loss_matches_oracle(H, W, seed):
    # one pixel, images smaller than the window, one tile, ragged multi-tile grids
    x, y = ss.image_pair(np.random.default_rng(seed), H, W)
    _compare(x, y)


@pytest.mark.parametrize("lam", [0.0, 1.0, 0.5])
def test_loss_weight_extremes(lam):
    x, y = ss.image_pair(np.random.default_rng(10), 45, 77)
    g, ref = _compare(x, y, lam)
    if lam == 0.0:
        # the L1 term alone: sign(x - y) / (3 H W), exact up to the fp32 weight
        inv = np.float32(1.0 / x.size)
        np.testing.assert_array_equal(g, (np.sign(x.astype(np.float64) - y) * inv).astype(
            np.float32))


def test_identical_images_zero_gradient():
    x, _ = ss.image_pair(np.random.default_rng(11), 40, 50)
    g, out = _gpu_loss(x, x)
    # SSIM(x, x) = 1 up to rounding; the gradient vanishes to rounding of its terms
    ref = oracle.loss_l1_ssim(x, x, want_map=True)
    assert abs(out[2] - 1.0) <= EPS and abs(out[1]) == 0.0
    assert (np.abs(g) <= G_RTOL * ref.mag + G_ATOL * ref.mag.max()).all()


def test_constant_images_closed_form():
    # flat images: SSIM of each interior pixel is (2ab + c1) / (a^2 + b^2 + c1)
    H, W = 70, 90
    a = np.array([0.25, 0.7, 0.5], np.float32)
    b = np.array([0.6, 0.2, 0.5], np.float32)
    x = np.broadcast_to(a, (H, W, 3)).copy()
    y = np.broadcast_to(b, (H, W, 3)).copy()
    _compare(x, y)


def test_deterministic():
    x, y = ss.image_pair(np.random.default_rng(12), 130, 260)
    g1, o1 = _gpu_loss(x, y)
    g2, o2 = _gpu_loss(x, y)
    np.testing.assert_array_equal(g1, g2)
    np.testing.assert_array_equal(o1, o2)


def test_full_size_image():
    # the 1297 x 840 image of the 1.5M-Gaussian scene, every element against the oracle
    x, y = ss.image_pair(np.random.default_rng(13), 840, 1297)
    _compare(x, y)


def test_argument_errors():
    import torch

    import differentiable_gaussian_splatting_gb300 as gs

    x = torch.zeros((8, 8, 3), device="cuda")
    y = torch.zeros_like(x)
    d = torch.zeros_like(x)
    out = torch.zeros(4, device="cuda")
    ws = torch.empty(gs.gs_loss_workspace_bytes(8, 8), dtype=torch.uint8, device="cuda")
    with pytest.raises(gs.GSError):
        gs.gs_loss_l1_ssim(8, 8, x, y, x, out, ws)  # gradient over the image
    bad = gs.LossSettings.default()
    bad.lambda_ = 1.5
    with pytest.raises(gs.GSError):
        gs.gs_loss_l1_ssim(8, 8, x, y, d, out, ws, bad)
    small = torch.empty(0, dtype=torch.uint8, device="cuda")
    with pytest.raises(gs.GSError):
        gs.gs_loss_l1_ssim(8, 8, x, y, d, out, small)
    gs.gs_loss_l1_ssim(8, 8, x, y, d, out, ws)
    torch.cuda.synchronize()
