"""Pins of the oracle's projection (Ryu & Yoo, Sec. 2.1, Eq. 1) against closed forms,
library routines and numerical differentiation -- never against its own formulas."""

import mpmath
import numpy as np
import pytest
from scipy.spatial.transform import Rotation

import oracle
from oracle import definitional as D
import synthetic_scenes as ss


def _one(mean, scale, quat, opac, W=64, H=48, f=60.0, deg=0, viewmat=None):
    sc = ss.Scene(np.array([mean], np.float32), np.array([scale], np.float32),
                  np.array([quat], np.float32), np.array([opac], np.float32),
                  np.zeros((1, (deg + 1) ** 2, 3), np.float32), deg)
    cam = ss.pinhole(np.eye(4) if viewmat is None else viewmat, f, W, H)
    return sc, cam


def test_conic_inverts_projected_covariance():
    rng = np.random.default_rng(1)
    sc, cam = ss.random_scene(rng, 400, 96, 80, sh_degree=0)
    p = oracle.project(sc, cam)
    v = p.visible
    assert v.sum() > 300
    a, b, c = p.splat[v, 2], p.splat[v, 3], p.splat[v, 4]
    P00, P01, P11 = p.splat[v, 8], p.splat[v, 9], p.splat[v, 10]
    # Lambda Sigma' = I; each entry is a two-term sum evaluated from fp32 values
    e00 = a * P00 + b * P01
    e01 = a * P01 + b * P11
    e11 = b * P01 + c * P11
    s00 = np.abs(a * P00) + np.abs(b * P01)
    s01 = np.abs(a * P01) + np.abs(b * P11)
    s11 = np.abs(b * P01) + np.abs(c * P11)
    tol = 2e-6
    assert np.all(np.abs(e00 - 1) <= tol * s00)
    assert np.all(np.abs(e11 - 1) <= tol * s11)
    assert np.all(np.abs(e01) <= tol * s01)


def test_isotropic_gaussian_on_axis():
    # an isotropic Gaussian on the optical axis projects to (cx, cy) with
    # Sigma' = (f s / z)^2 I, whatever its rotation
    for z, s, f in [(3.0, 0.1, 60.0), (10.0, 0.5, 200.0), (2.5, 0.02, 1000.0)]:
        q = np.random.default_rng(int(z * 10)).standard_normal(4)
        sc, cam = _one([0, 0, z], [s, s, s], q / np.linalg.norm(q), 0.9, f=f, W=64, H=64)
        p = oracle.project(sc, cam)
        assert p.tiles_touched[0] > 0
        exp_var = (f * s / z) ** 2
        np.testing.assert_allclose(p.splat[0, :2], [32.0, 32.0], rtol=0, atol=1e-5)
        np.testing.assert_allclose(p.splat[0, [8, 10]], [exp_var, exp_var], rtol=3e-6)
        assert abs(p.splat[0, 9]) <= 3e-6 * exp_var


def _numerical_jacobian(cam, m, h=1e-6):
    J = np.zeros((2, 3))
    for k in range(3):
        e = np.zeros(3)
        e[k] = h * max(1.0, abs(m[k]))
        J[:, k] = (D.pinhole(cam, m + e) - D.pinhole(cam, m - e)) / (2 * e[k])
    return J


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_projection_is_linearised_pinhole(seed):
    """Sigma' equals J_num Sigma J_num^T with J_num the numerical Jacobian of the
    pinhole map and Sigma = R S^2 R^T built with scipy's rotation (f64 oracle build).
    The focal lengths differ and the principal point is off the image centre, so that
    Eq. 1's two rows (fx / t_z, fy / t_z) and the two offsets cannot stand in for each
    other."""
    rng = np.random.default_rng(seed)
    eye = rng.uniform(-1, 1, 3) + np.array([0, 0, -5.0])
    V = ss.look_at(eye, rng.uniform(-0.3, 0.3, 3))
    cam = ss.Camera(V, 300.0, 230.0, 150.0, 130.0, 320, 240, 0.2)
    n = 50
    means = rng.uniform(-0.6, 0.6, (n, 3))
    scales = np.exp(rng.normal(-3, 0.5, (n, 3)))
    quats = rng.standard_normal((n, 4))
    sc = ss.Scene(means.astype(np.float32), scales.astype(np.float32),
                  quats.astype(np.float32), np.full(n, 0.8, np.float32),
                  np.zeros((n, 1, 3), np.float32), 0)
    p = oracle.project(sc, cam, variant="f64")
    checked = 0
    for i in range(n):
        if not p.visible[i]:
            continue
        m = sc.means[i].astype(np.float64)
        Jn = _numerical_jacobian(cam, m)
        q = sc.quats[i].astype(np.float64)
        Rm = Rotation.from_quat([q[1], q[2], q[3], q[0]]).as_matrix()
        Sig = Rm @ np.diag(sc.scales[i].astype(np.float64) ** 2) @ Rm.T
        P = Jn @ Sig @ Jn.T
        np.testing.assert_allclose(p.splat[i, [8, 9, 10]], [P[0, 0], P[0, 1], P[1, 1]],
                                   rtol=2e-6, atol=2e-8 * np.abs(P).max())
        np.testing.assert_allclose(p.splat[i, :2], D.pinhole(cam, m), rtol=1e-12)
        np.testing.assert_allclose(p.splat[i, 7], (np.asarray(V, np.float64)[:3, :3] @ m +
                                                   np.asarray(V, np.float64)[:3, 3])[2], rtol=1e-12)
        checked += 1
    assert checked > 30


def test_projected_covariance_monte_carlo():
    # a small, far Gaussian: the sample covariance of projected points approaches Sigma'
    rng = np.random.default_rng(7)
    q = np.array([0.9, 0.2, -0.3, 0.25])
    q /= np.linalg.norm(q)
    s = np.array([0.02, 0.05, 0.01])
    m = np.array([0.3, -0.2, 8.0])
    sc, cam = _one(m, s, q, 0.9, W=200, H=200, f=500.0)
    p = oracle.project(sc, cam, variant="f64")
    Rm = Rotation.from_quat([q[1], q[2], q[3], q[0]]).as_matrix()
    pts = m + (rng.standard_normal((200_000, 3)) * s) @ Rm.T
    uv = np.stack([500.0 * pts[:, 0] / pts[:, 2] + 100, 500.0 * pts[:, 1] / pts[:, 2] + 100], 1)
    cov = np.cov(uv.T)
    np.testing.assert_allclose([cov[0, 0], cov[0, 1], cov[1, 1]], p.splat[0, [8, 9, 10]],
                               rtol=0.02, atol=0.02 * cov.max())


def test_quaternion_sign_and_scale_invariance():
    q = np.array([0.25, -0.5, 0.75, 0.125])  # exact in fp32
    outs = []
    for qq in (q, -q, 2.0 * q):
        sc, cam = _one([0.2, -0.1, 4.0], [0.1, 0.3, 0.05], qq, 0.7)
        outs.append(oracle.project(sc, cam, variant="f64").splat[0, 8:11])
    np.testing.assert_allclose(outs[1], outs[0], rtol=1e-12)
    np.testing.assert_allclose(outs[2], outs[0], rtol=1e-12)


def _round_f32(x: mpmath.mpf) -> np.float32:
    f = np.float32(float(x))
    cands = [np.nextafter(f, np.float32(-np.inf)), f, np.nextafter(f, np.float32(np.inf))]
    return min(cands, key=lambda c: abs(mpmath.mpf(float(c)) - x))


def test_tau_is_correctly_rounded_2ln255o():
    rng = np.random.default_rng(3)
    ops = np.concatenate([rng.uniform(1 / 255, 1, 300), [0.004, 0.5, 0.99, 0.9999]]).astype(np.float32)
    mpmath.mp.dps = 60
    n = len(ops)
    sc = ss.Scene(np.tile([[0, 0, 3.0]], (n, 1)).astype(np.float32),
                  np.full((n, 3), 0.2, np.float32), np.tile([[1, 0, 0, 0]], (n, 1)).astype(np.float32),
                  ops, np.zeros((n, 1, 3), np.float32), 0)
    cam = ss.pinhole(np.eye(4), 60.0, 64, 64)
    p = oracle.project(sc, cam)
    for i, o in enumerate(ops):
        exact = 2 * mpmath.log(255 * mpmath.mpf(float(o)))
        assert p.splat[i, 6] == float(_round_f32(exact)), (o, p.splat[i, 6])


def test_support_half_extents_and_radii():
    """rx = max |dx| over the ellipse q(d) = tau, from a parametrisation of the ellipse."""
    rng = np.random.default_rng(5)
    sc, cam = ss.random_scene(rng, 100, 128, 96, sh_degree=0)
    p = oracle.project(sc, cam)
    th = np.linspace(0, 2 * np.pi, 20001)
    for i in np.nonzero(p.visible)[0][:40]:
        P = np.array([[p.splat[i, 8], p.splat[i, 9]], [p.splat[i, 9], p.splat[i, 10]]])
        L = np.linalg.cholesky(P)
        pts = np.sqrt(p.splat[i, 6]) * (L @ np.stack([np.cos(th), np.sin(th)]))
        rx, ry = np.abs(pts[0]).max(), np.abs(pts[1]).max()
        assert p.radii[i, 0] == int(np.ceil(rx * (1 - 1e-6))) or p.radii[i, 0] == int(np.ceil(rx))
        assert p.radii[i, 1] == int(np.ceil(ry * (1 - 1e-6))) or p.radii[i, 1] == int(np.ceil(ry))


def test_culling_cases():
    base = dict(scale=[0.1, 0.1, 0.1], quat=[1, 0, 0, 0])
    # behind the near plane and behind the camera
    for z in (0.1, 0.2, -3.0):
        sc, cam = _one([0, 0, z], base["scale"], base["quat"], 0.9)
        assert oracle.project(sc, cam).tiles_touched[0] == 0
    # opacity at or below the 1/255 cutoff (tau <= 0)
    for o in (0.0039, 1.0 / 256):
        sc, cam = _one([0, 0, 3.0], base["scale"], base["quat"], o)
        assert oracle.project(sc, cam).tiles_touched[0] == 0
    # just above the cutoff the support is tiny (rx ~ 0.4 px): centre it on a pixel centre
    sc, cam = _one([0.025, 0.025, 3.0], base["scale"], base["quat"], 0.004)
    assert oracle.project(sc, cam).tiles_touched[0] == 1
    # far outside the image: no tile
    sc, cam = _one([50.0, 0, 3.0], base["scale"], base["quat"], 0.9)
    assert oracle.project(sc, cam).tiles_touched[0] == 0
    # degenerate: zero scales, zero quaternion, non-finite mean
    for scale, quat, mean in (([0, 0, 0], [1, 0, 0, 0], [0, 0, 3.0]),
                              ([0.1] * 3, [0, 0, 0, 0], [0, 0, 3.0]),
                              ([0.1] * 3, [1, 0, 0, 0], [np.nan, 0, 3.0])):
        sc, cam = _one(mean, scale, quat, 0.9)
        p = oracle.project(sc, cam)
        assert p.tiles_touched[0] == 0 and np.all(p.splat[0] == 0)


def test_sh_degree0_is_constant_colour():
    rng = np.random.default_rng(11)
    sc, cam = ss.random_scene(rng, 50, 64, 64, sh_degree=0)
    p = oracle.project(sc, cam)
    v = p.visible
    # degree-0 colour = Y_00 s_0 with Y_00 = 1 / (2 sqrt(pi))
    np.testing.assert_allclose(p.rgb[v], sc.sh[v, 0, :] / (2 * np.sqrt(np.pi)), rtol=1e-6)


def test_colour_follows_the_direction_from_the_camera_centre():
    """A camera placed at C and turned by R has the view matrix [R | -R C]. Each colour is
    then sum_k Y_k(d) s_k with d the unit vector from C to the mean (Kopanas, Step 3),
    here built from C itself rather than recovered from the view matrix."""
    rng = np.random.default_rng(11)
    sc, cam = ss.random_scene(rng, 60, 64, 48, sh_degree=3)
    R = Rotation.random(random_state=5).as_matrix()
    C = np.array([0.7, -1.3, 2.1])
    means_cam = sc.means.astype(np.float64)
    sc.means = (means_cam @ R + C).astype(np.float32)  # world = R^T m_cam + C
    V = np.eye(4)
    V[:3, :3] = R
    V[:3, 3] = -R @ C
    cam = ss.pinhole(V.astype(np.float32), cam.fx, cam.width, cam.height)
    proj = oracle.project(sc, cam)
    vis = proj.visible
    assert vis.sum() >= 30
    d = sc.means.astype(np.float64) - C
    d /= np.linalg.norm(d, axis=1, keepdims=True)
    Y, _ = oracle.sh_basis(d)
    expect = np.einsum("nk,nkc->nc", Y, sc.sh.astype(np.float64))
    np.testing.assert_allclose(proj.rgb[vis], expect[vis], rtol=1e-5, atol=1e-6)
    assert np.all(proj.rgb[~vis] == 0)
