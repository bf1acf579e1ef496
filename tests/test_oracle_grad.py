"""Pins of the oracle's backward pass by central finite differences of its own forward
(f64 build, where the quadratic, the spans and the hit test are smooth in the inputs):
the nine screen-space derivatives per splat (Kopanas, Step 1 (a)) and the 59 per-Gaussian
parameter gradients (means 3, scales 3, quaternion 4, opacity 1, SH 48; Kopanas, Step 3).
A finite difference is used only where the perturbation leaves every hit and stop decision
unchanged (same n_contrib and last_idx maps)."""

import copy

import numpy as np
import pytest

import oracle
import synthetic_scenes as ss

V64 = "f64"


def _scene(seed, n=40, W=64, H=48, deg=3):
    rng = np.random.default_rng(seed)
    sc, _ = ss.random_scene(rng, n, W, H, sh_degree=deg, log_scale=(-2.3, 0.4), logit_std=1.5)
    eye = np.array([0.3, -0.2, -0.5])
    V = ss.look_at(eye, np.array([0.0, 0.0, 4.0]), up=(0.05, -1.0, 0.0))
    # fx != fy and an off-centre principal point: the chain rule's two Jacobian rows
    # and the two offsets are told apart
    cam = ss.Camera(V, 64.0, 52.0, 0.47 * W, 0.53 * H, W, H, 0.2)
    w = rng.standard_normal((H, W, 3))
    v = rng.standard_normal((H, W))
    return sc, cam, w, v


def _refactor(proj, g):
    """Cholesky factor of the (perturbed) conic a, b, c of splat g, in float64."""
    a, b, c = proj.splat[g, 2:5]
    l11 = np.sqrt(a)
    l12 = b / l11
    proj.splat[g, 13:16] = [l11, l12, np.sqrt(c - l12 * l12)]


def _loss_from_records(cam, proj, b, w, v):
    im = oracle.blend(cam, proj, b, V64)
    return float((w * im.img).sum() + (v * im.T).sum()), im


def _fd_screen_space(cam, proj, b, w, v, im0, g2, splats):
    """Central differences of the loss in each record entry of the given splats, against
    the analytic nine derivatives; returns the number of entries checked (an entry is
    skipped when a perturbation changes a hit or stop decision)."""
    # record columns: 0 mux, 1 muy, 2 a, 3 b, 4 c, 5 opacity; rgb separately
    cols = [(0, 0), (1, 1), (2, 2), (3, 3), (4, 4), (5, 5)]
    checked = 0
    for g in splats:
        for col, gi in cols + [("rgb", 6), ("rgb", 7), ("rgb", 8)]:
            p_hi, p_lo = copy.deepcopy(proj), copy.deepcopy(proj)
            if col == "rgb":
                h = 1e-4
                p_hi.rgb[g, gi - 6] += h
                p_lo.rgb[g, gi - 6] -= h
            else:
                x = proj.splat[g, col]
                h = 1e-5 * max(abs(x), 1e-3) if col in (2, 3, 4, 5) else 1e-5
                p_hi.splat[g, col] = x + h
                p_lo.splat[g, col] = x - h
                if col in (2, 3, 4):  # the quadratic reads the conic through its factor
                    for pp in (p_hi, p_lo):
                        _refactor(pp, g)
            L1, i1 = _loss_from_records(cam, p_hi, b, w, v)
            L2, i2 = _loss_from_records(cam, p_lo, b, w, v)
            if not (np.array_equal(i1.n_contrib, im0.n_contrib) and
                    np.array_equal(i2.n_contrib, im0.n_contrib) and
                    np.array_equal(i1.last_idx, im0.last_idx) and
                    np.array_equal(i2.last_idx, im0.last_idx)):
                continue
            fd = (L1 - L2) / (2 * h)
            assert abs(g2[g, gi] - fd) <= 1e-6 + 2e-6 * abs(fd), (g, gi, g2[g, gi], fd)
            checked += 1
    return checked


@pytest.mark.parametrize("seed", [0, 1])
def test_screen_space_gradients_match_finite_differences(seed):
    sc, cam, w, v = _scene(seed)
    proj = oracle.project(sc, cam, V64)
    b = oracle.bin_sort(cam, proj, None, V64)
    _, im0 = _loss_from_records(cam, proj, b, w, v)
    g2, _ = oracle.blend_bwd(cam, proj, b, w, v, V64)
    gs = np.nonzero(np.abs(g2).sum(1) > 0)[0]
    assert len(gs) >= 10
    assert _fd_screen_space(cam, proj, b, w, v, im0, g2, gs[:15]) >= 100


def _front_clamped(cam, proj):
    """Splats whose alpha reaches the 0.99 clamp at a pixel where they are the front-most
    hit (so they blend there at T = 1), from the records' conics in numpy."""
    ys, xs = np.mgrid[0:cam.height, 0:cam.width]
    px, py = xs + 0.5, ys + 0.5
    front = np.full((cam.height, cam.width), np.inf)
    who = np.full((cam.height, cam.width), -1)
    raw = np.zeros((cam.height, cam.width))
    for g in np.nonzero(proj.visible)[0]:
        mx, my, a, bb, c, o, tau, z = proj.splat[g, :8]
        dx, dy = px - mx, py - my
        q = a * dx * dx + 2 * bb * dx * dy + c * dy * dy
        hit = (q <= tau) & (z < front)
        front[hit], who[hit], raw[hit] = z, g, o * np.exp(-0.5 * q[hit])
    return np.unique(who[(who >= 0) & (raw > 0.99 * (1 + 1e-4))])


def test_clamped_alphas_carry_no_geometry_or_opacity_gradient():
    """Where o exp(-q/2) exceeds 0.99 the alpha is the constant 0.99, so that pixel adds
    nothing to the derivatives of the splat's mean, conic and opacity; only its colour
    term remains. Large splats of opacity 0.995-0.999 are clamped near their centres,
    and central differences, which see the clamp, must agree with the backward."""
    for seed in range(20, 40):
        rng = np.random.default_rng(seed)
        sc, cam, w, v = _scene(seed, n=10)
        sc.scales *= np.float32(4.0)
        sc.opacities[:] = rng.uniform(0.995, 0.999, sc.n).astype(np.float32)
        proj = oracle.project(sc, cam, V64)
        b = oracle.bin_sort(cam, proj, None, V64)
        _, im0 = _loss_from_records(cam, proj, b, w, v)
        if np.any(im0.flags & 2):  # an alpha within rounding of the clamp: resample
            continue
        clamped = _front_clamped(cam, proj)
        if len(clamped) >= 3:
            break
    else:
        pytest.fail("no scene with clamped splats and no alpha near the clamp")
    g2, _ = oracle.blend_bwd(cam, proj, b, w, v, V64)
    assert _fd_screen_space(cam, proj, b, w, v, im0, g2, clamped[:6]) >= 25


def _perturbed(sc, field, idx, delta):
    s2 = copy.deepcopy(sc)
    arr = getattr(s2, field)
    flat = arr.reshape(arr.shape[0], -1)
    old = flat[idx]
    flat[idx] = np.float32(old + delta)
    return s2, float(flat[idx]) - float(old)


@pytest.mark.parametrize("seed", [0, 1])
def test_parameter_gradients_match_finite_differences(seed):
    sc, cam, w, v = _scene(seed, n=25)
    L0, r0, g2, pg = oracle.loss_and_grads(sc, cam, w, v, V64)
    live = np.nonzero(np.abs(g2).sum(1) > 0)[0]
    assert len(live) >= 8
    fields = [("means", pg.means, 3, 1e-4), ("scales", pg.scales, 3, 1e-3),
              ("quats", pg.quats, 4, 1e-3), ("opacities", pg.opacities.reshape(-1, 1), 1, 1e-3),
              ("sh", pg.sh.reshape(sc.n, -1), sc.sh.shape[1] * 3, 1e-2)]
    checked = 0
    for g in live[:8]:
        for name, grad, width, rel in fields:
            arr = getattr(sc, name).reshape(sc.n, -1)
            for j in range(width):
                x = float(arr[g, j])
                h = rel * max(abs(x), 1e-2)
                s_hi, d_hi = _perturbed(sc, name, (g, j), +h)
                s_lo, d_lo = _perturbed(sc, name, (g, j), -h)
                r_hi = oracle.render(s_hi, cam, None, V64)
                r_lo = oracle.render(s_lo, cam, None, V64)
                same = all(np.array_equal(r.image.n_contrib, r0.image.n_contrib) and
                           np.array_equal(r.image.last_idx, r0.image.last_idx)
                           for r in (r_hi, r_lo))
                if not same:
                    continue
                L_hi = float((w * r_hi.image.img).sum() + (v * r_hi.image.T).sum())
                L_lo = float((w * r_lo.image.img).sum() + (v * r_lo.image.T).sum())
                fd = (L_hi - L_lo) / (d_hi - d_lo)
                an = grad[g, j]
                assert abs(an - fd) <= 1e-6 + 1e-4 * abs(fd), (name, g, j, an, fd)
                checked += 1
    assert checked >= 300


def test_parameter_gradient_magnitudes_bound_the_gradients():
    """The running-error magnitudes of the chain rule dominate |gradient| (the triangle
    inequality applied stage by stage)."""
    sc, cam, w, v = _scene(3, n=30)
    L0, r0, g2, pg = oracle.loss_and_grads(sc, cam, w, v)
    mag = oracle.project_bwd_magnitude(sc, cam, r0.proj, np.abs(g2))
    for k in ("means", "scales", "quats", "opacities", "sh"):
        assert np.all(getattr(mag, k) >= np.abs(getattr(pg, k)) * (1 - 1e-9) - 1e-15), k
