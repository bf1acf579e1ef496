"""Pins of the oracle's forward blending (Ryu & Yoo, Eq. 2-3 and the 1e-4 stop; Kopanas,
Step 1 (b) support, 0.99 clamp) against a float64 brute force without tiles, hand-worked
cases and invariants."""

import numpy as np
import pytest

import oracle
from oracle import definitional as D
import synthetic_scenes as ss


@pytest.mark.parametrize("seed,W,H,n,deg", [(0, 37, 53, 300, 0), (1, 64, 64, 400, 3),
                                            (2, 150, 97, 900, 1), (3, 48, 32, 400, 2)])
def test_tiled_blend_equals_brute_force(seed, W, H, n, deg):
    rng = np.random.default_rng(seed)
    sc, cam = ss.random_scene(rng, n, W, H, sh_degree=deg, log_scale=(-2.5, 0.7), logit_std=2.5)
    r = oracle.render(sc, cam)
    C, T, nc, amb = D.brute_force_blend(cam, r.proj.splat, r.proj.rgb, r.proj.visible)
    ok = ~amb
    assert ok.mean() > 0.98
    np.testing.assert_allclose(r.image.img[ok], C[ok], rtol=0, atol=1e-12)
    np.testing.assert_allclose(r.image.T[ok], T[ok], rtol=1e-12, atol=1e-15)
    np.testing.assert_array_equal(r.image.n_contrib[ok], nc[ok])
    assert (r.image.n_contrib > 3).any()
    if seed in (1, 2):  # dense enough that some pixels stop early
        assert (r.image.T < 1e-4).any()
    # and the fp32 quadratic of the definition is the exact quadratic up to rounding
    C64, T64, nc64, amb64 = D.brute_force_blend(cam, r.proj.splat, r.proj.rgb, r.proj.visible,
                                                fp32_quadratic=False)
    ok = ~(amb | amb64)
    np.testing.assert_allclose(r.image.img[ok], C64[ok], rtol=1e-5, atol=1e-6)
    np.testing.assert_array_equal(r.image.n_contrib[ok], nc64[ok])


def test_fp32_fma_emulation_against_exact_rationals():
    from fractions import Fraction
    rng = np.random.default_rng(4)
    x, y, z = (rng.standard_normal(4000).astype(np.float32) * np.float32(s)
               for s in (1.0, 3.0, 1e-3))
    # include exact halfway cases: z chosen so x*y + z sits between two fp32 values
    r = D.fma_f32(x, y, z)
    for i in range(0, 4000, 7):
        exact = Fraction(float(x[i])) * Fraction(float(y[i])) + Fraction(float(z[i]))
        cands = [np.nextafter(r[i], np.float32(-np.inf)), r[i], np.nextafter(r[i], np.float32(np.inf))]
        errs = [abs(Fraction(float(cc)) - exact) for cc in cands]
        assert errs[1] <= min(errs)


def _stack_scene(opacities, colours, W=32, H=32, f=32.0):
    """Splats centred exactly on the centre of pixel (16, 16), at increasing depths."""
    n = len(opacities)
    z = 2.0 + np.arange(n, dtype=np.float64)
    # mu' = f x / z + W/2 = 16.5  ->  x = 0.5 z / f
    means = np.stack([0.5 * z / f, 0.5 * z / f, z], 1)
    rgb = np.asarray(colours, np.float64).reshape(n, 1, 3)
    sc = ss.Scene(means.astype(np.float32), np.full((n, 3), 0.05, np.float32),
                  np.tile([[1, 0, 0, 0]], (n, 1)).astype(np.float32),
                  np.asarray(opacities, np.float32), (rgb * 2 * np.sqrt(np.pi)).astype(np.float32), 0)
    return sc, ss.pinhole(np.eye(4), f, W, H)


def test_single_opaque_splat_is_clamped_to_099():
    sc, cam = _stack_scene([0.9999], [[0.2, 0.4, 0.8]])
    r = oracle.render(sc, cam)
    col = r.proj.rgb[0]
    np.testing.assert_allclose(r.image.img[16, 16], 0.99 * col, rtol=1e-12)
    np.testing.assert_allclose(r.image.T[16, 16], 0.01, rtol=1e-12)
    assert r.image.n_contrib[16, 16] == 1 and r.image.last_idx[16, 16] >= 0


def test_two_splats_hand_formula():
    sc, cam = _stack_scene([0.6, 0.5], [[1, 0, 0], [0, 1, 0]])
    r = oracle.render(sc, cam)
    c1, c2 = r.proj.rgb
    a1, a2 = np.float32(0.6), np.float32(0.5)
    np.testing.assert_allclose(r.image.img[16, 16], c1 * a1 + c2 * a2 * (1 - a1), rtol=1e-12)
    np.testing.assert_allclose(r.image.T[16, 16], (1 - a1) * (1 - a2), rtol=1e-12)


def test_early_termination_includes_crossing_splat():
    # ten splats of alpha 0.8 at the pixel: T = 0.2^k; 0.2^5 = 3.2e-4 >= 1e-4,
    # 0.2^6 = 6.4e-5 < 1e-4  ->  six splats blend, the sixth is the one that crosses
    sc, cam = _stack_scene([0.8] * 10, [[0.5, 0.25, 1.0]] * 10)
    r = oracle.render(sc, cam)
    a = float(np.float32(0.8))
    assert r.image.n_contrib[16, 16] == 6
    np.testing.assert_allclose(r.image.T[16, 16], (1 - a) ** 6, rtol=1e-12)
    np.testing.assert_allclose(r.image.img[16, 16], r.proj.rgb[0] * (1 - (1 - a) ** 6), rtol=1e-12)
    t = (16 // 16) * oracle.n_tiles(cam)[0] + 16 // 16
    assert r.image.last_idx[16, 16] == r.binning.ranges[t, 0] + 5


def test_invariants_on_random_scenes():
    for seed in range(4):
        rng = np.random.default_rng(10 + seed)
        sc, cam = ss.random_scene(rng, 300, 80, 72, sh_degree=2, log_scale=(-2.5, 0.8),
                                  logit_std=3.0)
        r = oracle.render(sc, cam)
        T, nc, last = r.image.T, r.image.n_contrib, r.image.last_idx
        assert np.all((T >= 0) & (T <= 1))
        assert np.all((nc == 0) == (last == -1))
        assert np.all(r.image.img[nc == 0] == 0) and np.all(T[nc == 0] == 1)
        # the final transmittance is at least (1 - 0.99)^n
        assert np.all(T >= 0.01 ** nc.astype(np.float64) * (1 - 1e-12))
        # once T < 1e-4 the pixel stopped: exactly one blend took it below (T >= 1e-6)
        stopped = T < 1e-4
        assert np.all(T[stopped] >= 1e-4 * 0.01 * (1 - 1e-12))
        # last_idx lies in the pixel's tile range
        ntx, _ = oracle.n_tiles(cam)
        ys, xs = np.nonzero(nc > 0)
        t = (ys // 16) * ntx + xs // 16
        assert np.all(last[ys, xs] >= r.binning.ranges[t, 0])
        assert np.all(last[ys, xs] < r.binning.ranges[t, 1])


def test_empty_and_fully_culled_scenes():
    cam = ss.pinhole(np.eye(4), 50.0, 40, 30)
    empty = ss.Scene(np.zeros((0, 3), np.float32), np.zeros((0, 3), np.float32),
                     np.zeros((0, 4), np.float32), np.zeros(0, np.float32),
                     np.zeros((0, 1, 3), np.float32), 0)
    r = oracle.render(empty, cam)
    assert r.binning.n_pairs == 0 and np.all(r.image.T == 1) and np.all(r.image.img == 0)
    behind = ss.random_scene(np.random.default_rng(0), 20, 40, 30, sh_degree=0)[0]
    behind.means[:, 2] = -behind.means[:, 2]
    r = oracle.render(behind, cam)
    assert r.binning.n_pairs == 0 and np.all(r.image.T == 1)
