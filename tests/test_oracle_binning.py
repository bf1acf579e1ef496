"""Pins of the oracle's tile binning (Kopanas, Step 1 (b): exact conic-tile spans) and of
its pair ordering (Step 1 (d)) and LPT order (Ryu & Yoo, Sec. 4.1)."""

import numpy as np
import pytest

import oracle
from oracle import definitional as D
import synthetic_scenes as ss

CASES = [(0, 37, 53, 60), (1, 128, 128, 120), (2, 150, 97, 140), (3, 64, 40, 300)]


def _scene(seed, W, H, n):
    rng = np.random.default_rng(seed)
    # a mix of tiny, medium and large, strongly anisotropic splats
    sc, cam = ss.random_scene(rng, n, W, H, sh_degree=0, log_scale=(-3.0, 1.0), spread=1.2)
    return sc, cam


@pytest.mark.parametrize("seed,W,H,n", CASES)
def test_emitted_tiles_are_exact_and_complete(seed, W, H, n):
    """A tile is emitted iff the support ellipse q(d) <= tau meets the hull of its pixel
    centres -- decided here by the exact minimum of q over the rectangle, not by spans.
    Emitted tiles may lie within the documented widening (the ellipse q <= tau (1 + 2^-21),
    grown by 2^-8 px + r 2^-20); tiles that truly meet the ellipse are always emitted."""
    sc, cam = _scene(seed, W, H, n)
    p = oracle.project(sc, cam)
    ntx, nty = oracle.n_tiles(cam)
    nvis = 0
    for g in range(sc.n):
        rec = p.splat[g]
        if p.tiles_touched[g] == 0:
            # culled: either invisible, or the ellipse meets no tile
            if rec[6] > 0 and rec[13] > 0:
                a, b, c = p.conic_of_factor()[g]
                for t in range(ntx * nty):
                    x0, x1, y0, y1 = D.tile_hull(cam, t)
                    qmin = D.rect_min_q(a, b, c, x0 - rec[0], x1 - rec[0],
                                        y0 - rec[1], y1 - rec[1])
                    assert qmin > rec[6] * (1 - 1e-5)
            continue
        nvis += 1
        tiles = set(oracle.splat_tiles(cam, rec).tolist())
        assert len(tiles) == p.tiles_touched[g]
        # the quadratic is evaluated through its Cholesky factor: its conic
        a, b, c = p.conic_of_factor()[g]
        tau = rec[6]
        rx, ry = rec[11], rec[12]
        padx = 2.0 ** -8 + rx * 2.0 ** -20 + 1e-4
        pady = 2.0 ** -8 + ry * 2.0 ** -20 + 1e-4
        for t in range(ntx * nty):
            x0, x1, y0, y1 = D.tile_hull(cam, t)
            qmin = D.rect_min_q(a, b, c, x0 - rec[0], x1 - rec[0], y0 - rec[1], y1 - rec[1])
            if t in tiles:
                qpad = D.rect_min_q(a, b, c, x0 - padx - rec[0], x1 + padx - rec[0],
                                    y0 - pady - rec[1], y1 + pady - rec[1])
                assert qpad <= tau * (1 + 1e-5), (g, t)
            else:
                assert qmin > tau * (1 - 1e-5), (g, t)
    assert nvis > n // 3


@pytest.mark.parametrize("seed,W,H,n", CASES)
def test_sorted_pairs_ranges_and_lpt_order(seed, W, H, n):
    sc, cam = _scene(seed, W, H, n)
    p = oracle.project(sc, cam)
    b = oracle.bin_sort(cam, p)
    ntx, nty = oracle.n_tiles(cam)
    # reference ordering: Python's sort over (tile, depth, id)
    pairs = []
    for g in np.nonzero(p.visible)[0]:
        for t in oracle.splat_tiles(cam, p.splat[g]):
            pairs.append((int(t), float(p.splat[g, 7]), int(g)))
    pairs.sort()
    ref_ids = np.array([g for _, _, g in pairs], np.int32)
    ref_tiles = np.array([t for t, _, _ in pairs], np.int64)
    np.testing.assert_array_equal(b.ids, ref_ids)
    counts = np.bincount(ref_tiles, minlength=ntx * nty)
    np.testing.assert_array_equal(b.counts, counts)
    ends = np.cumsum(counts)
    np.testing.assert_array_equal(b.ranges[:, 1], ends)
    np.testing.assert_array_equal(b.ranges[:, 0], ends - counts)
    lpt = sorted(range(ntx * nty), key=lambda t: (-counts[t], t))
    np.testing.assert_array_equal(b.lpt_order, lpt)
    assert b.n_pairs == int(p.tiles_touched.sum())


def test_tile_selection_matches_full_list():
    sc, cam = _scene(2, 150, 97, 140)
    p = oracle.project(sc, cam)
    full = oracle.bin_sort(cam, p)
    sel = np.zeros(len(full.counts), np.uint8)
    sel[[0, 3, 7, 20, 41]] = 1
    part = oracle.bin_sort(cam, p, sel)
    for t in np.nonzero(sel)[0]:
        s, e = full.ranges[t]
        np.testing.assert_array_equal(part.tile_ids(t), full.ids[s:e])
    np.testing.assert_array_equal(part.counts, full.counts)


def test_three_sigma_square_contains_emitted_tiles_when_tau_le_9():
    """With tau <= 9 (o <= e^4.5 / 255) the support ellipse lies inside the 3-sigma
    circle of the classic conservative bound, so every emitted tile meets that square."""
    sc, cam = _scene(1, 128, 128, 200)
    p = oracle.project(sc, cam)
    checked = 0
    for g in np.nonzero(p.visible & (p.splat[:, 6] <= 9.0))[0]:
        P = np.array([[p.splat[g, 8], p.splat[g, 9]], [p.splat[g, 9], p.splat[g, 10]]])
        r3 = 3.0 * np.sqrt(np.linalg.eigvalsh(P).max()) * (1 + 2.0 ** -8) + 2.0 ** -8 + 0.01
        for t in oracle.splat_tiles(cam, p.splat[g]):
            x0, x1, y0, y1 = D.tile_hull(cam, int(t))
            assert x0 <= p.splat[g, 0] + r3 and x1 >= p.splat[g, 0] - r3
            assert y0 <= p.splat[g, 1] + r3 and y1 >= p.splat[g, 1] - r3
            checked += 1
    assert checked > 50


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_every_fp32_hit_pixel_lies_in_an_emitted_tile(seed):
    """Completeness against the hit test itself (the fp32 round-to-nearest quadratic,
    emulated exactly), on huge and needle-like splats whose tips are ill-conditioned."""
    rng = np.random.default_rng(100 + seed)
    W, H, n = 300, 200, 60
    sc, cam = ss.random_scene(rng, n, W, H, sh_degree=0, log_scale=(-1.0, 1.2), depth=(1.0, 4.0))
    # a third of them needles: one long axis, two very short ones
    k = n // 3
    sc.scales[:k] = np.stack([rng.uniform(0.5, 3.0, k), np.full(k, 1e-3), np.full(k, 2e-3)],
                             1).astype(np.float32)
    p = oracle.project(sc, cam)
    ntx, _ = oracle.n_tiles(cam)
    ys, xs = np.mgrid[0:H, 0:W]
    px = xs.astype(np.float32) + np.float32(0.5)
    py = ys.astype(np.float32) + np.float32(0.5)
    tile_of = (ys // 16) * ntx + xs // 16
    checked = 0
    for g in np.nonzero(p.visible)[0]:
        r = p.splat[g]
        dx = px - np.float32(r[0])
        dy = py - np.float32(r[1])
        q = D.quad_f32(r[13], r[14], r[15], dx, dy)
        hit = q <= np.float32(r[6])
        need = set(np.unique(tile_of[hit]).tolist())
        have = set(oracle.splat_tiles(cam, r).tolist())
        assert need <= have, (g, sorted(need - have)[:5])
        checked += int(hit.sum())
    assert checked > 100000


def test_completeness_for_ground_splats_under_the_camera():
    """Flat Gaussians on a ground plane just below and ahead of the camera project to
    huge, thin ellipses centred far outside the image (the street workload has many);
    every pixel their fp32 hit test accepts must lie in an emitted tile."""
    rng = np.random.default_rng(7)
    n, W, H = 400, 320, 240
    means = np.stack([rng.uniform(-8, 8, n), np.full(n, 1.6), rng.uniform(0.21, 1.0, n)], 1)
    scales = np.stack([np.exp(rng.normal(0.0, 1.0, n)), np.full(n, 2e-3),
                       np.exp(rng.normal(0.0, 1.0, n))], 1)
    ax = rng.normal(0, 0.05, (n, 3))  # nearly horizontal discs
    quats = np.concatenate([np.ones((n, 1)), ax], 1)
    quats /= np.linalg.norm(quats, axis=1, keepdims=True)
    sc = ss.Scene(means.astype(np.float32), scales.astype(np.float32), quats.astype(np.float32),
                  rng.uniform(0.05, 0.99, n).astype(np.float32), np.zeros((n, 1, 3), np.float32), 0)
    cam = ss.pinhole(np.eye(4), 200.0, W, H)
    p = oracle.project(sc, cam)
    ntx, _ = oracle.n_tiles(cam)
    ys, xs = np.mgrid[0:H, 0:W]
    px = xs.astype(np.float32) + np.float32(0.5)
    py = ys.astype(np.float32) + np.float32(0.5)
    tile_of = (ys // 16) * ntx + xs // 16
    far = thin = 0
    for g in np.nonzero(p.visible)[0]:
        r = p.splat[g]
        P = np.array([[r[8], r[9]], [r[9], r[10]]])
        ev = np.linalg.eigvalsh(P)
        thin += ev[1] / ev[0] > 1e4
        far += abs(r[0]) > 3 * W or abs(r[1]) > 3 * H
        q = D.quad_f32(r[13], r[14], r[15], px - np.float32(r[0]), py - np.float32(r[1]))
        need = set(np.unique(tile_of[q <= np.float32(r[6])]).tolist())
        assert need <= set(oracle.splat_tiles(cam, r).tolist()), g
    assert thin > 50 and far > 200, (thin, far)


def test_equal_depths_are_listed_by_ascending_id():
    """Splats at exactly the same depth keep ascending Gaussian id within each tile: the id
    is the tie-break of the (tile, depth, id) order, which a stable depth sort of the
    id-ordered splats followed by a stable tile sort gives (Kopanas, Step 1 (d))."""
    rng = np.random.default_rng(7)
    sc, cam = ss.random_scene(rng, 300, 64, 48, sh_degree=0, log_scale=(-2.0, 0.3))
    # the identity camera makes each depth t_z equal to the mean's z: all exactly 3
    sc.means[:, 2] = np.float32(3.0)
    proj = oracle.project(sc, cam)
    assert np.all(proj.splat[proj.visible, 7] == 3.0)
    b = oracle.bin_sort(cam, proj, None)
    crowded = 0
    for t in range(len(b.counts)):
        s, e = b.ranges[t]
        ids = b.ids[s:e]
        assert np.all(np.diff(ids) > 0), t
        crowded += len(ids) >= 5
    assert crowded >= 10  # of the 12 tiles


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_every_fp32_hit_lies_in_an_emitted_tile_for_thin_splats(seed):
    """Completeness where the spans are least certain: long, thin, rotated splats (aspect
    about 100-400), whose boundary near the tips moves by about sqrt(u) r under fp32
    rounding.  Every pixel whose fp32 hit test (q <= tau, the renderer's own test) passes
    must lie in one of the splat's emitted tiles."""
    rng = np.random.default_rng(40 + seed)
    W, H, n = 320, 256, 60
    sc, cam = ss.random_scene(rng, n, W, H, sh_degree=0, log_scale=(-1.8, 0.3),
                              logit_std=1.0)
    thin = rng.uniform(100.0, 400.0, n).astype(np.float32)
    sc.scales[:, 1] = sc.scales[:, 0] / thin
    sc.scales[:, 2] = sc.scales[:, 0] / thin
    p = oracle.project(sc, cam)
    ntx = (W + 15) // 16
    ys, xs = np.mgrid[0:H, 0:W]
    px = xs.astype(np.float32) + np.float32(0.5)
    py = ys.astype(np.float32) + np.float32(0.5)
    tile_of = (ys // 16) * ntx + xs // 16
    checked = 0
    for g in range(n):
        rec = p.splat[g]
        if p.tiles_touched[g] == 0 and not (rec[6] > 0 and rec[13] > 0):
            continue
        dx = px - np.float32(rec[0])
        dy = py - np.float32(rec[1])
        q = D.quad_f32(rec[13], rec[14], rec[15], dx, dy)
        hit = q <= np.float32(rec[6])
        if not hit.any():
            continue
        tiles = set(oracle.splat_tiles(cam, rec).tolist())
        missing = set(np.unique(tile_of[hit]).tolist()) - tiles
        assert not missing, (g, sorted(missing)[:5])
        checked += 1
    assert checked > n // 3
