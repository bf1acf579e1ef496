"""GPU parity of the whole hot path, through the C ABI, against the CPU oracle.

Small cases run the oracle on every pixel and Gaussian; they span several tiles and
ragged image edges.  The full-size workloads run in the same launch configuration as
the benchmark and compare sampled tiles and Gaussians that the oracle computes one by
one (every tile of a sampled Gaussian is blended, so its gradient is complete): small
splats, the largest splats (longest per-quadrant reductions, most atomics), and members
of the heaviest tiles, which the auto policy splits into depth chunks on the 3M and 6M
scenes (their backward runs through the chunked state).  The loss weights are used as
they are: near-tie pixels are compared against the outcome the GPU took (gpu_util)."""

import numpy as np
import pytest

import oracle
import synthetic_scenes as ss
from gpu_util import (CHAIN_ROUNDINGS, TIER2_MAX_SHARE, TIER2_MAX_SHARE_LARGE, U,
                      assert_grads_tiered, check_binning, check_forward,
                      check_projection, grad2d_bounds, param_bounds, run_backward, run_forward)

pytestmark = pytest.mark.gpu


def _check_param_grads(sc, cam, proj, pg, r2, bound2d, gabs, rows=None, name="",
                       max_share=TIER2_MAX_SHARE):
    """End to end: GPU chain(GPU grad2d) vs oracle chain(oracle grad2d), held to the
    chain's magnitudes of the grad2d bound (gpu_util)."""
    rows = np.arange(sc.n) if rows is None else rows
    sub = sc.subset(rows)
    p = oracle.Projection(proj.splat[rows], proj.rgb[rows], proj.radii[rows],
                          proj.tiles_touched[rows])
    rp = oracle.project_bwd(sub, cam, p, r2[rows])
    pb, pm = param_bounds(sub, cam, p, bound2d[rows], gabs[rows])
    for k in ("means", "scales", "quats", "opacities", "sh"):
        assert_grads_tiered(pg[k][rows], getattr(rp, k), name + k, pb[k], getattr(pm, k),
                            max_share=max_share)


def _check_project_bwd_alone(sc, cam, proj, r2, name=""):
    """The chain rule by itself: the GPU's gs_project_bwd fed the oracle's grad2d, held to
    the chain's own roundings."""
    import torch

    import differentiable_gaussian_splatting_gb300 as gs
    from gpu_util import t

    n, K = sc.n, (sc.sh_degree + 1) ** 2
    outs = [torch.empty((n, 3), device="cuda"), torch.empty((n, 3), device="cuda"),
            torch.empty((n, 4), device="cuda"), torch.empty(n, device="cuda"),
            torch.empty((n, K, 3), device="cuda")]
    r32 = r2.astype(np.float32)
    gs.gs_project_bwd(gs.Camera.of(cam), n, sc.sh_degree, t(sc.means), t(sc.scales),
                      t(sc.quats), t(sc.opacities), t(sc.sh), t(proj.tiles_touched),
                      t(r32), None, *outs)
    torch.cuda.synchronize()
    rp = oracle.project_bwd(sc, cam, proj, r32.astype(np.float64))
    pm = oracle.project_bwd_magnitude(sc, cam, proj, np.abs(r32.astype(np.float64)))
    for k, o in zip(("means", "scales", "quats", "opacities", "sh"), outs):
        m = getattr(pm, k)
        assert_grads_tiered(o.cpu().numpy(), getattr(rp, k), name + "alone:" + k,
                            CHAIN_ROUNDINGS * U * m, m)


def _full_parity(sc, cam, w, v=None, settings=None, capacity=None, sh_bf16=False, name=""):
    g = run_forward(sc, cam, settings=settings, capacity=capacity, sh_bf16=sh_bf16)
    ref = oracle.render(sc, cam)
    check_projection(g, ref.proj, sc)
    check_binning(g, ref.binning)
    stop_last = check_forward(g, cam, ref.proj, ref.binning, ref.image, name=name + "forward")
    g2, touched, pg = run_backward(g, w, v)
    r, bound = grad2d_bounds(cam, ref.proj, ref.binning, w, v, stop_last)
    assert_grads_tiered(g2, r.grad2d, name + "grad2d", bound, r.gabs)
    _check_param_grads(sc, cam, ref.proj, pg, r.grad2d, bound, r.gabs, name=name)
    _check_project_bwd_alone(sc, cam, ref.proj, r.grad2d, name=name)
    return g, ref


def test_tiny_config1_full():
    sc, cam = ss.make_config(1)
    w = ss.loss_weights(1, cam.height, cam.width)
    _full_parity(sc, cam, w)


@pytest.mark.parametrize("seed,W,H,n,deg", [(0, 37, 53, 300, 0), (1, 150, 97, 900, 3),
                                            (2, 200, 120, 3000, 1), (3, 64, 40, 600, 2)])
def test_random_ragged_scenes_full(seed, W, H, n, deg):
    rng = np.random.default_rng(seed)
    sc, cam = ss.random_scene(rng, n, W, H, sh_degree=deg, log_scale=(-2.8, 0.8), logit_std=2.5)
    w = rng.standard_normal((H, W, 3))
    v = rng.standard_normal((H, W))
    _full_parity(sc, cam, w, v)


@pytest.mark.parametrize("W,H", [(1, 1), (1, 37), (45, 1), (16, 16), (17, 16), (16, 33),
                                 (1000, 3), (32768, 2), (3, 32768)])
def test_degenerate_image_shapes_full(W, H):
    # one pixel, one column, one row, exactly one tile, one tile plus a one-pixel
    # ragged column or row, a long strip of tiles, and strips at the largest image
    # side the calls accept (32768 pixels, 2048 tiles in one row or column); with
    # f = 60 the splats are several pixels wide, so the single pixels saturate and
    # stop early
    rng = np.random.default_rng(40 + W + H)
    sc, cam = ss.random_scene(rng, 200, W, H, f=60.0, sh_degree=1, log_scale=(-2.8, 0.8),
                              logit_std=2.5)
    w = rng.standard_normal((H, W, 3))
    v = rng.standard_normal((H, W))
    _full_parity(sc, cam, w, v)


def test_anisotropic_intrinsics_rotated_camera_full():
    # fx != fy and a principal point off the image centre, seen from a camera turned
    # and moved off the origin: a swapped focal length, principal-point coordinate or
    # view-matrix row in the projection, its Jacobian or its chain rule shows here (the
    # other scenes have fx = fy and the principal point at the centre)
    rng = np.random.default_rng(61)
    W, H = 120, 90
    sc, _ = ss.random_scene(rng, 800, W, H, f=100.0, sh_degree=3, log_scale=(-2.8, 0.7),
                            logit_std=2.0)
    V = ss.look_at(np.array([1.2, -0.7, -1.5]), np.array([0.0, 0.0, 4.0]))
    cam = ss.Camera(V, 115.0, 80.0, 0.42 * W, 0.61 * H, W, H, 0.2)
    w = rng.standard_normal((H, W, 3))
    v = rng.standard_normal((H, W))
    g, ref = _full_parity(sc, cam, w, v)
    assert ref.binning.n_pairs > 1000


def test_non_finite_parameters_are_culled_full():
    # NaN and infinite means, scales, quaternions and opacity, and a zero quaternion:
    # each such Gaussian is culled (no tiles, zero records and gradients) on both sides,
    # and the rest of the view renders and differentiates as without them
    rng = np.random.default_rng(71)
    W, H = 80, 60
    sc, cam = ss.random_scene(rng, 300, W, H, sh_degree=2, log_scale=(-2.8, 0.7),
                              logit_std=2.0)
    nan, inf = np.float32(np.nan), np.float32(np.inf)
    sc.means[0] = [nan, 0.0, 3.0]
    sc.means[1] = [inf, 0.0, 3.0]
    sc.scales[2] = [inf, 0.1, 0.1]
    sc.scales[3] = [0.1, nan, 0.1]
    sc.quats[4] = [nan, 0.0, 0.0, 0.0]
    sc.quats[5] = [0.0, 0.0, 0.0, 0.0]
    sc.opacities[6] = nan
    sc.means[7, 2] = inf
    w = rng.standard_normal((H, W, 3))
    g, ref = _full_parity(sc, cam, w)
    assert np.all(ref.proj.tiles_touched[:8] == 0)
    assert np.all(np.asarray(g.tiles_touched)[:8] == 0)
    assert np.isfinite(g.img).all() and ref.binning.n_pairs > 200


def test_cull_boundaries_full_parity():
    """The two cull decisions at their boundaries, in fp32 steps: view depths one
    step below, at and above the near plane (in front means strictly beyond it),
    and opacities around 1/255, where tau = 2 ln(255 o) changes sign (the oracle
    culls the two lower ones and keeps fp32(1/255) with tau about 1.2e-7), beside
    the smallest and the largest opacity below 1."""
    rng = np.random.default_rng(51)
    f32 = np.float32
    sc, cam = ss.random_scene(rng, 400, 96, 64, sh_degree=2, log_scale=(-2.8, 0.8),
                              logit_std=2.5)
    zn = f32(cam.znear)
    depths = [np.nextafter(zn, f32(0)), zn, np.nextafter(zn, f32(1)), zn * f32(1.001)]
    o1 = f32(1.0) / f32(255.0)
    below = np.nextafter(o1, f32(0))
    above = np.nextafter(o1, f32(1))
    opac = [np.nextafter(below, f32(0)), below, o1, above, np.nextafter(above, f32(1)),
            f32(1e-7), np.nextafter(f32(1), f32(0)), f32(0.5)]
    for i, z in enumerate(depths):
        sc.means[i] = [0.02 * (i - 1.5) * z, 0.01 * z, z]
        sc.scales[i] = [4e-4, 3e-4, 5e-4]
        sc.opacities[i] = 0.6
    for j, o in enumerate(opac):
        k = len(depths) + j
        sc.means[k] = [(j - 3.5) * 0.3, 0.2, 3.0]
        sc.scales[k] = [0.03, 0.02, 0.025]
        sc.opacities[k] = o
    w = rng.standard_normal((64, 96, 3))
    g, ref = _full_parity(sc, cam, w)
    tt = ref.proj.tiles_touched
    # the boundaries are where the oracle puts them, so the comparison is not vacuous
    assert list(tt[:2]) == [0, 0] and np.all(tt[2:4] > 0)
    k = len(depths)
    assert list(tt[k:k + 2]) == [0, 0] and np.all(tt[k + 2:k + 5] > 0)


def test_clamp_near_ties_full_parity():
    """Splats centred on pixel centres with opacities inside the fp32 band of the 0.99
    clamp, in front of ordinary splats: at those pixels the GPU's image must equal the
    oracle's with one of the two clamp decisions, and its gradients stay within the
    bound that spans both (galt)."""
    rng = np.random.default_rng(31)
    sc, cam = ss.random_scene(rng, 600, 64, 48, sh_degree=1, log_scale=(-2.6, 0.5),
                              logit_std=2.0)
    V = np.asarray(cam.viewmat, np.float64)
    R, tv = V[:3, :3], V[:3, 3]
    z = float(((R @ sc.means.T.astype(np.float64)).T[:, 2] + tv[2]).min()) - 0.3
    for i, d in enumerate([3e-6, -3e-6, 1e-6, -1e-6, 5e-6, -5e-6]):
        sc.opacities[i] = np.float32(0.99 + d)
        px, py = 8 + 9 * i + 0.5, 20.5
        t = np.array([(px - cam.cx) * z / cam.fx, (py - cam.cy) * z / cam.fy, z])
        sc.means[i] = (R.T @ (t - tv)).astype(np.float32)
    ref = oracle.render(sc, cam)
    assert np.count_nonzero(ref.image.flags & oracle.FLAG_CLAMP_TIE) >= 3
    w = rng.standard_normal((48, 64, 3))
    v = rng.standard_normal((48, 64))
    _full_parity(sc, cam, w, v, name="clamp ties:")


def test_forced_split_tiles_match_sequential():
    import differentiable_gaussian_splatting_gb300 as gs

    rng = np.random.default_rng(5)
    sc, cam = ss.random_scene(rng, 4000, 96, 64, sh_degree=1, log_scale=(-2.4, 0.6), logit_std=2.0)
    w = rng.standard_normal((64, 96, 3))
    for h, k in ((6, 4), (2, 16), (24, 2)):
        s = gs.gs_default_settings()
        s.split_mode, s.force_h, s.force_k = 2, h, k
        g, ref = _full_parity(sc, cam, w, settings=s, name=f"split{h}x{k}:")
        st = g.r.stats()
        assert (st["h"], st["k"]) == (h, k)
        # every 256-splat batch of every chunk is blended or skipped, and counted once
        counts = (g.ranges[:, 1] - g.ranges[:, 0])[g.lpt].astype(np.int64)
        want = 0
        for t in range(h):
            lo = [(int(counts[t]) * p) // k for p in range(k + 1)]
            want += sum(-(-(lo[p + 1] - lo[p]) // 256) for p in range(k))
        got = (st["batches_chunks"] + st["batches_skipped_on_flag"] +
               st["batches_skipped_done"])
        assert got == want, (st, want)
        assert 0 <= st["batches_discarded"] <= st["batches_chunks"]
        assert st["batches_tiles"] <= sum(-(-int(c) // 256) for c in counts[h:])


@pytest.mark.parametrize("h_max", [256, 4096, 65536])
def test_policy_matches_oracle_eq6(h_max):
    """(h, k) of the 8-block policy search equals the oracle's Eq. 6 on the same counts;
    h_max 4096 and 65536 (every one of the 8,160 tiles a candidate: 32,640 candidates,
    several per thread) exercise the search loop and its cross-block minimum."""
    import differentiable_gaussian_splatting_gb300 as gs

    sc, cam = ss.make_config(4, n=300_000)
    s = gs.gs_default_settings()
    s.h_max = h_max
    g = run_forward(sc, cam, settings=s)
    st = g.r.stats()
    counts = (g.ranges[:, 1] - g.ranges[:, 0])[g.lpt].astype(np.int64)
    h, k, _ = oracle.policy(counts, st["resident_ctas"], lam=float(np.float32(s.policy_lambda)),
                            beta=float(np.float32(s.policy_beta)),
                            eps=float(np.float32(s.policy_eps)), h_max=s.h_max)
    assert (st["h"], st["k"]) == (h, k)
    # the per-frame tile load the policy saw
    nz = counts[counts > 0]
    assert (st["n_max"], st["n_total"]) == (int(counts.max()), int(counts.sum()))
    assert (st["n_min_nonempty"], st["nonempty_tiles"]) == (int(nz.min()), len(nz))


def test_config2_full():
    sc, cam = ss.make_config(2)
    w = ss.loss_weights(2, cam.height, cam.width)
    _full_parity(sc, cam, w)


def _sampled_parity(c, n_gauss=48, n_large=12, n_rand_tiles=12, n_heavy=6, heavy_members=3,
                    per_heavy=8):
    """Full-size workload; the oracle computes all projections, all tile counts, the
    LPT order, and the pixels and gradients of sampled tiles / Gaussians: small splats
    (<= 4 tiles), the largest ones (top 0.1 % and 1 % of tiles touched) and members of the
    heaviest tiles."""
    sc, cam = ss.make_config(c)
    w = ss.loss_weights(c, cam.height, cam.width)
    g = run_forward(sc, cam)
    proj = oracle.project(sc, cam)
    check_projection(g, proj, sc)
    rng = np.random.default_rng(1000 + c)
    ntx, nty = oracle.n_tiles(cam)
    tt = proj.tiles_touched
    live = tt[tt > 0]
    small = np.nonzero((tt > 0) & (tt <= 4))[0]
    q99, q999 = np.quantile(live, 0.99), np.quantile(live, 0.999)
    top = np.nonzero(tt >= q999)[0]
    upper = np.nonzero((tt >= q99) & (tt < q999))[0]
    full_counts = oracle.bin_sort(cam, proj, np.zeros(ntx * nty, np.uint8))
    np.testing.assert_array_equal(g.lpt, full_counts.lpt_order)
    heavy = []
    for tl in full_counts.lpt_order[:heavy_members]:
        s_, e_ = g.ranges[tl]
        heavy.append(rng.choice(g.sorted_ids[s_:e_], min(per_heavy, e_ - s_), replace=False))
    sample = np.unique(np.concatenate([
        rng.choice(small, size=min(n_gauss, len(small)), replace=False),
        rng.choice(top, size=min(n_large, len(top)), replace=False),
        rng.choice(upper, size=min(n_large, len(upper)), replace=False), *heavy]))
    sel = np.zeros(ntx * nty, np.uint8)
    for gi in sample:
        sel[oracle.splat_tiles(cam, proj.splat[gi])] = 1
    sel[full_counts.lpt_order[:n_heavy]] = 1
    sel[rng.choice(ntx * nty, n_rand_tiles, replace=False)] = 1
    b = oracle.bin_sort(cam, proj, sel)
    check_binning(g, b)
    im = oracle.blend_parallel(cam, proj, b)
    name = f"c{c}:"
    stop_last = check_forward(g, cam, proj, b, im, name=name + "forward")
    g2, _, pg = run_backward(g, w)
    r, bound = grad2d_bounds(cam, proj, b, w, None, stop_last)
    # the sample is weighted toward the largest splats, whose long sums cancel most
    assert_grads_tiered(g2[sample], r.grad2d[sample], name + "grad2d", bound[sample],
                        r.gabs[sample], max_share=TIER2_MAX_SHARE_LARGE)
    _check_param_grads(sc, cam, proj, pg, r.grad2d, bound, r.gabs, rows=sample, name=name,
                       max_share=TIER2_MAX_SHARE_LARGE)
    culled = proj.tiles_touched == 0
    for k in ("means", "scales", "quats", "opacities", "sh"):
        assert np.all(pg[k][culled] == 0), k
    return g, sample, tt


@pytest.mark.parametrize("c", [3, 4, 5])
def test_full_size_sampled(c):
    g, sample, tt = _sampled_parity(c)
    # the sample holds splats of hundreds of tiles, and on the heavy-tailed scenes the
    # heaviest tiles are split into depth chunks by the auto policy
    assert tt[sample].max() >= 100
    st = g.r.stats()
    if c in (4, 5):
        assert st["h"] >= 3 and st["k"] >= 2, st


def test_edge_cases():
    # empty scene, all culled, identical depths, a huge splat, degenerate scales
    cam = ss.pinhole(np.eye(4), 60.0, 70, 50)
    rng = np.random.default_rng(9)
    sc, _ = ss.random_scene(rng, 200, 70, 50, sh_degree=0)
    sc.means[:60, 2] = 3.0                       # equal depths: id order decides
    sc.scales[60:64] = [[2.0, 2.0, 2.0]]         # covers the whole image
    sc.scales[64:70] = [[0.0, 0.1, 0.1]]         # degenerate
    sc.means[70:80, 2] = -1.0                    # behind the camera
    w = rng.standard_normal((50, 70, 3))
    _full_parity(sc, cam, w)
    empty = sc.subset(np.arange(0))
    g = run_forward(empty, cam)
    assert g.n_pairs == 0 and np.all(g.T == 1) and np.all(g.img == 0)
    culled = sc.subset(np.arange(70, 80))
    g = run_forward(culled, cam)
    assert g.n_pairs == 0 and np.all(g.T == 1)


def test_binning_on_a_large_tile_grid():
    # 275 x 263 = 72325 tiles: more than the tile-count scan keeps in registers, so
    # its looping path runs; many tiles are empty
    rng = np.random.default_rng(11)
    sc, cam = ss.random_scene(rng, 20_000, 4400, 4200, sh_degree=0, log_scale=(-5.0, 0.5))
    g = run_forward(sc, cam)
    proj = oracle.project(sc, cam)
    check_projection(g, proj, sc)
    check_binning(g, oracle.bin_sort(cam, proj))


# pair capacities from this size on take gs_bin_sort's two-stage radix sort
RADIX_CAPACITY = 8 << 20


@pytest.mark.parametrize("seed,W,H,n,deg", [(1, 150, 97, 900, 3), (2, 200, 120, 3000, 1)])
def test_radix_path_full_parity(seed, W, H, n, deg):
    rng = np.random.default_rng(seed)
    sc, cam = ss.random_scene(rng, n, W, H, sh_degree=deg, log_scale=(-2.8, 0.8), logit_std=2.5)
    w = rng.standard_normal((H, W, 3))
    _full_parity(sc, cam, w, capacity=RADIX_CAPACITY)


@pytest.mark.parametrize("capacity", [None, RADIX_CAPACITY], ids=["buckets", "radix"])
def test_equal_depths_full_parity(capacity):
    # every splat at exactly the same depth (identity camera, z = 3): only the id
    # tie-break orders each tile's list, and overlapping splats blend in id order
    rng = np.random.default_rng(9)
    sc, cam = ss.random_scene(rng, 800, 100, 70, sh_degree=1, log_scale=(-2.6, 0.6),
                              logit_std=2.0)
    sc.means[:, 2] = np.float32(3.0)
    w = rng.standard_normal((70, 100, 3))
    _full_parity(sc, cam, w, capacity=capacity)


@pytest.mark.parametrize("target", [1, 2, 3, 4, 5, 7, 4095, 4096, 4097, 4099])
def test_radix_path_small_and_ragged_pair_counts(target):
    """The radix path on pair lists of a few pairs and around one 4096-key block: the
    passes' partial blocks and the four-keys-per-thread tile ranges' tails."""
    rng = np.random.default_rng(21)
    sc, cam = ss.random_scene(rng, 6000, 256, 160, sh_degree=0, log_scale=(-5.5, 0.3))
    cum = np.cumsum(oracle.project(sc, cam).tiles_touched)
    sub = sc.subset(np.arange(int(np.searchsorted(cum, target)) + 1))
    g = run_forward(sub, cam, capacity=RADIX_CAPACITY)
    ref = oracle.project(sub, cam)
    check_projection(g, ref, sub)
    check_binning(g, oracle.bin_sort(cam, ref))
    assert g.n_pairs == target  # every prefix count is hit on this scene


def test_radix_and_bucket_paths_agree():
    sc, cam = ss.make_config(2)
    a = run_forward(sc, cam)
    b = run_forward(sc, cam, capacity=RADIX_CAPACITY)
    assert a.n_pairs == b.n_pairs
    for f in ("sorted_ids", "ranges", "lpt", "n_contrib", "last_idx"):
        np.testing.assert_array_equal(getattr(a, f), getattr(b, f), err_msg=f)
    np.testing.assert_array_equal(a.img, b.img)


def test_radix_path_capacity_overflow():
    import torch

    import differentiable_gaussian_splatting_gb300 as gs
    from gpu_util import t

    # the heavy-tailed 3M scene has about 30M pairs: more than the capacity
    sc, cam = ss.make_config(4)
    r = gs.Rasterizer(cam, sc.sh_degree, sc.n, capacity=RADIX_CAPACITY)
    gs.gs_project(r.cam, sc.n, sc.sh_degree, t(sc.means), t(sc.scales), t(sc.quats),
                  t(sc.opacities), t(sc.sh), r.splats, r.depths, r.radii, r.tiles_touched)
    with pytest.raises(gs.GSError):
        gs.gs_bin_sort(r.cam, sc.n, r.splats, r.depths, r.tiles_touched, r.bin_ws, r.sorted_ids,
                       r.capacity, r.tile_ranges, r.lpt_order)
    torch.cuda.synchronize()
    rg = r.tile_ranges.cpu().numpy()
    assert np.all(rg == 0), "every tile range is empty when the list does not fit"


def _bf16_values(a):
    """a rounded to bfloat16 (round to nearest even), as float32 values."""
    import torch

    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16).float().numpy()


@pytest.mark.parametrize("seed,W,H,n,deg", [(0, 37, 53, 300, 0), (5, 80, 60, 700, 1),
                                            (3, 64, 40, 600, 2), (1, 150, 97, 900, 3)])
def test_bf16_sh_full_parity(seed, W, H, n, deg):
    # SH stored as bfloat16: the oracle gets the same (widened) values, so the
    # tolerances are those of the fp32 path
    rng = np.random.default_rng(seed)
    sc, cam = ss.random_scene(rng, n, W, H, sh_degree=deg, log_scale=(-2.8, 0.8), logit_std=2.5)
    sc.sh = _bf16_values(sc.sh).astype(sc.sh.dtype)
    w = rng.standard_normal((H, W, 3))
    v = rng.standard_normal((H, W))
    _full_parity(sc, cam, w, v, sh_bf16=True)


def test_bf16_sh_config2_full():
    sc, cam = ss.make_config(2, n=20_000)
    sc.sh = _bf16_values(sc.sh).astype(sc.sh.dtype)
    w = ss.loss_weights(2, cam.height, cam.width)
    _full_parity(sc, cam, w, sh_bf16=True)


def test_repeatable_integer_outputs():
    sc, cam = ss.make_config(2, n=50_000)
    a = run_forward(sc, cam)
    b = run_forward(sc, cam)
    for f in ("tiles_touched", "radii", "sorted_ids", "ranges", "lpt", "n_contrib", "last_idx"):
        np.testing.assert_array_equal(getattr(a, f), getattr(b, f))
    np.testing.assert_array_equal(a.img, b.img)


def test_capacity_overflow_is_reported_and_recovered():
    import torch

    import differentiable_gaussian_splatting_gb300 as gs
    from gpu_util import t

    sc, cam = ss.make_config(1)
    r = gs.Rasterizer(cam, sc.sh_degree, sc.n, capacity=16)
    gs.gs_project(r.cam, sc.n, sc.sh_degree, t(sc.means), t(sc.scales), t(sc.quats),
                  t(sc.opacities), t(sc.sh), r.splats, r.depths, r.radii, r.tiles_touched)
    with pytest.raises(gs.GSError):
        gs.gs_bin_sort(r.cam, sc.n, r.splats, r.depths, r.tiles_touched, r.bin_ws, r.sorted_ids,
                       r.capacity, r.tile_ranges, r.lpt_order)
    r.forward(t(sc.means), t(sc.scales), t(sc.quats), t(sc.opacities), t(sc.sh))
    torch.cuda.synchronize()
    assert r.capacity >= r.n_pairs > 16
