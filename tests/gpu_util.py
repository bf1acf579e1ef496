"""Helpers for the GPU parity tests: run the C-ABI path on the device and compare it with
the CPU oracle.

Tolerances (bit-exact integers; RGB and final transmittance within 1e-5 relative / 1e-6
absolute; gradients within 1e-4 relative / 1e-6 absolute):
* Forward: every pixel is compared.  Where the oracle flags the 1e-4 stop as a fp32
  near-tie, the oracle replays the stop the GPU took (its last_idx) and must admit it as
  an outcome of the stop rule within the fp32 band; the GPU then equals that outcome.
  Where an alpha lies within the band of the 0.99 clamp, the GPU must equal the oracle's
  rendering with either clamp decision.
* Gradients: |gpu - ref| <= 1e-6 + 1e-4 |ref| for every element, except elements whose
  derived fp32 error bound exceeds 1e-4 |ref| (cancellation, or an alpha error amplified
  by 1 / (1 - alpha) behind near-opaque splats).  Those are held to that bound:
    grad2d:  gamma_n gabs + grho + galt,  n = 6 + 4 tiles_touched (the warp's two rows
             and five shuffle levels, then one atomic per 8 x 8 quadrant of every tile),
             gamma_n = n u / (1 - n u), u = 2^-24; gabs, grho, galt from the oracle
             (oracle.blend_bwd_bounds);
    the 59 parameter gradients:  the chain rule's magnitudes (oracle.project_bwd_magnitude)
             of that grad2d bound, plus 64 u times those of gabs (the chain's own roundings).
  Every check counts the elements that pass only under the derived bound and asserts a
  ceiling on their share, and records the worst err / |ref|, err / magnitude and
  err / bound (printed in the session summary)."""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

import oracle

RGB_RTOL, RGB_ATOL = 1e-5, 1e-6
GRAD_RTOL, GRAD_ATOL = 1e-4, 1e-6
U = 2.0 ** -24
CHAIN_ROUNDINGS = 64          # the chain rule's own roundings, in units of u
TIER2_MAX_SHARE = 0.02        # elements passing only under the derived bound (whole scenes)
TIER2_MAX_SHARE_LARGE = 0.10  # the same in samples weighted toward the largest splats
STOP_TIE_MAX_SHARE = 0.01     # pixels whose stop the oracle flags as a fp32 near-tie
STATS: list = []              # per check: counts and worst ratios (session summary)


def t(a, dev="cuda"):
    import torch

    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


@dataclass
class GpuResult:
    r: object                # the Rasterizer
    splats: np.ndarray
    depths: np.ndarray
    radii: np.ndarray
    tiles_touched: np.ndarray
    n_pairs: int
    sorted_ids: np.ndarray
    ranges: np.ndarray
    lpt: np.ndarray
    img: np.ndarray
    T: np.ndarray
    n_contrib: np.ndarray
    last_idx: np.ndarray


def run_forward(sc, cam, settings=None, capacity=None, sh_bf16=False):
    import torch

    import differentiable_gaussian_splatting_gb300 as gs

    r = gs.Rasterizer(cam, sc.sh_degree, sc.n, capacity=capacity, settings=settings)
    sh = t(sc.sh)
    if sh_bf16:
        sh = sh.to(torch.bfloat16)  # the scene's SH must be bfloat16 values already
        assert torch.equal(sh.float(), t(sc.sh).float())
    r.forward(t(sc.means), t(sc.scales), t(sc.quats), t(sc.opacities), sh)
    torch.cuda.synchronize()
    I = r.n_pairs
    return GpuResult(r, r.splats.cpu().numpy(), r.depths.cpu().numpy(), r.radii.cpu().numpy(),
                  r.tiles_touched.cpu().numpy(), I, r.sorted_ids[:I].cpu().numpy(),
                  r.tile_ranges.cpu().numpy(), r.lpt_order.cpu().numpy(), r.image.cpu().numpy(),
                  r.t_final.cpu().numpy(), r.n_contrib.cpu().numpy(), r.last_idx.cpu().numpy())


def run_backward(g: GpuResult, w, v=None):
    import torch

    grads = g.r.backward(t(w.astype(np.float32)), None if v is None else t(v.astype(np.float32)))
    torch.cuda.synchronize()
    return (g.r.grad2d.cpu().numpy(), g.r.touched.cpu().numpy(),
            {k: getattr(grads, k).cpu().numpy() for k in ("means", "scales", "quats", "opacities", "sh")})


def check_projection(g: GpuResult, ref: oracle.Projection, sc, rows=None):
    """Integer outputs and the decision chain bit-exact; colour within tolerance."""
    rows = np.arange(sc.n) if rows is None else rows
    np.testing.assert_array_equal(g.tiles_touched[rows], ref.tiles_touched[rows])
    np.testing.assert_array_equal(g.radii[rows], ref.radii[rows])
    vis = rows[ref.tiles_touched[rows] > 0]
    gs_ = g.splats[vis]
    rs = ref.splat[vis].astype(np.float32)
    # record: mux, muy, l11, l12 | l22, tau, log2 o, rx | r, g, b, ry
    for gi, ri, name in ((0, 0, "mux"), (1, 1, "muy"), (2, 13, "l11"), (3, 14, "l12"),
                         (4, 15, "l22"), (5, 6, "tau"), (7, 11, "rx"), (11, 12, "ry")):
        bad = np.nonzero(gs_[:, gi] != rs[:, ri])[0]
        assert len(bad) == 0, f"{name} differs at {len(bad)} Gaussians, e.g. {vis[bad[:5]]}"
    np.testing.assert_array_equal(g.depths[vis], rs[:, 7])
    np.testing.assert_allclose(gs_[:, 6], np.log2(ref.splat[vis, 5]), rtol=0, atol=2e-6)
    np.testing.assert_allclose(gs_[:, 8:11], ref.rgb[vis], rtol=RGB_RTOL, atol=RGB_ATOL)
    culled = rows[ref.tiles_touched[rows] == 0]
    assert np.all(g.splats[culled] == 0)


def check_binning(g: GpuResult, ref: oracle.Binning, tiles=None):
    assert g.n_pairs == ref.n_pairs
    np.testing.assert_array_equal(g.ranges[:, 0], ref.ranges[:, 0])
    np.testing.assert_array_equal(g.ranges[:, 1], ref.ranges[:, 1])
    np.testing.assert_array_equal(g.lpt, ref.lpt_order)
    tiles = np.nonzero(ref.sel)[0] if ref.sel is not None else range(len(ref.counts))
    for tt in tiles:
        s, e = g.ranges[tt]
        np.testing.assert_array_equal(g.sorted_ids[s:e], ref.tile_ids(tt), err_msg=f"tile {tt}")


def check_forward(g: GpuResult, cam, proj, b, im: oracle.Image, name="forward"):
    """Every computed pixel against the oracle: at the oracle's stop near-ties, the outcome
    the GPU took (its last_idx), which the oracle must admit; at clamp near-ties, either
    clamp decision.  Returns stop_last for the backward: the GPU's last_idx at the
    near-ties, oracle.RULE elsewhere."""
    m = im.tile_mask
    tie = ((im.flags & oracle.FLAG_STOP_TIE) != 0) & m
    clamp = ((im.flags & oracle.FLAG_CLAMP_TIE) != 0) & m
    stop_last = np.where(tie, g.last_idx, oracle.RULE).astype(np.int32)
    fw = oracle.blend_parallel(cam, proj, b, stop_last=stop_last)
    bad = np.count_nonzero((fw.flags & oracle.FLAG_NOT_ADMISSIBLE) != 0)
    assert bad == 0, f"{name}: the GPU's stop is not an admissible outcome at {bad} pixels"
    other = int(np.count_nonzero(tie & (g.last_idx != im.last_idx)))
    np.testing.assert_array_equal(g.n_contrib[m], fw.n_contrib[m])
    np.testing.assert_array_equal(g.last_idx[m], fw.last_idx[m])

    def close(a, ref):
        return np.abs(a - ref) <= RGB_ATOL + RGB_RTOL * np.abs(ref)

    ok_img = np.all(close(g.img, fw.img), axis=2) & close(g.T, fw.T)
    if clamp.any():
        fl = oracle.blend_parallel(cam, proj, b, stop_last=stop_last, clamp_flip=True)
        ok_img |= clamp & np.all(close(g.img, fl.img), axis=2) & close(g.T, fl.T)
    nbad = int(np.count_nonzero(m & ~ok_img))
    assert nbad == 0, f"{name}: RGB / T outside tolerance at {nbad} pixels"
    n_pix = int(m.sum())
    STATS.append(dict(check=name, kind="pixels", n=n_pix, stop_ties=int(tie.sum()),
                      other_stop=other, clamp_ties=int(clamp.sum())))
    assert tie.sum() <= STOP_TIE_MAX_SHARE * n_pix, (name, int(tie.sum()), n_pix)
    return stop_last


def grad2d_bounds(cam, proj, b, w, v=None, stop_last=None):
    """The oracle's grad2d at the GPU's stop outcomes, and each element's derived fp32
    error bound gamma_n gabs + grho + galt (module docstring)."""
    r = oracle.blend_bwd_parallel(cam, proj, b, w, v, stop_last=stop_last)
    n = 6.0 + 4.0 * proj.tiles_touched.astype(np.float64)[:, None]
    bound = n * U / (1.0 - n * U) * r.gabs + r.grho + r.galt
    return r, bound


def param_bounds(scene, cam, proj, bound2d, gabs):
    """Derived error bounds of the 59 parameter gradients (module docstring)."""
    pb = oracle.project_bwd_magnitude(scene, cam, proj, bound2d)
    pm = oracle.project_bwd_magnitude(scene, cam, proj, gabs)
    return {k: getattr(pb, k) + CHAIN_ROUNDINGS * U * getattr(pm, k)
            for k in ("means", "scales", "quats", "opacities", "sh")}, pm


def assert_grads_tiered(gpu, ref, name, bound, mag=None, rtol=GRAD_RTOL, atol=GRAD_ATOL,
                        max_share=TIER2_MAX_SHARE):
    """|gpu - ref| <= atol + max(rtol |ref|, bound) element by element; the elements that
    pass only under the bound (the second tier) may be at most max_share of them.  The
    worst err / magnitude is taken over the elements whose error exceeds atol, the worst
    err / |ref| over the second tier with |ref| floored at atol."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    bound = np.broadcast_to(np.asarray(bound, np.float64), ref.shape)
    err = np.abs(gpu - ref)
    tier1 = err <= atol + rtol * np.abs(ref)
    lim = atol + np.maximum(rtol * np.abs(ref), bound)
    bad = err > lim
    if bad.any():
        i = np.argmax(err / lim)
        raise AssertionError(f"{name}: {bad.sum()} / {bad.size} outside tolerance; worst "
                             f"gpu={gpu.flat[i]:.9g} ref={ref.flat[i]:.9g} bound "
                             f"{bound.flat[i]:.4g} (|err| / tolerance {(err / lim).flat[i]:.3g})")
    t2 = ~tier1
    st = dict(check=name, kind="elements", n=int(err.size), tier2=int(t2.sum()),
              worst_rel=float((err / np.maximum(np.abs(ref), atol))[t2].max()) if t2.any() else 0.0,
              worst_err_over_bound=float((err / np.maximum(bound, 1e-300))[t2].max()) if t2.any()
              else 0.0)
    if mag is not None:
        m = np.broadcast_to(np.asarray(mag, np.float64), ref.shape)
        live = (m > 0) & (err > atol)
        st["worst_err_over_mag"] = float((err[live] / m[live]).max()) if live.any() else 0.0
    STATS.append(st)
    assert st["tier2"] <= max_share * err.size, st
    return st
