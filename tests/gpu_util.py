"""Helpers for the GPU parity tests: run the C-ABI path on the device and compare it with
the CPU oracle.  Tolerances: bit-exact integers; RGB and final
transmittance within 1e-5 relative / 1e-6 absolute; gradients within 1e-4 relative /
1e-6 absolute, relative to the magnitude of what each gradient sums (the oracle's sum of
the absolute values of every product and addend; it equals |gradient| when nothing
cancels, and a floating-point sum's error is bounded in proportion to it).  Pixels whose
stop decision the oracle flags as a fp32 near-tie are excluded from the forward comparison
and have dL/dC = 0 for the backward."""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

import oracle

RGB_RTOL, RGB_ATOL = 1e-5, 1e-6
GRAD_RTOL, GRAD_ATOL = 1e-4, 1e-6


def t(a, dev="cuda"):
    import torch

    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


@dataclass
class GpuRun:
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
    return GpuRun(r, r.splats.cpu().numpy(), r.depths.cpu().numpy(), r.radii.cpu().numpy(),
                  r.tiles_touched.cpu().numpy(), I, r.sorted_ids[:I].cpu().numpy(),
                  r.tile_ranges.cpu().numpy(), r.lpt_order.cpu().numpy(), r.image.cpu().numpy(),
                  r.t_final.cpu().numpy(), r.n_contrib.cpu().numpy(), r.last_idx.cpu().numpy())


def run_backward(g: GpuRun, w, v=None):
    import torch

    grads = g.r.backward(t(w.astype(np.float32)), None if v is None else t(v.astype(np.float32)))
    torch.cuda.synchronize()
    return (g.r.grad2d.cpu().numpy(), g.r.touched.cpu().numpy(),
            {k: getattr(grads, k).cpu().numpy() for k in ("means", "scales", "quats", "opacities", "sh")})


def check_projection(g: GpuRun, ref: oracle.Projection, sc, rows=None):
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


def check_binning(g: GpuRun, ref: oracle.Binning, tiles=None):
    assert g.n_pairs == ref.n_pairs
    np.testing.assert_array_equal(g.ranges[:, 0], ref.ranges[:, 0])
    np.testing.assert_array_equal(g.ranges[:, 1], ref.ranges[:, 1])
    np.testing.assert_array_equal(g.lpt, ref.lpt_order)
    tiles = np.nonzero(ref.sel)[0] if ref.sel is not None else range(len(ref.counts))
    for tt in tiles:
        s, e = g.ranges[tt]
        np.testing.assert_array_equal(g.sorted_ids[s:e], ref.tile_ids(tt), err_msg=f"tile {tt}")


def check_forward(g: GpuRun, im: oracle.Image):
    """Returns the mask of compared pixels."""
    ok = im.tile_mask & ((im.flags & oracle.FLAG_STOP_TIE) == 0)
    np.testing.assert_allclose(g.img[ok], im.img[ok], rtol=RGB_RTOL, atol=RGB_ATOL)
    np.testing.assert_allclose(g.T[ok], im.T[ok], rtol=RGB_RTOL, atol=RGB_ATOL)
    bad = np.nonzero(g.n_contrib[ok] != im.n_contrib[ok])[0]
    assert len(bad) == 0, f"n_contrib differs at {len(bad)} pixels"
    np.testing.assert_array_equal(g.last_idx[ok], im.last_idx[ok])
    return ok


def masked_weights(w, im: oracle.Image):
    """dL/dC with the oracle's near-tie pixels zeroed (both decisions are then valid)."""
    return (w * (im.flags == 0)[..., None]).astype(np.float32)


def assert_grads_close(gpu, ref, name, mag=None, rtol=GRAD_RTOL, atol=GRAD_ATOL):
    """|gpu - ref| <= atol + rtol * magnitude, the magnitude being the oracle's magnitude of
    the summed terms (>= |ref|; equal to it when nothing cancels), or |ref| if not given."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    scale = np.abs(ref) if mag is None else np.maximum(np.asarray(mag, np.float64), np.abs(ref))
    err = np.abs(gpu - ref)
    lim = atol + rtol * scale
    bad = err > lim
    if bad.any():
        i = np.argmax(err / lim)
        raise AssertionError(f"{name}: {bad.sum()} / {bad.size} outside tolerance; worst "
                             f"gpu={gpu.flat[i]:.9g} ref={ref.flat[i]:.9g} magnitude "
                             f"{scale.flat[i]:.4g} (|err|/tol {(err / lim).flat[i]:.3g})")
    return float((err / np.maximum(scale, 1e-30)).max()) if err.size else 0.0
