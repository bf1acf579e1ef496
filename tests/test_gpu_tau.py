"""The opacity threshold tau = 2 ln(255 o) of gs_project, over millions of opacities: it
must be the fp32 rounding of the value in double precision (the kernel computes it in
float-float and falls back to double only when the rounding is undecided), and
Gaussians with 255 o <= 1 must be culled."""

import ctypes as C

import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def _project_opacities(o):
    import torch

    import differentiable_gaussian_splatting_gb300 as gs

    n = o.size
    # every Gaussian in front of the camera, projected onto the pixel centre (64.5, 64.5),
    # so that any tau > 0 hits that pixel and the Gaussian stays visible
    vm = (C.c_float * 16)(*[1, 0, 0, 0, 0, 1, 0, 0, 0, 0, 1, 0, 0, 0, 0, 1])
    cam = gs.Camera(vm, 100.0, 100.0, 64.5, 64.5, 129, 129, 0.2)
    dev = "cuda"
    means = torch.zeros((n, 3), device=dev)
    means[:, 2] = 4.0
    scales = torch.full((n, 3), 0.01, device=dev)
    quats = torch.zeros((n, 4), device=dev)
    quats[:, 0] = 1.0
    opac = torch.from_numpy(o).to(dev)
    sh = torch.zeros((n, 1, 3), device=dev)
    splats = torch.empty((n, gs.SPLAT_FLOATS), device=dev)
    depths = torch.empty(n, device=dev)
    radii = torch.empty((n, 2), dtype=torch.int32, device=dev)
    tt = torch.empty(n, dtype=torch.int32, device=dev)
    gs.gs_project(cam, n, 0, means, scales, quats, opac, sh, splats, depths, radii, tt)
    torch.cuda.synchronize()
    return splats[:, 5].cpu().numpy(), tt.cpu().numpy()


def _reference(o):
    x = 255.0 * o.astype(np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        d = 2.0 * np.log(x)
    return d, x > 1.0


def test_tau_is_the_fp32_rounding_of_the_double_value():
    rng = np.random.default_rng(7)
    lo = np.float32(1.0 / 255.0)
    o = np.concatenate([
        rng.uniform(lo, 1.0, 2_000_000).astype(np.float32),
        # just above the cut-off 1/255, where tau is tiny
        (lo * (1.0 + rng.uniform(0.0, 1e-3, 200_000))).astype(np.float32),
        # the floats adjacent to 1/255 and to 1, and powers of two
        np.nextafter(lo, np.float32(0), dtype=np.float32) * np.ones(1, np.float32),
        lo * np.ones(1, np.float32), np.nextafter(lo, np.float32(1), dtype=np.float32) * np.ones(1, np.float32),
        np.float32([1.0, np.nextafter(np.float32(1), np.float32(0)), 0.5, 0.25, 0.125, 2 * lo, 4 * lo]),
    ])
    tau, tt = _project_opacities(o)
    d, positive = _reference(o)
    # culling: tau > 0 exactly when 255 o > 1
    np.testing.assert_array_equal(tt > 0, positive)
    vis = positive
    want = d[vis].astype(np.float32)
    got = tau[vis]
    bad = np.nonzero(got != want)[0]
    # a mismatch is admissible only where the double value lies within a few double ulps
    # of an fp32 rounding midpoint (double rounding of the reference itself)
    for b in bad:
        v = d[vis][b]
        f = np.float32(v)
        up = np.nextafter(f, np.float32(np.inf))
        dn = np.nextafter(f, np.float32(-np.inf))
        mid = min(abs(v - (float(f) + float(up)) / 2), abs(v - (float(f) + float(dn)) / 2))
        assert mid <= 8 * np.spacing(v), (o[vis][b], got[b], want[b])
    assert len(bad) <= 2
