"""gs_bin_sort_noalloc, the binning and sort on the library's fixed device scratch, against
gs_bin_sort on its caller-given workspace.  Both are integer work, so the outputs must agree
bit for bit, on consecutive calls of different sizes (the fixed scratch keeps the previous
call's contents).  This file sorts last so that it runs both after the other tests and,
alone, in a fresh process."""

import ctypes as C

import numpy as np
import pytest

import synthetic_scenes as ss

LIMIT_N, LIMIT_CAP = 1 << 16, 1 << 18
SCRATCH_BYTES = 7 << 20  # the library's fixed scratch array


def _cam(width=64, height=64):
    import differentiable_gaussian_splatting_gb300 as gs

    vm = (C.c_float * 16)(*[1, 0, 0, 0, 0, 1, 0, 0, 0, 0, 1, 0, 0, 0, 0, 1])
    return gs.Camera(vm, 100.0, 100.0, 32.0, 32.0, width, height, 0.2)


def test_sizes_beyond_the_fixed_scratch_are_rejected_on_the_host():
    from differentiable_gaussian_splatting_gb300 import build

    build.build()
    import differentiable_gaussian_splatting_gb300 as gs

    lib = gs.library()
    fake = C.c_void_p(0x100000)  # never dereferenced: the size check fails first

    def call(cam, n, cap):
        return lib.gs_bin_sort_noalloc(C.byref(cam), n, fake, fake, fake, fake, cap, fake, fake,
                                       None, None, None)

    assert call(_cam(), LIMIT_N + 1, 1000) == 5
    assert call(_cam(), 1000, LIMIT_CAP + 1) == 5
    assert call(_cam(2049, 2048), 1000, 1000) == 5   # 129 x 128 tiles > 16384
    assert call(_cam(), 1000, 0) == 1
    assert call(_cam(0, 64), 1000, 1000) == 1
    assert call(_cam(), -1, 1000) == 1
    # the camera is checked before the sizes: a width far beyond the image limit is an
    # invalid argument, not a size the scratch cannot hold
    assert call(_cam(2_000_000_000, 64), 1000, 1000) == 1


def test_every_limit_at_once_fits_the_fixed_scratch():
    import differentiable_gaussian_splatting_gb300 as gs

    # 2048 x 2048 is 16384 tiles, the tile limit; the layout grows with each size
    need = gs.gs_bin_sort_workspace_bytes(LIMIT_N, LIMIT_CAP, 2048, 2048)
    assert 0 < need <= SCRATCH_BYTES
    assert gs.gs_bin_sort_workspace_bytes(LIMIT_N, LIMIT_CAP, 16384, 256) <= SCRATCH_BYTES


def _project(sc, cam):
    import torch

    import differentiable_gaussian_splatting_gb300 as gs
    from gpu_util import t

    n = sc.n
    splats = torch.empty((n, gs.SPLAT_FLOATS), device="cuda")
    depths = torch.empty(n, device="cuda")
    radii = torch.empty((n, 2), dtype=torch.int32, device="cuda")
    tt = torch.empty(n, dtype=torch.int32, device="cuda")
    gs.gs_project(gs.Camera.of(cam), n, sc.sh_degree, t(sc.means), t(sc.scales), t(sc.quats),
                  t(sc.opacities), t(sc.sh), splats, depths, radii, tt)
    return splats, depths, tt


def _outputs(cam, capacity):
    import torch

    import differentiable_gaussian_splatting_gb300 as gs

    c = gs.Camera.of(cam)
    nt = gs.library().gs_num_tiles(c.width, c.height)
    return dict(ids=torch.full((capacity,), -7, dtype=torch.int32, device="cuda"),
                ranges=torch.full((nt, 2), -7, dtype=torch.int32, device="cuda"),
                lpt=torch.full((nt,), -7, dtype=torch.int32, device="cuda"),
                counts=torch.full((2,), -7, dtype=torch.int64, device="cuda"))


def _sort_with_workspace(cam, n, splats, depths, tt, capacity):
    import torch

    import differentiable_gaussian_splatting_gb300 as gs

    c = gs.Camera.of(cam)
    ws = torch.empty(gs.gs_bin_sort_workspace_bytes(n, capacity, c.width, c.height),
                     dtype=torch.uint8, device="cuda")
    o = _outputs(cam, capacity)
    I = gs.gs_bin_sort(c, n, splats, depths, tt, ws, o["ids"], capacity, o["ranges"], o["lpt"],
                       counts_device=o["counts"])
    return I, o


def _sort_noalloc(cam, n, splats, depths, tt, capacity):
    import differentiable_gaussian_splatting_gb300 as gs

    o = _outputs(cam, capacity)
    I = gs.gs_bin_sort_noalloc(gs.Camera.of(cam), n, splats, depths, tt, o["ids"], capacity,
                               o["ranges"], o["lpt"], counts_device=o["counts"])
    return I, o


def _same(a, b):
    I_a, oa = a
    I_b, ob = b
    assert I_a == I_b
    np.testing.assert_array_equal(oa["counts"].cpu().numpy(), ob["counts"].cpu().numpy())
    np.testing.assert_array_equal(oa["ids"][:I_a].cpu().numpy(), ob["ids"][:I_b].cpu().numpy())
    np.testing.assert_array_equal(oa["ranges"].cpu().numpy(), ob["ranges"].cpu().numpy())
    np.testing.assert_array_equal(oa["lpt"].cpu().numpy(), ob["lpt"].cpu().numpy())


@pytest.mark.gpu
def test_noalloc_sort_matches_gs_bin_sort_on_consecutive_calls():
    import torch

    # a large case near the limits (1297 x 840 image, 4346 tiles), then a small one, then
    # the large one again: each call must be unaffected by what the last left behind
    big_sc, big_cam = ss.make_config(3, n=60_000, seed=11)
    small_sc, small_cam = ss.make_config(1, n=2_000, seed=12)
    big = _project(big_sc, big_cam)
    small = _project(small_sc, small_cam)
    cases = [(big_cam, big_sc.n, big, LIMIT_CAP), (small_cam, small_sc.n, small, 20_000),
             (big_cam, big_sc.n, big, LIMIT_CAP)]
    for cam, n, (splats, depths, tt), cap in cases:
        want = _sort_with_workspace(cam, n, splats, depths, tt, cap)
        got = _sort_noalloc(cam, n, splats, depths, tt, cap)
        torch.cuda.synchronize()
        assert 0 < got[0] <= cap
        _same(want, got)


@pytest.mark.gpu
def test_noalloc_sort_with_every_limit_at_its_maximum():
    import torch

    # 65536 Gaussians, a 262144-pair capacity and 16384 tiles in one call (about 161k
    # pairs), twice in a row
    rng = np.random.default_rng(14)
    sc, cam = ss.random_scene(rng, LIMIT_N, 2048, 2048, sh_degree=0, log_scale=(-6.0, 0.5))
    splats, depths, tt = _project(sc, cam)
    for _ in range(2):
        want = _sort_with_workspace(cam, sc.n, splats, depths, tt, LIMIT_CAP)
        got = _sort_noalloc(cam, sc.n, splats, depths, tt, LIMIT_CAP)
        torch.cuda.synchronize()
        assert 100_000 < got[0] <= LIMIT_CAP
        _same(want, got)


@pytest.mark.gpu
def test_noalloc_sort_reports_capacity_and_empty_scenes():
    import torch

    import differentiable_gaussian_splatting_gb300 as gs

    sc, cam = ss.make_config(1, n=2_000, seed=13)
    splats, depths, tt = _project(sc, cam)
    I, _ = _sort_with_workspace(cam, sc.n, splats, depths, tt, LIMIT_CAP)
    with pytest.raises(gs.GSError) as e:
        _sort_noalloc(cam, sc.n, splats, depths, tt, I - 1)
    assert e.value.status == 3
    # no Gaussians: every tile range is empty
    got = _sort_noalloc(cam, 0, None, None, None, 16)
    want = _sort_with_workspace(cam, 0, None, None, None, 16)
    torch.cuda.synchronize()
    assert got[0] == 0
    _same(want, got)
