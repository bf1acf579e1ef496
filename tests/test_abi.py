"""The C ABI library loads and exports every entry point include/gs.h declares; host-side
argument validation rejects bad calls before touching a device (no GPU needed)."""

import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gs.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gs_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from differentiable_gaussian_splatting_gb300 import build

    build.build()
    import differentiable_gaussian_splatting_gb300 as gs

    return gs.library()


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert {"gs_project", "gs_bin_sort", "gs_rasterize_fwd", "gs_rasterize_bwd",
            "gs_project_bwd"} <= set(names)
    for name in names:
        assert hasattr(lib, name), name


def test_python_binding_has_the_c_names():
    import differentiable_gaussian_splatting_gb300 as gs

    for name in _declared():
        assert callable(getattr(gs, name, None)), name
        assert name in gs.__all__, name
    assert gs.gs_num_tiles(1297, 840) == 82 * 53 and gs.gs_num_tiles(0, 5) == 0
    assert gs.gs_status_string(3) == gs.STATUS[3]


def test_host_queries(lib):
    import differentiable_gaussian_splatting_gb300 as gs

    assert lib.gs_num_tiles(1297, 840) == 82 * 53
    assert lib.gs_num_tiles(128, 128) == 64
    assert lib.gs_num_tiles(0, 5) == 0
    s = lib.gs_default_settings()
    assert (s.split_mode, s.h_max, s.policy_lambda) == (0, 256, 256.0)
    assert abs(s.policy_eps - 0.1) < 1e-7
    assert lib.gs_status_string(3) == b"pair list capacity exceeded"
    assert gs.gs_bin_sort_workspace_bytes(1000, 4000, 128, 128) > 4000 * 16
    assert gs.gs_bin_sort_workspace_bytes(-1, 10, 128, 128) == 0
    assert gs.gs_raster_workspace_bytes(64, 64, 1000) > 1000
    assert gs.gs_raster_workspace_bytes(64, 64, 0) == 0
    bad = gs.Settings(7, 0, 0, 256, 256.0, 0.05, 0.1)
    assert lib.gs_raster_workspace_bytes(64, 64, 1000, C.byref(bad)) == 0


def _cam(**kw):
    import differentiable_gaussian_splatting_gb300 as gs

    vm = (C.c_float * 16)(*[1, 0, 0, 0, 0, 1, 0, 0, 0, 0, 1, 0, 0, 0, 0, 1])
    c = gs.Camera(vm, 100.0, 100.0, 32.0, 32.0, 64, 64, 0.2)
    for k, v in kw.items():
        setattr(c, k, v)
    return c


@pytest.mark.parametrize("bad", [dict(width=0), dict(height=-3), dict(znear=0.0),
                                 dict(znear=float("nan")), dict(fx=float("inf"))])
def test_invalid_cameras_are_rejected_on_the_host(lib, bad):
    cam = _cam(**bad)
    fake = C.c_void_p(0x100000)  # never dereferenced: validation fails first
    st = lib.gs_project(C.byref(cam), 10, 0, *([fake] * 9), None)
    assert st == 1


def test_invalid_sizes_and_pointers_are_rejected_on_the_host(lib):
    cam = _cam()
    fake = C.c_void_p(0x100000)
    assert lib.gs_project(C.byref(cam), -1, 0, *([fake] * 9), None) == 1
    assert lib.gs_project(C.byref(cam), 10, 4, *([fake] * 9), None) == 1
    assert lib.gs_project(C.byref(cam), 10, 0, *([None] + [fake] * 8), None) == 1
    mis = C.c_void_p(0x100004)  # not 16-byte aligned
    assert lib.gs_project(C.byref(cam), 10, 0, *([mis] + [fake] * 8), None) == 1
    assert lib.gs_project(C.byref(cam), 0, 0, *([None] * 9), None) == 0  # empty: nothing to do
    # bin sort: zero capacity; workspace too small
    assert lib.gs_bin_sort(C.byref(cam), 10, fake, fake, fake, fake, 1 << 20, fake, 0, fake, fake,
                           None, None, None) == 1
    assert lib.gs_bin_sort(C.byref(cam), 10, fake, fake, fake, fake, 16, fake, 100, fake, fake,
                           None, None, None) == 5
    # bad settings
    import differentiable_gaussian_splatting_gb300 as gs

    for bad in (gs.Settings(2, 5, 1, 256, 256.0, 0.05, 0.1),    # k < 2
                gs.Settings(2, 300, 4, 256, 256.0, 0.05, 0.1),  # h > h_max
                gs.Settings(0, 0, 4, 0, 256.0, 0.05, 0.1),      # h_max < 1
                gs.Settings(0, 0, 4, 256, -1.0, 0.05, 0.1),     # lambda < 0
                gs.Settings(0, 0, 4, 256, 256.0, 0.05, 1.5)):   # eps >= 1
        assert lib.gs_rasterize_fwd(C.byref(cam), C.byref(bad), 10, fake, fake, 100, fake,
                                    fake, fake, 1 << 30, *([fake] * 4), None) == 1


def test_loss_arguments_are_checked_on_the_host(lib):
    import differentiable_gaussian_splatting_gb300 as gs

    fake = C.c_void_p(0x100000)
    mis = C.c_void_p(0x100004)
    ok = gs.LossSettings.default()
    ws = lib.gs_loss_workspace_bytes(100, 60)
    assert ws == 4 * 2 * 8  # one float2 per 32x32 tile: 4 x 2 tiles
    assert lib.gs_loss_workspace_bytes(0, 60) == 0

    def call(w=100, h=60, img=fake, tgt=fake, s=ok, d=C.c_void_p(0x200000), out=fake,
             wsp=fake, wsb=ws):
        return lib.gs_loss_l1_ssim(w, h, img, tgt, C.byref(s) if s is not None else None, d, out,
                                   wsp, wsb, None)

    assert call(w=0) == 1 and call(h=-3) == 1
    assert call(s=None) == 1
    for field, value in (("lambda_", -0.1), ("lambda_", 1.5), ("c1", 0.0), ("c2", -1.0),
                         ("sigma", 0.0), ("sigma", float("inf"))):
        bad = gs.LossSettings.default()
        setattr(bad, field, value)
        assert call(s=bad) == 1, field
    assert call(img=None) == 1 and call(out=mis) == 1
    # the gradient may not overlap either image
    assert call(d=C.c_void_p(0x100000 + 16)) == 1
    assert call(wsb=ws - 1) == 5  # workspace too small


def test_adam_arguments_are_checked_on_the_host(lib):
    import differentiable_gaussian_splatting_gb300 as gs

    cam = _cam()
    fake = C.c_void_p(0x100000)
    mom = gs.AdamMoments()
    for k in range(5):
        mom.m[k] = 0x100000
        mom.v[k] = 0x100000
    good = dict(lr_means=1e-4, lr_scales=5e-3, lr_quats=1e-3, lr_opacities=5e-2, lr_sh0=2.5e-3,
                lr_shN=1.25e-4, beta1=0.9, beta2=0.999, eps=1e-15, step=1)

    def call(s, moments=mom, n=10, act=None):
        return lib.gs_project_bwd_adam(C.byref(cam), n, 3, *([fake] * 8),
                                       C.byref(moments) if moments is not None else None,
                                       C.byref(gs.AdamSettings(**s)), act, None, None)

    for field, value in (("beta1", 1.0), ("beta2", -0.1), ("eps", 0.0), ("step", 0),
                         ("lr_sh0", -1.0), ("lr_means", float("nan"))):
        assert call({**good, field: value}) == 1, field
    assert call(good, moments=None) == 1
    assert call(good, act=C.c_void_p(0x100004)) == 1  # activated scales misaligned
    assert call(good, n=-1) == 1
    empty = gs.AdamMoments()
    assert call(good, moments=empty) == 1  # null moment pointers


def test_capacity_error_carries_the_pairs_needed():
    """A pair list too short for the view raises GSError status 3 naming the pairs needed,
    which the Rasterizer reads to re-allocate before it retries the sort."""
    import differentiable_gaussian_splatting_gb300 as gs

    with pytest.raises(gs.GSError) as e:
        gs._check("gs_bin_sort", 3, "; pairs needed: 1234567")
    assert e.value.status == 3
    assert gs.Rasterizer._needed(e.value) == 1234567
    gs._check("gs_bin_sort", 0)  # GS_OK raises nothing
