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

    for name in ("gs_project", "gs_bin_sort", "gs_rasterize_fwd", "gs_rasterize_bwd",
                 "gs_project_bwd"):
        assert callable(getattr(gs, name))


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
