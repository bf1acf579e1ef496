"""Differentiable 3D Gaussian splatting rasterizer for NVIDIA GB300 (sm_103a).

Thin Python binding of the C ABI in ``include/gs.h`` (library ``libgs.so``).
The five calls of the hot path keep their C names:

    gs_project, gs_bin_sort, gs_rasterize_fwd, gs_rasterize_bwd, gs_project_bwd

Each takes torch CUDA tensors (or raw device addresses), checks shapes and
dtypes, and passes plain pointers to the library; every step of the path runs
in the library's CUDA kernels.  PyTorch only provides device memory and
streams.  There is no CPU fallback: if ``libgs.so`` is missing or no CUDA
device is present, the calls raise.

``Rasterizer`` is a convenience that allocates the outputs and workspaces of
one view and runs the five calls in order.
"""

from __future__ import annotations

import ctypes as C
import os
import threading
from dataclasses import dataclass

from . import build as _build

__all__ = [
    "gs_project", "gs_bin_sort", "gs_rasterize_fwd", "gs_rasterize_bwd", "gs_project_bwd",
    "gs_project_sh16", "gs_project_bwd_sh16", "gs_project_bwd_adam", "AdamSettings",
    "gs_loss_l1_ssim", "gs_loss_workspace_bytes", "LossSettings",
    "gs_bin_sort_workspace_bytes", "gs_raster_workspace_bytes", "gs_bin_sort_noalloc",
    "gs_raster_stats", "gs_default_settings", "gs_status_string", "gs_num_tiles",
    "Camera", "Settings", "Rasterizer", "library",
    "GSError", "TILE", "GRAD2D", "SPLAT_FLOATS",
]

TILE = 16
GRAD2D = 9
SPLAT_FLOATS = 12
STATUS = {0: "ok", 1: "invalid argument", 2: "CUDA error", 3: "pair list capacity exceeded",
          4: "device wait timed out", 5: "workspace too small"}


class GSError(RuntimeError):
    def __init__(self, fn: str, status: int, extra: str = ""):
        self.status = status
        super().__init__(f"{fn}: {STATUS.get(status, status)} ({status}){extra}")


class Camera(C.Structure):
    """gs_camera: row-major 4x4 world->camera matrix, intrinsics, image size, near plane."""
    _fields_ = [("viewmat", C.c_float * 16), ("fx", C.c_float), ("fy", C.c_float),
                ("cx", C.c_float), ("cy", C.c_float), ("width", C.c_int32),
                ("height", C.c_int32), ("znear", C.c_float)]

    @classmethod
    def of(cls, cam) -> "Camera":
        """From any object with viewmat, fx, fy, cx, cy, width, height, znear."""
        if isinstance(cam, cls):
            return cam
        vm = [float(v) for v in _flat16(cam.viewmat)]
        return cls((C.c_float * 16)(*vm), float(cam.fx), float(cam.fy), float(cam.cx),
                   float(cam.cy), int(cam.width), int(cam.height), float(getattr(cam, "znear", 0.2)))


def _flat16(vm):
    try:
        import numpy as np
        return np.asarray(vm, dtype=np.float64).reshape(16).tolist()
    except ImportError:  # pragma: no cover
        return [x for row in vm for x in row]


class Settings(C.Structure):
    """gs_settings: scheduling of the blending kernels (never changes results)."""
    _fields_ = [("split_mode", C.c_int32), ("force_h", C.c_int32), ("force_k", C.c_int32),
                ("h_max", C.c_int32), ("policy_lambda", C.c_float), ("policy_beta", C.c_float),
                ("policy_eps", C.c_float)]


class AdamSettings(C.Structure):
    """gs_adam_settings: learning rates per parameter group, Adam's betas and eps, step t."""
    _fields_ = [("lr_means", C.c_float), ("lr_scales", C.c_float), ("lr_quats", C.c_float),
                ("lr_opacities", C.c_float), ("lr_sh0", C.c_float), ("lr_shN", C.c_float),
                ("beta1", C.c_float), ("beta2", C.c_float), ("eps", C.c_float),
                ("step", C.c_int32)]


class AdamMoments(C.Structure):
    """gs_adam_moments: device pointers of the first and second moments, one per
    parameter (means, log-scales, quaternions, opacity logits, SH)."""
    _fields_ = [("m", C.c_void_p * 5), ("v", C.c_void_p * 5)]


class LossSettings(C.Structure):
    """gs_loss_settings: weight of the SSIM term, the SSIM constants, the window's sigma."""
    _fields_ = [("lambda_", C.c_float), ("c1", C.c_float), ("c2", C.c_float),
                ("sigma", C.c_float)]

    @classmethod
    def default(cls) -> "LossSettings":
        return cls(0.2, 0.01 ** 2, 0.03 ** 2, 1.5)


_lib = None
_lib_lock = threading.Lock()
_P = C.c_void_p
_I64 = C.c_int64


def library() -> C.CDLL:
    """Load libgs.so (building it first when the sources are newer)."""
    global _lib
    with _lib_lock:
        if _lib is None:
            path = _build.LIB
            if not _build.up_to_date():
                _build.build()
            if not os.path.exists(path):
                raise RuntimeError("libgs.so is not built; run differentiable_gaussian_splatting_gb300.build")
            lib = C.CDLL(path)
            _declare(lib)
            _lib = lib
        return _lib


def _declare(lib: C.CDLL) -> None:
    st = C.c_int
    lib.gs_default_settings.restype = Settings
    lib.gs_status_string.restype = C.c_char_p
    lib.gs_status_string.argtypes = [st]
    lib.gs_num_tiles.restype = _I64
    lib.gs_num_tiles.argtypes = [C.c_int32, C.c_int32]
    lib.gs_project.restype = st
    lib.gs_project.argtypes = [C.POINTER(Camera), _I64, C.c_int32] + [_P] * 9 + [_P]
    lib.gs_bin_sort_workspace_bytes.restype = C.c_size_t
    lib.gs_bin_sort_workspace_bytes.argtypes = [_I64, _I64, C.c_int32, C.c_int32]
    lib.gs_bin_sort.restype = st
    lib.gs_bin_sort.argtypes = [C.POINTER(Camera), _I64, _P, _P, _P, _P, C.c_size_t, _P, _I64,
                                _P, _P, _P, _P, _P]
    lib.gs_raster_workspace_bytes.restype = C.c_size_t
    lib.gs_raster_workspace_bytes.argtypes = [C.c_int32, C.c_int32, _I64, C.POINTER(Settings)]
    lib.gs_rasterize_fwd.restype = st
    lib.gs_rasterize_fwd.argtypes = [C.POINTER(Camera), C.POINTER(Settings), _I64, _P, _P, _I64,
                                     _P, _P, _P, C.c_size_t, _P, _P, _P, _P, _P]
    lib.gs_rasterize_bwd.restype = st
    lib.gs_rasterize_bwd.argtypes = [C.POINTER(Camera), C.POINTER(Settings), _I64, _P, _P, _I64,
                                     _P, _P, _P, C.c_size_t, _P, _P, _P, _P, _P, _P, _P]
    lib.gs_project_bwd.restype = st
    lib.gs_project_bwd.argtypes = [C.POINTER(Camera), _I64, C.c_int32] + [_P] * 13 + [_P]
    lib.gs_raster_stats.restype = st
    lib.gs_raster_stats.argtypes = [_P, C.c_size_t, _P, _P]
    lib.gs_project_sh16.restype = st
    lib.gs_project_sh16.argtypes = [C.POINTER(Camera), _I64, C.c_int32] + [_P] * 9 + [_P]
    lib.gs_project_bwd_sh16.restype = st
    lib.gs_project_bwd_sh16.argtypes = [C.POINTER(Camera), _I64, C.c_int32] + [_P] * 13 + [_P]
    lib.gs_project_bwd_adam.restype = st
    lib.gs_project_bwd_adam.argtypes = ([C.POINTER(Camera), _I64, C.c_int32] + [_P] * 8 +
                                        [C.POINTER(AdamMoments), C.POINTER(AdamSettings), _P,
                                         _P, _P])
    lib.gs_loss_workspace_bytes.restype = C.c_size_t
    lib.gs_loss_workspace_bytes.argtypes = [C.c_int32, C.c_int32]
    lib.gs_loss_l1_ssim.restype = st
    lib.gs_loss_l1_ssim.argtypes = [C.c_int32, C.c_int32, _P, _P, C.POINTER(LossSettings), _P, _P,
                                    _P, C.c_size_t, _P]
    lib.gs_bin_sort_noalloc.restype = st
    lib.gs_bin_sort_noalloc.argtypes = [C.POINTER(Camera), _I64, _P, _P, _P, _P, _I64, _P, _P, _P,
                                        _P, _P]


# ---------------------------------------------------------------------------
# argument marshalling
# ---------------------------------------------------------------------------
def _is_bf16(t) -> bool:
    import torch

    return isinstance(t, torch.Tensor) and t.dtype == torch.bfloat16


def _ptr(t, name, dtype=None, numel=None, optional=False):
    """Device address of a tensor (checked), an int address, or None."""
    if t is None:
        if optional:
            return None
        raise ValueError(f"{name} is required")
    if isinstance(t, int):
        return t
    import torch

    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch tensor or a device address")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name}: expected {dtype}, got {t.dtype}")
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{name}: needs at least {numel} elements, has {t.numel()}")
    return t.data_ptr() if t.numel() > 0 else None


def _stream(stream):
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, status: int, extra: str = "") -> None:
    if status != 0:
        raise GSError(fn, status, extra)


def _settings(settings) -> Settings:
    return settings if settings is not None else gs_default_settings()


def gs_default_settings() -> Settings:
    return library().gs_default_settings()


def gs_status_string(status: int) -> str:
    """The library's text for a gs_status code."""
    return library().gs_status_string(int(status)).decode()


def gs_num_tiles(width: int, height: int) -> int:
    """Number of 16 x 16 tiles covering a width x height image (0 for an empty image)."""
    return int(library().gs_num_tiles(int(width), int(height)))


def _f32():
    import torch

    return torch.float32


def _i32():
    import torch

    return torch.int32


def gs_project(cam, n, sh_degree, means, scales, quats, opacities, sh, splats, depths, radii,
               tiles_touched, stream=None):
    """Projection + SH colour + tile counts (see gs.h)."""
    K = (int(sh_degree) + 1) ** 2
    f, i = _f32(), _i32()
    st = library().gs_project(
        C.byref(Camera.of(cam)), int(n), int(sh_degree), _ptr(means, "means", f, 3 * n),
        _ptr(scales, "scales", f, 3 * n), _ptr(quats, "quats", f, 4 * n),
        _ptr(opacities, "opacities", f, n), _ptr(sh, "sh", f, 3 * K * n),
        _ptr(splats, "splats", f, SPLAT_FLOATS * n), _ptr(depths, "depths", f, n),
        _ptr(radii, "radii", i, 2 * n), _ptr(tiles_touched, "tiles_touched", i, n), _stream(stream))
    _check("gs_project", st)


def gs_project_sh16(cam, n, sh_degree, means, scales, quats, opacities, sh, splats, depths, radii,
                    tiles_touched, stream=None):
    """gs_project with the SH coefficients as a torch.bfloat16 tensor (see gs.h)."""
    import torch

    K = (int(sh_degree) + 1) ** 2
    f, i = _f32(), _i32()
    st = library().gs_project_sh16(
        C.byref(Camera.of(cam)), int(n), int(sh_degree), _ptr(means, "means", f, 3 * n),
        _ptr(scales, "scales", f, 3 * n), _ptr(quats, "quats", f, 4 * n),
        _ptr(opacities, "opacities", f, n), _ptr(sh, "sh", torch.bfloat16, 3 * K * n),
        _ptr(splats, "splats", f, SPLAT_FLOATS * n), _ptr(depths, "depths", f, n),
        _ptr(radii, "radii", i, 2 * n), _ptr(tiles_touched, "tiles_touched", i, n), _stream(stream))
    _check("gs_project_sh16", st)


def gs_bin_sort_workspace_bytes(n, capacity, width, height) -> int:
    return int(library().gs_bin_sort_workspace_bytes(int(n), int(capacity), int(width), int(height)))


def gs_bin_sort(cam, n, splats, depths, tiles_touched, workspace, sorted_ids, capacity,
                tile_ranges, lpt_order, counts_device=None, sync_pairs=True, stream=None):
    """Tile binning and sort into (tile, depth, id) order, with tile ranges and LPT order
    (per-tile buckets below 8 Mi pairs of capacity, a two-stage radix sort from there);
    returns the pair count I when sync_pairs (GSError status 3 names the count needed)."""
    import torch

    cam_c = Camera.of(cam)
    nt = library().gs_num_tiles(cam_c.width, cam_c.height)
    host = C.c_int64(-1)
    st = library().gs_bin_sort(
        C.byref(cam_c), int(n), _ptr(splats, "splats", _f32(), SPLAT_FLOATS * n, optional=n == 0),
        _ptr(depths, "depths", _f32(), n, optional=n == 0),
        _ptr(tiles_touched, "tiles_touched", _i32(), n, optional=n == 0),
        _ptr(workspace, "workspace", torch.uint8), workspace.numel(),
        _ptr(sorted_ids, "sorted_ids", _i32(), capacity), int(capacity),
        _ptr(tile_ranges, "tile_ranges", _i32(), 2 * nt), _ptr(lpt_order, "lpt_order", _i32(), nt),
        _ptr(counts_device, "counts_device", torch.int64, 2, optional=True),
        C.byref(host) if sync_pairs else None, _stream(stream))
    _check("gs_bin_sort", st, f"; pairs needed: {host.value}" if st == 3 else "")
    return int(host.value) if sync_pairs else None


def gs_bin_sort_noalloc(cam, n, splats, depths, tiles_touched, sorted_ids, capacity, tile_ranges,
                        lpt_order, counts_device=None, sync_pairs=True, stream=None):
    """gs_bin_sort on the library's fixed scratch (allocates nothing; see gs.h for its limits)."""
    import torch

    cam_c = Camera.of(cam)
    nt = library().gs_num_tiles(cam_c.width, cam_c.height)
    host = C.c_int64(-1)
    st = library().gs_bin_sort_noalloc(
        C.byref(cam_c), int(n), _ptr(splats, "splats", _f32(), SPLAT_FLOATS * n, optional=n == 0),
        _ptr(depths, "depths", _f32(), n, optional=n == 0),
        _ptr(tiles_touched, "tiles_touched", _i32(), n, optional=n == 0),
        _ptr(sorted_ids, "sorted_ids", _i32(), capacity), int(capacity),
        _ptr(tile_ranges, "tile_ranges", _i32(), 2 * nt), _ptr(lpt_order, "lpt_order", _i32(), nt),
        _ptr(counts_device, "counts_device", torch.int64, 2, optional=True),
        C.byref(host) if sync_pairs else None, _stream(stream))
    _check("gs_bin_sort_noalloc", st, f"; pairs needed: {host.value}" if st == 3 else "")
    return int(host.value) if sync_pairs else None


def gs_raster_workspace_bytes(width, height, capacity, settings=None) -> int:
    return int(library().gs_raster_workspace_bytes(int(width), int(height), int(capacity),
                                                   C.byref(_settings(settings))))


def gs_rasterize_fwd(cam, n, splats, sorted_ids, tile_ranges, lpt_order, workspace, image,
                     t_final, n_contrib, last_idx, settings=None, stream=None):
    """Forward blend (see gs.h); the pair capacity is sorted_ids' length."""
    import torch

    cam_c = Camera.of(cam)
    P = cam_c.width * cam_c.height
    st = library().gs_rasterize_fwd(
        C.byref(cam_c), C.byref(_settings(settings)), int(n),
        _ptr(splats, "splats", _f32(), SPLAT_FLOATS * n, optional=n == 0),
        _ptr(sorted_ids, "sorted_ids", _i32()), sorted_ids.numel(),
        _ptr(tile_ranges, "tile_ranges", _i32()),
        _ptr(lpt_order, "lpt_order", _i32()), _ptr(workspace, "workspace", torch.uint8),
        workspace.numel(), _ptr(image, "image", _f32(), 3 * P), _ptr(t_final, "t_final", _f32(), P),
        _ptr(n_contrib, "n_contrib", _i32(), P), _ptr(last_idx, "last_idx", _i32(), P),
        _stream(stream))
    _check("gs_rasterize_fwd", st)


def gs_rasterize_bwd(cam, n, splats, sorted_ids, tile_ranges, lpt_order, workspace, t_final,
                     last_idx, dL_dimage, dL_dt_final, grad2d, touched=None, settings=None,
                     stream=None):
    import torch

    cam_c = Camera.of(cam)
    P = cam_c.width * cam_c.height
    st = library().gs_rasterize_bwd(
        C.byref(cam_c), C.byref(_settings(settings)), int(n),
        _ptr(splats, "splats", _f32(), SPLAT_FLOATS * n, optional=n == 0),
        _ptr(sorted_ids, "sorted_ids", _i32()), sorted_ids.numel(),
        _ptr(tile_ranges, "tile_ranges", _i32()),
        _ptr(lpt_order, "lpt_order", _i32()), _ptr(workspace, "workspace", torch.uint8),
        workspace.numel(), _ptr(t_final, "t_final", _f32(), P),
        _ptr(last_idx, "last_idx", _i32(), P), _ptr(dL_dimage, "dL_dimage", _f32(), 3 * P),
        _ptr(dL_dt_final, "dL_dt_final", _f32(), P, optional=True),
        _ptr(grad2d, "grad2d", _f32(), GRAD2D * n, optional=n == 0),
        _ptr(touched, "touched", torch.uint8, n, optional=True), _stream(stream))
    _check("gs_rasterize_bwd", st)


def gs_project_bwd(cam, n, sh_degree, means, scales, quats, opacities, sh, tiles_touched, grad2d,
                   touched, dmeans, dscales, dquats, dopacities, dsh, stream=None):
    import torch

    K = (int(sh_degree) + 1) ** 2
    f, i = _f32(), _i32()
    st = library().gs_project_bwd(
        C.byref(Camera.of(cam)), int(n), int(sh_degree), _ptr(means, "means", f, 3 * n),
        _ptr(scales, "scales", f, 3 * n), _ptr(quats, "quats", f, 4 * n),
        _ptr(opacities, "opacities", f, n, optional=True), _ptr(sh, "sh", f, 3 * K * n),
        _ptr(tiles_touched, "tiles_touched", i, n), _ptr(grad2d, "grad2d", f, GRAD2D * n),
        _ptr(touched, "touched", torch.uint8, n, optional=True), _ptr(dmeans, "dmeans", f, 3 * n),
        _ptr(dscales, "dscales", f, 3 * n), _ptr(dquats, "dquats", f, 4 * n),
        _ptr(dopacities, "dopacities", f, n), _ptr(dsh, "dsh", f, 3 * K * n), _stream(stream))
    _check("gs_project_bwd", st)


def gs_project_bwd_sh16(cam, n, sh_degree, means, scales, quats, opacities, sh, tiles_touched,
                        grad2d, touched, dmeans, dscales, dquats, dopacities, dsh, stream=None):
    """gs_project_bwd with the SH coefficients as a torch.bfloat16 tensor; dsh is fp32."""
    import torch

    K = (int(sh_degree) + 1) ** 2
    f, i = _f32(), _i32()
    st = library().gs_project_bwd_sh16(
        C.byref(Camera.of(cam)), int(n), int(sh_degree), _ptr(means, "means", f, 3 * n),
        _ptr(scales, "scales", f, 3 * n), _ptr(quats, "quats", f, 4 * n),
        _ptr(opacities, "opacities", f, n, optional=True),
        _ptr(sh, "sh", torch.bfloat16, 3 * K * n),
        _ptr(tiles_touched, "tiles_touched", i, n), _ptr(grad2d, "grad2d", f, GRAD2D * n),
        _ptr(touched, "touched", torch.uint8, n, optional=True), _ptr(dmeans, "dmeans", f, 3 * n),
        _ptr(dscales, "dscales", f, 3 * n), _ptr(dquats, "dquats", f, 4 * n),
        _ptr(dopacities, "dopacities", f, n), _ptr(dsh, "dsh", f, 3 * K * n), _stream(stream))
    _check("gs_project_bwd_sh16", st)


def gs_project_bwd_adam(cam, n, sh_degree, means, log_scales, quats, opacity_logits, sh,
                        tiles_touched, grad2d, touched, m, v, settings: AdamSettings,
                        scales_out=None, opacities_out=None, stream=None):
    """gs_project_bwd fused with one Adam step on the raw parameters, in place (see gs.h).
    m and v: five tensors each, shaped like (means, log_scales, quats, opacity_logits, sh).
    scales_out / opacities_out (optional) receive exp(log_scales) and sigmoid(logits)
    after the step."""
    import torch

    K = (int(sh_degree) + 1) ** 2
    f, i = _f32(), _i32()
    sizes = (3 * n, 3 * n, 4 * n, n, 3 * K * n)
    names = ("means", "log_scales", "quats", "opacity_logits", "sh")
    if len(m) != 5 or len(v) != 5:
        raise ValueError("m and v need five tensors each")
    mom = AdamMoments()
    for k in range(5):
        mom.m[k] = _ptr(m[k], "m." + names[k], f, sizes[k])
        mom.v[k] = _ptr(v[k], "v." + names[k], f, sizes[k])
    params = (means, log_scales, quats, opacity_logits, sh)
    st = library().gs_project_bwd_adam(
        C.byref(Camera.of(cam)), int(n), int(sh_degree),
        *[_ptr(t, names[k], f, sizes[k]) for k, t in enumerate(params)],
        _ptr(tiles_touched, "tiles_touched", i, n), _ptr(grad2d, "grad2d", f, GRAD2D * n),
        _ptr(touched, "touched", torch.uint8, n, optional=True), C.byref(mom),
        C.byref(settings), _ptr(scales_out, "scales_out", f, 3 * n, optional=True),
        _ptr(opacities_out, "opacities_out", f, n, optional=True), _stream(stream))
    _check("gs_project_bwd_adam", st)


def gs_loss_workspace_bytes(width, height) -> int:
    return int(library().gs_loss_workspace_bytes(int(width), int(height)))


def gs_loss_l1_ssim(width, height, image, target, dL_dimage, loss_out, workspace,
                    settings: LossSettings | None = None, stream=None):
    """The L1 + SSIM loss of image against target and its gradient (see gs.h).
    loss_out: device float32[3] = (L, mean |x - y|, mean SSIM)."""
    import torch

    P = 3 * int(width) * int(height)
    f = _f32()
    ls = settings if settings is not None else LossSettings.default()
    st = library().gs_loss_l1_ssim(
        int(width), int(height), _ptr(image, "image", f, P), _ptr(target, "target", f, P),
        C.byref(ls), _ptr(dL_dimage, "dL_dimage", f, P), _ptr(loss_out, "loss_out", f, 3),
        _ptr(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream))
    _check("gs_loss_l1_ssim", st)


def gs_raster_stats(workspace, stream=None) -> dict:
    out = (C.c_int64 * 16)()
    st = library().gs_raster_stats(_ptr(workspace, "workspace"), workspace.numel(), out,
                                   _stream(stream))
    _check("gs_raster_stats", st)
    return {"h": out[0], "k": out[1], "resident_ctas": out[2], "work_items": out[3],
            "device_error": out[4], "n_max": out[5], "n_min_nonempty": out[6],
            "n_total": out[7], "nonempty_tiles": out[8], "batches_tiles": out[9],
            "batches_chunks": out[10], "batches_skipped_on_flag": out[11],
            "batches_skipped_done": out[12], "batches_discarded": out[13]}


# ---------------------------------------------------------------------------
# convenience: one view, buffers allocated with torch
# ---------------------------------------------------------------------------
@dataclass
class Grads:
    means: "object"
    scales: "object"
    quats: "object"
    opacities: "object"
    sh: "object"


class Rasterizer:
    """Owns the device buffers of one view and runs the five calls in order.

    forward(means, scales, quats, opacities, sh) -> (image [H, W, 3], t_final [H, W])
    backward(dL_dimage, dL_dt_final=None) -> Grads
    Tensors are float32 CUDA tensors of the shapes documented in gs.h.
    """

    def __init__(self, cam, sh_degree: int, n: int, capacity: int | None = None,
                 settings: Settings | None = None, device="cuda"):
        import torch

        self.cam = Camera.of(cam)
        self.sh_degree = int(sh_degree)
        self.n = int(n)
        self.settings = settings if settings is not None else gs_default_settings()
        self.device = torch.device(device)
        W, H = self.cam.width, self.cam.height
        self.n_tiles = int(library().gs_num_tiles(W, H))
        dev, f, i = self.device, torch.float32, torch.int32
        self.splats = torch.empty((self.n, SPLAT_FLOATS), dtype=f, device=dev)
        self.depths = torch.empty(self.n, dtype=f, device=dev)
        self.radii = torch.empty((self.n, 2), dtype=i, device=dev)
        self.tiles_touched = torch.empty(self.n, dtype=i, device=dev)
        self.tile_ranges = torch.empty((self.n_tiles, 2), dtype=i, device=dev)
        self.lpt_order = torch.empty(self.n_tiles, dtype=i, device=dev)
        self.counts = torch.zeros(2, dtype=torch.int64, device=dev)
        self.image = torch.empty((H, W, 3), dtype=f, device=dev)
        self.t_final = torch.empty((H, W), dtype=f, device=dev)
        self.n_contrib = torch.empty((H, W), dtype=i, device=dev)
        self.last_idx = torch.empty((H, W), dtype=i, device=dev)
        self.grad2d = torch.empty((self.n, GRAD2D), dtype=f, device=dev)
        self.touched = torch.empty(self.n, dtype=torch.uint8, device=dev)
        self._alloc_pairs(capacity if capacity else max(4 * self.n, 1 << 16))
        self.n_pairs = None
        self._inputs = None

    def _alloc_pairs(self, capacity: int):
        import torch

        self.capacity = int(capacity)
        self.sorted_ids = torch.empty(self.capacity, dtype=torch.int32, device=self.device)
        self.bin_ws = torch.empty(gs_bin_sort_workspace_bytes(self.n, self.capacity, self.cam.width,
                                                              self.cam.height),
                                  dtype=torch.uint8, device=self.device)
        self.raster_ws = torch.empty(gs_raster_workspace_bytes(self.cam.width, self.cam.height,
                                                               self.capacity, self.settings),
                                     dtype=torch.uint8, device=self.device)

    def forward(self, means, scales, quats, opacities, sh, sync_pairs: bool = True):
        n = self.n
        # SH coefficients as torch.bfloat16 take the bfloat16-storage calls
        project = gs_project_sh16 if _is_bf16(sh) else gs_project
        project(self.cam, n, self.sh_degree, means, scales, quats, opacities, sh, self.splats,
                self.depths, self.radii, self.tiles_touched)
        while True:
            try:
                self.n_pairs = gs_bin_sort(self.cam, n, self.splats, self.depths,
                                           self.tiles_touched, self.bin_ws, self.sorted_ids,
                                           self.capacity, self.tile_ranges, self.lpt_order,
                                           self.counts, sync_pairs=sync_pairs)
                break
            except GSError as e:
                if e.status != 3:
                    raise
                self._alloc_pairs(int(self._needed(e) * 1.25) + 1)
        gs_rasterize_fwd(self.cam, n, self.splats, self.sorted_ids, self.tile_ranges,
                         self.lpt_order, self.raster_ws, self.image, self.t_final, self.n_contrib,
                         self.last_idx, self.settings)
        self._inputs = (means, scales, quats, opacities, sh)
        return self.image, self.t_final

    @staticmethod
    def _needed(e: GSError) -> int:
        return int(str(e).rsplit("pairs needed:", 1)[1].strip())

    def backward(self, dL_dimage, dL_dt_final=None) -> Grads:
        import torch

        n, K = self.n, (self.sh_degree + 1) ** 2
        means, scales, quats, opacities, sh = self._inputs
        gs_rasterize_bwd(self.cam, n, self.splats, self.sorted_ids, self.tile_ranges,
                         self.lpt_order, self.raster_ws, self.t_final, self.last_idx, dL_dimage,
                         dL_dt_final, self.grad2d, self.touched, self.settings)
        dev, f = self.device, torch.float32
        g = Grads(torch.empty((n, 3), dtype=f, device=dev), torch.empty((n, 3), dtype=f, device=dev),
                  torch.empty((n, 4), dtype=f, device=dev), torch.empty(n, dtype=f, device=dev),
                  torch.empty((n, K, 3), dtype=f, device=dev))
        project_bwd = gs_project_bwd_sh16 if _is_bf16(sh) else gs_project_bwd
        project_bwd(self.cam, n, self.sh_degree, means, scales, quats, opacities, sh,
                    self.tiles_touched, self.grad2d, self.touched, g.means, g.scales, g.quats,
                    g.opacities, g.sh)
        return g

    def stats(self) -> dict:
        return gs_raster_stats(self.raster_ws)
