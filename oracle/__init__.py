"""CPU oracle for the differentiable Gaussian splatting rasterizer.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product library (``differentiable_gaussian_splatting_gb300``)
never imports it, and this package never imports the product library: the two
share no code.  Inputs come from ``synthetic_scenes`` (random numbers only).

The arithmetic lives in ``gs_oracle.c`` (plain C, compiled with
``-O2 -ffp-contract=off``, no fast-math).  Two builds are made:

* ``f32``: the chain that decides integers (projected centre, conic, tau,
  radii, row spans, the per-pixel hit test) in fp32 with one fixed operation
  order, as the pages require for a reproducible hit test (Kopanas, "What the
  3DGS Literature Left on the Table", Step 5); colours, alphas, transmittance
  and every gradient in double.  This is the oracle.
* ``f64``: the same source with that chain in double, used only as the smooth
  function for central finite differences that pin the analytic backward.

Every function here is argument marshalling around the C entry points; the
docstrings of ``gs_oracle.c`` cite the passages each one follows.

The training step after the chain rule (``raw_grads``, ``adam_step``) sits here
too: the GPU's fused chain rule + Adam call is compared with it; so does the
L1 + SSIM loss before the backward (``loss_l1_ssim``).

Parity pins: every function is pinned by a ``-m "not gpu"`` test under
``tests/`` (closed forms, library special cases, brute force, finite
differences); see the test names in ``tests/test_oracle_*.py``.  The chunking
policy choice (h*, k*) is pinned on hand-worked cases only.
"""

from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gs_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LOCK = threading.Lock()
_LIBS: dict[str, C.CDLL] = {}

TILE = 16
T_MIN = 1e-4
ALPHA_MAX = 0.99
REC = 16  # doubles per projected splat record


def lib_path(variant: str) -> str:
    return os.path.join(_BUILD, f"libgs_oracle_{variant}.so")


def build(force: bool = False) -> None:
    """Compile both oracle variants with gcc (plain C, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    for variant, extra in (("f32", []), ("f64", ["-DORACLE_F64"])):
        out = lib_path(variant)
        if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
            continue
        tmp = out + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
               "-shared", "-Wall", *extra, "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)


def _lib(variant: str = "f32") -> C.CDLL:
    with _LOCK:
        if variant not in _LIBS:
            build()
            lib = C.CDLL(lib_path(variant))
            _declare(lib)
            _LIBS[variant] = lib
        return _LIBS[variant]


_P = C.c_void_p
_I64 = C.c_int64
_I32 = C.c_int


def _declare(lib: C.CDLL) -> None:
    lib.ora_is_f64.restype = C.c_int
    lib.ora_sh_basis.argtypes = [_I64, _P, _P, _P]
    lib.ora_project.argtypes = [_I64, _I32, _P, _P, _I32, _I32, C.c_float,
                                _P, _P, _P, _P, _P, _P, _P, _P, _P]
    lib.ora_splat_tiles.argtypes = [_P, _P, _I32, _I32, C.c_float, _P, _P, _I64]
    lib.ora_splat_tiles.restype = _I64
    lib.ora_bin.argtypes = [_I64, _P, _P, _I32, _I32, C.c_float, _P, _P, _P,
                            _P, _P, _P, _P, _P, _I64]
    lib.ora_bin.restype = _I64
    lib.ora_blend.argtypes = [_I32, _I32, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]
    lib.ora_blend2.argtypes = [_I32, _I32, _P, _P, _P, _P, _P, _P, _P, _I32, _P, _P, _P, _P, _P]
    lib.ora_blend_bwd.argtypes = [_I32, _I32, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]
    lib.ora_blend_bwd2.argtypes = [_I32, _I32, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                   _P]
    lib.ora_project_bwd.argtypes = [_I64, _I32, _P, _P, _I32, _I32, C.c_float,
                                    _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]
    lib.ora_project_bwd_mag.argtypes = [_I64, _I32, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                        _P, _P]
    lib.ora_policy.argtypes = [_I64, _P, _I64, C.c_double, C.c_double, C.c_double, _I64, _P, _P]
    lib.ora_raw_grads.restype = None
    lib.ora_raw_grads.argtypes = [_I64, _P, _P, _P, _P, _P, _P]
    lib.ora_adam_step.restype = None
    lib.ora_adam_step.argtypes = [_I64, _P, _P, _P, _P, C.c_double, C.c_double, C.c_double,
                                  C.c_double, _I64]
    lib.ora_policy.restype = C.c_double
    lib.ora_loss_l1_ssim.restype = None
    lib.ora_loss_l1_ssim.argtypes = [_I32, _I32, _P, _P, C.c_double, C.c_double, C.c_double,
                                     C.c_double, _P, _P, _P, _P]


def _p(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32)


def _cam_args(cam):
    vm = _f32(np.asarray(cam.viewmat).reshape(16))
    intr = _f32([cam.fx, cam.fy, cam.cx, cam.cy])
    return vm, intr, int(cam.width), int(cam.height), float(cam.znear)


def n_tiles(cam) -> tuple[int, int]:
    return (int(cam.width) + TILE - 1) // TILE, (int(cam.height) + TILE - 1) // TILE


# --------------------------------------------------------------------------
# projection
# --------------------------------------------------------------------------
@dataclass
class Projection:
    splat: np.ndarray          # [N, 16] mux, muy, a, b, c, opacity, tau, depth, P00, P01, P11,
    #                            rx, ry, l11, l12, l22 (conic = L^T L, L = [[l11, l12], [0, l22]])
    rgb: np.ndarray            # [N, 3] float64
    radii: np.ndarray          # [N, 2] int32
    tiles_touched: np.ndarray  # [N] int32

    @property
    def visible(self) -> np.ndarray:
        return self.tiles_touched > 0

    def conic_of_factor(self) -> np.ndarray:
        """[N, 3] conic (a, b, c) of the evaluated quadratic, from its Cholesky factor."""
        l11, l12, l22 = self.splat[:, 13], self.splat[:, 14], self.splat[:, 15]
        return np.stack([l11 * l11, l11 * l12, l12 * l12 + l22 * l22], 1)


def project(scene, cam, variant: str = "f32") -> Projection:
    """Projection + SH colour of every Gaussian (Ryu & Yoo Eq. 1; Kopanas Step 1 (b), Step 3)."""
    lib = _lib(variant)
    n = int(scene.means.shape[0])
    vm, intr, W, H, zn = _cam_args(cam)
    means, scales, quats = _f32(scene.means), _f32(scene.scales), _f32(scene.quats)
    opac, sh = _f32(scene.opacities), _f32(scene.sh)
    splat = np.zeros((n, REC), np.float64)
    rgb = np.zeros((n, 3), np.float64)
    radii = np.zeros((n, 2), np.int32)
    tt = np.zeros(n, np.int32)
    lib.ora_project(n, int(scene.sh_degree), _p(vm), _p(intr), W, H, zn, _p(means), _p(scales),
                    _p(quats), _p(opac), _p(sh), _p(splat), _p(rgb), _p(radii), _p(tt))
    return Projection(splat, rgb, radii, tt)


def splat_tiles(cam, record: np.ndarray, variant: str = "f32") -> np.ndarray:
    """Tile ids covered by one projected splat record (row by row)."""
    lib = _lib(variant)
    vm, intr, W, H, zn = _cam_args(cam)
    rec = np.ascontiguousarray(record, dtype=np.float64)
    n = lib.ora_splat_tiles(_p(vm), _p(intr), W, H, zn, _p(rec), None, 0)
    out = np.zeros(max(n, 1), np.int32)
    lib.ora_splat_tiles(_p(vm), _p(intr), W, H, zn, _p(rec), _p(out), n)
    return out[:n]


# --------------------------------------------------------------------------
# binning + sort
# --------------------------------------------------------------------------
@dataclass
class Binning:
    counts: np.ndarray     # [n_tiles] int64, pairs per tile
    ranges: np.ndarray     # [n_tiles, 2] int64, [start, end) in the full sorted list
    lpt_order: np.ndarray  # [n_tiles] int32, descending count, ties by tile id
    sel: np.ndarray | None  # [n_tiles] uint8 selection (None = all tiles)
    sel_off: np.ndarray    # [n_tiles] int64, offset of tile t in `ids`
    ids: np.ndarray        # sorted Gaussian ids of the selected tiles, tile after tile

    @property
    def n_pairs(self) -> int:
        return int(self.counts.sum())

    def tile_ids(self, t: int) -> np.ndarray:
        o = int(self.sel_off[t])
        return self.ids[o:o + int(self.counts[t])]


def bin_sort(cam, proj: Projection, sel: np.ndarray | None = None, variant: str = "f32") -> Binning:
    """Pairs per tile in (tile, depth, id) order; ranges; LPT order (Kopanas Step 1 (b),(d);
    Ryu & Yoo Sec. 4.1)."""
    lib = _lib(variant)
    vm, intr, W, H, zn = _cam_args(cam)
    ntx, nty = n_tiles(cam)
    nt = ntx * nty
    n = int(proj.splat.shape[0])
    counts = np.zeros(nt, np.int64)
    ranges = np.zeros((nt, 2), np.int64)
    lpt = np.zeros(nt, np.int32)
    sel_off = np.zeros(nt, np.int64)
    sel_a = None if sel is None else np.ascontiguousarray(sel, dtype=np.uint8)
    args = (n, _p(vm), _p(intr), W, H, zn, _p(proj.splat), _p(proj.tiles_touched), _p(sel_a),
            _p(counts), _p(ranges), _p(lpt), _p(sel_off))
    # every Gaussian gives at most tiles_touched pairs, so one call usually suffices
    cap = int(np.clip(np.asarray(proj.tiles_touched, np.int64), 0, None).sum())
    ids = np.zeros(max(cap, 1), np.int32)
    need = lib.ora_bin(*args, _p(ids), cap)
    if need > cap:
        ids = np.zeros(need, np.int32)
        lib.ora_bin(*args, _p(ids), need)
    return Binning(counts, ranges, lpt, sel_a, sel_off, ids[:need])


# --------------------------------------------------------------------------
# blending
# --------------------------------------------------------------------------
@dataclass
class Image:
    img: np.ndarray        # [H, W, 3] float64
    T: np.ndarray          # [H, W] float64 final transmittance
    n_contrib: np.ndarray  # [H, W] int32
    last_idx: np.ndarray   # [H, W] int32, -1 = none
    flags: np.ndarray      # [H, W] uint8: bit0 stop near-tie, bit1 clamp near-tie
    tile_mask: np.ndarray  # [H, W] bool, pixels this call computed


FLAG_STOP_TIE = 1
FLAG_CLAMP_TIE = 2


def _pixel_mask(cam, sel: np.ndarray | None) -> np.ndarray:
    W, H = int(cam.width), int(cam.height)
    ntx, nty = n_tiles(cam)
    if sel is None:
        return np.ones((H, W), bool)
    m = np.asarray(sel, bool).reshape(nty, ntx)
    return np.repeat(np.repeat(m, TILE, 0), TILE, 1)[:H, :W]


RULE = -(1 << 31)  # stop_last entry: apply the stop rule at this pixel
FLAG_NOT_ADMISSIBLE = 4


def blend(cam, proj: Projection, b: Binning, variant: str = "f32",
          stop_last: np.ndarray | None = None, clamp_flip: bool = False) -> Image:
    """Front-to-back blending of the selected tiles (Ryu & Yoo Eq. 2-3).

    The other admissible outcomes of fp32 near-ties: stop_last [H, W] int32 holds, per
    pixel, RULE (apply the 1e-4 stop rule) or the list position of the last splat a
    renderer blended (-1 for none); that pixel then blends every hit up to it and its
    flags get FLAG_NOT_ADMISSIBLE when the stop rule does not admit the outcome.
    clamp_flip takes the other decision at every alpha within the band of the 0.99
    clamp (FLAG_CLAMP_TIE pixels)."""
    lib = _lib(variant)
    W, H = int(cam.width), int(cam.height)
    img = np.zeros((H, W, 3), np.float64)
    T = np.ones((H, W), np.float64)
    nc = np.zeros((H, W), np.int32)
    last = np.full((H, W), -1, np.int32)
    flags = np.zeros((H, W), np.uint8)
    sl = None if stop_last is None else np.ascontiguousarray(stop_last, np.int32).reshape(H, W)
    lib.ora_blend2(W, H, _p(proj.splat), _p(proj.rgb), _p(b.ranges), _p(b.sel_off), _p(b.ids),
                   _p(b.sel), _p(sl), int(bool(clamp_flip)), _p(img), _p(T), _p(nc), _p(last),
                   _p(flags))
    return Image(img, T, nc, last, flags, _pixel_mask(cam, b.sel))


@dataclass
class BlendGrads:
    grad2d: np.ndarray  # [N, 9] (mux, muy, a, b, c, opacity, r, g, b)
    gabs: np.ndarray    # [N, 9] magnitude: every term in absolute value, down to the inputs
    grho: np.ndarray    # [N, 9] the terms' magnitudes weighted by their pixel's fp32 error bound
    galt: np.ndarray    # [N, 9] spread of the admissible results at clamp near-ties


def blend_bwd(cam, proj: Projection, b: Binning, dL_dimg: np.ndarray,
              dL_dT: np.ndarray | None = None, variant: str = "f32"):
    """Nine screen-space derivatives per splat, summed over the selected tiles.

    Returns (grad2d [N, 9], gmag [N, 9]) with columns (mux, muy, a, b, c, opacity, r, g, b);
    gmag is the magnitude of what each element sums (every product and every addend, down
    to the inputs, in absolute value); it equals |grad2d| when nothing cancels."""
    r = blend_bwd_bounds(cam, proj, b, dL_dimg, dL_dT, variant=variant)
    return r.grad2d, r.gabs


def blend_bwd_bounds(cam, proj: Projection, b: Binning, dL_dimg: np.ndarray,
                     dL_dT: np.ndarray | None = None, stop_last: np.ndarray | None = None,
                     variant: str = "f32", bounds: bool = True) -> BlendGrads:
    """blend_bwd with the outcome a renderer took at stop near-ties (stop_last as for
    blend) and the quantities that bound an fp32 evaluation's error (BlendGrads; with
    bounds=False only grad2d is formed, the other fields are None)."""
    lib = _lib(variant)
    W, H = int(cam.width), int(cam.height)
    n = int(proj.splat.shape[0])
    out = BlendGrads(*(np.zeros((n, 9), np.float64) if bounds or i == 0 else None
                       for i in range(4)))
    dimg = np.ascontiguousarray(dL_dimg, dtype=np.float64).reshape(H, W, 3)
    dT = None if dL_dT is None else np.ascontiguousarray(dL_dT, dtype=np.float64).reshape(H, W)
    sl = None if stop_last is None else np.ascontiguousarray(stop_last, np.int32).reshape(H, W)
    lib.ora_blend_bwd2(W, H, _p(proj.splat), _p(proj.rgb), _p(b.ranges), _p(b.sel_off),
                       _p(b.ids), _p(b.sel), _p(sl), _p(dimg), _p(dT), _p(out.grad2d),
                       _p(out.gabs), _p(out.grho), _p(out.galt))
    return out


# --------------------------------------------------------------------------
# the same calls over disjoint tile sets on several host threads
# --------------------------------------------------------------------------
def tile_parts(b: Binning, parts: int) -> list[Binning]:
    """Split the selected tiles of b into up to `parts` disjoint sets of similar pair
    counts (largest tiles first, each to the lightest set).  Each part is b with its own
    selection mask: the calls below then blend only that part's tiles."""
    tiles = np.nonzero(b.sel)[0] if b.sel is not None else np.arange(len(b.counts))
    parts = max(1, min(int(parts), len(tiles)))
    order = tiles[np.argsort(-b.counts[tiles], kind="stable")]
    load = np.zeros(parts)
    masks = np.zeros((parts, len(b.counts)), np.uint8)
    for t in order:
        j = int(np.argmin(load))
        masks[j, t] = 1
        load[j] += 256 + b.counts[t]
    return [Binning(b.counts, b.ranges, b.lpt_order, m, b.sel_off, b.ids) for m in masks]


def _threads(fn, items, workers):
    from concurrent.futures import ThreadPoolExecutor

    # the C calls release the GIL (ctypes), so the parts run on separate cores
    with ThreadPoolExecutor(max_workers=workers) as ex:
        return list(ex.map(fn, items))


def blend_parallel(cam, proj: Projection, b: Binning, workers: int | None = None,
                   stop_last: np.ndarray | None = None, clamp_flip: bool = False) -> Image:
    """blend() of b's tiles split over `workers` host threads; every pixel's result comes
    from the one part that holds its tile, so the outputs equal blend()'s."""
    workers = workers or os.cpu_count() or 1
    outs = _threads(lambda p: blend(cam, proj, p, stop_last=stop_last, clamp_flip=clamp_flip),
                    tile_parts(b, workers), workers)
    res = outs[0]
    for o in outs[1:]:
        m = o.tile_mask
        for f in ("img", "T", "n_contrib", "last_idx", "flags"):
            getattr(res, f)[m] = getattr(o, f)[m]
        res.tile_mask = res.tile_mask | m
    return res


def blend_bwd_parallel(cam, proj: Projection, b: Binning, dL_dimg: np.ndarray,
                       dL_dT: np.ndarray | None = None, stop_last: np.ndarray | None = None,
                       workers: int | None = None, bounds: bool = True) -> BlendGrads:
    """blend_bwd_bounds() of b's tiles split over `workers` host threads; each part's
    per-Gaussian sums (float64) are added, so the result equals the single call's up to
    the order of those additions."""
    workers = workers or os.cpu_count() or 1
    outs = _threads(lambda p: blend_bwd_bounds(cam, proj, p, dL_dimg, dL_dT, stop_last,
                                               bounds=bounds),
                    tile_parts(b, workers), workers)
    res = outs[0]
    for o in outs[1:]:
        for f in ("grad2d", "gabs", "grho", "galt"):
            if getattr(res, f) is not None:
                getattr(res, f).__iadd__(getattr(o, f))
    return res


@dataclass
class ParamGrads:
    means: np.ndarray      # [N, 3]
    scales: np.ndarray     # [N, 3]
    quats: np.ndarray      # [N, 4]
    opacities: np.ndarray  # [N]
    sh: np.ndarray         # [N, K, 3]


def project_bwd_magnitude(scene, cam, proj: Projection, gmag: np.ndarray) -> ParamGrads:
    """Magnitudes of the 59 parameter gradients: the chain rule of project_bwd evaluated
    stage by stage on absolute values, from the magnitudes gmag [N, 9] of grad2d (a
    running error bound: a floating-point evaluation errs by a small multiple of u
    times these)."""
    lib = _lib("f32")
    n = int(scene.means.shape[0])
    K = (int(scene.sh_degree) + 1) ** 2
    vm, intr, W, H, zn = _cam_args(cam)
    out = ParamGrads(np.zeros((n, 3)), np.zeros((n, 3)), np.zeros((n, 4)), np.zeros(n),
                     np.zeros((n, K, 3)))
    gm = np.ascontiguousarray(np.abs(gmag), dtype=np.float64)
    lib.ora_project_bwd_mag(n, int(scene.sh_degree), _p(vm), _p(intr), _p(_f32(scene.means)),
                            _p(_f32(scene.scales)), _p(_f32(scene.quats)), _p(_f32(scene.sh)),
                            _p(proj.tiles_touched), _p(gm), _p(out.means), _p(out.scales),
                            _p(out.quats), _p(out.opacities), _p(out.sh))
    return out


def project_bwd(scene, cam, proj: Projection, grad2d: np.ndarray, variant: str = "f32") -> ParamGrads:
    """Chain rule from the nine screen-space derivatives to the 3D parameters."""
    lib = _lib(variant)
    n = int(scene.means.shape[0])
    K = (int(scene.sh_degree) + 1) ** 2
    vm, intr, W, H, zn = _cam_args(cam)
    out = ParamGrads(np.zeros((n, 3)), np.zeros((n, 3)), np.zeros((n, 4)), np.zeros(n),
                     np.zeros((n, K, 3)))
    g2 = np.ascontiguousarray(grad2d, dtype=np.float64)
    lib.ora_project_bwd(n, int(scene.sh_degree), _p(vm), _p(intr), W, H, zn,
                        _p(_f32(scene.means)), _p(_f32(scene.scales)), _p(_f32(scene.quats)),
                        _p(_f32(scene.opacities)), _p(_f32(scene.sh)), _p(proj.tiles_touched),
                        _p(g2), _p(out.means), _p(out.scales), _p(out.quats), _p(out.opacities),
                        _p(out.sh))
    return out


# --------------------------------------------------------------------------
# policy, SH basis
# --------------------------------------------------------------------------
def policy(counts_desc, K: int, lam: float = 256.0, beta: float = 0.05, eps: float = 0.10,
           h_max: int = 1 << 30) -> tuple[int, int, float]:
    """Per-frame chunking choice (h*, k*) of Ryu & Yoo Eq. 6."""
    lib = _lib("f32")
    c = np.ascontiguousarray(counts_desc, dtype=np.int64)
    h = C.c_int64(0)
    k = C.c_int64(0)
    cost = lib.ora_policy(len(c), _p(c), int(K), lam, beta, eps, int(h_max), C.byref(h), C.byref(k))
    return int(h.value), int(k.value), float(cost)


def raw_grads(scales: np.ndarray, opacities: np.ndarray, pg: ParamGrads):
    """Gradients w.r.t. log-scales and opacity logits from those w.r.t. the activated
    scales and opacities (the training step after the chain rule)."""
    lib = _lib("f64")
    s = np.ascontiguousarray(scales, np.float64)
    o = np.ascontiguousarray(opacities, np.float64).reshape(-1)
    ds = np.ascontiguousarray(pg.scales, np.float64)
    do = np.ascontiguousarray(pg.opacities, np.float64).reshape(-1)
    dls = np.empty_like(ds)
    dlo = np.empty_like(do)
    lib.ora_raw_grads(len(o), _p(s), _p(o), _p(ds), _p(do), _p(dls), _p(dlo))
    return dls, dlo


def adam_step(p: np.ndarray, m: np.ndarray, v: np.ndarray, g: np.ndarray, lr: float,
              b1: float, b2: float, eps: float, t: int) -> None:
    """One Adam step t >= 1 on float64 arrays, in place (p, m, v)."""
    for a in (p, m, v):
        assert a.dtype == np.float64 and a.flags.c_contiguous
    gg = np.ascontiguousarray(g, np.float64)
    assert gg.size == p.size == m.size == v.size
    _lib("f64").ora_adam_step(p.size, _p(p), _p(m), _p(v), _p(gg), lr, b1, b2, eps, int(t))


SSIM_C1 = 0.01 ** 2
SSIM_C2 = 0.03 ** 2
SSIM_SIGMA = 1.5


@dataclass
class Loss:
    loss: float        # (1 - lambda) mean|x - y| + lambda (1 - mean SSIM)
    l1: float          # mean |x - y|
    ssim: float        # mean SSIM
    dL_dimg: np.ndarray  # [H, W, 3] float64
    ssim_map: np.ndarray | None  # [H, W, 3] float64 per-pixel SSIM (when asked for)
    mag: np.ndarray | None  # [H, W, 3] the gradient's terms summed in absolute value (when asked for)


def loss_l1_ssim(img: np.ndarray, target: np.ndarray, lam: float = 0.2, c1: float = SSIM_C1,
                 c2: float = SSIM_C2, sigma: float = SSIM_SIGMA, want_map: bool = False) -> Loss:
    """The L1 + SSIM training loss of two [H, W, 3] float32 images and its gradient
    w.r.t. the first (11 x 11 Gaussian window, zero outside the image)."""
    x = _f32(img)
    y = _f32(target)
    assert x.shape == y.shape and x.ndim == 3 and x.shape[2] == 3
    H, W = x.shape[:2]
    out = np.zeros(3, np.float64)
    g = np.empty((H, W, 3), np.float64)
    smap = np.empty((H, W, 3), np.float64) if want_map else None
    mag = np.empty((H, W, 3), np.float64) if want_map else None
    _lib("f64").ora_loss_l1_ssim(W, H, _p(x), _p(y), lam, c1, c2, sigma, _p(out), _p(g),
                                 _p(smap), _p(mag))
    return Loss(float(out[0]), float(out[1]), float(out[2]), g, smap, mag)


def sh_basis(dirs: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """The 16 real SH basis values and Cartesian gradients at unit directions [n, 3]."""
    lib = _lib("f32")
    d = np.ascontiguousarray(dirs, dtype=np.float64).reshape(-1, 3)
    Y = np.zeros((len(d), 16))
    dY = np.zeros((len(d), 16, 3))
    lib.ora_sh_basis(len(d), _p(d), _p(Y), _p(dY))
    return Y, dY


# --------------------------------------------------------------------------
# convenience: the whole forward + backward on the CPU
# --------------------------------------------------------------------------
@dataclass
class Render:
    proj: Projection
    binning: Binning
    image: Image


def render(scene, cam, sel: np.ndarray | None = None, variant: str = "f32") -> Render:
    proj = project(scene, cam, variant)
    b = bin_sort(cam, proj, sel, variant)
    return Render(proj, b, blend(cam, proj, b, variant))


def loss_and_grads(scene, cam, w: np.ndarray, v: np.ndarray | None = None,
                   variant: str = "f32"):
    """L = sum(w * img) + sum(v * T_final) and its gradients w.r.t. every parameter."""
    r = render(scene, cam, None, variant)
    L = float((w * r.image.img).sum())
    if v is not None:
        L += float((v * r.image.T).sum())
    g2, _ = blend_bwd(cam, r.proj, r.binning, w, v, variant)
    return L, r, g2, project_bwd(scene, cam, r.proj, g2, variant)
