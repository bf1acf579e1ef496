"""Seeded synthetic inputs for the Gaussian splatting rasterizer.

This module is shared by the tests, the benchmark, the smoke check, the
oracle and the CUDA library's callers.  It holds none of the method's
arithmetic: it only draws random Gaussian parameters and builds pinhole
cameras.  Scales and opacities are returned *activated* (exp of a log-scale,
sigmoid of a logit), quaternions as unit vectors (w, x, y, z).

The pages measure on datasets that are not available here (Mip-NeRF 360
garden/room, Tanks & Temples, Hier-3DGS, Waymo, nuScenes); the five configs
below stand in for them with the shapes the pages give (Gaussian counts,
image sizes, SH degree, heavy tile skew).  All draws use numpy's PCG64
generator in float64 and are cast to float32.

Config 1  tiny:   2,000 Gaussians, 128x128, SH degree 0
Config 2  object: 100k Gaussians on a shell, 800x800, SH degree 3
Config 3  scene:  1.5M Gaussians (2,000-component mixture + ground plane),
                  1297x840, SH degree 3
Config 4  skewed: 3M Gaussians, 20 % packed into 5 tight clusters, 1920x1080
Config 5  street: 6M Gaussians along a 400 m corridor, 3840x2160
"""

from __future__ import annotations

import math
from dataclasses import dataclass, replace

import numpy as np


@dataclass
class Camera:
    viewmat: np.ndarray  # [4, 4] float32, world -> camera, OpenCV axes (x right, y down, z forward)
    fx: float
    fy: float
    cx: float
    cy: float
    width: int
    height: int
    znear: float = 0.2


@dataclass
class Scene:
    means: np.ndarray      # [N, 3] float32
    scales: np.ndarray     # [N, 3] float32, > 0
    quats: np.ndarray      # [N, 4] float32, unit (w, x, y, z)
    opacities: np.ndarray  # [N] float32, in (0, 1)
    sh: np.ndarray         # [N, K, 3] float32, K = (sh_degree + 1)^2
    sh_degree: int

    @property
    def n(self) -> int:
        return int(self.means.shape[0])

    def subset(self, idx) -> "Scene":
        return replace(self, means=self.means[idx], scales=self.scales[idx],
                       quats=self.quats[idx], opacities=self.opacities[idx], sh=self.sh[idx])


CONFIG_NAMES = {
    1: "tiny-2k-128x128-sh0",
    2: "shell-100k-800x800-sh3",
    3: "scene-1.5M-1297x840-sh3",
    4: "clustered-3M-1920x1080-sh3",
    5: "street-6M-3840x2160-sh3",
}
CONFIG_N = {1: 2_000, 2: 100_000, 3: 1_500_000, 4: 3_000_000, 5: 6_000_000}


def look_at(eye, target, up=(0.0, -1.0, 0.0)) -> np.ndarray:
    """World->camera matrix with OpenCV axes: z towards the target, y down."""
    eye = np.asarray(eye, np.float64)
    f = np.asarray(target, np.float64) - eye
    f /= np.linalg.norm(f)
    down = -np.asarray(up, np.float64)
    r = np.cross(down, f)
    r /= np.linalg.norm(r)
    d = np.cross(f, r)
    Rm = np.stack([r, d, f])  # rows: camera axes in world coordinates
    V = np.eye(4)
    V[:3, :3] = Rm
    V[:3, 3] = -Rm @ eye
    return V.astype(np.float32)


def pinhole(viewmat, f, width, height, znear=0.2) -> Camera:
    return Camera(np.asarray(viewmat, np.float32), float(f), float(f), width / 2.0, height / 2.0,
                  int(width), int(height), float(znear))


def _unit_quats(rng, n):
    q = rng.standard_normal((n, 4))
    q /= np.linalg.norm(q, axis=1, keepdims=True)
    return q


def _sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def _sh_deg3(rng, n, dc_mean=0.5, dc_std=0.3, rest_std=0.2):
    sh = np.empty((n, 16, 3))
    sh[:, 0, :] = rng.normal(dc_mean, dc_std, (n, 3))
    sh[:, 1:, :] = rng.normal(0.0, rest_std, (n, 15, 3))
    return sh


def _shell(rng, n, r0=0.9, r1=1.0):
    u = rng.standard_normal((n, 3))
    u /= np.linalg.norm(u, axis=1, keepdims=True)
    return u * rng.uniform(r0, r1, (n, 1))


def _pack(means, log_scales, quats, logits, sh, deg) -> Scene:
    return Scene(means.astype(np.float32), np.exp(log_scales).astype(np.float32),
                 quats.astype(np.float32), _sigmoid(logits).astype(np.float32),
                 sh.astype(np.float32), deg)


def config1(rng, n):
    means = np.stack([rng.uniform(-1, 1, n), rng.uniform(-1, 1, n), rng.uniform(2, 6, n)], 1)
    log_scales = rng.normal(-3.0, 0.5, (n, 3))
    quats = _unit_quats(rng, n)
    logits = rng.normal(0.0, 1.0, n)
    rgb = rng.uniform(0.0, 1.0, (n, 1, 3))
    # the degree-0 basis function is the constant 1 / (2 sqrt(pi)): scale the
    # coefficient so that the colour itself is U[0, 1]
    sh = rgb * (2.0 * math.sqrt(math.pi))
    cam = pinhole(np.eye(4), 128.0, 128, 128)
    return _pack(means, log_scales, quats, logits, sh, 0), cam


def config2(rng, n):
    means = _shell(rng, n)
    log_scales = rng.normal(-4.5, 0.7, (n, 3))
    quats = _unit_quats(rng, n)
    logits = rng.normal(0.0, 1.5, n)
    sh = _sh_deg3(rng, n)
    cam = pinhole(look_at((0, 0, -4), (0, 0, 0)), 1100.0, 800, 800)
    return _pack(means, log_scales, quats, logits, sh, 3), cam


def config3(rng, n):
    n_ground = n // 5
    n_mix = n - n_ground
    comps = 2000
    centres = np.stack([rng.uniform(-8, 8, comps), rng.uniform(-3, 1, comps),
                        rng.uniform(-8, 8, comps)], 1)
    sig = rng.uniform(0.1, 1.0, comps)
    weights = rng.dirichlet(np.ones(comps))
    which = rng.choice(comps, n_mix, p=weights)
    mix = centres[which] + rng.standard_normal((n_mix, 3)) * sig[which, None]
    ground = np.stack([rng.uniform(-10, 10, n_ground), 1.5 + rng.normal(0, 0.01, n_ground),
                       rng.uniform(-10, 10, n_ground)], 1)
    means = np.concatenate([mix, ground])
    log_scales = rng.normal(-5.0, 1.0, (n, 3))
    quats = _unit_quats(rng, n)
    logits = rng.normal(0.0, 2.0, n)
    sh = _sh_deg3(rng, n)
    # inside the scene's extent (z in [-8, 8]) at z = -6 looking +z: about a third of the
    # Gaussians are visible, as in the garden scene of the pages (507K of 1.5M)
    cam = pinhole(look_at((0, 0, -6), (0, 0, 0)), 1150.0, 1297, 840)
    return _pack(means, log_scales, quats, logits, sh, 3), cam


def config4(rng, n):
    n_cl = n // 5
    n_shell = n - n_cl
    shell = _shell(rng, n_shell)
    # 5 cluster centres on the camera-facing half of the shell, near the view axis
    c = np.stack([rng.uniform(-0.5, 0.5, 5), rng.uniform(-0.5, 0.5, 5), np.zeros(5)], 1)
    c[:, 2] = -np.sqrt(np.maximum(0.0, 0.95 ** 2 - (c[:, :2] ** 2).sum(1)))
    which = rng.integers(0, 5, n_cl)
    cl = c[which] + rng.normal(0.0, 0.02, (n_cl, 3))
    means = np.concatenate([shell, cl])
    log_scales = rng.normal(-5.0, 1.2, (n, 3))
    quats = _unit_quats(rng, n)
    logits = rng.normal(0.0, 1.5, n)
    sh = _sh_deg3(rng, n)
    cam = pinhole(look_at((0, 0, -4), (0, 0, 0)), 1485.0, 1920, 1080)
    return _pack(means, log_scales, quats, logits, sh, 3), cam


def config5(rng, n):
    n_ground = (2 * n) // 5
    n_left = n // 5
    n_right = n // 5
    n_clut = n - n_ground - n_left - n_right
    ground = np.stack([rng.uniform(-10, 10, n_ground), np.full(n_ground, 1.6),
                       rng.uniform(0, 400, n_ground)], 1)
    left = np.stack([np.full(n_left, -10.0), rng.uniform(-13.4, 1.6, n_left),
                     rng.uniform(0, 400, n_left)], 1)
    right = np.stack([np.full(n_right, 10.0), rng.uniform(-13.4, 1.6, n_right),
                      rng.uniform(0, 400, n_right)], 1)
    blobs = 200
    bc = np.stack([rng.uniform(-8, 8, blobs), rng.uniform(-3.0, 1.6, blobs),
                   rng.uniform(0, 400, blobs)], 1)
    which = rng.integers(0, blobs, n_clut)
    clutter = bc[which] + rng.normal(0.0, 2.0, (n_clut, 3))
    means = np.concatenate([ground, left, right, clutter])
    log_scales = rng.normal(-4.0, 1.5, (n, 3))
    quats = _unit_quats(rng, n)
    logits = rng.normal(0.0, 2.0, n)
    sh = _sh_deg3(rng, n)
    cam = pinhole(np.eye(4), 2200.0, 3840, 2160)
    return _pack(means, log_scales, quats, logits, sh, 3), cam


_MAKERS = {1: config1, 2: config2, 3: config3, 4: config4, 5: config5}


def make_config(c: int, n: int | None = None, seed: int | None = None) -> tuple[Scene, Camera]:
    """Scene and camera of config c (1..5); n overrides the Gaussian count."""
    rng = np.random.default_rng(c if seed is None else seed)
    return _MAKERS[c](rng, CONFIG_N[c] if n is None else int(n))


def loss_weights(c: int, height: int, width: int, seed: int | None = None) -> np.ndarray:
    """dL/dimg for L = sum(w * img), w ~ N(0, 1) [H, W, 3] float32 (seed 100 + c)."""
    rng = np.random.default_rng(100 + c if seed is None else seed)
    return rng.standard_normal((height, width, 3)).astype(np.float32)


def random_scene(rng, n, width, height, f=None, sh_degree=3, depth=(2.0, 6.0),
                 log_scale=(-3.0, 0.5), logit_std=1.5, spread=1.0) -> tuple[Scene, Camera]:
    """Small random scenes for the tests: Gaussians in front of an identity camera."""
    f = float(f if f is not None else max(width, height))
    z = rng.uniform(depth[0], depth[1], n)
    x = rng.uniform(-spread, spread, n) * z * (width / 2.0) / f
    y = rng.uniform(-spread, spread, n) * z * (height / 2.0) / f
    means = np.stack([x, y, z], 1)
    log_scales = rng.normal(log_scale[0], log_scale[1], (n, 3))
    quats = _unit_quats(rng, n)
    logits = rng.normal(0.0, logit_std, n)
    K = (sh_degree + 1) ** 2
    sh = rng.normal(0.0, 0.3, (n, K, 3))
    sh[:, 0, :] = rng.uniform(0.0, 1.0, (n, 3)) * (2.0 * math.sqrt(math.pi))
    cam = pinhole(np.eye(4), f, width, height)
    return _pack(means, log_scales, quats, logits, sh, sh_degree), cam


def _smooth_field(rng, height, width, cell):
    """Random values on a coarse grid, bilinearly interpolated to height x width x 3."""
    gh, gw = height // cell + 2, width // cell + 2
    g = rng.random((gh, gw, 3))
    ys = np.arange(height) / cell
    xs = np.arange(width) / cell
    y0 = np.floor(ys).astype(int)
    x0 = np.floor(xs).astype(int)
    fy = (ys - y0)[:, None, None]
    fx = (xs - x0)[None, :, None]
    a = g[y0][:, x0]
    b = g[y0][:, x0 + 1]
    c = g[y0 + 1][:, x0]
    d = g[y0 + 1][:, x0 + 1]
    return (a * (1 - fx) + b * fx) * (1 - fy) + (c * (1 - fx) + d * fx) * fy


def image_pair(rng, height, width) -> tuple[np.ndarray, np.ndarray]:
    """A rendered image and its target for the photometric loss, [H, W, 3] float32 in
    [0, 1]: smooth content at two scales with sharp-edged rectangles and a black
    region (where a render without background shows nothing); the target is the
    same content with a shifted edge, added texture and noise."""
    base = 0.6 * _smooth_field(rng, height, width, 24) + 0.4 * _smooth_field(rng, height, width, 5)
    img = base.copy()
    tgt = base.copy()
    for _ in range(max(1, (height * width) // 4000)):
        h = int(rng.integers(2, max(3, height // 3)))
        w = int(rng.integers(2, max(3, width // 3)))
        y = int(rng.integers(0, height))
        x = int(rng.integers(0, width))
        col = rng.random(3)
        img[y:y + h, x:x + w] = col
        dy, dx = rng.integers(-2, 3, size=2)
        tgt[max(0, y + dy):y + dy + h, max(0, x + dx):x + dx + w] = col
    tgt = tgt + 0.15 * (_smooth_field(rng, height, width, 3) - 0.5)
    tgt = tgt + 0.03 * rng.standard_normal(tgt.shape)
    # black where nothing is rendered: a band along the top
    band = int(0.15 * height)
    img[:band] = 0.0
    tgt[: band // 2] = 0.0
    return (np.clip(img, 0, 1).astype(np.float32), np.clip(tgt, 0, 1).astype(np.float32))
