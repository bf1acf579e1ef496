"""Float64 definitional checks for the oracle (test infrastructure only).

Independent restatements, in numpy float64, of what the pages define, used to
pin ``gs_oracle.c`` on tiny inputs:

* ``brute_force_blend``: per pixel, every visible splat in (depth, id) order,
  with no tiles, no binning and no spans (Ryu & Yoo Eq. 2-3; Kopanas Step 1 (b)
  for the q <= 2 ln(255 o) support; the 1e-4 stop after Eq. 3).
* ``rect_min_q``: the exact minimum of the quadratic form q(d) over an
  axis-aligned rectangle, which decides whether a tile meets a support
  ellipse without using the closed-form row spans.
* ``pinhole``: the camera map whose numerical Jacobian pins the projection.
"""

from __future__ import annotations

import numpy as np

TILE = 16
T_MIN = 1e-4
ALPHA_MAX = 0.99


def fma_f32(x, y, z):
    """Correctly rounded fp32 fused multiply-add of fp32 arrays, emulated exactly.

    x*y is exact in float64 (48 significant bits); s = fl64(x*y + z) has error e
    (TwoSum).  Rounding s to fp32 equals rounding the exact x*y + z except when s
    is exactly halfway between two fp32 values; then the sign of e decides."""
    x, y, z = (np.asarray(v, np.float32).astype(np.float64) for v in (x, y, z))
    p = x * y
    s = p + z
    bb = s - p
    e = (p - (s - bb)) + (z - bb)
    r = s.astype(np.float32)
    up = np.nextafter(r, np.float32(np.inf))
    dn = np.nextafter(r, np.float32(-np.inf))
    # s exactly at a midpoint between r and a neighbour, and e pushes away from r
    mid_up = (up.astype(np.float64) + r.astype(np.float64)) * 0.5
    mid_dn = (dn.astype(np.float64) + r.astype(np.float64)) * 0.5
    r = np.where((s == mid_up) & (e > 0), up, r)
    r = np.where((s == mid_dn) & (e < 0), dn, r)
    return r


def quad_f32(l11, l12, l22, dx, dy):
    """q = fma(u1, u1, u2 u2), u1 = fma(l11, dx, l12 dy), u2 = l22 dy, in fp32
    round-to-nearest: d^T Lambda d through the Cholesky factor of the conic (the
    reproducible evaluation of the quadratic that Kopanas, Step 5, requires)."""
    f = np.float32
    l11, l12, l22, dx, dy = (np.asarray(v, f) for v in (l11, l12, l22, dx, dy))
    u1 = fma_f32(l11, dx, l12 * dy)
    u2 = l22 * dy
    return fma_f32(u1, u1, u2 * u2)


def brute_force_blend(cam, splat: np.ndarray, rgb: np.ndarray, visible: np.ndarray,
                      tie_rel: float = 1e-5, fp32_quadratic: bool = True):
    """Blend every visible splat over every pixel, front to back.

    splat rows: the oracle's record (mux, muy, a, b, c, opacity, tau, depth, ...,
    l11, l12, l22 in columns 13..15).
    With fp32_quadratic the quadratic form is the fp32 round-to-nearest
    evaluation of ``quad_f32``; otherwise plain float64.
    Returns img [H, W, 3], T [H, W], n_contrib [H, W], ambiguous [H, W] where
    ambiguous marks pixels at which some q lies within tie_rel of tau or some
    stop decision within tie_rel of 1e-4."""
    W, H = int(cam.width), int(cam.height)
    ids = np.nonzero(visible)[0]
    order = ids[np.lexsort((ids, splat[ids, 7]))]
    ys, xs = np.mgrid[0:H, 0:W]
    px = xs.astype(np.float32) + np.float32(0.5)
    py = ys.astype(np.float32) + np.float32(0.5)
    C = np.zeros((H, W, 3))
    T = np.ones((H, W))
    n = np.zeros((H, W), np.int32)
    done = np.zeros((H, W), bool)
    amb = np.zeros((H, W), bool)
    for g in order:
        mux, muy, a, b, c, o, tau = splat[g, :7]
        l11, l12, l22 = splat[g, 13:16]
        if fp32_quadratic:
            dx = px - np.float32(mux)
            dy = py - np.float32(muy)
            q = quad_f32(l11, l12, l22, dx, dy).astype(np.float64)
        else:
            a, b, c = l11 * l11, l11 * l12, l12 * l12 + l22 * l22
            dx = px.astype(np.float64) - mux
            dy = py.astype(np.float64) - muy
            q = a * dx * dx + 2.0 * b * dx * dy + c * dy * dy
        live = ~done
        amb |= live & (np.abs(q - tau) <= tie_rel * tau)
        hit = live & (q <= tau)
        alpha = np.minimum(ALPHA_MAX, o * np.exp(-0.5 * q))
        alpha = np.where(hit, alpha, 0.0)
        C += rgb[g][None, None, :] * (alpha * T)[..., None]
        T = T * (1.0 - alpha)
        n += hit
        amb |= live & (np.abs(T - T_MIN) <= tie_rel * T_MIN)
        done |= T < T_MIN
    return C, T, n, amb


def rect_min_q(a, b, c, x0, x1, y0, y1):
    """min over d in [x0, x1] x [y0, y1] of a dx^2 + 2 b dx dy + c dy^2 (a, c > 0, ac > b^2).

    The form is convex: the minimum is 0 at the origin if the rectangle holds
    it, else on the boundary, where each edge is a 1D quadratic."""
    if x0 <= 0.0 <= x1 and y0 <= 0.0 <= y1:
        return 0.0
    best = np.inf
    for y in (y0, y1):  # horizontal edges: minimise over x at fixed y
        x = min(max(-b * y / a, x0), x1)
        best = min(best, a * x * x + 2 * b * x * y + c * y * y)
    for x in (x0, x1):  # vertical edges
        y = min(max(-b * x / c, y0), y1)
        best = min(best, a * x * x + 2 * b * x * y + c * y * y)
    return best


def tile_hull(cam, t: int):
    """Closed hull of the pixel centres of tile t, clipped to the image."""
    ntx = (int(cam.width) + TILE - 1) // TILE
    tx, ty = t % ntx, t // ntx
    x0 = TILE * tx + 0.5
    x1 = min(TILE * tx + TILE - 0.5, cam.width - 0.5)
    y0 = TILE * ty + 0.5
    y1 = min(TILE * ty + TILE - 0.5, cam.height - 0.5)
    return x0, x1, y0, y1


def pinhole(cam, m: np.ndarray) -> np.ndarray:
    """World point -> pixel coordinates (float64)."""
    V = np.asarray(cam.viewmat, np.float64)
    t = V[:3, :3] @ m + V[:3, 3]
    return np.array([cam.fx * t[0] / t[2] + cam.cx, cam.fy * t[1] / t[2] + cam.cy])
