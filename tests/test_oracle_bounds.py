"""Pins of the oracle quantities that set the GPU gradient tolerance, and of the other
admissible outcomes of its fp32 near-ties.

* ``gabs`` (the magnitude of what each screen-space gradient sums), ``grho`` (those
  magnitudes weighted by each pixel's fp32 error bound) and ``galt`` (the spread of the
  admissible results at near-ties of the 0.99 clamp) are checked for EQUALITY against a
  restatement in Python: the per-pixel backward of the blend written with the pages'
  formulas over numbers that carry their own magnitude (every product the product of the
  factors' magnitudes, every sum or difference the sum of the terms' magnitudes), on
  splat lists built without tiles.  An oracle that over- or understates any of them fails.
* The bound itself: an fp32 evaluation of the same backward, with every alpha perturbed
  within the band the oracle assumes for a renderer's alpha, stays within
  gamma_n gabs + grho of the oracle's float64 gradient.
* Forced stop outcomes (Ryu & Yoo, Eq. 3 and the stop rule after it): replaying the
  rule's own outcome changes nothing; an outcome the rule forbids outside the fp32 band is
  flagged; at a constructed near-tie both outcomes are admitted.
"""

import math

import numpy as np
import pytest

import oracle
import synthetic_scenes as ss
from oracle.definitional import quad_f32

U = 2.0 ** -24
E_ALPHA = 2.0 ** -17
ALPHA_MAX = 0.99
T_MIN = 1e-4


class A:
    """A value with its magnitude: |x| for an input, propagated through + - * /."""

    __slots__ = ("v", "m")

    def __init__(self, v, m=None):
        self.v = float(v)
        self.m = abs(self.v) if m is None else float(m)

    @staticmethod
    def of(x):
        return x if isinstance(x, A) else A(x)

    def __add__(self, o):
        o = A.of(o)
        return A(self.v + o.v, self.m + o.m)

    def __sub__(self, o):
        o = A.of(o)
        return A(self.v - o.v, self.m + o.m)

    def __mul__(self, o):
        o = A.of(o)
        return A(self.v * o.v, self.m * o.m)

    def __truediv__(self, o):  # divisors here are positive inputs (1 - alpha)
        o = A.of(o)
        return A(self.v / o.v, self.m / abs(o.v))

    __radd__ = __add__
    __rmul__ = __mul__


def _pixel_lists(cam, proj, clamp_flip=False):
    """Per pixel, the blended splats front to back over ALL visible splats in (depth, id)
    order (no tiles): (g, alpha, T before, dx, dy, q, clamped, near_clamp)."""
    W, H = int(cam.width), int(cam.height)
    vis = np.nonzero(proj.tiles_touched > 0)[0]
    order = vis[np.lexsort((vis, proj.splat[vis, 7]))]
    out = {}
    f = np.float32
    for py in range(H):
        for px in range(W):
            T, lst = 1.0, []
            for g in order:
                if T < T_MIN:
                    break
                s = proj.splat[g]
                dx = f(f(px) + f(0.5)) - f(s[0])
                dy = f(f(py) + f(0.5)) - f(s[1])
                q = float(quad_f32(s[13], s[14], s[15], dx, dy))
                if not q <= float(f(s[6])):
                    continue
                araw = s[5] * math.exp(-0.5 * q)
                near = abs(araw - ALPHA_MAX) <= 2.0 * E_ALPHA * ALPHA_MAX
                clamped = not araw < ALPHA_MAX
                if clamp_flip and near:
                    clamped = not clamped
                alpha = ALPHA_MAX if clamped else araw
                lst.append((g, alpha, T, float(dx), float(dy), q, clamped, near))
                T *= 1.0 - alpha
            out[(py, px)] = (lst, T)
    return out


def _terms(proj, lst, Tfin, G, gT):
    """{g: [9 A]} -- the pages' per-pixel backward (Kopanas, Step 1 (a)) over A numbers."""
    Gs = [A(x) for x in G]
    behind = [A(0.0, 0.0)] * 3
    res = {}
    for g, alpha, T, dx, dy, q, clamped, _ in reversed(lst):
        s, col = proj.splat[g], [A(c) for c in proj.rgb[g]]
        a_, T_, om = A(alpha), A(T), 1.0 - alpha
        w = a_ * T_
        cG = col[0] * Gs[0] + col[1] * Gs[1] + col[2] * Gs[2]
        bG = behind[0] * Gs[0] + behind[1] * Gs[1] + behind[2] * Gs[2]
        dalpha = T_ * cG - bG / om - A(gT) * A(Tfin) / om
        t = [A(0.0, 0.0)] * 9
        for ch in range(3):
            t[6 + ch] = w * Gs[ch]
        behind = [behind[ch] + col[ch] * w for ch in range(3)]
        if not clamped:
            dq = A(-0.5) * a_ * dalpha
            l11, l12, l22 = s[13], s[14], s[15]
            a, b, c = A(l11 * l11), A(l11 * l12), A(l12 * l12 + l22 * l22)
            DX, DY = A(dx), A(dy)
            t[5] = A(math.exp(-0.5 * q)) * dalpha
            t[0] = A(-2.0) * (a * DX + b * DY) * dq
            t[1] = A(-2.0) * (b * DX + c * DY) * dq
            t[2] = DX * DX * dq
            t[3] = A(2.0) * DX * DY * dq
            t[4] = DY * DY * dq
        res[g] = t
    return res


def _eps(lst):
    """Relative error bound of a pixel's fp32 backward, as the oracle documents it."""
    return 2.0 * E_ALPHA + 32.0 * U + sum(2.0 * (E_ALPHA * a / (1.0 - a) + 8.0 * U)
                                          for _, a, *_ in lst)


def _restated(cam, proj, w, v):
    n = proj.splat.shape[0]
    g2, gabs, grho, galt = (np.zeros((n, 9)) for _ in range(4))
    lists = _pixel_lists(cam, proj)
    flipped = _pixel_lists(cam, proj, clamp_flip=True)
    for (py, px), (lst, Tfin) in lists.items():
        G, gT = w[py, px], (0.0 if v is None else v[py, px])
        e = _eps(lst)
        terms = _terms(proj, lst, Tfin, G, gT)
        for g, t in terms.items():
            g2[g] += [x.v for x in t]
            gabs[g] += [x.m for x in t]
            grho[g] += [e * x.m for x in t]
        if any(x[7] for x in lst):
            lst2, T2 = flipped[(py, px)]
            alt = _terms(proj, lst2, T2, G, gT)
            for g, t in terms.items():
                galt[g] += [abs(a.v - b.v) for a, b in zip(alt[g], t)]
    return g2, gabs, grho, galt


def _scene(seed, n, W, H, deg, logit_std=2.0):
    rng = np.random.default_rng(seed)
    sc, cam = ss.random_scene(rng, n, W, H, sh_degree=deg, log_scale=(-2.3, 0.5),
                              logit_std=logit_std)
    w = rng.standard_normal((H, W, 3))
    v = rng.standard_normal((H, W))
    return sc, cam, w, v


def _near_clamp_scene():
    """Splats centred on pixel centres (q about 0 there) with opacities within the clamp
    band, on both sides of 0.99, in front of ordinary splats."""
    sc, cam, w, v = _scene(21, 30, 40, 32, 1)
    V = np.asarray(cam.viewmat, np.float64)
    R, tv = V[:3, :3], V[:3, 3]
    z = (R @ sc.means.T.astype(np.float64)).T[:, 2].min() + tv[2] - 0.3  # in front
    for i, o in enumerate([0.99 + 3e-6, 0.99 - 3e-6, 0.99 + 1e-6]):
        sc.opacities[i] = np.float32(o)
        px, py = 10 + 9 * i + 0.5, 12.5
        t = np.array([(px - cam.cx) * z / cam.fx, (py - cam.cy) * z / cam.fy, z])
        sc.means[i] = (R.T @ (t - tv)).astype(np.float32)
    return sc, cam, w, v


@pytest.mark.parametrize("seed,n,W,H,deg", [(1, 40, 48, 32, 3), (2, 25, 33, 27, 0),
                                            (3, 60, 40, 40, 1)])
def test_magnitudes_equal_the_abs_arithmetic_restatement(seed, n, W, H, deg):
    sc, cam, w, v = _scene(seed, n, W, H, deg)
    proj = oracle.project(sc, cam)
    b = oracle.bin_sort(cam, proj)
    r = oracle.blend_bwd_bounds(cam, proj, b, w, v)
    g2, gabs, grho, _ = _restated(cam, proj, w, v)
    assert np.count_nonzero(gabs) > 50
    np.testing.assert_allclose(r.grad2d, g2, rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(r.gabs, gabs, rtol=1e-12, atol=0)
    np.testing.assert_allclose(r.grho, grho, rtol=1e-12, atol=0)
    # gabs is a magnitude: never below |grad2d|, and strictly above it where terms cancel
    assert np.all(r.gabs >= np.abs(r.grad2d) * (1 - 1e-12))
    assert np.any(r.gabs > 2 * np.abs(r.grad2d))


def test_clamp_spread_equals_the_restatement():
    sc, cam, w, v = _near_clamp_scene()
    proj = oracle.project(sc, cam)
    b = oracle.bin_sort(cam, proj)
    im = oracle.blend(cam, proj, b)
    assert np.count_nonzero(im.flags & oracle.FLAG_CLAMP_TIE) >= 3
    r = oracle.blend_bwd_bounds(cam, proj, b, w, v)
    g2, gabs, grho, galt = _restated(cam, proj, w, v)
    assert np.count_nonzero(galt) >= 3
    np.testing.assert_allclose(r.galt, galt, rtol=1e-10, atol=1e-15)
    np.testing.assert_allclose(r.gabs, gabs, rtol=1e-12, atol=0)
    # the flipped rendering is the other clamp decision at exactly the flagged pixels
    alt = oracle.blend(cam, proj, b, clamp_flip=True)
    same = np.all(alt.img == im.img, axis=2) & (alt.T == im.T)
    flagged = (im.flags & oracle.FLAG_CLAMP_TIE) != 0
    assert np.all(same[~flagged]) and not np.any(same[flagged])


def _fp32_backward(cam, proj, w, v, rng):
    """An fp32 evaluation of the blend backward in a renderer's order (transmittance
    recovered back to front by division, the colour behind as a running sum, sums of
    contributions in float32), with every alpha perturbed by a relative error of up to
    E_ALPHA / 2 the way an approximate exponential would; returns grad2d and the number
    of contributions summed into each element."""
    f = np.float32
    n = proj.splat.shape[0]
    acc = np.zeros((n, 9), np.float32)
    cnt = np.zeros(n, np.int64)
    for (py, px), (lst, _) in _pixel_lists(cam, proj).items():
        if not lst:
            continue
        al = [f(a * (1.0 + rng.uniform(-0.5, 0.5) * E_ALPHA)) if not cl else f(ALPHA_MAX)
              for _, a, _, _, _, _, cl, _ in lst]
        T = f(1.0)
        for a in al:
            T = f(T * f(f(1.0) - a))
        G = [f(x) for x in w[py, px]]
        gT = f(0.0 if v is None else v[py, px])
        accg = f(gT * T)
        for (g, _, _, dx, dy, q, clamped, _), a in zip(reversed(lst), reversed(al)):
            s, col = proj.splat[g], [f(c) for c in proj.rgb[g]]
            inv = f(f(1.0) / f(f(1.0) - a))
            Tb = f(T * inv)
            wt = f(a * Tb)
            cG = f(f(f(col[0] * G[0]) + f(col[1] * G[1])) + f(col[2] * G[2]))
            dal = f(f(Tb * cG) - f(accg * inv))
            accg = f(accg + f(cG * wt))
            T = Tb
            t = np.zeros(9, np.float32)
            for ch in range(3):
                t[6 + ch] = f(wt * G[ch])
            if not clamped:
                l11, l12, l22 = f(s[13]), f(s[14]), f(s[15])
                DX, DY = f(dx), f(dy)
                gs = f(a * dal)
                dq = f(f(-0.5) * gs)
                u1 = f(f(l11 * DX) + f(l12 * DY))
                t[5] = f(gs / f(s[5]))
                t[0] = f(f(f(-2.0) * f(l11 * u1)) * dq)
                t[1] = f(f(f(-2.0) * f(f(l12 * u1) + f(f(l22 * l22) * DY))) * dq)
                t[2] = f(f(DX * DX) * dq)
                t[3] = f(f(f(2.0) * f(DX * DY)) * dq)
                t[4] = f(f(DY * DY) * dq)
            acc[g] = acc[g] + t
            cnt[g] += 1
    return acc.astype(np.float64), cnt


@pytest.mark.parametrize("seed", [4, 5])
def test_error_bound_covers_an_fp32_evaluation(seed):
    sc, cam, w, v = _scene(seed, 50, 40, 32, 2, logit_std=3.0)  # many near-opaque splats
    proj = oracle.project(sc, cam)
    b = oracle.bin_sort(cam, proj)
    r = oracle.blend_bwd_bounds(cam, proj, b, w, v)
    g32, cnt = _fp32_backward(cam, proj, w, v, np.random.default_rng(seed))
    nsum = cnt[:, None] + 8
    bound = nsum * U / (1 - nsum * U) * r.gabs + r.grho
    err = np.abs(g32 - r.grad2d)
    assert np.all(err <= bound), float((err / np.maximum(bound, 1e-300)).max())
    # and the bound is not vacuous: it is below a few hundredths of the magnitude
    live = r.gabs > 0
    assert np.median((bound[live] / r.gabs[live])) < 1e-3


def _near_stop_scene():
    """Two clamped splats over the same pixels take T to 1e-4 to within the band, so the
    stop before the third one behind them is a near-tie; where the third is dense, T then
    falls well below 1e-4 and the rule stops before a fourth."""
    W = H = 24
    cam = ss.pinhole(np.eye(4), 40.0, W, H)
    means = np.array([[0, 0, 2.0], [0, 0, 2.5], [0, 0, 3.0], [0, 0, 3.5]], np.float32)
    scales = np.array([[3.0] * 3, [3.0] * 3, [0.3] * 3, [0.3] * 3], np.float32)
    quats = np.tile(np.array([1, 0, 0, 0], np.float32), (4, 1))
    opac = np.array([0.9999, 0.9999, 0.6, 0.6], np.float32)
    sh = np.full((4, 1, 3), 1.0, np.float32)
    return ss.Scene(means, scales, quats, opac, sh, 0), cam


def test_forced_stop_outcomes():
    sc, cam = _near_stop_scene()
    proj = oracle.project(sc, cam)
    b = oracle.bin_sort(cam, proj)
    im = oracle.blend(cam, proj, b)
    tie = (im.flags & oracle.FLAG_STOP_TIE) != 0
    assert tie.sum() > 10
    # replaying the rule's own outcome everywhere changes nothing and is admitted
    same = oracle.blend(cam, proj, b, stop_last=im.last_idx)
    for f in ("img", "T", "n_contrib", "last_idx"):
        np.testing.assert_array_equal(getattr(same, f), getattr(im, f), err_msg=f)
    assert not np.any(same.flags & oracle.FLAG_NOT_ADMISSIBLE)
    # at the near-ties the other decision (blend the third splat too) is admitted; every
    # tile lists the three splats in depth order
    assert np.all(b.counts == 4)
    ys, xs = np.mgrid[0:cam.height, 0:cam.width]
    start = b.ranges[(ys // 16) * ((cam.width + 15) // 16) + xs // 16, 0]
    # the other decision: stop before the third splat where the rule blends it, blend it
    # where the rule stops before it
    cand = tie & (((im.n_contrib == 2) & (im.last_idx == start + 1)) |
                  ((im.n_contrib == 3) & (im.last_idx == start + 2)))
    py, px = np.nonzero(cand)
    assert len(py) > 10
    forced = np.full(im.last_idx.shape, oracle.RULE, np.int32)
    forced[py, px] = np.where(im.n_contrib[py, px] == 3, start[py, px] + 1, start[py, px] + 2)
    alt = oracle.blend(cam, proj, b, stop_last=forced)
    assert np.all(alt.n_contrib[py, px] == 5 - im.n_contrib[py, px])
    assert not np.any(alt.flags & oracle.FLAG_NOT_ADMISSIBLE)
    assert np.all(alt.T[py, px] != im.T[py, px])
    # outside the band: stopping early, or naming a position that is not a hit, is not
    ok = (im.flags == 0) & (im.n_contrib >= 2)
    qy, qx = np.nonzero(ok)
    assert len(qy) > 10
    early = np.full(im.last_idx.shape, oracle.RULE, np.int32)
    tiles = (qy // 16) * ((cam.width + 15) // 16) + qx // 16
    early[qy, qx] = b.ranges[tiles, 0]  # only the first splat
    bad = oracle.blend(cam, proj, b, stop_last=early)
    assert np.all(bad.flags[qy, qx] & oracle.FLAG_NOT_ADMISSIBLE)
    beyond = np.full(im.last_idx.shape, oracle.RULE, np.int32)
    beyond[qy, qx] = b.ranges[tiles, 1] + 5
    bad = oracle.blend(cam, proj, b, stop_last=beyond)
    assert np.all(bad.flags[qy, qx] & oracle.FLAG_NOT_ADMISSIBLE)
    # blending a hit after T fell well below 1e-4 (the fourth splat) is not admitted either
    ry, rx = np.nonzero((im.n_contrib == 3) & (im.last_idx == start + 2) & (im.T < 5e-5))
    past = np.full(im.last_idx.shape, oracle.RULE, np.int32)
    past[ry, rx] = start[ry, rx] + 3
    bad = oracle.blend(cam, proj, b, stop_last=past)
    hit4 = bad.n_contrib[ry, rx] == 4
    assert hit4.sum() > 5
    assert np.all(bad.flags[ry[hit4], rx[hit4]] & oracle.FLAG_NOT_ADMISSIBLE)


def test_forced_stop_backward():
    sc, cam = _near_stop_scene()
    proj = oracle.project(sc, cam)
    b = oracle.bin_sort(cam, proj)
    im = oracle.blend(cam, proj, b)
    rng = np.random.default_rng(3)
    w = rng.standard_normal((cam.height, cam.width, 3))
    base = oracle.blend_bwd_bounds(cam, proj, b, w)
    same = oracle.blend_bwd_bounds(cam, proj, b, w, stop_last=im.last_idx)
    np.testing.assert_array_equal(same.grad2d, base.grad2d)
    # forcing the other stop decision at every near-tie pixel changes the third splat's
    # gradient, which it receives or loses at those pixels
    tie = (im.flags & oracle.FLAG_STOP_TIE) != 0
    ys, xs = np.mgrid[0:cam.height, 0:cam.width]
    start = b.ranges[(ys // 16) * ((cam.width + 15) // 16) + xs // 16, 0]
    py, px = np.nonzero(tie & (im.n_contrib >= 2) & (im.last_idx >= start + 1))
    forced = np.full(im.last_idx.shape, oracle.RULE, np.int32)
    forced[py, px] = np.where(im.n_contrib[py, px] == 3, start[py, px] + 1, start[py, px] + 2)
    alt = oracle.blend_bwd_bounds(cam, proj, b, w, stop_last=forced)
    assert np.any(alt.grad2d[2] != base.grad2d[2])


def _chain_restated(sc, cam, tt, g2v, g2m):
    """The chain rule of the projection (grad2d -> means, scales, quats, opacities, SH), in
    the oracle's order of operations, over A numbers: the forward quantities it multiplies
    by are inputs (a rotation entry, a Jacobian entry, an element of Sigma'), except Sigma =
    M M^T and T = J W, whose sums carry their terms' magnitudes; grad2d enters with the
    magnitudes g2m.  Returns {name: (values, magnitudes)}."""
    n, K = sc.n, (sc.sh_degree + 1) ** 2
    Vm = np.asarray(cam.viewmat, np.float32).astype(np.float64).reshape(16)
    V = Vm[:12]
    fx, fy = float(np.float32(cam.fx)), float(np.float32(cam.fy))
    cw = -np.array([Vm[j] * Vm[3] + Vm[4 + j] * Vm[7] + Vm[8 + j] * Vm[11] for j in range(3)])
    out = {k: (np.zeros(s), np.zeros(s)) for k, s in
           (("means", (n, 3)), ("scales", (n, 3)), ("quats", (n, 4)), ("opacities", (n,)),
            ("sh", (n, K, 3)))}

    def put(name, i, vals):
        v, m = out[name]
        flat = [a for a in np.ravel(np.array(vals, dtype=object))]
        v[i] = np.reshape([a.v for a in flat], v[i].shape)
        m[i] = np.reshape([a.m for a in flat], m[i].shape)

    for i in range(n):
        if tt[i] <= 0 or not np.any(g2v[i] != 0):
            continue
        g = [A(g2v[i, r], g2m[i, r]) for r in range(9)]
        m = sc.means[i].astype(np.float64)
        t = [V[4 * r] * m[0] + V[4 * r + 1] * m[1] + V[4 * r + 2] * m[2] + V[4 * r + 3]
             for r in range(3)]
        qr = sc.quats[i].astype(np.float64)
        qn = math.sqrt(qr[0] * qr[0] + qr[1] * qr[1] + qr[2] * qr[2] + qr[3] * qr[3])
        w, x, y, z = qr / qn
        R = [1 - 2 * (y * y + z * z), 2 * (x * y - w * z), 2 * (x * z + w * y),
             2 * (x * y + w * z), 1 - 2 * (x * x + z * z), 2 * (y * z - w * x),
             2 * (x * z - w * y), 2 * (y * z + w * x), 1 - 2 * (x * x + y * y)]
        s = sc.scales[i].astype(np.float64)
        M = [A(R[3 * r + c] * s[c]) for r in range(3) for c in range(3)]
        S = [M[3 * r] * M[3 * c] + M[3 * r + 1] * M[3 * c + 1] + M[3 * r + 2] * M[3 * c + 2]
             for r in range(3) for c in range(3)]
        tx, ty, tz = t
        j00, j11, j02, j12 = fx / tz, fy / tz, -fx * tx / (tz * tz), -fy * ty / (tz * tz)
        Tm = [[A(j00) * A(V[k]) + A(j02) * A(V[8 + k]) for k in range(3)],
              [A(j11) * A(V[4 + k]) + A(j12) * A(V[8 + k]) for k in range(3)]]
        P = [[sum(Tm[a][r].v * S[3 * r + c].v * Tm[b][c].v for r in range(3) for c in range(3))
              for b in range(2)] for a in range(2)]
        P00, P01, P11 = P[0][0], P[0][1], P[1][1]
        det = P00 * P11 - P01 * P01
        det2 = det * det
        ga, gb, gc = g[2], g[3], g[4]
        dP00 = (ga * A(-P11 * P11 / det2) + gb * A(P01 * P11 / det2) +
                gc * (A(1.0 / det) - A(P00 * P11 / det2)))
        dP11 = (ga * (A(1.0 / det) - A(P11 * P00 / det2)) + gb * A(P01 * P00 / det2) +
                gc * A(-P00 * P00 / det2))
        dP01 = (ga * A(2.0 * P01 * P11 / det2) + gb * (A(-1.0 / det) - A(2.0 * P01 * P01 / det2)) +
                gc * A(2.0 * P00 * P01 / det2))
        dS = [dP00 * Tm[0][r] * Tm[0][c] + dP01 * Tm[0][r] * Tm[1][c] + dP11 * Tm[1][r] * Tm[1][c]
              for r in range(3) for c in range(3)]
        dT = [[None] * 3, [None] * 3]
        for r in range(3):
            ST0 = S[3 * r] * Tm[0][0] + S[3 * r + 1] * Tm[0][1] + S[3 * r + 2] * Tm[0][2]
            ST1 = S[3 * r] * Tm[1][0] + S[3 * r + 1] * Tm[1][1] + S[3 * r + 2] * Tm[1][2]
            dT[0][r] = A(2.0) * dP00 * ST0 + dP01 * ST1
            dT[1][r] = dP01 * ST0 + A(2.0) * dP11 * ST1
        dj00 = dT[0][0] * A(V[0]) + dT[0][1] * A(V[1]) + dT[0][2] * A(V[2])
        dj02 = dT[0][0] * A(V[8]) + dT[0][1] * A(V[9]) + dT[0][2] * A(V[10])
        dj11 = dT[1][0] * A(V[4]) + dT[1][1] * A(V[5]) + dT[1][2] * A(V[6])
        dj12 = dT[1][0] * A(V[8]) + dT[1][1] * A(V[9]) + dT[1][2] * A(V[10])
        tz2, tz3 = tz * tz, tz * tz * tz
        dt0 = g[0] * A(fx / tz) + dj02 * A(-fx / tz2)
        dt1 = g[1] * A(fy / tz) + dj12 * A(-fy / tz2)
        dt2 = (g[0] * A(-fx * tx / tz2) + g[1] * A(-fy * ty / tz2) + dj00 * A(-fx / tz2) +
               dj02 * A(2.0 * fx * tx / tz3) + dj11 * A(-fy / tz2) + dj12 * A(2.0 * fy * ty / tz3))
        dm = [A(V[c]) * dt0 + A(V[4 + c]) * dt1 + A(V[8 + c]) * dt2 for c in range(3)]
        dM = [sum(((dS[3 * r + j] + dS[3 * j + r]) * M[3 * j + k] for j in range(3)),
                  A(0.0, 0.0)) for r in range(3) for k in range(3)]
        ds = [sum((dM[3 * r + k] * A(R[3 * r + k]) for r in range(3)), A(0.0, 0.0))
              for k in range(3)]
        dR = [dM[3 * r + k] * A(s[k]) for r in range(3) for k in range(3)]
        co = {  # dR[e] -> (dw, dx, dy, dz) coefficients of R(w, x, y, z)
            0: (0, 0, -4 * y, -4 * z), 1: (-2 * z, 2 * y, 2 * x, -2 * w),
            2: (2 * y, 2 * z, 2 * w, 2 * x), 3: (2 * z, 2 * y, 2 * x, 2 * w),
            4: (0, -4 * x, 0, -4 * z), 5: (-2 * x, -2 * w, 2 * z, 2 * y),
            6: (-2 * y, 2 * z, -2 * w, 2 * x), 7: (2 * x, 2 * w, 2 * z, 2 * y),
            8: (0, -4 * x, -4 * y, 0)}
        dqh = [sum((dR[e] * A(co[e][k]) for e in range(9) if co[e][k] != 0), A(0.0, 0.0))
               for k in range(4)]
        qh = [A(w), A(x), A(y), A(z)]
        dotq = qh[0] * dqh[0] + qh[1] * dqh[1] + qh[2] * dqh[2] + qh[3] * dqh[3]
        dq = [(dqh[k] - qh[k] * dotq) / A(qn) for k in range(4)]
        d = m - cw
        ln = math.sqrt(d[0] * d[0] + d[1] * d[1] + d[2] * d[2])
        dhat = d / ln
        Y, dY = oracle.sh_basis(dhat[None])
        gcol = g[6:9]
        dsh = [[A(Y[0, k]) * gcol[ch] for ch in range(3)] for k in range(K)]
        gd = [A(0.0, 0.0)] * 3
        for k in range(K):
            proj = gcol[0] * A(float(sc.sh[i, k, 0])) + gcol[1] * A(float(sc.sh[i, k, 1])) + \
                gcol[2] * A(float(sc.sh[i, k, 2]))
            gd = [gd[j] + proj * A(dY[0, k, j]) for j in range(3)]
        dotd = A(dhat[0]) * gd[0] + A(dhat[1]) * gd[1] + A(dhat[2]) * gd[2]
        dm = [dm[j] + (gd[j] - A(dhat[j]) * dotd) / A(ln) for j in range(3)]
        put("means", i, dm)
        put("scales", i, ds)
        put("quats", i, dq)
        put("opacities", i, [g[5]])
        put("sh", i, dsh)
    return out


@pytest.mark.parametrize("seed,deg", [(6, 3), (7, 1)])
def test_parameter_magnitudes_equal_the_abs_arithmetic_restatement(seed, deg):
    sc, cam, w, v = _scene(seed, 30, 40, 32, deg)
    V = ss.look_at(np.array([0.4, -0.3, -0.6]), np.array([0.0, 0.0, 4.0]), up=(0.1, -1.0, 0.0))
    # a rotated camera (every view-matrix entry matters) with fx != fy
    cam = ss.Camera(V, 48.0, 40.0, 0.47 * 40, 0.55 * 32, 40, 32, 0.2)
    proj = oracle.project(sc, cam)
    b = oracle.bin_sort(cam, proj)
    r = oracle.blend_bwd_bounds(cam, proj, b, w, v)
    assert np.count_nonzero(proj.tiles_touched) > 10
    pg = oracle.project_bwd(sc, cam, proj, r.grad2d)
    pm = oracle.project_bwd_magnitude(sc, cam, proj, r.gabs)
    ref = _chain_restated(sc, cam, proj.tiles_touched, r.grad2d, r.gabs)
    for k, (val, mag) in ref.items():
        np.testing.assert_allclose(getattr(pg, k), val, rtol=1e-9, atol=1e-12, err_msg=k)
        np.testing.assert_allclose(getattr(pm, k), mag, rtol=1e-9, atol=1e-12, err_msg=k)
        assert np.all(mag >= np.abs(val) * (1 - 1e-12)), k


def test_parallel_tile_parts_equal_the_single_call():
    """The oracle's calls run over disjoint tile sets on host threads give the single
    call's results: the same pixels, and per-Gaussian sums up to their order."""
    sc, cam, w, v = _scene(8, 400, 120, 90, 2)
    proj = oracle.project(sc, cam)
    b = oracle.bin_sort(cam, proj)
    parts = oracle.tile_parts(b, 5)
    sel = np.zeros(len(b.counts), int)
    for p in parts:
        sel += p.sel
    assert np.all(sel == 1)  # disjoint, and together every tile
    im, par = oracle.blend(cam, proj, b), oracle.blend_parallel(cam, proj, b, workers=5)
    for f in ("img", "T", "n_contrib", "last_idx", "flags", "tile_mask"):
        np.testing.assert_array_equal(getattr(par, f), getattr(im, f), err_msg=f)
    r = oracle.blend_bwd_bounds(cam, proj, b, w, v)
    rp = oracle.blend_bwd_parallel(cam, proj, b, w, v, workers=5)
    for f in ("grad2d", "gabs", "grho", "galt"):
        a, c = getattr(rp, f), getattr(r, f)
        np.testing.assert_allclose(a, c, rtol=1e-9, atol=1e-12 * np.abs(c).max(), err_msg=f)


def _stop_band_scene(o2):
    """Three large splats centred on pixel (12, 12)'s centre, front to back: a clamped
    one (alpha 0.99), one of opacity o2 (its alpha at the centre pixel is o2) and one
    behind them, so that the stop test runs once more after the second."""
    W = H = 25  # cx = cy = 12.5, the centre of pixel (12, 12)
    cam = ss.pinhole(np.eye(4), 40.0, W, H)
    means = np.array([[0, 0, 2.0], [0, 0, 2.5], [0, 0, 3.0]], np.float32)
    scales = np.full((3, 3), 1.0, np.float32)
    quats = np.tile(np.array([1, 0, 0, 0], np.float32), (3, 1))
    opac = np.array([0.9999, o2, 0.5], np.float32)
    sh = np.full((3, 1, 3), 1.0, np.float32)
    return ss.Scene(means, scales, quats, opac, sh, 0), cam


def _stop_band_ratio(o2):
    """|T - 1e-4| / (err T) after the two front splats at the centre pixel, with the
    band's definition: err = sum over the blended splats of 2^-17 alpha / (1 - alpha)
    (the renderer's alpha error, amplified by the transmittance update) + 2^-23 (two
    fp32 roundings of the update)."""
    T, err = 1.0, 0.0
    for a in (ALPHA_MAX, float(np.float32(o2))):
        T *= 1.0 - a
        err += E_ALPHA * a / (1.0 - a) + 2.0 ** -23
    return abs(T - T_MIN) / (err * T)


def test_stop_band_is_twice_the_accumulated_error():
    """A stop decision is a near-tie when the transmittance lies within 2 err T of 1e-4:
    at the centre pixel, T at 1.5 err T from 1e-4 is flagged, at 3 err T it is not
    (the second splat's opacity sets T; neither alpha is near the clamp's band)."""
    # opacities whose T after two splats sits at the wanted multiple of err T
    def o2_for(ratio):
        lo, hi = 0.9899, 0.98998  # T falls as o2 rises, and the ratio with it
        for _ in range(60):
            mid = 0.5 * (lo + hi)
            if _stop_band_ratio(mid) > ratio:
                lo = mid
            else:
                hi = mid
        return np.float32(0.5 * (lo + hi))
    for ratio, flagged in ((1.5, True), (3.0, False)):
        o2 = o2_for(ratio)
        r = _stop_band_ratio(o2)
        assert abs(r - ratio) < 0.05 and abs(float(o2) - ALPHA_MAX) > 2 * E_ALPHA * ALPHA_MAX
        sc, cam = _stop_band_scene(o2)
        proj = oracle.project(sc, cam)
        im = oracle.blend(cam, proj, oracle.bin_sort(cam, proj))
        assert im.n_contrib[12, 12] == 3  # T stays above 1e-4: the third splat blends
        assert bool(im.flags[12, 12] & oracle.FLAG_STOP_TIE) == flagged, (ratio, r)


def test_clamp_band_is_twice_the_alpha_error():
    """An alpha is a clamp near-tie when o exp(-q/2) lies within 2 E_alpha 0.99 of 0.99
    (E_alpha = 2^-17, the renderer's alpha error): one splat centred on pixel (12, 12)'s
    centre (q = 0 there, so its raw alpha is its opacity) at 1.5 and at 3 band units
    above and below 0.99 is flagged, and not flagged."""
    unit = E_ALPHA * ALPHA_MAX
    for ratio, flagged in ((1.5, True), (-1.5, True), (3.0, False), (-3.0, False)):
        o = np.float32(ALPHA_MAX + ratio * unit)
        assert abs(abs(float(o) - ALPHA_MAX) / unit - abs(ratio)) < 0.05
        W = H = 25
        cam = ss.pinhole(np.eye(4), 40.0, W, H)
        sc = ss.Scene(np.array([[0, 0, 2.0]], np.float32), np.full((1, 3), 1.0, np.float32),
                      np.array([[1, 0, 0, 0]], np.float32), np.array([o], np.float32),
                      np.full((1, 1, 3), 1.0, np.float32), 0)
        proj = oracle.project(sc, cam)
        im = oracle.blend(cam, proj, oracle.bin_sort(cam, proj))
        assert im.n_contrib[12, 12] == 1
        assert bool(im.flags[12, 12] & oracle.FLAG_CLAMP_TIE) == flagged, ratio
