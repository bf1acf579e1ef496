"""Pins of the oracle's training step after the chain rule: the gradients of the raw
parameters (log-scales, opacity logits) and one Adam step (Kingma & Ba), against closed
forms, the step-size bound of the Adam paper (Sec. 2.1) and central finite differences of
the oracle's own forward."""

import copy

import numpy as np
import pytest

import oracle
import synthetic_scenes as ss

B1, B2, EPS = 0.9, 0.999, 1e-15


def _arrays(rng, n):
    p = rng.standard_normal(n)
    return p, np.zeros(n), np.zeros(n)


def test_first_step_is_a_normalised_sign_step():
    # t = 1 with zero moments: the bias-corrected moments are g and g^2 exactly
    rng = np.random.default_rng(0)
    p, m, v = _arrays(rng, 1000)
    g = rng.standard_normal(1000) * 10.0 ** rng.uniform(-6, 3, 1000)
    g[:10] = 0.0
    p0 = p.copy()
    oracle.adam_step(p, m, v, g, 0.01, B1, B2, EPS, 1)
    np.testing.assert_allclose(m, (1 - B1) * g, rtol=1e-14)
    np.testing.assert_allclose(v, (1 - B2) * g * g, rtol=1e-14)
    np.testing.assert_allclose(p, p0 - 0.01 * g / (np.abs(g) + EPS), rtol=1e-12, atol=1e-15)
    np.testing.assert_array_equal(p[:10], p0[:10])


def test_constant_gradient_moves_linearly():
    # a constant gradient keeps the bias-corrected moments at g and g^2 for every t
    rng = np.random.default_rng(1)
    p, m, v = _arrays(rng, 200)
    g = rng.standard_normal(200)
    p0 = p.copy()
    for t in range(1, 51):
        oracle.adam_step(p, m, v, g, 1e-3, B1, B2, EPS, t)
    np.testing.assert_allclose(p, p0 - 50 * 1e-3 * np.sign(g), rtol=0, atol=1e-11)


@pytest.mark.parametrize("b1,b2", [(0.9, 0.999), (0.5, 0.99), (0.99, 0.9)])
def test_step_size_bound(b1, b2):
    # Cauchy-Schwarz on m_t = (1 - b1) sum_k b1^k g_{t-k} against v_t = (1 - b2) sum_k
    # b2^k g_{t-k}^2 bounds the step of any gradient sequence (eps = 0):
    # |step_t| <= lr (1 - b1) / (1 - b1^t) sqrt((1 - b2^t) / (1 - b2) sum_{k<t} (b1^2 / b2)^k);
    # for b1^2 < b2 and large t this tends to the Adam paper's (1 - b1) / sqrt(1 - b2 - ...)
    rng = np.random.default_rng(2)
    n, lr = 500, 0.1
    p, m, v = _arrays(rng, n)
    for t in range(1, 40):
        g = rng.standard_normal(n) * 10.0 ** rng.uniform(-3, 3, n)
        g[rng.random(n) < 0.2] = 0.0
        before = p.copy()
        oracle.adam_step(p, m, v, g, lr, b1, b2, 0.0, t)
        S = sum((b1 * b1 / b2) ** k for k in range(t))
        bound = lr * (1 - b1) / (1 - b1 ** t) * np.sqrt((1 - b2 ** t) / (1 - b2) * S)
        step = np.abs(p - before)
        ok = np.isfinite(step)  # 0 / 0 where every gradient so far was zero
        assert np.all(step[ok] <= bound * (1 + 1e-9)), (t, step[ok].max(), bound)
        assert np.sum(ok) > n // 2


def _scene(seed, n=25, W=64, H=48):
    rng = np.random.default_rng(seed)
    sc, _ = ss.random_scene(rng, n, W, H, sh_degree=1, log_scale=(-2.3, 0.4), logit_std=1.5)
    eye = np.array([0.3, -0.2, -0.5])
    V = ss.look_at(eye, np.array([0.0, 0.0, 4.0]), up=(0.05, -1.0, 0.0))
    cam = ss.pinhole(V, 64.0, W, H)
    return sc, cam, rng.standard_normal((H, W, 3)), rng.standard_normal((H, W))


@pytest.mark.parametrize("seed", [0, 1])
def test_raw_gradients_match_finite_differences(seed):
    # loss as a function of the raw parameters: scales = exp(log s), opacity = sigmoid(logit)
    sc, cam, w, v = _scene(seed)
    L0, r0, g2, pg = oracle.loss_and_grads(sc, cam, w, v, "f64")
    dls, dlo = oracle.raw_grads(sc.scales, sc.opacities, pg)
    live = np.nonzero(np.abs(g2).sum(1) > 0)[0]
    assert len(live) >= 8
    log_s = np.log(sc.scales.astype(np.float64))
    o = sc.opacities.astype(np.float64).reshape(-1)
    logit = np.log(o / (1 - o))

    def loss(s2):
        r = oracle.render(s2, cam, None, "f64")
        same = (np.array_equal(r.image.n_contrib, r0.image.n_contrib) and
                np.array_equal(r.image.last_idx, r0.image.last_idx))
        return float((w * r.image.img).sum() + (v * r.image.T).sum()), same

    checked = 0
    for g in live[:8]:
        for j in range(3):
            h = 1e-3
            vals = []
            for d in (+h, -h):
                s2 = copy.deepcopy(sc)
                s2.scales[g, j] = np.float32(np.exp(log_s[g, j] + d))
                vals.append((loss(s2), float(np.log(np.float64(s2.scales[g, j])))))
            (Lh, sh_), xh = vals[0]
            (Ll, sl_), xl = vals[1]
            if sh_ and sl_:
                fd = (Lh - Ll) / (xh - xl)
                assert abs(dls[g, j] - fd) <= 1e-6 + 1e-4 * abs(fd), ("log-scale", g, j, dls[g, j], fd)
                checked += 1
        vals = []
        for d in (+1e-3, -1e-3):
            s2 = copy.deepcopy(sc)
            s2.opacities.reshape(-1)[g] = np.float32(1 / (1 + np.exp(-(logit[g] + d))))
            o2 = np.float64(s2.opacities.reshape(-1)[g])
            vals.append((loss(s2), float(np.log(o2 / (1 - o2)))))
        (Lh, sh_), xh = vals[0]
        (Ll, sl_), xl = vals[1]
        if sh_ and sl_:
            fd = (Lh - Ll) / (xh - xl)
            assert abs(dlo[g] - fd) <= 1e-6 + 1e-4 * abs(fd), ("logit", g, dlo[g], fd)
            checked += 1
    assert checked >= 20
