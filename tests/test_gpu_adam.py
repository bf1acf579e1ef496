"""The chain rule fused with one Adam step (gs_project_bwd_adam) against the oracle: the
oracle's parameter gradients carried to the raw parameters (log-scales, opacity logits)
and its Adam step, from the same parameters and moments.  The gradients are compared
through the first moment, m_new = b1 m + (1 - b1) g, at the gradient tolerances (1e-4
relative, or the derived fp32 bound where that is larger; gpu_util)."""

import numpy as np
import pytest

import oracle
import synthetic_scenes as ss
from gpu_util import (GRAD_ATOL, GRAD_RTOL, assert_grads_tiered, grad2d_bounds, param_bounds,
                      t)

pytestmark = pytest.mark.gpu

B1, B2, EPS, STEP = 0.9, 0.999, 1e-15, 3
LR = dict(lr_means=1.6e-4, lr_scales=5e-3, lr_quats=1e-3, lr_opacities=5e-2, lr_sh0=2.5e-3,
          lr_shN=1.25e-4)


def _raw_scene(seed, W, H, n, deg):
    rng = np.random.default_rng(seed)
    sc, cam = ss.random_scene(rng, n, W, H, sh_degree=deg, log_scale=(-2.8, 0.8), logit_std=2.5)
    log_s = np.log(sc.scales.astype(np.float64)).astype(np.float32)
    o = sc.opacities.astype(np.float64).reshape(-1)
    logit = np.log(o / (1 - o)).astype(np.float32)
    # the activated values both sides see: exp and sigmoid of the fp32 raw values
    sc.scales = np.exp(log_s.astype(np.float64)).astype(np.float32)
    sc.opacities = (1 / (1 + np.exp(-logit.astype(np.float64)))).astype(np.float32).reshape(
        sc.opacities.shape)
    return sc, cam, log_s, logit, rng


@pytest.mark.parametrize("seed,W,H,n,deg", [(0, 37, 53, 300, 0), (5, 80, 60, 700, 1),
                                            (3, 64, 40, 600, 2), (1, 150, 97, 900, 3)])
def test_fused_adam_step_matches_oracle(seed, W, H, n, deg):
    import torch

    import differentiable_gaussian_splatting_gb300 as gs

    sc, cam, log_s, logit, rng = _raw_scene(seed, W, H, n, deg)
    ref = oracle.render(sc, cam)
    wm = rng.standard_normal((H, W, 3)).astype(np.float32)
    # GPU: forward on the activated values, the raster backward, then the fused step
    r = gs.Rasterizer(cam, sc.sh_degree, sc.n)
    r.forward(t(sc.means), t(sc.scales), t(sc.quats), t(sc.opacities), t(sc.sh))
    r.backward(t(wm))
    # the oracle takes the GPU's stop where the oracle flags it as a fp32 near-tie
    tie = (ref.image.flags & oracle.FLAG_STOP_TIE) != 0
    stop_last = np.where(tie, r.last_idx.cpu().numpy(), oracle.RULE).astype(np.int32)
    raw = [sc.means.astype(np.float32), log_s, sc.quats.astype(np.float32), logit,
           sc.sh.astype(np.float32)]
    m0 = [rng.standard_normal(a.shape).astype(np.float32) * 1e-3 for a in raw]
    v0 = [(rng.random(a.shape) * 1e-5).astype(np.float32) for a in raw]
    P = [t(a.copy()) for a in raw]
    M = [t(a.copy()) for a in m0]
    Vv = [t(a.copy()) for a in v0]
    s = gs.AdamSettings(**LR, beta1=B1, beta2=B2, eps=EPS, step=STEP)
    act_s = torch.full((sc.n, 3), float("nan"), device="cuda")
    act_o = torch.full((sc.n,), float("nan"), device="cuda")
    gs.gs_project_bwd_adam(r.cam, sc.n, sc.sh_degree, *P, r.tiles_touched, r.grad2d, r.touched,
                           M, Vv, s, scales_out=act_s, opacities_out=act_o)
    torch.cuda.synchronize()
    # oracle: gradients of the activated parameters, carried to the raw ones, then Adam
    rb, bound = grad2d_bounds(cam, ref.proj, ref.binning, wm, None, stop_last)
    pg = oracle.project_bwd(sc, cam, ref.proj, rb.grad2d)
    pb, pm = param_bounds(sc, cam, ref.proj, bound, rb.gabs)
    dls, dlo = oracle.raw_grads(sc.scales, sc.opacities, pg)
    s_abs = np.abs(sc.scales.astype(np.float64))
    o = sc.opacities.astype(np.float64).reshape(-1)
    grads = [pg.means, dls, pg.quats, dlo, pg.sh]
    mags = [pm.means, s_abs * pm.scales, pm.quats, o * (1 - o) * np.abs(pm.opacities.reshape(-1)),
            pm.sh]
    # the raw gradients are exact scalings of the activated ones: so are their bounds
    bounds = [pb["means"], s_abs * pb["scales"], pb["quats"],
              o * (1 - o) * pb["opacities"].reshape(-1), pb["sh"]]
    lrs = [LR["lr_means"], LR["lr_scales"], LR["lr_quats"], LR["lr_opacities"]]
    names = ["means", "log_scales", "quats", "logits", "sh"]
    for k in range(5):
        g = np.asarray(grads[k], np.float64).reshape(raw[k].shape)
        p_ref = raw[k].astype(np.float64).copy()
        m_ref = m0[k].astype(np.float64).copy()
        v_ref = v0[k].astype(np.float64).copy()
        if k < 4:
            oracle.adam_step(p_ref.reshape(-1), m_ref.reshape(-1), v_ref.reshape(-1),
                             g.reshape(-1), lrs[k], B1, B2, EPS, STEP)
            lr_el = np.full(raw[k].shape, lrs[k])
        else:  # SH: band 0 (the first three values of a row) and bands 1-3 take two rates
            flat_p, flat_m, flat_v = (a.reshape(sc.n, -1) for a in (p_ref, m_ref, v_ref))
            gf = g.reshape(sc.n, -1)
            for cols, lr in ((slice(0, 3), LR["lr_sh0"]), (slice(3, None), LR["lr_shN"])):
                pp, mm, vv = (np.ascontiguousarray(a[:, cols]) for a in (flat_p, flat_m, flat_v))
                oracle.adam_step(pp.reshape(-1), mm.reshape(-1), vv.reshape(-1),
                                 np.ascontiguousarray(gf[:, cols]).reshape(-1), lr, B1, B2, EPS, STEP)
                flat_p[:, cols], flat_m[:, cols], flat_v[:, cols] = pp, mm, vv
            lr_el = np.zeros((sc.n, gf.shape[1]))
            lr_el[:, :3], lr_el[:, 3:] = LR["lr_sh0"], LR["lr_shN"]
            lr_el = lr_el.reshape(raw[k].shape)
        p_gpu = P[k].cpu().numpy().astype(np.float64)
        m_gpu = M[k].cpu().numpy().astype(np.float64)
        v_gpu = Vv[k].cpu().numpy().astype(np.float64)
        # the gradient the step used, read back from the first moment
        g_gpu = (m_gpu - B1 * m0[k].astype(np.float64)) / (1 - B1)
        assert_grads_tiered(g_gpu, g, "adam:" + names[k], np.asarray(bounds[k]).reshape(g.shape),
                            np.asarray(mags[k]).reshape(g.shape), rtol=GRAD_RTOL,
                            atol=GRAD_ATOL + 4e-7 * np.abs(m0[k]).max())
        np.testing.assert_allclose(v_gpu, v_ref, rtol=1e-3, atol=1e-12, err_msg=names[k])
        # the step itself: within a thousandth of its rate, plus the parameter's rounding
        lim = 1e-3 * lr_el + 2e-7 * np.maximum(1.0, np.abs(p_ref))
        bad = np.abs(p_gpu - p_ref) > lim
        assert not bad.any(), (names[k], int(bad.sum()), float((np.abs(p_gpu - p_ref) / lim).max()))
        if k == 1:  # the next forward's scales: exp of the updated log-scales
            np.testing.assert_allclose(act_s.cpu().numpy(), np.exp(p_gpu), rtol=1e-6)
            np.testing.assert_allclose(act_s.cpu().numpy(), np.exp(p_ref),
                                       rtol=2e-6 + float(lim.max()))
        if k == 3:  # and opacities: sigmoid of the updated logits
            sg = 1 / (1 + np.exp(-p_gpu))
            np.testing.assert_allclose(act_o.cpu().numpy(), sg, rtol=1e-6, atol=1e-7)
