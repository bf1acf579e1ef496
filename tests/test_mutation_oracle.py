"""Mutation check of the oracle's pins: each entry below plants one plausible mistake
in a copy of ``oracle/gs_oracle.c`` (a flipped sign, a dropped term or factor, a wrong
or transposed index, a reversed order) and runs the oracle's own pin tests
(``tests/test_oracle_*.py``) against that copy.  A mutant that no pin rejects marks
arithmetic the pins do not fix.

The table is checked against the source on every CPU run (each planted text must occur
exactly once, so the table follows the source as it changes), and a sample of eight
mutants, one from each part of the oracle, runs every time.  Running the whole table
takes about five minutes on eight cores and is opt-in:

    GS_ORACLE_MUTANTS=1 python -m pytest tests/test_mutation_oracle.py -n 8 -q

Everything happens on the CPU, in a temporary copy: the repository's oracle is never
modified.
"""

import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "gs_oracle.c")

# (name, text in gs_oracle.c, replacement)
MUTANTS = [
    # ---- projection: camera transform, rotation, Jacobian, Eq. 1, conic, tau, extents
    ("camera_row_index", "dreal ty = ((V[4] * mx + V[5] * my) + V[6] * mz) + V[7];",
     "dreal ty = ((V[4] * mx + V[5] * my) + V[2] * mz) + V[7];"),
    ("rotation_sign_r01", "R[1] = 2 * (x * y - w * z);", "R[1] = 2 * (x * y + w * z);"),
    ("rotation_index_r12", "R[5] = 2 * (y * z - w * x);", "R[5] = 2 * (y * z - w * y);"),
    ("jacobian_sign_j02", "dreal j02 = -(j00 * u);", "dreal j02 = (j00 * u);"),
    ("jacobian_row_t1", "T1[k] = j11 * V[4 + k] + j12 * V[8 + k];",
     "T1[k] = j11 * V[4 + k] + j12 * V[4 + k];"),
    ("scale_index_n1", "T1[2] * R[6 + k]) * s3[k];", "T1[2] * R[6 + k]) * s3[(k + 1) % 3];"),
    ("determinant_scale_e0", "dreal e0 = (s1 * s2) * c0;", "dreal e0 = (s0 * s2) * c0;"),
    ("conic_sign_b", "dreal b = -(P01 / det);", "dreal b = (P01 / det);"),
    ("cholesky_sign_l12", "dreal l12 = -((P01 / P11) * l11);", "dreal l12 = ((P01 / P11) * l11);"),
    ("tau_factor_two", "double t = 2.0 * log(CUTOFF_INV * (double)o);",
     "double t = log(CUTOFF_INV * (double)o);"),
    ("extent_rx_uses_p11", "dreal rx = sqrt(tau * P00);", "dreal rx = sqrt(tau * P11);"),
    ("near_plane_ignored", "if (!(tz > cam->znear) ||", "if (!(tz > 0) ||"),
    ("principal_point_swapped", "dreal mux = cam->fx * u + cam->cx;",
     "dreal mux = cam->fx * u + cam->cy;"),
    ("jacobian_focal_swapped", "dreal j11 = cam->fy / tz;", "dreal j11 = cam->fx / tz;"),
    ("alpha_cutoff_256", "#define CUTOFF_INV 255.0", "#define CUTOFF_INV 256.0"),
    # ---- exact row spans and tile rows
    ("span_boundary_sign", "return (sqrt(disc) - s->l12 * dy) / s->l11;",
     "return (sqrt(disc) + s->l12 * dy) / s->l11;"),
    ("span_vertex_sign", "return -((sqrt(s->tau) * s->l12) / (s->l22 * h));",
     "return ((sqrt(s->tau) * s->l12) / (s->l22 * h));"),
    ("span_left_not_mirrored", "dmax(dyv, -hi), -lo)", "dmax(dyv, lo), hi)"),
    ("span_last_column_dropped", "dreal f1 = floor((Xhi - (dreal)0.5) * (dreal)0.0625) + 1;",
     "dreal f1 = floor((Xhi - (dreal)0.5) * (dreal)0.0625);"),
    ("span_first_column_late", "dreal f0 = ceil((Xlo - (dreal)15.5) * (dreal)0.0625);",
     "dreal f0 = ceil((Xlo - (dreal)0.5) * (dreal)0.0625);"),
    ("span_right_edge_unclipped", "if (Xlo > (dreal)cam->W - (dreal)0.5 || Xhi < (dreal)0.5) return 0;",
     "if (Xlo > (dreal)cam->W + (dreal)0.5 || Xhi < (dreal)0.5) return 0;"),
    ("radius_rounded_down", "radii[2 * i] = to_int_clamped(ceil(s.rx), 0, RADIUS_MAX);",
     "radii[2 * i] = to_int_clamped(floor(s.rx), 0, RADIUS_MAX);"),
    ("rows_first_row_late", "ceil(((s->muy - ryp) - (dreal)15.5)",
     "ceil(((s->muy - ryp) - (dreal)0.5)"),
    ("rows_last_row_dropped", "dreal f1 = floor(((s->muy + ryp) - (dreal)0.5) * (dreal)0.0625) + 1;",
     "dreal f1 = floor(((s->muy + ryp) - (dreal)0.5) * (dreal)0.0625);"),
    ("tile_band_not_clipped",
     "dmin((dreal)(16 * ty) + (dreal)15.5, (dreal)cam->H - (dreal)0.5)",
     "((dreal)(16 * ty) + (dreal)15.5)"),
    # ---- spherical harmonics and the view direction
    ("sh_sign_y1", "Y[1] = k1 * y;", "Y[1] = -(k1 * y);"),
    ("sh_sign_y6", "Y[6] = k2b * (3 * z * z - 1);", "Y[6] = -(k2b * (3 * z * z - 1));"),
    ("sh_sign_y10", "Y[10] = k3b * x * y * z;", "Y[10] = -(k3b * x * y * z);"),
    ("sh_sign_y2", "Y[2] = k1 * z;", "Y[2] = -k1 * z;"),
    ("sh_sign_y15", "Y[15] = k3a * x * (x * x - 3 * y * y);",
     "Y[15] = -k3a * x * (x * x - 3 * y * y);"),
    ("sh_y12_constant", "Y[12] = k3d * z * (5 * z * z - 3);", "Y[12] = k3d * z * (5 * z * z - 1);"),
    ("sh_gradient_y9", "dY[9][1] = k3a * (3 * x * x - 3 * y * y);",
     "dY[9][1] = k3a * (3 * x * x - y * y);"),
    ("sh_normalisation_k2b", "double k2b = sqrt(5.0 / (16 * PI));",
     "double k2b = sqrt(5.0 / (4 * PI));"),
    ("camera_centre_sign", "cw[j] = -((double)viewmat[0 + j] * viewmat[3]",
     "cw[j] = ((double)viewmat[0 + j] * viewmat[3]"),
    ("camera_centre_transposed",
     "(double)viewmat[4 + j] * viewmat[7] +", "(double)viewmat[1 + 4 * j] * viewmat[7] +"),
    ("colour_channel_dropped", "acc += Y[k] * (double)sh[(i * K + k) * 3 + ch];",
     "acc += Y[k] * (double)sh[(i * K + k) * 3];"),
]
MUTANTS += [
    # ---- binning, (tile, depth, id) order, ranges, LPT order
    ("sort_depth_reversed", "if (x->depth_d != y->depth_d) return x->depth_d < y->depth_d ? -1 : 1;",
     "if (x->depth_d != y->depth_d) return x->depth_d > y->depth_d ? -1 : 1;"),
    ("sort_tie_break_reversed", "if (x->id != y->id) return x->id < y->id ? -1 : 1;",
     "if (x->id != y->id) return x->id > y->id ? -1 : 1;"),
    ("lpt_ascending", "if (x->count != y->count) return x->count > y->count ? -1 : 1;",
     "if (x->count != y->count) return x->count < y->count ? -1 : 1;"),
    ("lpt_tie_break_reversed", "return x->tile < y->tile ? -1 : (x->tile > y->tile);",
     "return x->tile > y->tile ? -1 : (x->tile < y->tile);"),
    ("range_end_off_by_one", "        ranges[2 * t + 1] = acc;\n",
     "        ranges[2 * t + 1] = acc - (acc > 0);\n"),
    # ---- forward blend
    ("pixel_centre_dropped", "dreal dx = ((dreal)px + (dreal)0.5) - mux;",
     "dreal dx = ((dreal)px) - mux;"),
    ("quadratic_form_term", "dreal q = fma(u1, u1, u2 * u2);", "dreal q = fma(u1, u1, u2);"),
    ("termination_threshold", "if (!forced && T < T_MIN) break;",
     "if (!forced && T < 1e-3) break;"),
    ("stop_exclusive", "blended_t* e = &(*list)[nb++];",
     "if (!forced && T * (1.0 - alpha) < T_MIN) break;\n        blended_t* e = &(*list)[nb++];"),
    ("stop_band_halved", "int near = fabs(T - T_MIN) <= 2.0 * err * T;",
     "int near = fabs(T - T_MIN) <= 0.5 * err * T;"),
    ("clamp_band_halved", "int near = fabs(araw - ALPHA_MAX) <= 2.0 * E_ALPHA * ALPHA_MAX;",
     "int near = fabs(araw - ALPHA_MAX) <= 0.5 * E_ALPHA * ALPHA_MAX;"),
    ("clamp_band_doubled", "int near = fabs(araw - ALPHA_MAX) <= 2.0 * E_ALPHA * ALPHA_MAX;",
     "int near = fabs(araw - ALPHA_MAX) <= 4.0 * E_ALPHA * ALPHA_MAX;"),
    ("stop_band_doubled", "int near = fabs(T - T_MIN) <= 2.0 * err * T;",
     "int near = fabs(T - T_MIN) <= 4.0 * err * T;"),
    ("stop_band_alpha_weight", "err += E_ALPHA * alpha / (1.0 - alpha) + 1.1920928955078125e-07;",
     "err += E_ALPHA * alpha + 1.1920928955078125e-07;"),
    ("alpha_clamp_dropped", "return c ? ALPHA_MAX : araw;", "return araw;"),
    ("colour_without_transmittance",
     "C[ch] += rgb[3 * (int64_t)e->g + ch] * e->alpha * e->T;",
     "C[ch] += rgb[3 * (int64_t)e->g + ch] * e->alpha;"),
    ("transmittance_update", "T *= (1.0 - alpha);\n        err +=",
     "T *= (1.0 - alpha) * (1.0 - alpha);\n        err +="),
    ("contributors_not_counted", "n_contrib[p] = (int32_t)nb;", "n_contrib[p] = 0;"),
    ("last_index_relative", "last_idx[p] = nb ? (int32_t)list[nb - 1].k : -1;",
     "last_idx[p] = nb ? (int32_t)(list[nb - 1].k - ranges[2 * t]) : -1;"),
    # ---- backward of the blend: the nine screen-space derivatives
    ("dalpha_behind_sign", "double dalpha = e->T * cG - bG / (1.0 - e->alpha) -",
     "double dalpha = e->T * cG + bG / (1.0 - e->alpha) -"),
    ("dalpha_final_t_factor", " gT * Tfin / (1.0 - e->alpha);", " gT * Tfin;"),
    ("behind_without_transmittance", "behind[ch] += col[ch] * w;",
     "behind[ch] += col[ch] * e->alpha;"),
    ("dq_alpha_dropped", "double dq = -0.5 * e->alpha * dalpha;", "double dq = -0.5 * dalpha;"),
    ("dopacity_factor", "tm[5] = exp(-0.5 * e->q) * dalpha;", "tm[5] = e->alpha * dalpha;"),
    ("dmux_conic_index", "tm[0] = -2.0 * (a * e->dx + b * e->dy) * dq;",
     "tm[0] = -2.0 * (a * e->dx + cc * e->dy) * dq;"),
    ("dmuy_sign", "tm[1] = -2.0 * (b * e->dx + cc * e->dy) * dq;",
     "tm[1] = 2.0 * (b * e->dx + cc * e->dy) * dq;"),
    ("dconic_b_factor", "tm[3] = 2.0 * e->dx * e->dy * dq;", "tm[3] = e->dx * e->dy * dq;"),
    ("conic_c_from_factor", "cc = l12 * l12 + l22 * l22;", "cc = l22 * l22;"),
    ("clamp_gate_dropped", "if (!e->clamped) {", "if (1) {"),
    ("dcolour_factor", "tm[6 + ch] = w * G[ch];", "tm[6 + ch] = e->alpha * G[ch];"),
    # ---- magnitudes and error bounds that set the GPU gradient tolerance
    ("magnitude_behind_doubled", "behind_mag += cG_mag * w;", "behind_mag += 2.0 * cG_mag * w;"),
    ("magnitude_conic_b_factor", "mg[3] = 2.0 * fabs(e->dx * e->dy) * dq_mag;",
     "mg[3] = 4.0 * fabs(e->dx * e->dy) * dq_mag;"),
    ("error_bound_base_dropped", "double eps = 2.0 * E_ALPHA + 32.0 * U32;", "double eps = 0.0;"),
    ("error_bound_rounding_term", "eps += 2.0 * (E_ALPHA * list[j].alpha / (1.0 - list[j].alpha) + 8.0 * U32);",
     "eps += 2.0 * (E_ALPHA * list[j].alpha / (1.0 - list[j].alpha) + U32);"),
    ("error_bound_alpha_weight",
     "eps += 2.0 * (E_ALPHA * list[j].alpha / (1.0 - list[j].alpha) + 8.0 * U32);",
     "eps += 2.0 * (E_ALPHA / (1.0 - list[j].alpha) + 8.0 * U32);"),
    ("clamp_spread_not_a_difference",
     "galt[9 * g + r] += fabs(term2[9 * j + r] - term[9 * j + r]);",
     "galt[9 * g + r] += fabs(term2[9 * j + r]) + fabs(term[9 * j + r]);"),
    ("forced_stop_not_checked", "if (T < T_MIN && !near) fl |= 4;", "if (0) fl |= 4;"),
    ("param_magnitude_quat_doubled", "double dw = 2 * (az * dR[1] + ay * dR[2]",
     "double dw = 4 * (az * dR[1] + ay * dR[2]"),
    ("param_magnitude_view_dir", "dm[j] += (gd[j] + ad[j] * dotd) / len;",
     "dm[j] += (2.0 * gd[j] + ad[j] * dotd) / len;"),
    # ---- projection backward (chain rule)
    ("dt_gmy_focal_swapped", "dt[1] += gmy * fy / tz;", "dt[1] += gmy * fx / tz;"),
    ("dj12_focal_swapped", "dt[1] += dj12 * (-fy / tz2);", "dt[1] += dj12 * (-fx / tz2);"),
    ("dP11_first_term_sign", "double dP11 = ga * (1.0 / det - P11 * P00 / det2)",
     "double dP11 = ga * (-1.0 / det - P11 * P00 / det2)"),
    ("magnitude_dt1_focal_swapped", "dt[1] = gmy * fabs(fy) / tz + dj12 * fabs(fy) / tz2;",
     "dt[1] = gmy * fabs(fx) / tz + dj12 * fabs(fy) / tz2;"),
    ("dP00_sign", "double dP00 = ga * (-P11 * P11 / det2) + gb * (P01 * P11 / det2) +",
     "double dP00 = ga * (-P11 * P11 / det2) + gb * (-P01 * P11 / det2) +"),
    ("dP01_sign", "gb * (-1.0 / det - 2.0 * P01 * P01 / det2)",
     "gb * (1.0 / det - 2.0 * P01 * P01 / det2)"),
    ("dT_operand",
     "S[3 * r + 2] * Tm[1][2];\n            dT[0][r] = 2.0 * dP00 * ST0 + dP01 * ST1;",
     "S[3 * r + 2] * Tm[1][2];\n            dT[0][r] = 2.0 * dP00 * ST0 + dP01 * ST0;"),
    ("dJ_index", "dj02 += dT[0][k] * V[8 + k];", "dj02 += dT[0][k] * V[k];"),
    ("dt_second_derivative", "dt[2] += dj02 * (2.0 * fx * tx / tz3);",
     "dt[2] += dj02 * (fx * tx / tz3);"),
    ("dt_mean_sign", "dt[2] += gmx * (-fx * tx / tz2);", "dt[2] += gmx * (fx * tx / tz2);"),
    ("dmeans_transposed", "dm[c] += V[c] * dt[0] + V[4 + c] * dt[1] + V[8 + c] * dt[2];",
     "dm[c] += V[4 * c] * dt[0] + V[4 * c + 1] * dt[1] + V[4 * c + 2] * dt[2];"),
    ("dM_not_symmetrised", "acc += (dS[3 * r + j] + dS[3 * j + r]) * M[3 * j + k];",
     "acc += 2.0 * dS[3 * r + j] * M[3 * j + k];"),
    ("dscale_transposed", "ds[k] += dM[3 * r + k] * R[3 * r + k];",
     "ds[k] += dM[3 * r + k] * R[3 * k + r];"),
    ("dquat_sign_w", "dw += dR[1] * (-2 * z);", "dw += dR[1] * (2 * z);"),
    ("dquat_sign_x", "dx += dR[5] * (-2 * w);", "dx += dR[5] * (2 * w);"),
    ("dquat_sign_y_r6", "dw += dR[6] * (-2 * y);  dx += dR[6] * (2 * z);  dy += dR[6] * (-2 * w);",
     "dw += dR[6] * (-2 * y);  dx += dR[6] * (2 * z);  dy += dR[6] * (2 * w);"),
    ("drot_scale_index", "dR[3 * r + k] = dM[3 * r + k] * s[k];", "dR[3 * r + k] = dM[3 * r + k] * s[r];"),
    ("dquat_not_projected", "dq[k] = (dqh[k] - qh[k] * dotq) / qn;", "dq[k] = dqh[k] / qn;"),
    ("dquat_norm_dropped", "dq[k] = (dqh[k] - qh[k] * dotq) / qn;", "dq[k] = (dqh[k] - qh[k] * dotq);"),
    ("dopacity_scaled", "dopac[i] = g2[5];", "dopac[i] = 0.5 * g2[5];"),
    ("dsh_channel", "dshi[3 * k + ch] = Y[k] * gcol[ch];", "dshi[3 * k + ch] = Y[k] * gcol[0];"),
    ("dmeans_sh_not_projected", "dm[j] += (gd[j] - dhat[j] * dotd) / len;",
     "dm[j] += gd[j] / len;"),
    # ---- chunking policy (Eq. 6)
    ("policy_chunk_cost_k", "double cost = fmax(total + lambda * (double)h * k, Kl) + beta * Kl;",
     "double cost = fmax(total + lambda * (double)h, Kl) + beta * Kl;"),
    ("policy_beta_term_dropped", "double cost = fmax(total + lambda * (double)h * k, Kl) + beta * Kl;",
     "double cost = fmax(total + lambda * (double)h * k, Kl);"),
    ("policy_k16_missing", "const int ks[4] = {2, 4, 8, 16};", "const int ks[4] = {2, 4, 8, 8};"),
    ("policy_tie_takes_later", "if (cost < best) {", "if (cost <= best) {"),
    ("policy_margin_dropped", "!(best <= (1.0 - eps) * base)", "!(best <= base)"),
    ("policy_next_tile_ignored", "double l = fmax(N1 / k, next);", "double l = N1 / k;"),
    ("policy_next_index", "double next = h < nt ? (double)counts_desc[h] : 0.0;",
     "double next = h < nt ? (double)counts_desc[h - 1] : 0.0;"),
    # ---- raw gradients and Adam
    ("adam_eps_inside_sqrt", "p[i] -= lr * (m[i] / c1) / (sqrt(v[i] / c2) + eps);",
     "p[i] -= lr * (m[i] / c1) / sqrt(v[i] / c2 + eps);"),
    ("loss_weights_swapped", "out[0] = (1.0 - lambda) * out[1] + lambda * (1.0 - out[2]);",
     "out[0] = lambda * out[1] + (1.0 - lambda) * (1.0 - out[2]);"),
    ("loss_grad_weights_swapped", "dL_dx[i] = (1.0 - lambda) * inv * sg - lambda * inv * ds;",
     "dL_dx[i] = lambda * inv * sg - (1.0 - lambda) * inv * ds;"),
    ("adam_first_moment_weight", "m[i] = b1 * m[i] + (1.0 - b1) * g[i];",
     "m[i] = b1 * m[i] + g[i];"),
    ("adam_bias_power", "double c1 = 1.0 - pow(b1, (double)t), c2 = 1.0 - pow(b2, (double)t);",
     "double c1 = 1.0 - pow(b1, (double)t), c2 = 1.0 - pow(b2, (double)(t + 1));"),
    ("adam_second_moment", "v[i] = b2 * v[i] + (1.0 - b2) * g[i] * g[i];",
     "v[i] = b2 * v[i] + (1.0 - b2) * g[i];"),
    ("adam_bias_correction", "p[i] -= lr * (m[i] / c1) / (sqrt(v[i] / c2) + eps);",
     "p[i] -= lr * m[i] / (sqrt(v[i]) + eps);"),
    ("raw_logit_factor", "dlogits[i] = opac[i] * (1.0 - opac[i]) * dopac[i];",
     "dlogits[i] = opac[i] * dopac[i];"),
    ("raw_log_scale_factor", "dlog_scales[i] = scales[i] * dscales[i];",
     "dlog_scales[i] = dscales[i];"),
    # ---- L1 + SSIM loss
    ("ssim_variance_term", "double vx = exx - mx * mx,", "double vx = exx,"),
    ("ssim_dmu_sign", "dmu[i] = (2.0 * my * (A2 - A1) - 2.0 * mx * s * (B2 - B1)) / D;",
     "dmu[i] = (2.0 * my * (A2 - A1) + 2.0 * mx * s * (B2 - B1)) / D;"),
    ("ssim_dxx_sign", "dxx[i] = -s / B2;", "dxx[i] = s / B2;"),
    ("ssim_chain_factor", "ds += w * (dmu[q] + 2.0 * xv * dxx[q] + yv * dxy[q]);",
     "ds += w * (dmu[q] + xv * dxx[q] + yv * dxy[q]);"),
    ("ssim_window_width", "g[k + SSIM_R] = exp(-(double)(k * k) / (2.0 * sigma * sigma));",
     "g[k + SSIM_R] = exp(-(double)(k * k) / (sigma * sigma));"),
    ("ssim_covariance_term", "cov = exy - mx * my", "cov = exy"),
    ("ssim_c2_as_c1", "A2 = 2.0 * cov + c2", "A2 = 2.0 * cov + c1"),
    ("ssim_dxy_factor", "dxy[i] = 2.0 * A1 / D;", "dxy[i] = A1 / D;"),
    ("loss_mean_over_pixels", "double inv = 1.0 / (double)(3 * np);", "double inv = 1.0 / (double)np;"),
    ("l1_sign", "double sg = xv > yv ? 1.0 : (xv < yv ? -1.0 : 0.0);", "double sg = 1.0;"),
]


def _source() -> str:
    with open(SRC) as f:
        return f.read()


def test_mutant_table_matches_the_source():
    src = _source()
    names = [m[0] for m in MUTANTS]
    assert len(set(names)) == len(names)
    for name, old, new in MUTANTS:
        assert src.count(old) == 1, f"{name}: planted text must occur exactly once"
        assert old != new, name


def _copy_tree(dst: str) -> None:
    os.makedirs(os.path.join(dst, "oracle"))
    for f in ("__init__.py", "definitional.py", "gs_oracle.c"):
        shutil.copy(os.path.join(ROOT, "oracle", f), os.path.join(dst, "oracle", f))
    for f in ("synthetic_scenes.py", "pytest.ini"):
        shutil.copy(os.path.join(ROOT, f), os.path.join(dst, f))
    os.makedirs(os.path.join(dst, "tests"))
    for f in os.listdir(os.path.join(ROOT, "tests")):
        if f == "conftest.py" or (f.startswith("test_oracle_") and f.endswith(".py")):
            shutil.copy(os.path.join(ROOT, "tests", f), os.path.join(dst, "tests", f))
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), os.path.join(dst, "tests", "golden"))


# One mutant from each part of the oracle, run on every CPU run (a few seconds each);
# the whole table stays opt-in.
SAMPLE = ("camera_row_index", "span_boundary_sign", "transmittance_update",
          "contributors_not_counted", "dalpha_behind_sign", "dconic_b_factor",
          "lpt_ascending", "adam_bias_correction")


@pytest.mark.parametrize("name", SAMPLE)
def test_sampled_mutants_fail_a_pin(tmp_path, name):
    (old, new), = [(o, n) for m, o, n in MUTANTS if m == name]
    _run_mutant(tmp_path, name, old, new)


@pytest.mark.skipif(os.environ.get("GS_ORACLE_MUTANTS") != "1",
                    reason="mutation run is opt-in: GS_ORACLE_MUTANTS=1")
@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_every_mutant_fails_a_pin(tmp_path, name, old, new):
    _run_mutant(tmp_path, name, old, new)


def _run_mutant(tmp_path, name, old, new):
    dst = str(tmp_path / "copy")
    _copy_tree(dst)
    path = os.path.join(dst, "oracle", "gs_oracle.c")
    with open(path) as f:
        src = f.read()
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    env = dict(os.environ, PYTHONPATH=dst, PYTHONDONTWRITEBYTECODE="1")
    env.pop("GS_ORACLE_MUTANTS", None)
    # the mutant must build: a planted mistake, not a syntax error
    b = subprocess.run([sys.executable, "-c", "import oracle; oracle.build(force=True)"],
                       cwd=dst, env=env, capture_output=True, text=True, timeout=300)
    assert b.returncode == 0, f"{name} does not compile:\n{b.stderr[-2000:]}"
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:xdist", "tests"],
                       cwd=dst, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 1, (
        f"mutant {name} survived every pin (pytest exit {r.returncode}):\n{r.stdout[-1500:]}")
