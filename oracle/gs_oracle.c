/*
 * gs_oracle.c -- plain, slow CPU oracle for the differentiable 3D Gaussian
 * splatting rasterizer (forward and backward).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link or call
 * this file; only the tests, the smoke check and the CPU-baseline leg of the
 * benchmark use it.  It shares no code, header, table or helper with the CUDA
 * library.
 *
 * What it computes, and where it comes from:
 *   - projection of a 3D Gaussian to a 2D splat: "Mitigating SM-Level Load
 *     Imbalance in 3D Gaussian Splatting on GPUs" (Ryu & Yoo), Sec. 2.1, Eq. 1
 *     (Sigma' = J W Sigma W^T J^T);
 *   - per-pixel opacity alpha = o exp(-q/2) (same paper, Eq. 2) with the
 *     opacity-aware support q <= 2 ln(255 o) of "What the 3DGS Literature Left
 *     on the Table" (Kopanas), Step 1 (b);
 *   - front-to-back blending C = sum c_i alpha_i T_i with the 1e-4 stop
 *     (Ryu & Yoo, Eq. 3 and the text after it);
 *   - exact row-span tile binning (Kopanas, Step 1 (b)) and the
 *     (tile, depth) ordering of the pair list (Kopanas, Step 1 (d));
 *   - view-dependent colour c = sum_k Y_k(d) s_k over 16 real spherical
 *     harmonics (Kopanas, Step 3);
 *   - the nine screen-space derivatives per splat (Kopanas, Step 1 (a)) and
 *     the chain rule back to means, scales, quaternions, opacities and SH
 *     coefficients (calculus; pinned by finite differences in the tests);
 *   - the per-frame chunking cost model (Ryu & Yoo, Sec. 4.4, Eq. 6);
 *   - the steps either side of the path in a training step (the pages' Metal
 *     port, "perf: rasterizer and pipeline optimizations", Breakdown and
 *     Queue): the raw-parameter gradients and one Adam step, and the
 *     L1 + SSIM photometric loss with its gradient.
 *
 * Precision.  The pages fix fp32 for the rasterizer and require the quadratic
 * to be evaluated with explicit round-to-nearest operations so that every
 * hit decision is reproducible (Kopanas, Step 5).  This oracle therefore
 * evaluates the chain that *decides integers* (projected centre, conic,
 * threshold tau, radii, row spans, the per-pixel hit test q <= tau) in the
 * type `dreal`, which is float in the default build and double in the
 * ORACLE_F64 build used only for finite-difference checks.  Every operation
 * of that chain is written in one fixed order; the file is compiled with
 * -ffp-contract=off so that no multiply-add is fused unless fma() is called.
 * Everything that does not decide an integer (colour, alpha, transmittance,
 * all gradients) is computed in double.
 *
 * tau is the fp32 rounding of the exact 2 ln(255 o), computed in double.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <tgmath.h>

#ifdef ORACLE_F64
typedef double dreal;
#define DREAL_IS_DOUBLE 1
#else
typedef float dreal;
#define DREAL_IS_DOUBLE 0
#endif

#define TILE 16
#define T_MIN 1e-4
#define ALPHA_MAX 0.99
#define CUTOFF_INV 255.0 /* alpha cutoff 1/255 */
#define RADIUS_MAX (1 << 30) /* radii are reported clamped to this */
#define REC 16               /* doubles per exported splat record */

/* ------------------------------------------------------------------------ */
/* Camera                                                                    */
/* ------------------------------------------------------------------------ */

typedef struct {
    dreal V[12];              /* rows 0..2 of the 4x4 world->camera matrix */
    dreal fx, fy, cx, cy;
    int W, H;
    dreal znear;
    int ntx, nty;
} camera_t;

static void make_camera(camera_t* cam, const float* viewmat, const float* intr, int W, int H,
                        float znear) {
    for (int i = 0; i < 12; ++i) cam->V[i] = (dreal)viewmat[i];
    cam->fx = (dreal)intr[0];
    cam->fy = (dreal)intr[1];
    cam->cx = (dreal)intr[2];
    cam->cy = (dreal)intr[3];
    cam->W = W;
    cam->H = H;
    cam->znear = (dreal)znear;
    cam->ntx = (W + TILE - 1) / TILE;
    cam->nty = (H + TILE - 1) / TILE;
}

/* ------------------------------------------------------------------------ */
/* Projection (Ryu & Yoo Eq. 1), fp32 fixed order                            */
/* ------------------------------------------------------------------------ */

typedef struct {
    int visible;
    dreal tx, ty, tz;
    dreal mux, muy;
    dreal P00, P01, P11; /* Sigma' */
    dreal a, b, c;       /* conic = inverse of Sigma'; q = a dx^2 + 2 b dx dy + c dy^2 */
    dreal l11, l12, l22; /* conic = L^T L, L = [[l11, l12], [0, l22]] */
    dreal tau;           /* support threshold 2 ln(255 o) */
    dreal rx, ry;        /* half extents of the support ellipse */
} splat_t;

static int finite_d(dreal x) { return isfinite(x); }

/* tau = 2 ln(255 o); in the fp32 build it is the correctly rounded fp32 value
 * of the double result. */
static dreal support_tau(float o) {
    double t = 2.0 * log(CUTOFF_INV * (double)o);
    return (dreal)t;
}

static void project_one(const camera_t* cam, const float* m3, const float* s3, const float* q4,
                        float opac, splat_t* sp) {
    const dreal* V = cam->V;
    memset(sp, 0, sizeof(*sp));
    dreal mx = m3[0], my = m3[1], mz = m3[2];
    /* camera-space position t = W m + t_v */
    dreal tx = ((V[0] * mx + V[1] * my) + V[2] * mz) + V[3];
    dreal ty = ((V[4] * mx + V[5] * my) + V[6] * mz) + V[7];
    dreal tz = ((V[8] * mx + V[9] * my) + V[10] * mz) + V[11];
    sp->tx = tx;
    sp->ty = ty;
    sp->tz = tz;
    if (!(tz > cam->znear) || !finite_d(tx) || !finite_d(ty) || !finite_d(tz)) return;

    /* normalised quaternion (w, x, y, z) */
    dreal qw = q4[0], qx = q4[1], qy = q4[2], qz = q4[3];
    dreal n2 = ((qw * qw + qx * qx) + qy * qy) + qz * qz;
    if (!(n2 > 0) || !finite_d(n2)) return;
    dreal nr = sqrt(n2);
    dreal w = qw / nr, x = qx / nr, y = qy / nr, z = qz / nr;
    dreal R[9];
    R[0] = 1 - 2 * (y * y + z * z);
    R[1] = 2 * (x * y - w * z);
    R[2] = 2 * (x * z + w * y);
    R[3] = 2 * (x * y + w * z);
    R[4] = 1 - 2 * (x * x + z * z);
    R[5] = 2 * (y * z - w * x);
    R[6] = 2 * (x * z - w * y);
    R[7] = 2 * (y * z + w * x);
    R[8] = 1 - 2 * (x * x + y * y);

    dreal s0 = s3[0], s1 = s3[1], s2 = s3[2];

    /* pinhole projection and its Jacobian J evaluated at t */
    dreal u = tx / tz, v = ty / tz;
    dreal mux = cam->fx * u + cam->cx;
    dreal muy = cam->fy * v + cam->cy;
    dreal j00 = cam->fx / tz;
    dreal j11 = cam->fy / tz;
    dreal j02 = -(j00 * u);
    dreal j12 = -(j11 * v);

    /* T = J W (2x3), W = rotation block of the view matrix */
    dreal T0[3], T1[3];
    for (int k = 0; k < 3; ++k) {
        T0[k] = j00 * V[k] + j02 * V[8 + k];
        T1[k] = j11 * V[4 + k] + j12 * V[8 + k];
    }
    /* Sigma' = J W R S S R^T W^T J^T = N N^T with N = (T R) diag(s):
     * n_ik = (T_i . R_col_k) s_k (Eq. 1 with Sigma = R S S^T R^T) */
    dreal n0[3], n1[3];
    for (int k = 0; k < 3; ++k) {
        n0[k] = ((T0[0] * R[k] + T0[1] * R[3 + k]) + T0[2] * R[6 + k]) * s3[k];
        n1[k] = ((T1[0] * R[k] + T1[1] * R[3 + k]) + T1[2] * R[6 + k]) * s3[k];
    }
    dreal P00 = (n0[0] * n0[0] + n0[1] * n0[1]) + n0[2] * n0[2];
    dreal P01 = (n0[0] * n1[0] + n0[1] * n1[1]) + n0[2] * n1[2];
    dreal P11 = (n1[0] * n1[0] + n1[1] * n1[1]) + n1[2] * n1[2];
    /* det Sigma' = |n0 x n1|^2 (Lagrange) and n0 x n1 = s0 s1 s2 S^-1 R^T (T0 x T1):
     * a sum of squares, free of the cancellation of P00 P11 - P01^2 */
    dreal w0 = T0[1] * T1[2] - T0[2] * T1[1];
    dreal w1 = T0[2] * T1[0] - T0[0] * T1[2];
    dreal w2 = T0[0] * T1[1] - T0[1] * T1[0];
    dreal c0 = (R[0] * w0 + R[3] * w1) + R[6] * w2;
    dreal c1 = (R[1] * w0 + R[4] * w1) + R[7] * w2;
    dreal c2 = (R[2] * w0 + R[5] * w1) + R[8] * w2;
    dreal e0 = (s1 * s2) * c0;
    dreal e1 = (s0 * s2) * c1;
    dreal e2 = (s0 * s1) * c2;
    dreal det = (e0 * e0 + e1 * e1) + e2 * e2;
    if (!(det > 0) || !(P00 > 0) || !(P11 > 0) || !finite_d(det)) return;
    dreal a = P11 / det;
    dreal b = -(P01 / det);
    dreal c = P00 / det;
    /* Cholesky factor of the conic, taken from Sigma' without cancellation:
     * l22 = 1/sqrt(P11), l11 = sqrt(P11/det), l12 = -(P01/P11) l11 */
    dreal l22 = 1 / sqrt(P11);
    dreal l11 = sqrt(P11 / det);
    dreal l12 = -((P01 / P11) * l11);

    dreal tau = support_tau(opac);
    if (!(tau > 0)) return;
    dreal rx = sqrt(tau * P00);
    dreal ry = sqrt(tau * P11);
    if (!finite_d(mux) || !finite_d(muy) || !finite_d(a) || !finite_d(b) || !finite_d(c) ||
        !finite_d(l11) || !finite_d(l12) || !finite_d(l22) || !finite_d(rx) || !finite_d(ry))
        return;

    sp->mux = mux;
    sp->muy = muy;
    sp->P00 = P00;
    sp->P01 = P01;
    sp->P11 = P11;
    sp->a = a;
    sp->b = b;
    sp->c = c;
    sp->l11 = l11;
    sp->l12 = l12;
    sp->l22 = l22;
    sp->tau = tau;
    sp->rx = rx;
    sp->ry = ry;
    sp->visible = 1;
}

/* ------------------------------------------------------------------------ */
/* Exact row spans (Kopanas, Step 1 (b))                                     */
/* ------------------------------------------------------------------------ */
/*
 * A tile's region is the closed hull of its pixel centres (x + 0.5, y + 0.5)
 * clipped to the image.  For each tile row, the support ellipse q(d) <= tau is
 * intersected with the row's band and the covered tile columns [tx0, tx1)
 * follow in closed form.  With q = (l11 dx + l12 dy)^2 + (l22 dy)^2 the right
 * boundary is x_r(dy) = (sqrt(tau - (l22 dy)^2) - l12 dy) / l11, concave in
 * dy with its vertex at dy = -sqrt(tau) l12 / (l22 h), h = sqrt(l12^2 +
 * l22^2); the left boundary is x_l(dy) = -x_r(-dy).  x_r is evaluated at the
 * band point nearest its vertex, clamped to |dy| <= ry.
 *
 * The fp32 evaluation is widened just enough that every pixel whose fp32 hit
 * test passes lies in an emitted tile (u = 2^-24):
 *   - the discriminant tau - (l22 dy)^2 carries an absolute error of about
 *     4 u tau, which near the tips (discriminant -> 0) moves the boundary by
 *     about sqrt(u) r; it is widened by 2^-21 tau = 8 u tau before the root,
 *     so the widening is about sqrt(8 u tau) / l11 at a tip and u-sized
 *     elsewhere;
 *   - the remaining roundings of the span and of the hit test's quadratic
 *     are a few u of the extent: padx = 2^-8 px + rx 2^-20 (and pady alike
 *     for the band), the 2^-8 px covering the rounding of mu' + x_r in
 *     pixel coordinates up to the 32768-pixel image limit.
 */

static dreal xr_at(const splat_t* s, dreal dy) {
    dreal t = s->l22 * dy;
    dreal disc = s->tau - t * t;
    if (!(disc > 0)) disc = 0;
    disc = disc + s->tau * (dreal)4.76837158203125e-07; /* + 2^-21 tau */
    return (sqrt(disc) - s->l12 * dy) / s->l11;
}

static dreal vertex_dy(const splat_t* s) {
    dreal h = sqrt(s->l12 * s->l12 + s->l22 * s->l22);
    return -((sqrt(s->tau) * s->l12) / (s->l22 * h));
}

static dreal dmin(dreal x, dreal y) { return x < y ? x : y; }
static dreal dmax(dreal x, dreal y) { return x > y ? x : y; }

/* Clamp a float to [lo, hi] before converting it to int. */
static int to_int_clamped(dreal f, int lo, int hi) {
    if (!(f >= (dreal)lo)) return lo;
    if (f > (dreal)hi) return hi;
    return (int)f;
}

/* rows [*ty0, *ty1) that the padded ellipse may cover */
static void row_range(const camera_t* cam, const splat_t* s, int* ty0, int* ty1) {
    const dreal pad_unit = (dreal)0.00390625;        /* 2^-8 */
    const dreal pad_scale = (dreal)9.5367431640625e-07; /* 2^-20 */
    dreal pady = pad_unit + s->ry * pad_scale;
    dreal ryp = s->ry + pady;
    dreal f0 = ceil(((s->muy - ryp) - (dreal)15.5) * (dreal)0.0625);
    dreal f1 = floor(((s->muy + ryp) - (dreal)0.5) * (dreal)0.0625) + 1;
    *ty0 = to_int_clamped(f0, 0, cam->nty);
    *ty1 = to_int_clamped(f1, 0, cam->nty);
}

/* span of tile columns [*tx0, *tx1) in row ty; returns 0 when empty */
static int row_span(const camera_t* cam, const splat_t* s, int ty, int* tx0, int* tx1) {
    const dreal pad_unit = (dreal)0.00390625;        /* 2^-8 */
    const dreal pad_scale = (dreal)9.5367431640625e-07; /* 2^-20 */
    dreal padx = pad_unit + s->rx * pad_scale;
    dreal pady = pad_unit + s->ry * pad_scale;
    dreal ryp = s->ry + pady;
    dreal y0 = (dreal)(16 * ty) + (dreal)0.5;
    dreal y1 = dmin((dreal)(16 * ty) + (dreal)15.5, (dreal)cam->H - (dreal)0.5);
    dreal lo = dmax(y0 - s->muy, -ryp);
    dreal hi = dmin(y1 - s->muy, ryp);
    if (!(lo <= hi)) return 0;
    dreal dyv = vertex_dy(s);
    /* evaluate x_r only on the ellipse itself: |dy| <= ry */
    dreal dh = dmin(dmax(dmin(dmax(dyv, lo), hi), -s->ry), s->ry);
    dreal dl = dmin(dmax(dmin(dmax(dyv, -hi), -lo), -s->ry), s->ry);
    dreal xhi = xr_at(s, dh) + padx;
    dreal xlo_neg = xr_at(s, dl) + padx;
    dreal Xhi = s->mux + xhi;
    dreal Xlo = s->mux - xlo_neg;
    if (Xlo > (dreal)cam->W - (dreal)0.5 || Xhi < (dreal)0.5) return 0;
    dreal f0 = ceil((Xlo - (dreal)15.5) * (dreal)0.0625);
    dreal f1 = floor((Xhi - (dreal)0.5) * (dreal)0.0625) + 1;
    *tx0 = to_int_clamped(f0, 0, cam->ntx);
    *tx1 = to_int_clamped(f1, 0, cam->ntx);
    return *tx0 < *tx1;
}

static int64_t count_tiles(const camera_t* cam, const splat_t* s) {
    int ty0, ty1, tx0, tx1;
    int64_t n = 0;
    row_range(cam, s, &ty0, &ty1);
    for (int ty = ty0; ty < ty1; ++ty)
        if (row_span(cam, s, ty, &tx0, &tx1)) n += tx1 - tx0;
    return n;
}

/* ------------------------------------------------------------------------ */
/* Real spherical harmonics, degree <= 3 (Kopanas, Step 3)                   */
/* ------------------------------------------------------------------------ */
/*
 * Orthonormal real basis in the order l = 0..3, m = -l..l, without the
 * Condon-Shortley phase: Y_{l,m<0} ~ sin(|m| phi), Y_{l,m>0} ~ cos(m phi).
 * Written as polynomials of the unit direction (x, y, z); Y[k] and its
 * Cartesian gradient dY[k][0..2].
 */
static void sh_basis(const double d[3], double Y[16], double dY[16][3]) {
    const double PI = 3.14159265358979323846;
    double x = d[0], y = d[1], z = d[2];
    double k0 = sqrt(1.0 / (4 * PI));
    double k1 = sqrt(3.0 / (4 * PI));
    double k2a = sqrt(15.0 / (4 * PI));
    double k2b = sqrt(5.0 / (16 * PI));
    double k2c = sqrt(15.0 / (16 * PI));
    double k3a = sqrt(35.0 / (32 * PI));
    double k3b = sqrt(105.0 / (4 * PI));
    double k3c = sqrt(21.0 / (32 * PI));
    double k3d = sqrt(7.0 / (16 * PI));
    double k3e = sqrt(105.0 / (16 * PI));
    memset(dY, 0, sizeof(double) * 48);
    Y[0] = k0;
    Y[1] = k1 * y;  dY[1][1] = k1;
    Y[2] = k1 * z;  dY[2][2] = k1;
    Y[3] = k1 * x;  dY[3][0] = k1;
    Y[4] = k2a * x * y;  dY[4][0] = k2a * y;  dY[4][1] = k2a * x;
    Y[5] = k2a * y * z;  dY[5][1] = k2a * z;  dY[5][2] = k2a * y;
    Y[6] = k2b * (3 * z * z - 1);  dY[6][2] = k2b * 6 * z;
    Y[7] = k2a * x * z;  dY[7][0] = k2a * z;  dY[7][2] = k2a * x;
    Y[8] = k2c * (x * x - y * y);  dY[8][0] = k2c * 2 * x;  dY[8][1] = -k2c * 2 * y;
    Y[9] = k3a * y * (3 * x * x - y * y);
    dY[9][0] = k3a * 6 * x * y;  dY[9][1] = k3a * (3 * x * x - 3 * y * y);
    Y[10] = k3b * x * y * z;
    dY[10][0] = k3b * y * z;  dY[10][1] = k3b * x * z;  dY[10][2] = k3b * x * y;
    Y[11] = k3c * y * (5 * z * z - 1);
    dY[11][1] = k3c * (5 * z * z - 1);  dY[11][2] = k3c * 10 * y * z;
    Y[12] = k3d * z * (5 * z * z - 3);
    dY[12][2] = k3d * (15 * z * z - 3);
    Y[13] = k3c * x * (5 * z * z - 1);
    dY[13][0] = k3c * (5 * z * z - 1);  dY[13][2] = k3c * 10 * x * z;
    Y[14] = k3e * z * (x * x - y * y);
    dY[14][0] = k3e * 2 * x * z;  dY[14][1] = -k3e * 2 * y * z;  dY[14][2] = k3e * (x * x - y * y);
    Y[15] = k3a * x * (x * x - 3 * y * y);
    dY[15][0] = k3a * (3 * x * x - 3 * y * y);  dY[15][1] = -k3a * 6 * x * y;
}

/* camera centre in world space, c_w = -W^T t_v */
static void camera_centre(const float* viewmat, double cw[3]) {
    for (int j = 0; j < 3; ++j)
        cw[j] = -((double)viewmat[0 + j] * viewmat[3] + (double)viewmat[4 + j] * viewmat[7] +
                  (double)viewmat[8 + j] * viewmat[11]);
}

static void view_dir(const float* m3, const double cw[3], double dhat[3], double* len) {
    double d[3] = {(double)m3[0] - cw[0], (double)m3[1] - cw[1], (double)m3[2] - cw[2]};
    double l = sqrt(d[0] * d[0] + d[1] * d[1] + d[2] * d[2]);
    *len = l;
    for (int j = 0; j < 3; ++j) dhat[j] = l > 0 ? d[j] / l : 0.0;
}

/* ------------------------------------------------------------------------ */
/* Exported: SH basis (for pinning against a library routine)                */
/* ------------------------------------------------------------------------ */
void ora_sh_basis(int64_t n, const double* dirs, double* Y, double* dY) {
    for (int64_t i = 0; i < n; ++i) {
        double y[16], dy[16][3];
        sh_basis(dirs + 3 * i, y, dy);
        memcpy(Y + 16 * i, y, sizeof(y));
        if (dY) memcpy(dY + 48 * i, dy, sizeof(dy));
    }
}

int ora_is_f64(void) { return DREAL_IS_DOUBLE; }

/* ------------------------------------------------------------------------ */
/* Exported: forward projection                                              */
/* ------------------------------------------------------------------------ */
/*
 * Outputs per Gaussian i (culled Gaussians get zeros and tiles_touched 0):
 *   splat[i][0..15] = mux, muy, a, b, c, opacity, tau, depth t_z, P00, P01, P11, rx, ry,
 *                     l11, l12, l22
 *   rgb[i][0..2]    = sum_k Y_k(d) s_k (double; no offset, no clamp)
 *   radii[i][0..1]  = ceil(rx), ceil(ry)
 *   tiles_touched[i]
 */
void ora_project(int64_t n, int sh_degree, const float* viewmat, const float* intr, int W, int H,
                 float znear, const float* means, const float* scales, const float* quats,
                 const float* opac, const float* sh, double* splat, double* rgb, int32_t* radii,
                 int32_t* tiles_touched) {
    camera_t cam;
    make_camera(&cam, viewmat, intr, W, H, znear);
    double cw[3];
    camera_centre(viewmat, cw);
    int K = (sh_degree + 1) * (sh_degree + 1);
    for (int64_t i = 0; i < n; ++i) {
        splat_t s;
        project_one(&cam, means + 3 * i, scales + 3 * i, quats + 4 * i, opac[i], &s);
        int64_t nt = s.visible ? count_tiles(&cam, &s) : 0;
        double* o = splat + REC * i;
        memset(o, 0, REC * sizeof(double));
        rgb[3 * i] = rgb[3 * i + 1] = rgb[3 * i + 2] = 0;
        radii[2 * i] = radii[2 * i + 1] = 0;
        tiles_touched[i] = 0;
        if (!s.visible || nt == 0) continue;
        o[0] = s.mux;  o[1] = s.muy;
        o[2] = s.a;  o[3] = s.b;  o[4] = s.c;
        o[5] = opac[i];  o[6] = s.tau;  o[7] = s.tz;
        o[8] = s.P00;  o[9] = s.P01;  o[10] = s.P11;
        o[11] = s.rx;  o[12] = s.ry;
        o[13] = s.l11;  o[14] = s.l12;  o[15] = s.l22;
        radii[2 * i] = to_int_clamped(ceil(s.rx), 0, RADIUS_MAX);
        radii[2 * i + 1] = to_int_clamped(ceil(s.ry), 0, RADIUS_MAX);
        tiles_touched[i] = (int32_t)nt;
        double dhat[3], len, Y[16], dY[16][3];
        view_dir(means + 3 * i, cw, dhat, &len);
        sh_basis(dhat, Y, dY);
        for (int ch = 0; ch < 3; ++ch) {
            double acc = 0;
            for (int k = 0; k < K; ++k) acc += Y[k] * (double)sh[(i * K + k) * 3 + ch];
            rgb[3 * i + ch] = acc;
        }
    }
}

/* Rebuild a splat_t from the exported record (values are exact in dreal). */
static void splat_from_record(const double* o, splat_t* s) {
    memset(s, 0, sizeof(*s));
    s->mux = (dreal)o[0];
    s->muy = (dreal)o[1];
    s->a = (dreal)o[2];
    s->b = (dreal)o[3];
    s->c = (dreal)o[4];
    s->tau = (dreal)o[6];
    s->tz = (dreal)o[7];
    s->P00 = (dreal)o[8];
    s->P01 = (dreal)o[9];
    s->P11 = (dreal)o[10];
    s->rx = (dreal)o[11];
    s->ry = (dreal)o[12];
    s->l11 = (dreal)o[13];
    s->l12 = (dreal)o[14];
    s->l22 = (dreal)o[15];
    s->visible = 1;
}

/* Exported: the tiles of one splat, row by row (for brute-force pins). */
int64_t ora_splat_tiles(const float* viewmat, const float* intr, int W, int H, float znear,
                        const double* record, int32_t* tiles, int64_t cap) {
    camera_t cam;
    make_camera(&cam, viewmat, intr, W, H, znear);
    splat_t s;
    splat_from_record(record, &s);
    int ty0, ty1, tx0, tx1;
    int64_t n = 0;
    row_range(&cam, &s, &ty0, &ty1);
    for (int ty = ty0; ty < ty1; ++ty)
        if (row_span(&cam, &s, ty, &tx0, &tx1))
            for (int tx = tx0; tx < tx1; ++tx) {
                if (n < cap) tiles[n] = ty * cam.ntx + tx;
                ++n;
            }
    return n;
}

/* ------------------------------------------------------------------------ */
/* Exported: binning and sort (Kopanas, Step 1 (b), (d))                     */
/* ------------------------------------------------------------------------ */
/*
 * counts[t]       : number of (tile, Gaussian) pairs of tile t (all tiles)
 * ranges[t]       : [start, end) of tile t in the full sorted pair list,
 *                   i.e. the exclusive prefix sum of counts
 * lpt_order[j]    : tiles by descending count, ties by ascending tile id
 *                   (Ryu & Yoo, Sec. 4.1, "LPT ordering")
 * For the tiles with sel[t] != 0 (sel may be NULL = all tiles) the sorted
 * Gaussian ids are written to ids[] tile after tile, tile t starting at
 * sel_off[t].  Pairs are ordered by (tile, depth, Gaussian id).
 * Returns the number of ids written (or needed, when ids is NULL).
 */
typedef struct {
    int32_t tile;
    float depth;
    double depth_d;
    int32_t id;
} pair_t;

static int cmp_pair(const void* pa, const void* pb) {
    const pair_t* x = (const pair_t*)pa;
    const pair_t* y = (const pair_t*)pb;
    if (x->tile != y->tile) return x->tile < y->tile ? -1 : 1;
    if (x->depth_d != y->depth_d) return x->depth_d < y->depth_d ? -1 : 1;
    if (x->id != y->id) return x->id < y->id ? -1 : 1;
    return 0;
}

typedef struct {
    int32_t tile;
    int64_t count;
} tcount_t;

static int cmp_tcount(const void* pa, const void* pb) {
    const tcount_t* x = (const tcount_t*)pa;
    const tcount_t* y = (const tcount_t*)pb;
    if (x->count != y->count) return x->count > y->count ? -1 : 1;
    return x->tile < y->tile ? -1 : (x->tile > y->tile);
}

int64_t ora_bin(int64_t n, const float* viewmat, const float* intr, int W, int H, float znear,
                const double* splat, const int32_t* tiles_touched, const uint8_t* sel,
                int64_t* counts, int64_t* ranges, int32_t* lpt_order, int64_t* sel_off,
                int32_t* ids, int64_t ids_cap) {
    camera_t cam;
    make_camera(&cam, viewmat, intr, W, H, znear);
    int64_t nt = (int64_t)cam.ntx * cam.nty;
    for (int64_t t = 0; t < nt; ++t) counts[t] = 0;
    int64_t nsel = 0;
    for (int64_t i = 0; i < n; ++i) {
        if (tiles_touched[i] <= 0) continue;
        splat_t s;
        splat_from_record(splat + REC * i, &s);
        int ty0, ty1, tx0, tx1;
        row_range(&cam, &s, &ty0, &ty1);
        for (int ty = ty0; ty < ty1; ++ty)
            if (row_span(&cam, &s, ty, &tx0, &tx1))
                for (int tx = tx0; tx < tx1; ++tx) {
                    int64_t t = (int64_t)ty * cam.ntx + tx;
                    counts[t]++;
                    if (!sel || sel[t]) nsel++;
                }
    }
    int64_t acc = 0, acc_sel = 0;
    for (int64_t t = 0; t < nt; ++t) {
        ranges[2 * t] = acc;
        acc += counts[t];
        ranges[2 * t + 1] = acc;
        sel_off[t] = acc_sel;
        if (!sel || sel[t]) acc_sel += counts[t];
    }
    tcount_t* tc = (tcount_t*)malloc(sizeof(tcount_t) * (size_t)(nt > 0 ? nt : 1));
    for (int64_t t = 0; t < nt; ++t) {
        tc[t].tile = (int32_t)t;
        tc[t].count = counts[t];
    }
    qsort(tc, (size_t)nt, sizeof(tcount_t), cmp_tcount);
    for (int64_t t = 0; t < nt; ++t) lpt_order[t] = tc[t].tile;
    free(tc);
    if (!ids || ids_cap < nsel) return nsel;

    pair_t* pairs = (pair_t*)malloc(sizeof(pair_t) * (size_t)(nsel > 0 ? nsel : 1));
    int64_t k = 0;
    for (int64_t i = 0; i < n; ++i) {
        if (tiles_touched[i] <= 0) continue;
        splat_t s;
        splat_from_record(splat + REC * i, &s);
        int ty0, ty1, tx0, tx1;
        row_range(&cam, &s, &ty0, &ty1);
        for (int ty = ty0; ty < ty1; ++ty)
            if (row_span(&cam, &s, ty, &tx0, &tx1))
                for (int tx = tx0; tx < tx1; ++tx) {
                    int64_t t = (int64_t)ty * cam.ntx + tx;
                    if (sel && !sel[t]) continue;
                    pairs[k].tile = (int32_t)t;
                    pairs[k].depth = (float)splat[REC * i + 7];
                    pairs[k].depth_d = splat[REC * i + 7];
                    pairs[k].id = (int32_t)i;
                    ++k;
                }
    }
    qsort(pairs, (size_t)k, sizeof(pair_t), cmp_pair);
    for (int64_t j = 0; j < k; ++j) ids[j] = pairs[j].id;
    free(pairs);
    return nsel;
}

/* ------------------------------------------------------------------------ */
/* Exported: forward blending (Ryu & Yoo, Eq. 2-3)                           */
/* ------------------------------------------------------------------------ */
/*
 * Per pixel of every selected tile, front to back over the tile's list:
 *   stop before a splat once T < 1e-4;
 *   hit iff q <= tau with q = fma(u1, u1, u2 u2), u1 = fma(l11, dx, l12 dy),
 *   u2 = l22 dy, dx = (x + 0.5) - mux, dy = (y + 0.5) - muy (all in dreal):
 *   the quadratic form d^T Lambda d evaluated through the Cholesky factor of
 *   the conic, a sum of non-negative terms (well conditioned for thin splats);
 *   alpha = min(0.99, o exp(-q/2));  C += c alpha T;  T *= 1 - alpha.
 * Outputs: img[H][W][3], T_final[H][W], n_contrib[H][W] (blended splats) and
 * last_idx[H][W] (position in the full sorted pair list of the last blended
 * splat, -1 if none).  flags[H][W] bit 0 marks a pixel whose stop decision
 * lies within the fp32 error band of the 1e-4 threshold (several fp32
 * results are then correct), bit 1 a pixel with an alpha within that band
 * of the 0.99 clamp.
 *
 * The error band: a fp32 renderer evaluates each alpha with a relative error
 * of at most E_ALPHA and each transmittance update with at most two roundings.
 * The relative error of T after k blends is then bounded by
 * sum_j (E_ALPHA alpha_j / (1 - alpha_j) + 2^-23); a decision is flagged when
 * T is within twice that bound of 1e-4.
 *
 * The other admissible outcomes of such near-ties are rendered on request:
 *   stop_last (may be NULL): per pixel ORA_RULE to apply the stop rule, or the
 *     list position of the last splat a renderer blended (-1 for none).  The
 *     pixel then blends every hit up to that position and stops, and flags
 *     bit 2 is set when the stop rule does not admit that outcome: a hit
 *     blended after T fell below 1e-4 outside the band, a stop before a hit
 *     with T at or above 1e-4 outside the band, or a position that is not a
 *     hit of the list.
 *   clamp_flip: nonzero takes the other clamp decision at every splat whose
 *     alpha lies within the band of 0.99 (bit 1): alpha = 0.99 where the rule
 *     leaves it unclamped, the unclamped o exp(-q/2) where the rule clamps.
 */
#define E_ALPHA 7.62939453125e-06 /* 2^-17 */
#define ORA_RULE INT32_MIN
#define U32 5.9604644775390625e-08 /* 2^-24, unit roundoff of fp32 */

typedef struct {
    int W, H, ntx;
    const double* splat;
    const double* rgb;
    const int64_t* ranges;
    const int64_t* sel_off;
    const int32_t* ids;
} blend_ctx_t;

static int hit_test(const double* rec, int px, int py, dreal* q_out, double* dx_out,
                    double* dy_out) {
    dreal mux = (dreal)rec[0], muy = (dreal)rec[1];
    dreal l11 = (dreal)rec[13], l12 = (dreal)rec[14], l22 = (dreal)rec[15];
    dreal tau = (dreal)rec[6];
    dreal dx = ((dreal)px + (dreal)0.5) - mux;
    dreal dy = ((dreal)py + (dreal)0.5) - muy;
    dreal u1 = fma(l11, dx, l12 * dy);
    dreal u2 = l22 * dy;
    dreal q = fma(u1, u1, u2 * u2);
    *q_out = q;
    *dx_out = (double)dx;
    *dy_out = (double)dy;
    return q <= tau;
}

/* alpha of a hit with the clamp decision; *near_clamp: alpha within the band */
static double alpha_of(const double* rec, double q, int clamp_flip, int* clamped,
                       int* near_clamp, double* araw_out) {
    double araw = rec[5] * exp(-0.5 * q);
    int near = fabs(araw - ALPHA_MAX) <= 2.0 * E_ALPHA * ALPHA_MAX;
    int c = !(araw < ALPHA_MAX);
    if (clamp_flip && near) c = !c;
    *clamped = c;
    *near_clamp = near;
    *araw_out = araw;
    return c ? ALPHA_MAX : araw;
}

/* One blended splat of a pixel (front to back), as the backward needs it. */
typedef struct {
    int32_t g;
    int64_t k;
    double alpha, araw, T, dx, dy, q;
    int clamped, near_clamp;
} blended_t;

/*
 * The splats a pixel blends, front to back, under the stop rule or the forced
 * outcome stop (ORA_RULE or a list position); returns their number, grows
 * *list as needed, writes the final transmittance and the flags (bits as
 * ora_blend's) and the fp32 band err of the stop decisions.
 */
static int64_t pixel_blend(const blend_ctx_t* c, int64_t t, int px, int py, int32_t stop,
                           int clamp_flip, blended_t** list, int64_t* cap, double* T_out,
                           uint8_t* flags_out) {
    int64_t s0 = c->ranges[2 * t], s1 = c->ranges[2 * t + 1];
    int forced = stop != ORA_RULE;
    double T = 1.0, err = 0;
    int64_t nb = 0, last = -1;
    uint8_t fl = 0;
    for (int64_t k = s0; k < s1; ++k) {
        int near = fabs(T - T_MIN) <= 2.0 * err * T;
        if (near) fl |= 1;
        if (!forced && T < T_MIN) break;
        int32_t g = c->ids[c->sel_off[t] + (k - s0)];
        const double* rec = c->splat + REC * (int64_t)g;
        dreal q;
        double dx, dy;
        if (!hit_test(rec, px, py, &q, &dx, &dy)) continue;
        if (forced) {
            if (k > (int64_t)stop) {
                if (!(T < T_MIN || near)) fl |= 4; /* stopped before a hit the rule blends */
                break;
            }
            if (T < T_MIN && !near) fl |= 4; /* blended past a stop outside the band */
        }
        int clamped, near_clamp;
        double araw;
        double alpha = alpha_of(rec, (double)q, clamp_flip, &clamped, &near_clamp, &araw);
        if (near_clamp) fl |= 2;
        if (nb == *cap) {
            *cap *= 2;
            *list = (blended_t*)realloc(*list, sizeof(blended_t) * (size_t)*cap);
        }
        blended_t* e = &(*list)[nb++];
        e->g = g;
        e->k = k;
        e->alpha = alpha;
        e->araw = araw;
        e->T = T;
        e->dx = dx;
        e->dy = dy;
        e->q = (double)q;
        e->clamped = clamped;
        e->near_clamp = near_clamp;
        T *= (1.0 - alpha);
        err += E_ALPHA * alpha / (1.0 - alpha) + 1.1920928955078125e-07;
        last = k;
    }
    if (forced && last != (int64_t)stop) fl |= 4; /* the given position is not a blended hit */
    *T_out = T;
    *flags_out = fl;
    return nb;
}

void ora_blend2(int W, int H, const double* splat, const double* rgb, const int64_t* ranges,
                const int64_t* sel_off, const int32_t* ids, const uint8_t* sel,
                const int32_t* stop_last, int clamp_flip, double* img, double* T_final,
                int32_t* n_contrib, int32_t* last_idx, uint8_t* flags) {
    int ntx = (W + TILE - 1) / TILE, nty = (H + TILE - 1) / TILE;
    blend_ctx_t c = {W, H, ntx, splat, rgb, ranges, sel_off, ids};
    int64_t cap = 64;
    blended_t* list = (blended_t*)malloc(sizeof(blended_t) * (size_t)cap);
    for (int ty = 0; ty < nty; ++ty)
        for (int tx = 0; tx < ntx; ++tx) {
            int64_t t = (int64_t)ty * ntx + tx;
            if (sel && !sel[t]) continue;
            for (int py = ty * TILE; py < ty * TILE + TILE && py < H; ++py)
                for (int px = tx * TILE; px < tx * TILE + TILE && px < W; ++px) {
                    int64_t p = (int64_t)py * W + px;
                    double T;
                    uint8_t fl;
                    int32_t stop = stop_last ? stop_last[p] : ORA_RULE;
                    int64_t nb = pixel_blend(&c, t, px, py, stop, clamp_flip, &list, &cap, &T, &fl);
                    double C[3] = {0, 0, 0};
                    for (int64_t j = 0; j < nb; ++j) {
                        const blended_t* e = &list[j];
                        for (int ch = 0; ch < 3; ++ch)
                            C[ch] += rgb[3 * (int64_t)e->g + ch] * e->alpha * e->T;
                    }
                    img[3 * p] = C[0];
                    img[3 * p + 1] = C[1];
                    img[3 * p + 2] = C[2];
                    T_final[p] = T;
                    n_contrib[p] = (int32_t)nb;
                    last_idx[p] = nb ? (int32_t)list[nb - 1].k : -1;
                    flags[p] = fl;
                }
        }
    free(list);
}

void ora_blend(int W, int H, const double* splat, const double* rgb, const int64_t* ranges,
               const int64_t* sel_off, const int32_t* ids, const uint8_t* sel, double* img,
               double* T_final, int32_t* n_contrib, int32_t* last_idx, uint8_t* flags) {
    ora_blend2(W, H, splat, rgb, ranges, sel_off, ids, sel, NULL, 0, img, T_final, n_contrib,
               last_idx, flags);
}

/* ------------------------------------------------------------------------ */
/* Exported: backward of the blend -> nine screen-space derivatives          */
/* ------------------------------------------------------------------------ */
/*
 * For the blended splats k of a pixel (in order), with T_k the transmittance
 * before k, G = dL/dC and gT = dL/dT_final:
 *   dL/dc_k     = alpha_k T_k G
 *   dL/dalpha_k = T_k (c_k . G) - (B_k . G) / (1 - alpha_k) - gT T_final / (1 - alpha_k)
 *   with B_k = sum_{j > k} c_j alpha_j T_j the colour behind k.
 * Unless the 0.99 clamp is active: dL/do += exp(-q/2) dL/dalpha and
 * dL/dq = -(alpha/2) dL/dalpha; with dx = px - mux, dy = py - muy:
 *   dL/dmux = -2 (a dx + b dy) dL/dq,  dL/dmuy = -2 (b dx + c dy) dL/dq,
 *   dL/da = dx^2 dL/dq,  dL/db = 2 dx dy dL/dq,  dL/dc = dy^2 dL/dq.
 * grad2d[g][0..8] = (mux, muy, a, b, c, opacity, r, g, b), accumulated in
 * double over every selected tile.
 *
 * Magnitudes (the scale of an fp32 evaluation's error), all optional:
 *   gabs[g][r]: every term above evaluated with each input replaced by its
 *     absolute value and every difference by a sum, down to the inputs (the
 *     dot products c . G and B . G as sums over channels of |c_ch G_ch|); it
 *     bounds the sum of absolute values of everything an evaluation adds and
 *     equals |grad2d| when nothing cancels.
 *   grho[g][r]: the same terms, each weighted by the relative error bound
 *     eps_p of its pixel's fp32 evaluation,
 *       eps_p = 2 sum_j (E_ALPHA alpha_j / (1 - alpha_j) + 8 u) + 2 E_ALPHA + 32 u,
 *     u = 2^-24, over the pixel's blended splats j: the transmittance in
 *     front of a splat and the colour behind it carry each alpha's error
 *     amplified by 1 / (1 - alpha) and a few roundings per blend (forward
 *     products, backward division and running sums); alpha itself (and the
 *     opacity it is divided by) carries E_ALPHA; a term's own products a few
 *     roundings.
 *   galt[g][r]: the spread of the admissible results at near-ties of the
 *     clamp: per pixel with an alpha in the band of 0.99 (ora_blend's bit 1),
 *     |terms with every such clamp decision taken the other way - terms as the
 *     rule takes them|, summed.
 * stop_last: as for ora_blend2 (NULL or per pixel ORA_RULE / a forced last
 *   position): the backward of the outcome a renderer took at a stop near-tie.
 */
static void pixel_terms(const blend_ctx_t* c, const blended_t* list, int64_t nb, double Tfin,
                        const double G[3], double gT, double* term, double* mag) {
    double behind[3] = {0, 0, 0};
    double behind_mag = 0;
    for (int64_t j = nb - 1; j >= 0; --j) {
        const blended_t* e = &list[j];
        const double* rec = c->splat + REC * (int64_t)e->g;
        const double* col = c->rgb + 3 * (int64_t)e->g;
        double* tm = term + 9 * j;
        double* mg = mag + 9 * j;
        for (int r = 0; r < 9; ++r) tm[r] = mg[r] = 0;
        double w = e->alpha * e->T;
        for (int ch = 0; ch < 3; ++ch) {
            tm[6 + ch] = w * G[ch];
            mg[6 + ch] = fabs(tm[6 + ch]);
        }
        double cG = col[0] * G[0] + col[1] * G[1] + col[2] * G[2];
        double cG_mag = fabs(col[0] * G[0]) + fabs(col[1] * G[1]) + fabs(col[2] * G[2]);
        double bG = behind[0] * G[0] + behind[1] * G[1] + behind[2] * G[2];
        double dalpha = e->T * cG - bG / (1.0 - e->alpha) - gT * Tfin / (1.0 - e->alpha);
        double dalpha_mag = e->T * cG_mag + behind_mag / (1.0 - e->alpha) +
                            fabs(gT) * Tfin / (1.0 - e->alpha);
        for (int ch = 0; ch < 3; ++ch) behind[ch] += col[ch] * w;
        behind_mag += cG_mag * w;
        if (!e->clamped) {
            double dq = -0.5 * e->alpha * dalpha;
            /* conic of the evaluated quadratic: a = l11^2, b = l11 l12,
             * c = l12^2 + l22^2 */
            double l11 = rec[13], l12 = rec[14], l22 = rec[15];
            double a = l11 * l11, b = l11 * l12, cc = l12 * l12 + l22 * l22;
            tm[5] = exp(-0.5 * e->q) * dalpha;
            tm[0] = -2.0 * (a * e->dx + b * e->dy) * dq;
            tm[1] = -2.0 * (b * e->dx + cc * e->dy) * dq;
            tm[2] = e->dx * e->dx * dq;
            tm[3] = 2.0 * e->dx * e->dy * dq;
            tm[4] = e->dy * e->dy * dq;
            double dq_mag = 0.5 * e->alpha * dalpha_mag;
            mg[5] = exp(-0.5 * e->q) * dalpha_mag;
            mg[0] = 2.0 * (fabs(a * e->dx) + fabs(b * e->dy)) * dq_mag;
            mg[1] = 2.0 * (fabs(b * e->dx) + fabs(cc * e->dy)) * dq_mag;
            mg[2] = e->dx * e->dx * dq_mag;
            mg[3] = 2.0 * fabs(e->dx * e->dy) * dq_mag;
            mg[4] = e->dy * e->dy * dq_mag;
        }
    }
}

void ora_blend_bwd2(int W, int H, const double* splat, const double* rgb, const int64_t* ranges,
                    const int64_t* sel_off, const int32_t* ids, const uint8_t* sel,
                    const int32_t* stop_last, const double* dL_dimg, const double* dL_dT,
                    double* grad2d, double* gabs, double* grho, double* galt) {
    int ntx = (W + TILE - 1) / TILE, nty = (H + TILE - 1) / TILE;
    blend_ctx_t c = {W, H, ntx, splat, rgb, ranges, sel_off, ids};
    int64_t cap = 64, tcap = 0;
    blended_t* list = (blended_t*)malloc(sizeof(blended_t) * (size_t)cap);
    double *term = NULL, *mag = NULL, *term2 = NULL, *mag2 = NULL;
    for (int ty = 0; ty < nty; ++ty)
        for (int tx = 0; tx < ntx; ++tx) {
            int64_t t = (int64_t)ty * ntx + tx;
            if (sel && !sel[t]) continue;
            for (int py = ty * TILE; py < ty * TILE + TILE && py < H; ++py)
                for (int px = tx * TILE; px < tx * TILE + TILE && px < W; ++px) {
                    int64_t p = (int64_t)py * W + px;
                    double Tfin;
                    uint8_t fl;
                    int32_t stop = stop_last ? stop_last[p] : ORA_RULE;
                    int64_t nb = pixel_blend(&c, t, px, py, stop, 0, &list, &cap, &Tfin, &fl);
                    if (nb == 0) continue;
                    if (nb > tcap) {
                        tcap = cap;
                        term = (double*)realloc(term, sizeof(double) * 9 * (size_t)tcap);
                        mag = (double*)realloc(mag, sizeof(double) * 9 * (size_t)tcap);
                        term2 = (double*)realloc(term2, sizeof(double) * 9 * (size_t)tcap);
                        mag2 = (double*)realloc(mag2, sizeof(double) * 9 * (size_t)tcap);
                    }
                    double G[3] = {dL_dimg[3 * p], dL_dimg[3 * p + 1], dL_dimg[3 * p + 2]};
                    double gT = dL_dT ? dL_dT[p] : 0.0;
                    pixel_terms(&c, list, nb, Tfin, G, gT, term, mag);
                    double eps = 2.0 * E_ALPHA + 32.0 * U32;
                    int any_near_clamp = 0;
                    for (int64_t j = 0; j < nb; ++j) {
                        eps += 2.0 * (E_ALPHA * list[j].alpha / (1.0 - list[j].alpha) + 8.0 * U32);
                        any_near_clamp |= list[j].near_clamp;
                    }
                    for (int64_t j = 0; j < nb; ++j) {
                        int64_t g = list[j].g;
                        for (int r = 0; r < 9; ++r) {
                            grad2d[9 * g + r] += term[9 * j + r];
                            if (gabs) gabs[9 * g + r] += mag[9 * j + r];
                            if (grho) grho[9 * g + r] += eps * mag[9 * j + r];
                        }
                    }
                    if (galt && any_near_clamp) {
                        /* the same splats with every near-tie clamp decision flipped */
                        double T = 1.0;
                        for (int64_t j = 0; j < nb; ++j) {
                            blended_t* e = &list[j];
                            if (e->near_clamp) {
                                e->clamped = !e->clamped;
                                e->alpha = e->clamped ? ALPHA_MAX : e->araw;
                            }
                            e->T = T;
                            T *= (1.0 - e->alpha);
                        }
                        pixel_terms(&c, list, nb, T, G, gT, term2, mag2);
                        for (int64_t j = 0; j < nb; ++j) {
                            int64_t g = list[j].g;
                            for (int r = 0; r < 9; ++r)
                                galt[9 * g + r] += fabs(term2[9 * j + r] - term[9 * j + r]);
                        }
                    }
                }
        }
    free(list);
    free(term);
    free(mag);
    free(term2);
    free(mag2);
}

void ora_blend_bwd(int W, int H, const double* splat, const double* rgb, const int64_t* ranges,
                   const int64_t* sel_off, const int32_t* ids, const uint8_t* sel,
                   const double* dL_dimg, const double* dL_dT, double* grad2d, double* gabs) {
    ora_blend_bwd2(W, H, splat, rgb, ranges, sel_off, ids, sel, NULL, dL_dimg, dL_dT, grad2d, gabs,
                   NULL, NULL);
}

/* ------------------------------------------------------------------------ */
/* Exported: backward of the projection (chain rule, double)                 */
/* ------------------------------------------------------------------------ */
/*
 * Inputs grad2d[n][9] as produced by ora_blend_bwd and touched[n] (nonzero
 * where the Gaussian received a gradient).  Outputs, zero for culled or
 * untouched Gaussians:
 *   dmeans[n][3], dscales[n][3], dquats[n][4] (w.r.t. the raw quaternion),
 *   dopac[n], dsh[n][K][3].
 * The forward quantities are recomputed in double from the inputs.
 */
void ora_project_bwd(int64_t n, int sh_degree, const float* viewmat, const float* intr, int W,
                     int H, float znear, const float* means, const float* scales,
                     const float* quats, const float* opac, const float* sh,
                     const int32_t* tiles_touched, const double* grad2d, double* dmeans,
                     double* dscales, double* dquats, double* dopac, double* dsh) {
    (void)W;
    (void)H;
    (void)znear;
    int K = (sh_degree + 1) * (sh_degree + 1);
    double V[12];
    for (int i = 0; i < 12; ++i) V[i] = viewmat[i];
    double fx = intr[0], fy = intr[1];
    double cw[3];
    camera_centre(viewmat, cw);
    for (int64_t i = 0; i < n; ++i) {
        double* dm = dmeans + 3 * i;
        double* ds = dscales + 3 * i;
        double* dq = dquats + 4 * i;
        double* dshi = dsh + (int64_t)K * 3 * i;
        dm[0] = dm[1] = dm[2] = 0;
        ds[0] = ds[1] = ds[2] = 0;
        dq[0] = dq[1] = dq[2] = dq[3] = 0;
        dopac[i] = 0;
        for (int k = 0; k < 3 * K; ++k) dshi[k] = 0;
        if (tiles_touched[i] <= 0) continue;
        const double* g2 = grad2d + 9 * i;
        int any = 0;
        for (int r = 0; r < 9; ++r) any |= (g2[r] != 0.0);
        if (!any) continue;

        /* forward recomputation in double */
        double m[3] = {means[3 * i], means[3 * i + 1], means[3 * i + 2]};
        double t[3];
        for (int r = 0; r < 3; ++r)
            t[r] = V[4 * r] * m[0] + V[4 * r + 1] * m[1] + V[4 * r + 2] * m[2] + V[4 * r + 3];
        double qr[4] = {quats[4 * i], quats[4 * i + 1], quats[4 * i + 2], quats[4 * i + 3]};
        double qn = sqrt(qr[0] * qr[0] + qr[1] * qr[1] + qr[2] * qr[2] + qr[3] * qr[3]);
        double w = qr[0] / qn, x = qr[1] / qn, y = qr[2] / qn, z = qr[3] / qn;
        double R[9] = {1 - 2 * (y * y + z * z), 2 * (x * y - w * z),     2 * (x * z + w * y),
                       2 * (x * y + w * z),     1 - 2 * (x * x + z * z), 2 * (y * z - w * x),
                       2 * (x * z - w * y),     2 * (y * z + w * x),     1 - 2 * (x * x + y * y)};
        double s[3] = {scales[3 * i], scales[3 * i + 1], scales[3 * i + 2]};
        double M[9], S[9];
        for (int r = 0; r < 3; ++r)
            for (int c = 0; c < 3; ++c) M[3 * r + c] = R[3 * r + c] * s[c];
        for (int r = 0; r < 3; ++r)
            for (int c = 0; c < 3; ++c)
                S[3 * r + c] = M[3 * r] * M[3 * c] + M[3 * r + 1] * M[3 * c + 1] +
                               M[3 * r + 2] * M[3 * c + 2];
        double tx = t[0], ty = t[1], tz = t[2];
        double j00 = fx / tz, j11 = fy / tz;
        double j02 = -fx * tx / (tz * tz), j12 = -fy * ty / (tz * tz);
        double Tm[2][3];
        for (int k = 0; k < 3; ++k) {
            Tm[0][k] = j00 * V[k] + j02 * V[8 + k];
            Tm[1][k] = j11 * V[4 + k] + j12 * V[8 + k];
        }
        double P[2][2];
        for (int a_ = 0; a_ < 2; ++a_)
            for (int b_ = 0; b_ < 2; ++b_) {
                double acc = 0;
                for (int r = 0; r < 3; ++r)
                    for (int c = 0; c < 3; ++c) acc += Tm[a_][r] * S[3 * r + c] * Tm[b_][c];
                P[a_][b_] = acc;
            }
        double P00 = P[0][0], P01 = P[0][1], P11 = P[1][1];
        double det = P00 * P11 - P01 * P01;
        double det2 = det * det;

        /* conic (a, b, c) = (P11, -P01, P00) / det  ->  dP00, dP01, dP11 */
        double ga = g2[2], gb = g2[3], gc = g2[4];
        double dP00 = ga * (-P11 * P11 / det2) + gb * (P01 * P11 / det2) +
                      gc * (1.0 / det - P00 * P11 / det2);
        double dP11 = ga * (1.0 / det - P11 * P00 / det2) + gb * (P01 * P00 / det2) +
                      gc * (-P00 * P00 / det2);
        double dP01 = ga * (2.0 * P01 * P11 / det2) + gb * (-1.0 / det - 2.0 * P01 * P01 / det2) +
                      gc * (2.0 * P00 * P01 / det2);

        /* Sigma' = T Sigma T^T: P00 = T0 S T0, P01 = T0 S T1, P11 = T1 S T1 */
        double dS[9], dT[2][3];
        for (int r = 0; r < 3; ++r)
            for (int c = 0; c < 3; ++c)
                dS[3 * r + c] = dP00 * Tm[0][r] * Tm[0][c] + dP01 * Tm[0][r] * Tm[1][c] +
                                dP11 * Tm[1][r] * Tm[1][c];
        for (int r = 0; r < 3; ++r) {
            double ST0 = S[3 * r] * Tm[0][0] + S[3 * r + 1] * Tm[0][1] + S[3 * r + 2] * Tm[0][2];
            double ST1 = S[3 * r] * Tm[1][0] + S[3 * r + 1] * Tm[1][1] + S[3 * r + 2] * Tm[1][2];
            dT[0][r] = 2.0 * dP00 * ST0 + dP01 * ST1;
            dT[1][r] = dP01 * ST0 + 2.0 * dP11 * ST1;
        }
        /* T = J W */
        double dj00 = 0, dj02 = 0, dj11 = 0, dj12 = 0;
        for (int k = 0; k < 3; ++k) {
            dj00 += dT[0][k] * V[k];
            dj02 += dT[0][k] * V[8 + k];
            dj11 += dT[1][k] * V[4 + k];
            dj12 += dT[1][k] * V[8 + k];
        }
        /* mu' and J as functions of t */
        double gmx = g2[0], gmy = g2[1];
        double dt[3] = {0, 0, 0};
        double tz2 = tz * tz, tz3 = tz2 * tz;
        dt[0] += gmx * fx / tz;
        dt[2] += gmx * (-fx * tx / tz2);
        dt[1] += gmy * fy / tz;
        dt[2] += gmy * (-fy * ty / tz2);
        dt[2] += dj00 * (-fx / tz2);
        dt[0] += dj02 * (-fx / tz2);
        dt[2] += dj02 * (2.0 * fx * tx / tz3);
        dt[2] += dj11 * (-fy / tz2);
        dt[1] += dj12 * (-fy / tz2);
        dt[2] += dj12 * (2.0 * fy * ty / tz3);
        /* t = W m + t_v */
        for (int c = 0; c < 3; ++c) dm[c] += V[c] * dt[0] + V[4 + c] * dt[1] + V[8 + c] * dt[2];

        /* Sigma = M M^T, M = R diag(s) */
        double dM[9];
        for (int r = 0; r < 3; ++r)
            for (int k = 0; k < 3; ++k) {
                double acc = 0;
                for (int j = 0; j < 3; ++j) acc += (dS[3 * r + j] + dS[3 * j + r]) * M[3 * j + k];
                dM[3 * r + k] = acc;
            }
        double dR[9];
        for (int r = 0; r < 3; ++r)
            for (int k = 0; k < 3; ++k) {
                ds[k] += dM[3 * r + k] * R[3 * r + k];
                dR[3 * r + k] = dM[3 * r + k] * s[k];
            }
        /* R(w, x, y, z) */
        double dw = 0, dx = 0, dy = 0, dz = 0;
        dy += dR[0] * (-4 * y);  dz += dR[0] * (-4 * z);
        dw += dR[1] * (-2 * z);  dx += dR[1] * (2 * y);  dy += dR[1] * (2 * x);  dz += dR[1] * (-2 * w);
        dw += dR[2] * (2 * y);   dx += dR[2] * (2 * z);  dy += dR[2] * (2 * w);  dz += dR[2] * (2 * x);
        dw += dR[3] * (2 * z);   dx += dR[3] * (2 * y);  dy += dR[3] * (2 * x);  dz += dR[3] * (2 * w);
        dx += dR[4] * (-4 * x);  dz += dR[4] * (-4 * z);
        dw += dR[5] * (-2 * x);  dx += dR[5] * (-2 * w); dy += dR[5] * (2 * z);  dz += dR[5] * (2 * y);
        dw += dR[6] * (-2 * y);  dx += dR[6] * (2 * z);  dy += dR[6] * (-2 * w); dz += dR[6] * (2 * x);
        dw += dR[7] * (2 * x);   dx += dR[7] * (2 * w);  dy += dR[7] * (2 * z);  dz += dR[7] * (2 * y);
        dx += dR[8] * (-4 * x);  dy += dR[8] * (-4 * y);
        /* normalisation q_hat = q / |q| */
        double qh[4] = {w, x, y, z}, dqh[4] = {dw, dx, dy, dz};
        double dotq = qh[0] * dqh[0] + qh[1] * dqh[1] + qh[2] * dqh[2] + qh[3] * dqh[3];
        for (int k = 0; k < 4; ++k) dq[k] = (dqh[k] - qh[k] * dotq) / qn;

        /* opacity */
        dopac[i] = g2[5];

        /* colour c = sum_k Y_k(d_hat) s_k */
        double dhat[3], len, Y[16], dY[16][3];
        view_dir(means + 3 * i, cw, dhat, &len);
        sh_basis(dhat, Y, dY);
        double gcol[3] = {g2[6], g2[7], g2[8]};
        double gd[3] = {0, 0, 0};
        for (int k = 0; k < K; ++k) {
            double proj = 0;
            for (int ch = 0; ch < 3; ++ch) {
                dshi[3 * k + ch] = Y[k] * gcol[ch];
                proj += gcol[ch] * (double)sh[(i * K + k) * 3 + ch];
            }
            for (int j = 0; j < 3; ++j) gd[j] += proj * dY[k][j];
        }
        double dotd = dhat[0] * gd[0] + dhat[1] * gd[1] + dhat[2] * gd[2];
        for (int j = 0; j < 3; ++j) dm[j] += (gd[j] - dhat[j] * dotd) / len;
    }
}

/* ------------------------------------------------------------------------ */
/* Exported: magnitudes of the projection backward (running error bound)     */
/* ------------------------------------------------------------------------ */
/*
 * The chain rule of ora_project_bwd evaluated on magnitudes: every input
 * gradient replaced by gmag[n][9] (>= |grad2d|), every factor by its absolute
 * value and every sum or difference by the sum of its terms' magnitudes,
 * stage by stage.  A floating-point evaluation of the chain has an error
 * bounded by a small multiple of u times these values (u the unit roundoff).
 */
void ora_project_bwd_mag(int64_t n, int sh_degree, const float* viewmat, const float* intr,
                         const float* means, const float* scales, const float* quats,
                         const float* sh, const int32_t* tiles_touched, const double* gmag,
                         double* mmeans, double* mscales, double* mquats, double* mopac,
                         double* msh) {
    int K = (sh_degree + 1) * (sh_degree + 1);
    double V[12], aV[12];
    for (int i = 0; i < 12; ++i) {
        V[i] = viewmat[i];
        aV[i] = fabs(V[i]);
    }
    double fx = intr[0], fy = intr[1];
    double cw[3];
    camera_centre(viewmat, cw);
    for (int64_t i = 0; i < n; ++i) {
        double* dm = mmeans + 3 * i;
        double* ds = mscales + 3 * i;
        double* dq = mquats + 4 * i;
        double* dshi = msh + (int64_t)K * 3 * i;
        dm[0] = dm[1] = dm[2] = 0;
        ds[0] = ds[1] = ds[2] = 0;
        dq[0] = dq[1] = dq[2] = dq[3] = 0;
        mopac[i] = 0;
        for (int k = 0; k < 3 * K; ++k) dshi[k] = 0;
        if (tiles_touched[i] <= 0) continue;
        const double* g2 = gmag + 9 * i;
        double m[3] = {means[3 * i], means[3 * i + 1], means[3 * i + 2]};
        double t[3];
        for (int r = 0; r < 3; ++r)
            t[r] = V[4 * r] * m[0] + V[4 * r + 1] * m[1] + V[4 * r + 2] * m[2] + V[4 * r + 3];
        double qr[4] = {quats[4 * i], quats[4 * i + 1], quats[4 * i + 2], quats[4 * i + 3]};
        double qn = sqrt(qr[0] * qr[0] + qr[1] * qr[1] + qr[2] * qr[2] + qr[3] * qr[3]);
        double w = qr[0] / qn, x = qr[1] / qn, y = qr[2] / qn, z = qr[3] / qn;
        double R[9] = {1 - 2 * (y * y + z * z), 2 * (x * y - w * z),     2 * (x * z + w * y),
                       2 * (x * y + w * z),     1 - 2 * (x * x + z * z), 2 * (y * z - w * x),
                       2 * (x * z - w * y),     2 * (y * z + w * x),     1 - 2 * (x * x + y * y)};
        double s[3] = {scales[3 * i], scales[3 * i + 1], scales[3 * i + 2]};
        double M[9], S[9], aM[9], aS[9];
        for (int r = 0; r < 3; ++r)
            for (int c = 0; c < 3; ++c) {
                M[3 * r + c] = R[3 * r + c] * s[c];
                aM[3 * r + c] = fabs(M[3 * r + c]);
            }
        for (int r = 0; r < 3; ++r)
            for (int c = 0; c < 3; ++c) {
                S[3 * r + c] = M[3 * r] * M[3 * c] + M[3 * r + 1] * M[3 * c + 1] +
                               M[3 * r + 2] * M[3 * c + 2];
                aS[3 * r + c] = aM[3 * r] * aM[3 * c] + aM[3 * r + 1] * aM[3 * c + 1] +
                                aM[3 * r + 2] * aM[3 * c + 2];
            }
        double tx = t[0], ty = t[1], tz = t[2];
        double j00 = fx / tz, j11 = fy / tz;
        double j02 = -fx * tx / (tz * tz), j12 = -fy * ty / (tz * tz);
        double Tm[2][3], aT[2][3];
        for (int k = 0; k < 3; ++k) {
            Tm[0][k] = j00 * V[k] + j02 * V[8 + k];
            Tm[1][k] = j11 * V[4 + k] + j12 * V[8 + k];
            aT[0][k] = fabs(j00) * aV[k] + fabs(j02) * aV[8 + k];
            aT[1][k] = fabs(j11) * aV[4 + k] + fabs(j12) * aV[8 + k];
        }
        double P[2][2];
        for (int a_ = 0; a_ < 2; ++a_)
            for (int b_ = 0; b_ < 2; ++b_) {
                double acc = 0;
                for (int r = 0; r < 3; ++r)
                    for (int c = 0; c < 3; ++c) acc += Tm[a_][r] * S[3 * r + c] * Tm[b_][c];
                P[a_][b_] = acc;
            }
        double P00 = P[0][0], P01 = P[0][1], P11 = P[1][1];
        double det = P00 * P11 - P01 * P01, det2 = det * det;
        double aP01 = fabs(P01);
        /* conic -> Sigma' */
        double ga = g2[2], gb = g2[3], gc = g2[4];
        double dP00 = ga * P11 * P11 / det2 + gb * aP01 * P11 / det2 + gc * (1.0 / det + P00 * P11 / det2);
        double dP11 = ga * (1.0 / det + P11 * P00 / det2) + gb * aP01 * P00 / det2 + gc * P00 * P00 / det2;
        double dP01 = ga * 2.0 * aP01 * P11 / det2 + gb * (1.0 / det + 2.0 * P01 * P01 / det2) +
                      gc * 2.0 * P00 * aP01 / det2;
        double dS[9], dT[2][3];
        for (int r = 0; r < 3; ++r)
            for (int c = 0; c < 3; ++c)
                dS[3 * r + c] = dP00 * aT[0][r] * aT[0][c] + dP01 * aT[0][r] * aT[1][c] +
                                dP11 * aT[1][r] * aT[1][c];
        for (int r = 0; r < 3; ++r) {
            double ST0 = aS[3 * r] * aT[0][0] + aS[3 * r + 1] * aT[0][1] + aS[3 * r + 2] * aT[0][2];
            double ST1 = aS[3 * r] * aT[1][0] + aS[3 * r + 1] * aT[1][1] + aS[3 * r + 2] * aT[1][2];
            dT[0][r] = 2.0 * dP00 * ST0 + dP01 * ST1;
            dT[1][r] = dP01 * ST0 + 2.0 * dP11 * ST1;
        }
        double dj00 = 0, dj02 = 0, dj11 = 0, dj12 = 0;
        for (int k = 0; k < 3; ++k) {
            dj00 += dT[0][k] * aV[k];
            dj02 += dT[0][k] * aV[8 + k];
            dj11 += dT[1][k] * aV[4 + k];
            dj12 += dT[1][k] * aV[8 + k];
        }
        double gmx = g2[0], gmy = g2[1];
        double atx = fabs(tx), aty = fabs(ty);
        double tz2 = tz * tz, tz3 = tz2 * tz;
        double dt[3];
        dt[0] = gmx * fabs(fx) / tz + dj02 * fabs(fx) / tz2;
        dt[1] = gmy * fabs(fy) / tz + dj12 * fabs(fy) / tz2;
        dt[2] = gmx * fabs(fx) * atx / tz2 + gmy * fabs(fy) * aty / tz2 + dj00 * fabs(fx) / tz2 +
                dj02 * 2.0 * fabs(fx) * atx / tz3 + dj11 * fabs(fy) / tz2 +
                dj12 * 2.0 * fabs(fy) * aty / tz3;
        for (int c = 0; c < 3; ++c) dm[c] += aV[c] * dt[0] + aV[4 + c] * dt[1] + aV[8 + c] * dt[2];
        double dM[9], dR[9];
        for (int r = 0; r < 3; ++r)
            for (int k = 0; k < 3; ++k) {
                double acc = 0;
                for (int j = 0; j < 3; ++j) acc += (dS[3 * r + j] + dS[3 * j + r]) * aM[3 * j + k];
                dM[3 * r + k] = acc;
            }
        for (int r = 0; r < 3; ++r)
            for (int k = 0; k < 3; ++k) {
                ds[k] += dM[3 * r + k] * fabs(R[3 * r + k]);
                dR[3 * r + k] = dM[3 * r + k] * fabs(s[k]);
            }
        double aw = fabs(w), ax = fabs(x), ay = fabs(y), az = fabs(z);
        double dw = 2 * (az * dR[1] + ay * dR[2] + az * dR[3] + ax * dR[5] + ay * dR[6] + ax * dR[7]);
        double dx = 2 * (ay * dR[1] + az * dR[2] + ay * dR[3] + 2 * ax * dR[4] + aw * dR[5] +
                         az * dR[6] + aw * dR[7] + 2 * ax * dR[8]);
        double dy = 2 * (2 * ay * dR[0] + ax * dR[1] + aw * dR[2] + ax * dR[3] + az * dR[5] +
                         aw * dR[6] + az * dR[7] + 2 * ay * dR[8]);
        double dz = 2 * (2 * az * dR[0] + aw * dR[1] + ax * dR[2] + aw * dR[3] + 2 * az * dR[4] +
                         ay * dR[5] + ax * dR[6] + ay * dR[7]);
        double qh[4] = {aw, ax, ay, az}, dqh[4] = {dw, dx, dy, dz};
        double dotq = qh[0] * dqh[0] + qh[1] * dqh[1] + qh[2] * dqh[2] + qh[3] * dqh[3];
        for (int k = 0; k < 4; ++k) dq[k] = (dqh[k] + qh[k] * dotq) / qn;
        mopac[i] = g2[5];
        double dhat[3], len, Y[16], dY[16][3];
        view_dir(means + 3 * i, cw, dhat, &len);
        sh_basis(dhat, Y, dY);
        double gd[3] = {0, 0, 0};
        for (int k = 0; k < K; ++k) {
            double proj = 0;
            for (int ch = 0; ch < 3; ++ch) {
                dshi[3 * k + ch] = fabs(Y[k]) * g2[6 + ch];
                proj += g2[6 + ch] * fabs((double)sh[(i * K + k) * 3 + ch]);
            }
            for (int j = 0; j < 3; ++j) gd[j] += proj * fabs(dY[k][j]);
        }
        double ad[3] = {fabs(dhat[0]), fabs(dhat[1]), fabs(dhat[2])};
        double dotd = ad[0] * gd[0] + ad[1] * gd[1] + ad[2] * gd[2];
        for (int j = 0; j < 3; ++j) dm[j] += (gd[j] + ad[j] * dotd) / len;
    }
}

/* ------------------------------------------------------------------------ */
/* Exported: per-frame chunking policy (Ryu & Yoo, Sec. 4.4, Eq. 6)          */
/* ------------------------------------------------------------------------ */
/*
 * counts_desc[0..nt-1] are the tile counts in descending order (N_1 >= N_2 ...),
 * K the number of concurrently resident CTAs.  For k in {2, 4, 8, 16} and
 * h = 0 .. min(nt, h_max):
 *   l(h, k) = max(N_1 / k, N_{h+1})  (l(0, k) = N_1; N_{nt+1} = 0)
 *   T(h, k) = max((N_total + lambda h k) / K, l) + beta l
 * The minimiser (lowest T; ties to the smaller h, then the smaller k) is
 * taken only if T <= (1 - eps) T(0); otherwise h = 0 (no chunking).  The
 * comparisons are made on K T (the same order, no division).
 * Writes (h*, k*) and returns T(h*, k*).
 */
double ora_policy(int64_t nt, const int64_t* counts_desc, int64_t K, double lambda, double beta,
                  double eps, int64_t h_max, int64_t* h_out, int64_t* k_out) {
    /* Eq. 6 multiplied by K > 0 (same minimiser, no division):
     * K T(h, k) = max(N_total + lambda h k, K l) + beta K l;  l = max(N_1 / k, N_{h+1}) */
    double total = 0;
    for (int64_t t = 0; t < nt; ++t) total += (double)counts_desc[t];
    double Kd = (double)K;
    double N1 = nt > 0 ? (double)counts_desc[0] : 0.0;
    double base = fmax(total, Kd * N1) + beta * (Kd * N1);
    double best = base;
    int64_t bh = 0, bk = 1;
    int64_t hm = nt < h_max ? nt : h_max;
    const int ks[4] = {2, 4, 8, 16};
    for (int64_t h = 1; h <= hm; ++h)
        for (int ki = 0; ki < 4; ++ki) {
            double k = ks[ki];
            double next = h < nt ? (double)counts_desc[h] : 0.0;
            double l = fmax(N1 / k, next);
            double Kl = Kd * l;
            double cost = fmax(total + lambda * (double)h * k, Kl) + beta * Kl;
            if (cost < best) {
                best = cost;
                bh = h;
                bk = ks[ki];
            }
        }
    if (bh > 0 && !(best <= (1.0 - eps) * base)) {
        bh = 0;
        bk = 1;
        best = base;
    }
    *h_out = bh;
    *k_out = bk;
    return best / Kd;
}

/*
 * The training step after the chain rule ("proj_sh_bwd_adam" of the pages' Metal
 * port, where the projection backward and the Adam step are one pass): the
 * gradients of the raw parameters a training loop optimises, then one Adam step.
 *
 * Raw gradients: scales are exp(log-scales) and opacities sigmoid(logits), so
 * dL/dlog s = s dL/ds and dL/dlogit = o (1 - o) dL/do.
 */
void ora_raw_grads(int64_t n, const double* scales, const double* opac, const double* dscales,
                   const double* dopac, double* dlog_scales, double* dlogits) {
    for (int64_t i = 0; i < 3 * n; ++i) dlog_scales[i] = scales[i] * dscales[i];
    for (int64_t i = 0; i < n; ++i) dlogits[i] = opac[i] * (1.0 - opac[i]) * dopac[i];
}

/*
 * Adam (Kingma & Ba), one step t >= 1 on count elements, in place:
 *   m <- b1 m + (1 - b1) g,  v <- b2 v + (1 - b2) g^2,
 *   p <- p - lr (m / (1 - b1^t)) / (sqrt(v / (1 - b2^t)) + eps)
 */
void ora_adam_step(int64_t count, double* p, double* m, double* v, const double* g, double lr,
                   double b1, double b2, double eps, int64_t t) {
    double c1 = 1.0 - pow(b1, (double)t), c2 = 1.0 - pow(b2, (double)t);
    for (int64_t i = 0; i < count; ++i) {
        m[i] = b1 * m[i] + (1.0 - b1) * g[i];
        v[i] = b2 * v[i] + (1.0 - b2) * g[i] * g[i];
        p[i] -= lr * (m[i] / c1) / (sqrt(v[i] / c2) + eps);
    }
}

/*
 * The photometric loss of a training step ("loss_fwd_bwd" of the pages' Metal
 * port, whose intermediates are five windowed moments for each of the three
 * colour channels), read as the usual 3DGS objective
 *
 *   L = (1 - lambda) mean |x - y| + lambda (1 - mean SSIM(x, y))
 *
 * over the H x W x 3 values of the rendered image x and the target y, with the
 * structural similarity of Wang et al. (2004) per pixel and channel:
 *
 *   mu_x = w * x,  mu_y = w * y,  e_xx = w * x^2,  e_yy = w * y^2,  e_xy = w * xy
 *   var_x = e_xx - mu_x^2,  var_y = e_yy - mu_y^2,  cov = e_xy - mu_x mu_y
 *   SSIM = (2 mu_x mu_y + c1)(2 cov + c2) / ((mu_x^2 + mu_y^2 + c1)(var_x + var_y + c2))
 *
 * "w *" is the weighted sum over the 11 x 11 window centred on the pixel with
 * weights g(a) g(b), g(k) = exp(-k^2 / (2 sigma^2)) normalised over k = -5..5,
 * and pixels outside the image count as zero.  Written as that 2D sum, not as
 * two 1D passes.
 *
 * The gradient dL/dx is the chain rule through those definitions.  Per pixel q
 * and channel the SSIM depends on x only through mu_x, e_xx and e_xy; with
 * A1 = 2 mu_x mu_y + c1, A2 = 2 cov + c2, B1 = mu_x^2 + mu_y^2 + c1,
 * B2 = var_x + var_y + c2 and D = B1 B2:
 *
 *   dS/dmu_x = (2 mu_y (A2 - A1) - 2 mu_x S (B2 - B1)) / D
 *   dS/de_xx = -S / B2
 *   dS/de_xy = 2 A1 / D
 *
 * and a pixel p enters mu_x(q), e_xx(q), e_xy(q) with weights w(q - p),
 * w(q - p) 2 x(p) and w(q - p) y(p), for every q of the image within the
 * window.  The L1 term's derivative is sign(x - y) (0 where x = y).
 *
 * out[0] = L, out[1] = mean |x - y|, out[2] = mean SSIM; dL_dx [H][W][3];
 * ssim_map [H][W][3] (optional, NULL = not written) the per-pixel SSIM; mag
 * [H][W][3] (optional) the same sums over absolute values of every term,
 * (1 - lambda) / (3HW) + lambda / (3HW) sum_q w(q - p) (|dS/dmu_x| +
 * 2 |x(p)| |dS/de_xx| + |y(p)| |dS/de_xy|): the scale that rounding errors of
 * an fp32 evaluation are proportional to.
 */
#define SSIM_R 5 /* window radius: 11 taps */

static void ssim_window(double sigma, double* g) {
    double s = 0.0;
    for (int k = -SSIM_R; k <= SSIM_R; ++k) {
        g[k + SSIM_R] = exp(-(double)(k * k) / (2.0 * sigma * sigma));
        s += g[k + SSIM_R];
    }
    for (int k = 0; k <= 2 * SSIM_R; ++k) g[k] /= s;
}

void ora_loss_l1_ssim(int W, int H, const float* x, const float* y, double lambda, double c1,
                      double c2, double sigma, double* out, double* dL_dx, double* ssim_map,
                      double* mag) {
    double g[2 * SSIM_R + 1];
    ssim_window(sigma, g);
    int64_t np = (int64_t)W * H;
    double inv = 1.0 / (double)(3 * np);
    /* per pixel and channel: dS/dmu_x, dS/de_xx, dS/de_xy */
    double* dmu = (double*)malloc(sizeof(double) * 3 * np);
    double* dxx = (double*)malloc(sizeof(double) * 3 * np);
    double* dxy = (double*)malloc(sizeof(double) * 3 * np);
    double l1 = 0.0, ssim = 0.0;
    for (int r = 0; r < H; ++r)
        for (int c = 0; c < W; ++c)
            for (int ch = 0; ch < 3; ++ch) {
                double mx = 0, my = 0, exx = 0, eyy = 0, exy = 0;
                for (int a = -SSIM_R; a <= SSIM_R; ++a)
                    for (int b = -SSIM_R; b <= SSIM_R; ++b) {
                        int rr = r + a, cc = c + b;
                        if (rr < 0 || rr >= H || cc < 0 || cc >= W) continue;
                        double w = g[a + SSIM_R] * g[b + SSIM_R];
                        double xv = x[((int64_t)rr * W + cc) * 3 + ch];
                        double yv = y[((int64_t)rr * W + cc) * 3 + ch];
                        mx += w * xv;
                        my += w * yv;
                        exx += w * xv * xv;
                        eyy += w * yv * yv;
                        exy += w * xv * yv;
                    }
                double vx = exx - mx * mx, vy = eyy - my * my, cov = exy - mx * my;
                double A1 = 2.0 * mx * my + c1, A2 = 2.0 * cov + c2;
                double B1 = mx * mx + my * my + c1, B2 = vx + vy + c2;
                double D = B1 * B2;
                double s = A1 * A2 / D;
                int64_t i = ((int64_t)r * W + c) * 3 + ch;
                if (ssim_map) ssim_map[i] = s;
                dmu[i] = (2.0 * my * (A2 - A1) - 2.0 * mx * s * (B2 - B1)) / D;
                dxx[i] = -s / B2;
                dxy[i] = 2.0 * A1 / D;
                ssim += s;
                l1 += fabs((double)x[i] - (double)y[i]);
            }
    out[1] = l1 * inv;
    out[2] = ssim * inv;
    out[0] = (1.0 - lambda) * out[1] + lambda * (1.0 - out[2]);
    for (int r = 0; r < H; ++r)
        for (int c = 0; c < W; ++c)
            for (int ch = 0; ch < 3; ++ch) {
                int64_t i = ((int64_t)r * W + c) * 3 + ch;
                double xv = x[i], yv = y[i];
                double ds = 0.0, da = 0.0;
                for (int a = -SSIM_R; a <= SSIM_R; ++a)
                    for (int b = -SSIM_R; b <= SSIM_R; ++b) {
                        int rr = r + a, cc = c + b;
                        if (rr < 0 || rr >= H || cc < 0 || cc >= W) continue;
                        double w = g[a + SSIM_R] * g[b + SSIM_R];
                        int64_t q = ((int64_t)rr * W + cc) * 3 + ch;
                        ds += w * (dmu[q] + 2.0 * xv * dxx[q] + yv * dxy[q]);
                        da += w * (fabs(dmu[q]) + 2.0 * fabs(xv) * fabs(dxx[q]) +
                                   fabs(yv) * fabs(dxy[q]));
                    }
                double sg = xv > yv ? 1.0 : (xv < yv ? -1.0 : 0.0);
                dL_dx[i] = (1.0 - lambda) * inv * sg - lambda * inv * ds;
                if (mag) mag[i] = (1.0 - lambda) * inv + lambda * inv * da;
            }
    free(dmu);
    free(dxx);
    free(dxy);
}
