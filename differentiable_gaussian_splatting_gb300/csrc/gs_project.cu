// gs_project.cu -- per-Gaussian projection (forward) and its chain rule
// (backward), one thread per Gaussian, streaming from HBM.
//
// Forward: "Mitigating SM-Level Load Imbalance in 3D Gaussian Splatting on
// GPUs" (Ryu & Yoo), Sec. 2.1, Eq. 1; "What the 3DGS Literature Left on the
// Table" (Kopanas), Step 1 (b) opacity-aware support and exact spans, (c)
// 48-byte record, (e) visibility-gated SH with 16-byte loads; Step 3 (SH
// streamed in groups of four basis functions).
// Backward: the chain rule of the same formulas (Kopanas, Step 3: 59 gradient
// floats per Gaussian; culled rows are written as zeros in-kernel).
#include <cuda_runtime.h>

#include "gs_device.cuh"
#include "gs_internal.h"
#include "gs_project_variants.h"

namespace gs {

// ---------------------------------------------------------------------------
// real spherical harmonics, degree <= 3, no Condon-Shortley phase, in the
// order l = 0..3, m = -l..l (polynomials of the unit view direction)
// ---------------------------------------------------------------------------
constexpr float kY0 = 0.28209479177387814f;   // sqrt(1 / 4pi)
constexpr float kY1 = 0.48860251190291992f;   // sqrt(3 / 4pi)
constexpr float kY2a = 1.0925484305920792f;   // sqrt(15 / 4pi)
constexpr float kY2b = 0.31539156525252005f;  // sqrt(5 / 16pi)
constexpr float kY2c = 0.54627421529603959f;  // sqrt(15 / 16pi)
constexpr float kY3a = 0.59004358992664352f;  // sqrt(35 / 32pi)
constexpr float kY3b = 2.8906114426405538f;   // sqrt(105 / 4pi)
constexpr float kY3c = 0.45704579946446572f;  // sqrt(21 / 32pi)
constexpr float kY3d = 0.37317633259011540f;  // sqrt(7 / 16pi)
constexpr float kY3e = 1.4453057213202769f;   // sqrt(105 / 16pi)

// SH coefficients are fp32, or bfloat16 (the upper half of an fp32, as raw
// 16-bit patterns; widening is exact)
__device__ __forceinline__ float sh_at(const float* p, int64_t j) { return __ldg(p + j); }
__device__ __forceinline__ float sh_at(const uint16_t* p, int64_t j) {
    return __uint_as_float((uint32_t)__ldg(p + j) << 16);
}
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ void sh_values(float x, float y, float z, float Y[16]) {
    float xx = x * x, yy = y * y, zz = z * z;
    Y[0] = kY0;
    Y[1] = kY1 * y;
    Y[2] = kY1 * z;
    Y[3] = kY1 * x;
    Y[4] = kY2a * x * y;
    Y[5] = kY2a * y * z;
    Y[6] = kY2b * (3.f * zz - 1.f);
    Y[7] = kY2a * x * z;
    Y[8] = kY2c * (xx - yy);
    Y[9] = kY3a * y * (3.f * xx - yy);
    Y[10] = kY3b * x * y * z;
    Y[11] = kY3c * y * (5.f * zz - 1.f);
    Y[12] = kY3d * z * (5.f * zz - 3.f);
    Y[13] = kY3c * x * (5.f * zz - 1.f);
    Y[14] = kY3e * z * (xx - yy);
    Y[15] = kY3a * x * (xx - 3.f * yy);
}

// Cartesian gradient of basis function k at (x, y, z).
__device__ __forceinline__ float3 sh_grad(int k, float x, float y, float z) {
    switch (k) {
        case 1: return make_float3(0.f, kY1, 0.f);
        case 2: return make_float3(0.f, 0.f, kY1);
        case 3: return make_float3(kY1, 0.f, 0.f);
        case 4: return make_float3(kY2a * y, kY2a * x, 0.f);
        case 5: return make_float3(0.f, kY2a * z, kY2a * y);
        case 6: return make_float3(0.f, 0.f, 6.f * kY2b * z);
        case 7: return make_float3(kY2a * z, 0.f, kY2a * x);
        case 8: return make_float3(2.f * kY2c * x, -2.f * kY2c * y, 0.f);
        case 9: return make_float3(6.f * kY3a * x * y, 3.f * kY3a * (x * x - y * y), 0.f);
        case 10: return make_float3(kY3b * y * z, kY3b * x * z, kY3b * x * y);
        case 11: return make_float3(0.f, kY3c * (5.f * z * z - 1.f), 10.f * kY3c * y * z);
        case 12: return make_float3(0.f, 0.f, kY3d * (15.f * z * z - 3.f));
        case 13: return make_float3(kY3c * (5.f * z * z - 1.f), 0.f, 10.f * kY3c * x * z);
        case 14: return make_float3(2.f * kY3e * x * z, -2.f * kY3e * y * z, kY3e * (x * x - y * y));
        case 15: return make_float3(3.f * kY3a * (x * x - y * y), -6.f * kY3a * x * y, 0.f);
        default: return make_float3(0.f, 0.f, 0.f);
    }
}

// ---------------------------------------------------------------------------
// tau = fp32 rounding of 2 ln(255 o), in float-float arithmetic
// ---------------------------------------------------------------------------
// The threshold must be the correctly rounded fp32 value, which a double
// evaluation gives; FP64 is slow on this part, so the value is computed in
// float-float (a pair hi + lo of floats, about 44 bits) with ln x =
// e ln 2 + 2 atanh((m - 1) / (m + 1)), x = 2^e m, m in [sqrt(1/2), sqrt(2))
// (argument reduction by a power of two and the odd atanh series), and the
// rounding to fp32 is accepted only when a bound on the error keeps the value
// inside one fp32 rounding interval; otherwise (about one case in 10^4) the
// caller evaluates it in double.  All operations are round-to-nearest and
// uncontracted, as the error-free transformations require.
struct FF {
    float h, l;
};
__device__ __forceinline__ FF two_sum(float a, float b) {
    const float s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    return FF{s, __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb))};
}
__device__ __forceinline__ FF fast_two_sum(float a, float b) {  // |a| >= |b|
    const float s = __fadd_rn(a, b);
    return FF{s, __fsub_rn(b, __fsub_rn(s, a))};
}
__device__ __forceinline__ FF two_prod(float a, float b) {
    const float p = __fmul_rn(a, b);
    return FF{p, __fmaf_rn(a, b, -p)};
}
__device__ __forceinline__ FF ff_add(FF a, FF b) {
    const FF s = two_sum(a.h, b.h);
    return fast_two_sum(s.h, __fadd_rn(__fadd_rn(a.l, b.l), s.l));
}
__device__ __forceinline__ FF ff_mul(FF a, FF b) {
    const FF p = two_prod(a.h, b.h);
    return fast_two_sum(p.h, __fmaf_rn(a.h, b.l, __fmaf_rn(a.l, b.h, p.l)));
}

// *tau and true when the fp32 rounding is certain, false otherwise
__device__ __forceinline__ bool tau_float_float(float o, float* tau) {
    if (!(o > 0.f) || !(o < 1.0e30f)) return false;
    // x = 255 o exactly, as xh + xl
    const float xh = __fmul_rn(255.f, o);
    const float xl = __fmaf_rn(255.f, o, -xh);
    if (!(xh > 1.f || (xh == 1.f && xl > 0.f))) {
        *tau = 0.f;  // 255 o <= 1: tau <= 0 (culled either way)
        return true;
    }
    // x = 2^e (mh + ml), mh in [sqrt(1/2), sqrt(2)); the scalings are exact
    const int bits = __float_as_int(xh);
    int e = ((bits >> 23) & 0xff) - 127;
    float mh = __int_as_float((bits & 0x7fffff) | 0x3f800000);
    if (mh > 0x1.6a09e6p+0f) {
        mh = __fmul_rn(mh, 0.5f);
        e += 1;
    }
    const float ml = __fmul_rn(xl, __int_as_float((127 - e) << 23));
    // s = (M - 1) / (M + 1), M = mh + ml (mh - 1 is exact)
    const FF num = two_sum(__fsub_rn(mh, 1.f), ml);
    const FF d0 = two_sum(mh, 1.f);
    const FF den = fast_two_sum(d0.h, __fadd_rn(d0.l, ml));
    const float sh = __fdiv_rn(num.h, den.h);
    float r = __fmaf_rn(-sh, den.h, num.h);  // exact remainder
    r = __fmaf_rn(-sh, den.l, __fadd_rn(r, num.l));
    const FF s = fast_two_sum(sh, __fdiv_rn(r, den.h));
    // ln M = 2 s (1 + z P(z)), z = s^2 <= 0.0295, P = 1/3 + z/5 + z^2/7 + ...
    const FF z = ff_mul(s, s);
    float R = 0x1.af286cp-5f;                  // 1/19
    R = __fmaf_rn(R, z.h, 0x1.e1e1e2p-5f);     // 1/17
    R = __fmaf_rn(R, z.h, 0x1.111112p-4f);     // 1/15
    R = __fmaf_rn(R, z.h, 0x1.3b13b2p-4f);     // 1/13
    R = __fmaf_rn(R, z.h, 0x1.745d18p-4f);     // 1/11
    R = __fmaf_rn(R, z.h, 0x1.c71c72p-4f);     // 1/9
    FF P = ff_add(FF{0x1.24924ap-3f, -0x1.b6db6ep-28f}, two_prod(z.h, R));     // 1/7 + z R
    P = ff_add(FF{0x1.99999ap-3f, -0x1.99999ap-29f}, ff_mul(z, P));             // 1/5 + z P
    P = ff_add(FF{0x1.555556p-2f, -0x1.555556p-27f}, ff_mul(z, P));             // 1/3 + z P
    const FF u = ff_mul(z, P);
    const FF w = fast_two_sum(1.f, u.h);
    const FF lnM = ff_mul(s, fast_two_sum(w.h, __fadd_rn(w.l, u.l)));          // ln M / 2
    // ln x / 2 = e ln2 / 2 + ln M / 2; ln 2 = hi (15 bits, so e hi is exact) + lo + lo2
    const float fe = (float)e;
    const FF eln2 = fast_two_sum(__fmul_rn(fe, 0x1.62e4p-1f),
                                 __fmaf_rn(fe, 0x1.7f7d1cp-20f, __fmul_rn(fe, 0x1.ef357ap-45f)));
    const FF half_e = FF{__fmul_rn(eln2.h, 0.5f), __fmul_rn(eln2.l, 0.5f)};
    const FF L = ff_add(half_e, lnM);          // ln(x) / 2
    // tau = 4 L (exact scaling); accept the fp32 rounding if the error bound
    // (2^-36 relative) cannot cross the half gap to a neighbouring float
    const float Th = __fmul_rn(L.h, 4.f), Tl = __fmul_rn(L.l, 4.f);
    const int tb = __float_as_int(Th);
    const float gap = Tl >= 0.f ? __fsub_rn(__int_as_float(tb + 1), Th)
                                : __fsub_rn(Th, __int_as_float(tb - 1));
    if (!(__fadd_rn(fabsf(Tl), __fmul_rn(Th, 0x1p-36f)) < __fmul_rn(gap, 0.5f))) return false;
    *tau = Th;
    return true;
}

// ---------------------------------------------------------------------------
// the fp32 projection chain (fixed order, round-to-nearest)
// ---------------------------------------------------------------------------
struct Projected {
    bool ok;
    float tx, ty, tz;
    float mux, muy, l11, l12, l22, tau, rx, ry;
};

__device__ __forceinline__ Projected project_chain(const CamParams& cam, float mx, float my,
                                                   float mz, float s0, float s1, float s2,
                                                   float4 q4, float opac) {
    Projected P;
    P.ok = false;
    const float* V = cam.V;
    float tx = radd(radd(radd(rmul(V[0], mx), rmul(V[1], my)), rmul(V[2], mz)), V[3]);
    float ty = radd(radd(radd(rmul(V[4], mx), rmul(V[5], my)), rmul(V[6], mz)), V[7]);
    float tz = radd(radd(radd(rmul(V[8], mx), rmul(V[9], my)), rmul(V[10], mz)), V[11]);
    P.tx = tx;
    P.ty = ty;
    P.tz = tz;
    if (!(tz > cam.znear) || !isfinite(tx) || !isfinite(ty) || !isfinite(tz)) return P;

    float n2 = radd(radd(radd(rmul(q4.x, q4.x), rmul(q4.y, q4.y)), rmul(q4.z, q4.z)),
                    rmul(q4.w, q4.w));
    if (!(n2 > 0.f) || !isfinite(n2)) return P;
    float nr = rsqrt_exact(n2);
    float w = rdiv(q4.x, nr), x = rdiv(q4.y, nr), y = rdiv(q4.z, nr), z = rdiv(q4.w, nr);
    float R[9];
    R[0] = rsub(1.f, rmul(2.f, radd(rmul(y, y), rmul(z, z))));
    R[1] = rmul(2.f, rsub(rmul(x, y), rmul(w, z)));
    R[2] = rmul(2.f, radd(rmul(x, z), rmul(w, y)));
    R[3] = rmul(2.f, radd(rmul(x, y), rmul(w, z)));
    R[4] = rsub(1.f, rmul(2.f, radd(rmul(x, x), rmul(z, z))));
    R[5] = rmul(2.f, rsub(rmul(y, z), rmul(w, x)));
    R[6] = rmul(2.f, rsub(rmul(x, z), rmul(w, y)));
    R[7] = rmul(2.f, radd(rmul(y, z), rmul(w, x)));
    R[8] = rsub(1.f, rmul(2.f, radd(rmul(x, x), rmul(y, y))));
    float u = rdiv(tx, tz), v = rdiv(ty, tz);
    float mux = radd(rmul(cam.fx, u), cam.cx);
    float muy = radd(rmul(cam.fy, v), cam.cy);
    float j00 = rdiv(cam.fx, tz), j11 = rdiv(cam.fy, tz);
    float j02 = -rmul(j00, u), j12 = -rmul(j11, v);
    float T0[3], T1[3];
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        T0[k] = radd(rmul(j00, V[k]), rmul(j02, V[8 + k]));
        T1[k] = radd(rmul(j11, V[4 + k]), rmul(j12, V[8 + k]));
    }
    // Sigma' = N N^T with N = (T R) diag(s), T = J W (Eq. 1 with Sigma = R S S^T R^T)
    const float sv[3] = {s0, s1, s2};
    float n0[3], n1[3];
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        n0[k] = rmul(radd(radd(rmul(T0[0], R[k]), rmul(T0[1], R[3 + k])), rmul(T0[2], R[6 + k])), sv[k]);
        n1[k] = rmul(radd(radd(rmul(T1[0], R[k]), rmul(T1[1], R[3 + k])), rmul(T1[2], R[6 + k])), sv[k]);
    }
    float P00 = radd(radd(rmul(n0[0], n0[0]), rmul(n0[1], n0[1])), rmul(n0[2], n0[2]));
    float P01 = radd(radd(rmul(n0[0], n1[0]), rmul(n0[1], n1[1])), rmul(n0[2], n1[2]));
    float P11 = radd(radd(rmul(n1[0], n1[0]), rmul(n1[1], n1[1])), rmul(n1[2], n1[2]));
    // A support that cannot reach the image gets no tile from the spans: cull it
    // before the threshold, the conic factor and the extents.  o < 1 gives
    // tau < 2 ln 255 < 11.1, so the padded half extents (the spans' widening
    // included) stay below sqrt(11.1 Sigma'xx) * 1.001 + 0.02 and likewise in y;
    // a box that misses the pixel-centre hull of the image by those bounds has
    // no tile, which the full chain would also find (the outputs are the same).
    if (P00 >= 0.f && P11 >= 0.f) {
        const float bx = fmaf(sqrt_approx(11.1f * P00), 1.001f, 0.02f);
        const float by = fmaf(sqrt_approx(11.1f * P11), 1.001f, 0.02f);
        if (mux + bx < 0.5f || mux - bx > (float)cam.W - 0.5f || muy + by < 0.5f ||
            muy - by > (float)cam.H - 0.5f)
            return P;
    }
    // det Sigma' = |n0 x n1|^2 (Lagrange's identity) with n0 x n1 = s0 s1 s2 S^-1 R^T (T0 x T1):
    // a sum of squares, free of the cancellation of P00 P11 - P01^2 for thin splats
    float w0 = rsub(rmul(T0[1], T1[2]), rmul(T0[2], T1[1]));
    float w1 = rsub(rmul(T0[2], T1[0]), rmul(T0[0], T1[2]));
    float w2 = rsub(rmul(T0[0], T1[1]), rmul(T0[1], T1[0]));
    float c0 = radd(radd(rmul(R[0], w0), rmul(R[3], w1)), rmul(R[6], w2));
    float c1 = radd(radd(rmul(R[1], w0), rmul(R[4], w1)), rmul(R[7], w2));
    float c2 = radd(radd(rmul(R[2], w0), rmul(R[5], w1)), rmul(R[8], w2));
    float e0 = rmul(rmul(s1, s2), c0);
    float e1 = rmul(rmul(s0, s2), c1);
    float e2 = rmul(rmul(s0, s1), c2);
    float det = radd(radd(rmul(e0, e0), rmul(e1, e1)), rmul(e2, e2));
    if (!(det > 0.f) || !(P00 > 0.f) || !(P11 > 0.f) || !isfinite(det)) return P;
    float a = rdiv(P11, det);
    float b = -rdiv(P01, det);
    float c = rdiv(P00, det);
    // Cholesky factor of the conic from Sigma' (no cancellation beyond det):
    // l22 = 1/sqrt(P11), l11 = sqrt(P11/det), l12 = -(P01/P11) l11
    float l22 = rdiv(1.f, rsqrt_exact(P11));
    float l11 = rsqrt_exact(rdiv(P11, det));
    float l12 = -rmul(rdiv(P01, P11), l11);
    // tau = fp32 rounding of 2 ln(255 o): float-float, in double when undecided
    float tau;
    if (!tau_float_float(opac, &tau)) tau = __double2float_rn(2.0 * log(255.0 * (double)opac));
    if (!(tau > 0.f)) return P;
    float rx = rsqrt_exact(rmul(tau, P00));
    float ry = rsqrt_exact(rmul(tau, P11));
    if (!isfinite(mux) || !isfinite(muy) || !isfinite(a) || !isfinite(b) || !isfinite(c) ||
        !isfinite(l11) || !isfinite(l12) || !isfinite(l22) || !isfinite(rx) || !isfinite(ry))
        return P;
    P.mux = mux;
    P.muy = muy;
    P.l11 = l11;
    P.l12 = l12;
    P.l22 = l22;
    P.tau = tau;
    P.rx = rx;
    P.ry = ry;
    P.ok = true;
    return P;
}

// ---------------------------------------------------------------------------
// forward projection kernel
// ---------------------------------------------------------------------------
// One thread per Gaussian for the chain and the colour.  The tile count is a
// sum over the tile rows a splat's support may cover; rows per splat range
// from 0 (culled) to the image height, so the block spreads all its
// (Gaussian, row) pairs evenly over its threads instead of looping per thread.
// The kernel is bound by the latency of its long chain, so it wants many warps in
// flight: 128-thread blocks at 12 per SM (40 registers) keep 48 warps per SM and
// wait on smaller blocks at the row pass's barriers.
constexpr int kProjThreads = 128;

struct ProjShared {
    float e[8][kProjThreads];      // Ellipse fields, structure of arrays
    float dyv[kProjThreads];       // vertex_dy of each splat
    int ty0[kProjThreads];         // first row
    int off[kProjThreads + 1];     // exclusive prefix of row counts
    int cnt[kProjThreads];         // tile count
    int wsum[kProjThreads / 32];
};

template <int K, typename ShT>
__global__ void __launch_bounds__(kProjThreads, 12) project_kernel(CamParams cam, int64_t n,
                                                      const float* __restrict__ means,
                                                      const float* __restrict__ scales,
                                                      const float4* __restrict__ quats,
                                                      const float* __restrict__ opac,
                                                      const ShT* __restrict__ sh,
                                                      float4* __restrict__ splats,
                                                      float* __restrict__ depths,
                                                      int2* __restrict__ radii,
                                                      int* __restrict__ tiles_touched) {
    grid_dep_sync();
    __shared__ ProjShared S;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t i = (int64_t)blockIdx.x * kProjThreads + tid;
    const bool in = i < n;
    float mx = 0.f, my = 0.f, mz = 0.f, o = 0.f;
    Projected P;
    P.ok = false;
    if (in) {
        mx = means[3 * i];
        my = means[3 * i + 1];
        mz = means[3 * i + 2];
        o = opac[i];
        P = project_chain(cam, mx, my, mz, scales[3 * i], scales[3 * i + 1], scales[3 * i + 2],
                          quats[i], o);
    }
    int nrows = 0;
    if (P.ok) {
        const Ellipse e{P.mux, P.muy, P.l11, P.l12, P.l22, P.tau, P.rx, P.ry};
        int ty0, ty1;
        row_range(e, cam.nty, &ty0, &ty1);
        nrows = max(ty1 - ty0, 0);
        S.e[0][tid] = e.mux;
        S.e[1][tid] = e.muy;
        S.e[2][tid] = e.l11;
        S.e[3][tid] = e.l12;
        S.e[4][tid] = e.l22;
        S.e[5][tid] = e.tau;
        S.e[6][tid] = e.rx;
        S.e[7][tid] = e.ry;
        S.dyv[tid] = nrows > 0 ? vertex_dy(e) : 0.f;
        S.ty0[tid] = ty0;
        // the colour needs the SH row of every visible Gaussian: bring the rows of
        // those whose padded box meets the image into L2 while the rows are walked
        const float px = radd(P.rx, pad_of(P.rx));
        if (nrows > 0 && P.mux + px >= 0.5f && P.mux - px <= (float)cam.W - 0.5f) {
            constexpr int kRowBytes = K * 3 * (int)sizeof(ShT);
            const char* row = reinterpret_cast<const char*>(sh + i * (K * 3));
            if constexpr (kRowBytes % 16 == 0) {
                // exactly the row's bytes (whole 128-byte lines would fetch a third
                // more for a 192-byte row); rows start on 16-byte boundaries
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(row),
                             "r"(kRowBytes)
                             : "memory");
            } else {
#pragma unroll
                for (int b = 0; b < kRowBytes; b += 128)
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(row + b));
                asm volatile("prefetch.global.L2 [%0];" ::"l"(row + kRowBytes - 1));
            }
        }
    }
    S.cnt[tid] = 0;
    // block exclusive scan of the row counts
    int incl = nrows;
#pragma unroll
    for (int o2 = 1; o2 < 32; o2 <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o2);
        if (lane >= o2) incl += v;
    }
    if (lane == 31) S.wsum[warp] = incl;
    __syncthreads();
    int wbase = 0, total = 0;
#pragma unroll
    for (int w = 0; w < kProjThreads / 32; ++w) {
        const int v = S.wsum[w];
        wbase += w < warp ? v : 0;
        total += v;
    }
    S.off[tid] = wbase + incl - nrows;
    if (tid == 0) S.off[kProjThreads] = total;
    __syncthreads();
    for (int r = tid; r < total; r += kProjThreads) {
        // owner: the last g with off[g] <= r (splats without rows share the next offset)
        int lo = 0, hi = kProjThreads;  // off[lo] <= r < off[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (S.off[mid] <= r) lo = mid; else hi = mid;
        }
        const int g = lo;
        const Ellipse e{S.e[0][g], S.e[1][g], S.e[2][g], S.e[3][g],
                        S.e[4][g], S.e[5][g], S.e[6][g], S.e[7][g]};
        const int ty = S.ty0[g] + (r - S.off[g]);
        int tx0, tx1;
        if (row_span(e, S.dyv[g], ty, cam.W, cam.H, cam.ntx, &tx0, &tx1))
            atomicAdd(&S.cnt[g], tx1 - tx0);
    }
    __syncthreads();
    if (!in) return;
    const int tiles = S.cnt[tid];
    float4* rec = splats + 3 * i;
    if (!P.ok || tiles == 0) {
        float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
        rec[0] = z;
        rec[1] = z;
        rec[2] = z;
        depths[i] = 0.f;
        radii[i] = make_int2(0, 0);
        tiles_touched[i] = 0;
        return;
    }
    // colour, only for visible Gaussians: c = sum_k Y_k(d) s_k
    float dx = mx - cam.cw[0], dy = my - cam.cw[1], dz = mz - cam.cw[2];
    float inv = rsqrtf(dx * dx + dy * dy + dz * dz);
    float Y[16];
    sh_values(dx * inv, dy * inv, dz * inv, Y);
    float cr = 0.f, cg = 0.f, cb = 0.f;
    const ShT* row = sh + (int64_t)i * (K * 3);
    if constexpr (sizeof(ShT) == 2 && (K * 3) % 24 == 0) {
        // bfloat16: groups of eight basis functions = three 16-byte loads
        const uint4* r4 = reinterpret_cast<const uint4*>(row);
#pragma unroll
        for (int g = 0; g < K / 8; ++g) {
            const uint4 a = __ldg(r4 + 3 * g), b = __ldg(r4 + 3 * g + 1), c = __ldg(r4 + 3 * g + 2);
            const uint32_t w[12] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w, c.x, c.y, c.z, c.w};
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                // coefficients 3q, 3q + 1, 3q + 2 of the group (two per 32-bit word)
                const int e0 = 3 * q, e1 = 3 * q + 1, e2 = 3 * q + 2;
                const float v0 = (e0 & 1) ? bf16_hi(w[e0 >> 1]) : bf16_lo(w[e0 >> 1]);
                const float v1 = (e1 & 1) ? bf16_hi(w[e1 >> 1]) : bf16_lo(w[e1 >> 1]);
                const float v2 = (e2 & 1) ? bf16_hi(w[e2 >> 1]) : bf16_lo(w[e2 >> 1]);
                const float y = Y[8 * g + q];
                cr += y * v0;
                cg += y * v1;
                cb += y * v2;
            }
        }
    } else if constexpr (sizeof(ShT) == 2) {
#pragma unroll
        for (int k = 0; k < K; ++k) {
            cr += Y[k] * sh_at(row, 3 * k);
            cg += Y[k] * sh_at(row, 3 * k + 1);
            cb += Y[k] * sh_at(row, 3 * k + 2);
        }
    } else if constexpr ((K * 3) % 4 == 0) {
        // groups of four basis functions = three float4 (Kopanas, Step 3)
        const float4* r4 = reinterpret_cast<const float4*>(row);
#pragma unroll
        for (int g = 0; g < K / 4; ++g) {
            float4 v0 = __ldg(r4 + 3 * g), v1 = __ldg(r4 + 3 * g + 1), v2 = __ldg(r4 + 3 * g + 2);
            float y0 = Y[4 * g], y1 = Y[4 * g + 1], y2 = Y[4 * g + 2], y3 = Y[4 * g + 3];
            cr += y0 * v0.x + y1 * v0.w + y2 * v1.z + y3 * v2.y;
            cg += y0 * v0.y + y1 * v1.x + y2 * v1.w + y3 * v2.z;
            cb += y0 * v0.z + y1 * v1.y + y2 * v2.x + y3 * v2.w;
        }
    } else {
#pragma unroll
        for (int k = 0; k < K; ++k) {
            cr += Y[k] * __ldg(row + 3 * k);
            cg += Y[k] * __ldg(row + 3 * k + 1);
            cb += Y[k] * __ldg(row + 3 * k + 2);
        }
    }
    rec[0] = make_float4(P.mux, P.muy, P.l11, P.l12);
    rec[1] = make_float4(P.l22, P.tau, log2f(o), P.rx);
    rec[2] = make_float4(cr, cg, cb, P.ry);
    depths[i] = P.tz;
    radii[i] = make_int2(to_int_clamped(ceilf(P.rx), 0, kRadiusMax),
                         to_int_clamped(ceilf(P.ry), 0, kRadiusMax));
    tiles_touched[i] = tiles;
}

template <typename ShT>
cudaError_t launch_project_t(const CamParams& cam, int64_t n, int sh_degree, const float* means,
                             const float* scales, const float* quats, const float* opacities,
                             const ShT* sh, float* splats, float* depths, int32_t* radii,
                             int32_t* tiles_touched, cudaStream_t st) {
    if (n == 0) return cudaSuccess;
    dim3 block(kProjThreads), grid((unsigned)((n + kProjThreads - 1) / kProjThreads));
    auto q4 = reinterpret_cast<const float4*>(quats);
    auto s4 = reinterpret_cast<float4*>(splats);
    auto r2 = reinterpret_cast<int2*>(radii);
    auto go = [&](auto kernel) {
        return launch(kernel, grid, block, 0, st, cam, n, means, scales, q4, opacities, sh, s4,
                      depths, r2, tiles_touched);
    };
    switch (sh_degree) {
        case 0: return go(project_kernel<1, ShT>);
        case 1: return go(project_kernel<4, ShT>);
        case 2: return go(project_kernel<9, ShT>);
        default: return go(project_kernel<16, ShT>);
    }
}

cudaError_t launch_project(const CamParams& cam, int64_t n, int sh_degree, const float* means,
                           const float* scales, const float* quats, const float* opacities,
                           const float* sh, float* splats, float* depths, int32_t* radii,
                           int32_t* tiles_touched, cudaStream_t st) {
    return launch_project_t(cam, n, sh_degree, means, scales, quats, opacities, sh, splats,
                            depths, radii, tiles_touched, st);
}

cudaError_t launch_project_sh16(const CamParams& cam, int64_t n, int sh_degree, const float* means,
                                const float* scales, const float* quats, const float* opacities,
                                const uint16_t* sh, float* splats, float* depths, int32_t* radii,
                                int32_t* tiles_touched, cudaStream_t st) {
    return launch_project_t(cam, n, sh_degree, means, scales, quats, opacities, sh, splats,
                            depths, radii, tiles_touched, st);
}

// ---------------------------------------------------------------------------
// backward: nine screen-space derivatives -> 59 parameter gradients
// ---------------------------------------------------------------------------
// One thread per Gaussian.  The SH rows (12 K bytes each) dominate the traffic:
// each warp copies the rows of its live Gaussians into shared memory with
// contiguous loads, every lane turns its row into the SH gradient in place, and
// the warp writes its 32 consecutive gradient rows (zeros for the others) with
// contiguous stores.
constexpr int kPbThreads = 128;

// A parameter read: through the read-only path, except when the kernel updates
// the parameters in place (the fused Adam step)
template <bool kInPlace, typename T>
__device__ __forceinline__ T ld_param(const T* p) {
    if constexpr (kInPlace) return *p;
    else return __ldg(p);
}

// One Adam step of one parameter (fp32): the moments are updated in place and
// the new parameter value is returned.  The step's square root and reciprocal
// are the hardware approximations (about one unit in the last place each): the
// step size needs no correct rounding, and the exact forms cost most of the
// kernel's instructions
__device__ __forceinline__ float adam1(float p, float& m, float& v, float g, float lr,
                                       const AdamArgs& a) {
    m = fmaf(a.b1, m, (1.f - a.b1) * g);
    v = fmaf(a.b2, v, (1.f - a.b2) * (g * g));
    return p - lr * (m * a.c1) * rcp_approx(sqrt_approx(v * a.c2) + a.eps);
}

__device__ __forceinline__ void adam_at(float* p, float* m, float* v, int64_t j, float g, float lr,
                                        const AdamArgs& a) {
    float mj = m[j], vj = v[j];
    p[j] = adam1(p[j], mj, vj, g, lr, a);
    m[j] = mj;
    v[j] = vj;
}

// kAdam: the parameters are the raw ones (means, log-scales, quaternions,
// opacity logits, SH in ad.p[]); instead of writing gradients the kernel takes
// one Adam step on them (scales = exp(log-scales), opacities = sigmoid(logits)).
template <int K, typename ShT, bool kAdam>
__global__ void __launch_bounds__(kPbThreads) project_bwd_kernel(
    CamParams cam, int64_t n, const float* means, const float* scales, const float4* quats,
    const ShT* sh, const int* __restrict__ tiles_touched, const float* __restrict__ grad2d,
    const uint8_t* __restrict__ touched, float* __restrict__ dmeans, float* __restrict__ dscales,
    float4* __restrict__ dquats, float* __restrict__ dopac, float* __restrict__ dsh, AdamArgs ad) {
    grid_dep_sync();
    constexpr int RW = K * 3;                       // floats per SH row
    constexpr bool kVec = (RW % 4) == 0;            // rows of whole float4
    // staged rows of whole float4 sit an odd number of float4 apart, so that the
    // lanes' 16-byte accesses to their own rows fall in distinct bank groups
    constexpr int R4 = kVec ? RW / 4 : 1;           // float4 per row
    constexpr int RS = kVec ? 4 * (R4 | 1) : RW;    // floats from one staged row to the next
    __shared__ __align__(16) float srow[kPbThreads / 32][32 * RS];
    __shared__ int slive[kPbThreads / 32][32];  // rank among the live lanes -> lane
    // bfloat16 rows of whole 16-byte words are staged in the upper part of the
    // lane's fp32 row, whose gradients are written from its start: a group's
    // coefficients are read before its gradients overwrite them
    constexpr bool kVec16 = sizeof(ShT) == 2 && (RW % 8) == 0;
    constexpr int R8 = kVec16 ? RW / 8 : 1;         // 16-byte words per bfloat16 row
    constexpr int kOff16 = RS / 4 - R8;             // its first word within the row
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t wbase = (int64_t)blockIdx.x * kPbThreads + warp * 32;
    const int64_t i = wbase + lane;
    const bool in = i < n;
    const bool live = in && tiles_touched[i] > 0 && (touched == nullptr || touched[i] != 0);
    float* my = srow[warp];
    // this lane's inputs, requested before the SH rows are staged
    float g[9], m[3], s[3];
    float4 q4 = make_float4(0.f, 0.f, 0.f, 0.f);
    float sig = 0.f;  // the opacity, for the logit's chain rule (fused Adam)
    if (live) {
#pragma unroll
        for (int r = 0; r < 9; ++r) g[r] = grad2d[9 * i + r];
#pragma unroll
        for (int r = 0; r < 3; ++r) {
            m[r] = ld_param<kAdam>(means + 3 * i + r);
            s[r] = ld_param<kAdam>(scales + 3 * i + r);
            if constexpr (kAdam) s[r] = expf(s[r]);
        }
        q4 = ld_param<kAdam>(quats + i);
        if constexpr (kAdam) sig = 1.f / (1.f + expf(-ad.p[3][i]));
    }

    // ---- stage the live rows (others read as zero and are never used)
    const uint32_t lmask = __ballot_sync(0xffffffffu, live);
    if constexpr (kVec16) {
        const uint4* sh16 = reinterpret_cast<const uint4*>(sh);
        uint4* my16 = reinterpret_cast<uint4*>(my);
        const int nl = __popc(lmask);
        if (live) slive[warp][__popc(lmask & ((1u << lane) - 1u))] = lane;
        __syncwarp();
        for (int f = lane; f < nl * R8; f += 32) {
            const int rank = f / R8, col = f - rank * R8;
            const int l = slive[warp][rank];
            cp_async16(&my16[l * (RS / 4) + kOff16 + col], sh16 + (wbase + l) * R8 + col);
        }
        cp_async_commit();  // waited for after the geometric part below
    } else if constexpr (sizeof(ShT) == 2) {
        if (live) {
#pragma unroll
            for (int j = 0; j < RW; ++j) my[lane * RS + j] = sh_at(sh, i * RW + j);
        }
    } else if constexpr (kVec) {
        const float4* sh4 = reinterpret_cast<const float4*>(sh);
        float4* my4 = reinterpret_cast<float4*>(my);
        const int nl = __popc(lmask);
        if (live) slive[warp][__popc(lmask & ((1u << lane) - 1u))] = lane;
        __syncwarp();
        for (int f = lane; f < nl * R4; f += 32) {
            const int rank = f / R4, col = f - rank * R4;
            const int l = slive[warp][rank];
            cp_async16(&my4[l * (RS / 4) + col], sh4 + (wbase + l) * R4 + col);
        }
        cp_async_commit();  // waited for after the geometric part below
    } else {
        if (live) {
#pragma unroll
            for (int j = 0; j < RW; ++j) my[lane * RW + j] = ld_param<kAdam>(sh + i * RW + j);
        }
    }

    // ---- the geometric part (no SH needed), while the SH rows arrive
    float dm[3] = {0.f, 0.f, 0.f}, ds[3] = {0.f, 0.f, 0.f};
    float4 dq = make_float4(0.f, 0.f, 0.f, 0.f);
    if (live) {
        const float* V = cam.V;

        // ---- forward recomputation (fp32) ----
        float t[3];
#pragma unroll
        for (int r = 0; r < 3; ++r) t[r] = V[4 * r] * m[0] + V[4 * r + 1] * m[1] + V[4 * r + 2] * m[2] + V[4 * r + 3];
        float qn = sqrtf(q4.x * q4.x + q4.y * q4.y + q4.z * q4.z + q4.w * q4.w);
        float iqn = 1.f / qn;
        float w = q4.x * iqn, x = q4.y * iqn, y = q4.z * iqn, z = q4.w * iqn;
        float R[9] = {1.f - 2.f * (y * y + z * z), 2.f * (x * y - w * z), 2.f * (x * z + w * y),
                      2.f * (x * y + w * z), 1.f - 2.f * (x * x + z * z), 2.f * (y * z - w * x),
                      2.f * (x * z - w * y), 2.f * (y * z + w * x), 1.f - 2.f * (x * x + y * y)};
        float tz = t[2], iz = 1.f / tz;
        float u = t[0] * iz, v = t[1] * iz;
        float j00 = cam.fx * iz, j11 = cam.fy * iz, j02 = -j00 * u, j12 = -j11 * v;
        float T0[3], T1[3];
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            T0[k] = j00 * V[k] + j02 * V[8 + k];
            T1[k] = j11 * V[4 + k] + j12 * V[8 + k];
        }
        // Sigma' = N N^T, N = A diag(s), A = T R
        float A0[3], A1[3], n0[3], n1[3];
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            A0[k] = T0[0] * R[k] + T0[1] * R[3 + k] + T0[2] * R[6 + k];
            A1[k] = T1[0] * R[k] + T1[1] * R[3 + k] + T1[2] * R[6 + k];
            n0[k] = A0[k] * s[k];
            n1[k] = A1[k] * s[k];
        }
        // nu = n0 x n1 = s0 s1 s2 S^-1 R^T (T0 x T1) and det Sigma' = |nu|^2 (see the forward)
        float w0 = T0[1] * T1[2] - T0[2] * T1[1];
        float w1 = T0[2] * T1[0] - T0[0] * T1[2];
        float w2 = T0[0] * T1[1] - T0[1] * T1[0];
        float nu[3] = {s[1] * s[2] * (R[0] * w0 + R[3] * w1 + R[6] * w2),
                       s[0] * s[2] * (R[1] * w0 + R[4] * w1 + R[7] * w2),
                       s[0] * s[1] * (R[2] * w0 + R[5] * w1 + R[8] * w2)};
        float idet = 1.f / (nu[0] * nu[0] + nu[1] * nu[1] + nu[2] * nu[2]);
        // dual basis of N's rows, M = Lambda N: m0 = (n1 x nu) / det, m1 = (nu x n0) / det;
        // Lambda = M M^T.  Forming Lambda a_k through adj(Sigma') cancels for thin splats.
        float m0[3] = {(n1[1] * nu[2] - n1[2] * nu[1]) * idet, (n1[2] * nu[0] - n1[0] * nu[2]) * idet,
                       (n1[0] * nu[1] - n1[1] * nu[0]) * idet};
        float m1[3] = {(nu[1] * n0[2] - nu[2] * n0[1]) * idet, (nu[2] * n0[0] - nu[0] * n0[2]) * idet,
                       (nu[0] * n0[1] - nu[1] * n0[0]) * idet};
        float L00 = m0[0] * m0[0] + m0[1] * m0[1] + m0[2] * m0[2];
        float L01 = m0[0] * m1[0] + m0[1] * m1[1] + m0[2] * m1[2];
        float L11 = m1[0] * m1[0] + m1[1] * m1[1] + m1[2] * m1[2];

        // ---- conic -> Sigma' = N N^T -> N: dL/dN = 2 dSigma' N = -2 Lambda G M,
        //      G = [[ga, gb/2], [gb/2, gc]] ----
        float ga = g[2], gbh = 0.5f * g[3], gc = g[4];
        // ---- N = A diag(s) -> ds, dA; A = T R -> dT, dR ----
        float dT0[3] = {0.f, 0.f, 0.f}, dT1[3] = {0.f, 0.f, 0.f};
        float dR[9];
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            const float gm0 = ga * m0[k] + gbh * m1[k];
            const float gm1 = gbh * m0[k] + gc * m1[k];
            const float dn0 = -2.f * (L00 * gm0 + L01 * gm1);
            const float dn1 = -2.f * (L01 * gm0 + L11 * gm1);
            ds[k] = dn0 * A0[k] + dn1 * A1[k];
            const float dA0 = dn0 * s[k], dA1 = dn1 * s[k];
#pragma unroll
            for (int r = 0; r < 3; ++r) {
                dT0[r] += R[3 * r + k] * dA0;
                dT1[r] += R[3 * r + k] * dA1;
                dR[3 * r + k] = T0[r] * dA0 + T1[r] * dA1;
            }
        }

        // ---- T = J W -> dJ; (mu', J) -> dt -> dm ----
        float dj00 = dT0[0] * V[0] + dT0[1] * V[1] + dT0[2] * V[2];
        float dj02 = dT0[0] * V[8] + dT0[1] * V[9] + dT0[2] * V[10];
        float dj11 = dT1[0] * V[4] + dT1[1] * V[5] + dT1[2] * V[6];
        float dj12 = dT1[0] * V[8] + dT1[1] * V[9] + dT1[2] * V[10];
        float gmx = g[0], gmy = g[1];
        float dtx = (gmx - dj02 * iz) * j00;
        float dty = (gmy - dj12 * iz) * j11;
        float dtz = -(gmx * j00 * u + gmy * j11 * v) - (dj00 * j00 + dj11 * j11) * iz +
                    2.f * (dj02 * j00 * u + dj12 * j11 * v) * iz;
#pragma unroll
        for (int c = 0; c < 3; ++c) dm[c] = V[c] * dtx + V[4 + c] * dty + V[8 + c] * dtz;

        // ---- R(w, x, y, z) -> normalised quaternion -> raw quaternion ----
        float dw = -2.f * z * dR[1] + 2.f * y * dR[2] + 2.f * z * dR[3] - 2.f * x * dR[5] -
                   2.f * y * dR[6] + 2.f * x * dR[7];
        float dx_ = 2.f * y * dR[1] + 2.f * z * dR[2] + 2.f * y * dR[3] - 4.f * x * dR[4] -
                    2.f * w * dR[5] + 2.f * z * dR[6] + 2.f * w * dR[7] - 4.f * x * dR[8];
        float dy_ = -4.f * y * dR[0] + 2.f * x * dR[1] + 2.f * w * dR[2] + 2.f * x * dR[3] +
                    2.f * z * dR[5] - 2.f * w * dR[6] + 2.f * z * dR[7] - 4.f * y * dR[8];
        float dz_ = -4.f * z * dR[0] - 2.f * w * dR[1] + 2.f * x * dR[2] + 2.f * w * dR[3] -
                    4.f * z * dR[4] + 2.f * y * dR[5] + 2.f * x * dR[6] + 2.f * y * dR[7];
        float dot = w * dw + x * dx_ + y * dy_ + z * dz_;
        dq = make_float4((dw - w * dot) * iqn, (dx_ - x * dot) * iqn, (dy_ - y * dot) * iqn,
                         (dz_ - z * dot) * iqn);
    }
    if constexpr (kVec || kVec16) cp_async_wait<0>();
    __syncwarp();

    if (live) {
        // ---- colour -> SH coefficients (in place in the staged row) and view direction ----
        float ex = m[0] - cam.cw[0], ey = m[1] - cam.cw[1], ez = m[2] - cam.cw[2];
        float ilen = rsqrtf(ex * ex + ey * ey + ez * ez);
        float hx = ex * ilen, hy = ey * ilen, hz = ez * ilen;
        float Y[16];
        sh_values(hx, hy, hz, Y);
        float gr = g[6], gg = g[7], gbl = g[8];
        float* row = my + lane * RS;
        float gdx = 0.f, gdy = 0.f, gdz = 0.f;
        auto basis = [&](int k, float c0, float c1, float c2) {
            const float p = gr * c0 + gg * c1 + gbl * c2;
            const float3 dY = sh_grad(k, hx, hy, hz);
            gdx += p * dY.x;
            gdy += p * dY.y;
            gdz += p * dY.z;
        };
        if constexpr (kVec16) {
            // bfloat16 coefficients from the staged row, eight basis functions
            // (three 16-byte words) at a time; their gradients into the fp32 row
            const uint4* s16 = reinterpret_cast<const uint4*>(row) + kOff16;
            float4* r4 = reinterpret_cast<float4*>(row);
#pragma unroll
            for (int q8 = 0; q8 < K / 8; ++q8) {
                const uint4 a = s16[3 * q8], b = s16[3 * q8 + 1], c = s16[3 * q8 + 2];
                const uint32_t wd[12] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w, c.x, c.y, c.z, c.w};
                float o[24];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int e = 3 * q;
                    const float c0 = (e & 1) ? bf16_hi(wd[e >> 1]) : bf16_lo(wd[e >> 1]);
                    const float c1 = ((e + 1) & 1) ? bf16_hi(wd[(e + 1) >> 1]) : bf16_lo(wd[(e + 1) >> 1]);
                    const float c2 = ((e + 2) & 1) ? bf16_hi(wd[(e + 2) >> 1]) : bf16_lo(wd[(e + 2) >> 1]);
                    const float y = Y[8 * q8 + q];
                    o[e] = y * gr;
                    o[e + 1] = y * gg;
                    o[e + 2] = y * gbl;
                    basis(8 * q8 + q, c0, c1, c2);
                }
#pragma unroll
                for (int f = 0; f < 6; ++f)
                    r4[6 * q8 + f] = make_float4(o[4 * f], o[4 * f + 1], o[4 * f + 2], o[4 * f + 3]);
            }
        } else if constexpr (kVec) {
            // groups of four basis functions = three float4 of the row
            float4* r4 = reinterpret_cast<float4*>(row);
#pragma unroll
            for (int q = 0; q < K / 4; ++q) {
                const float4 v0 = r4[3 * q], v1 = r4[3 * q + 1], v2 = r4[3 * q + 2];
                const float y0 = Y[4 * q], y1 = Y[4 * q + 1], y2 = Y[4 * q + 2], y3 = Y[4 * q + 3];
                r4[3 * q] = make_float4(y0 * gr, y0 * gg, y0 * gbl, y1 * gr);
                r4[3 * q + 1] = make_float4(y1 * gg, y1 * gbl, y2 * gr, y2 * gg);
                r4[3 * q + 2] = make_float4(y2 * gbl, y3 * gr, y3 * gg, y3 * gbl);
                basis(4 * q, v0.x, v0.y, v0.z);
                basis(4 * q + 1, v0.w, v1.x, v1.y);
                basis(4 * q + 2, v1.z, v1.w, v2.x);
                basis(4 * q + 3, v2.y, v2.z, v2.w);
            }
        } else {
#pragma unroll
            for (int k = 0; k < K; ++k) {
                const float c0 = row[3 * k], c1 = row[3 * k + 1], c2 = row[3 * k + 2];
                row[3 * k] = Y[k] * gr;
                row[3 * k + 1] = Y[k] * gg;
                row[3 * k + 2] = Y[k] * gbl;
                basis(k, c0, c1, c2);
            }
        }
        float dd = hx * gdx + hy * gdy + hz * gdz;
        dm[0] += (gdx - hx * dd) * ilen;
        dm[1] += (gdy - hy * dd) * ilen;
        dm[2] += (gdz - hz * dd) * ilen;

        if constexpr (!kAdam) {
            dmeans[3 * i] = dm[0];
            dmeans[3 * i + 1] = dm[1];
            dmeans[3 * i + 2] = dm[2];
            dscales[3 * i] = ds[0];
            dscales[3 * i + 1] = ds[1];
            dscales[3 * i + 2] = ds[2];
            dquats[i] = dq;
            dopac[i] = g[5];
        }
    } else if (in) {
        if constexpr (!kAdam) {
            dmeans[3 * i] = dmeans[3 * i + 1] = dmeans[3 * i + 2] = 0.f;
            dscales[3 * i] = dscales[3 * i + 1] = dscales[3 * i + 2] = 0.f;
            dquats[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            dopac[i] = 0.f;
        }
    }
    if constexpr (kAdam) {
        // every Gaussian takes the step (zero gradients where not live): the raw
        // gradients are dL/dlog s = s dL/ds and dL/dlogit = o (1 - o) dL/do
        if (in) {
            // the eleven geometric values: every load first, then the steps, then
            // every store (the compiler cannot reorder them across the stores)
            const int grp[11] = {0, 0, 0, 1, 1, 1, 2, 2, 2, 2, 3};
            const int64_t idx[11] = {3 * i, 3 * i + 1, 3 * i + 2, 3 * i, 3 * i + 1, 3 * i + 2,
                                     4 * i, 4 * i + 1, 4 * i + 2, 4 * i + 3, i};
            const float gv[11] = {dm[0], dm[1], dm[2], ds[0] * s[0], ds[1] * s[1], ds[2] * s[2],
                                  dq.x, dq.y, dq.z, dq.w, g[5] * sig * (1.f - sig)};
            float pv[11], mv[11], vv[11];
#pragma unroll
            for (int e = 0; e < 11; ++e) {
                pv[e] = ad.p[grp[e]][idx[e]];
                mv[e] = ad.m[grp[e]][idx[e]];
                vv[e] = ad.v[grp[e]][idx[e]];
            }
#pragma unroll
            for (int e = 0; e < 11; ++e)
                pv[e] = adam1(pv[e], mv[e], vv[e], live ? gv[e] : 0.f, ad.lr[grp[e]], ad);
#pragma unroll
            for (int e = 0; e < 11; ++e) {
                ad.p[grp[e]][idx[e]] = pv[e];
                ad.m[grp[e]][idx[e]] = mv[e];
                ad.v[grp[e]][idx[e]] = vv[e];
            }
            if (ad.act_scales) {
#pragma unroll
                for (int r = 0; r < 3; ++r) ad.act_scales[3 * i + r] = expf(pv[3 + r]);
            }
            if (ad.act_opacities) ad.act_opacities[i] = 1.f / (1.f + expf(-pv[10]));
        }
    }
    __syncwarp();

    // ---- the warp's gradient rows, contiguous (zeros for the rows not live)
    const int nrows = (int)min64(32, n - wbase);
    if (nrows <= 0) return;
    if constexpr (kAdam && kVec) {
        // the SH rows' Adam step over the warp's rows in 16-byte words, four words
        // a lane in flight (band 0 is the first three values of a row)
        float4* P = reinterpret_cast<float4*>(ad.p[4]) + wbase * R4;
        float4* M = reinterpret_cast<float4*>(ad.m[4]) + wbase * R4;
        float4* Vv = reinterpret_cast<float4*>(ad.v[4]) + wbase * R4;
        const float4* my4 = reinterpret_cast<const float4*>(my);
        const int nf = nrows * R4;
        for (int f0 = lane; f0 < nf; f0 += 4 * 32) {
            float4 pw[4], mw[4], vw[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int f = f0 + 32 * u;
                if (f < nf) {
                    pw[u] = P[f];
                    mw[u] = M[f];
                    vw[u] = Vv[f];
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int f = f0 + 32 * u;
                if (f < nf) {
                    const int l = f / R4, col = f - l * R4;
                    const float4 gw = ((lmask >> l) & 1u) ? my4[l * (RS / 4) + col]
                                                          : make_float4(0.f, 0.f, 0.f, 0.f);
                    const float l0 = ad.lr[5], lb = col == 0 ? ad.lr[4] : ad.lr[5];
                    pw[u].x = adam1(pw[u].x, mw[u].x, vw[u].x, gw.x, lb, ad);
                    pw[u].y = adam1(pw[u].y, mw[u].y, vw[u].y, gw.y, lb, ad);
                    pw[u].z = adam1(pw[u].z, mw[u].z, vw[u].z, gw.z, lb, ad);
                    pw[u].w = adam1(pw[u].w, mw[u].w, vw[u].w, gw.w, l0, ad);
                    P[f] = pw[u];
                    M[f] = mw[u];
                    Vv[f] = vw[u];
                }
            }
        }
    } else if constexpr (kAdam) {
        float* P = ad.p[4] + wbase * RW;
        float* M = ad.m[4] + wbase * RW;
        float* Vv = ad.v[4] + wbase * RW;
        for (int f = lane; f < nrows * RW; f += 32) {
            const int l = f / RW, j = f - l * RW;
            const float gv = ((lmask >> l) & 1u) ? my[l * RS + j] : 0.f;
            adam_at(P, M, Vv, f, gv, j < 3 ? ad.lr[4] : ad.lr[5], ad);
        }
    } else if constexpr (kVec) {
        const float4* my4 = reinterpret_cast<const float4*>(my);
        float4* d4 = reinterpret_cast<float4*>(dsh) + wbase * R4;
        for (int f = lane; f < nrows * R4; f += 32) {
            const int l = f / R4, col = f - l * R4;
            d4[f] = ((lmask >> l) & 1u) ? my4[l * (RS / 4) + col] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    } else {
        float* d = dsh + wbase * RW;
        for (int f = lane; f < nrows * RW; f += 32) {
            const int l = f / RW;
            d[f] = ((lmask >> l) & 1u) ? my[f] : 0.f;
        }
    }
}

template <typename ShT>
cudaError_t launch_project_bwd_t(const CamParams& cam, int64_t n, int sh_degree,
                                 const float* means, const float* scales, const float* quats,
                                 const ShT* sh, const int32_t* tiles_touched, const float* grad2d,
                                 const uint8_t* touched, float* dmeans, float* dscales,
                                 float* dquats, float* dopacities, float* dsh, cudaStream_t st) {
    if (n == 0) return cudaSuccess;
    dim3 block(kPbThreads), grid((unsigned)((n + kPbThreads - 1) / kPbThreads));
    auto q4 = reinterpret_cast<const float4*>(quats);
    auto dq4 = reinterpret_cast<float4*>(dquats);
    auto go = [&](auto kernel) {
        return launch(kernel, grid, block, 0, st, cam, n, means, scales, q4, sh, tiles_touched,
                      grad2d, touched, dmeans, dscales, dq4, dopacities, dsh, AdamArgs{});
    };
    switch (sh_degree) {
        case 0: return go(project_bwd_kernel<1, ShT, false>);
        case 1: return go(project_bwd_kernel<4, ShT, false>);
        case 2: return go(project_bwd_kernel<9, ShT, false>);
        default: return go(project_bwd_kernel<16, ShT, false>);
    }
}

cudaError_t launch_project_bwd(const CamParams& cam, int64_t n, int sh_degree, const float* means,
                               const float* scales, const float* quats, const float* opacities,
                               const float* sh, const int32_t* tiles_touched, const float* grad2d,
                               const uint8_t* touched, float* dmeans, float* dscales,
                               float* dquats, float* dopacities, float* dsh, cudaStream_t st) {
    (void)opacities;
    return launch_project_bwd_t(cam, n, sh_degree, means, scales, quats, sh, tiles_touched,
                                grad2d, touched, dmeans, dscales, dquats, dopacities, dsh, st);
}

cudaError_t launch_project_bwd_sh16(const CamParams& cam, int64_t n, int sh_degree,
                                    const float* means, const float* scales, const float* quats,
                                    const float* opacities, const uint16_t* sh,
                                    const int32_t* tiles_touched, const float* grad2d,
                                    const uint8_t* touched, float* dmeans, float* dscales,
                                    float* dquats, float* dopacities, float* dsh, cudaStream_t st) {
    (void)opacities;
    return launch_project_bwd_t(cam, n, sh_degree, means, scales, quats, sh, tiles_touched,
                                grad2d, touched, dmeans, dscales, dquats, dopacities, dsh, st);
}

cudaError_t launch_project_bwd_adam(const CamParams& cam, int64_t n, int sh_degree,
                                    const int32_t* tiles_touched, const float* grad2d,
                                    const uint8_t* touched, const AdamArgs& adam, cudaStream_t st) {
    if (n == 0) return cudaSuccess;
    dim3 block(kPbThreads), grid((unsigned)((n + kPbThreads - 1) / kPbThreads));
    const float* means = adam.p[0];
    const float* log_scales = adam.p[1];
    auto q4 = reinterpret_cast<const float4*>(adam.p[2]);
    const float* sh = adam.p[4];
    auto go = [&](auto kernel) {
        return launch(kernel, grid, block, 0, st, cam, n, means, log_scales, q4, sh, tiles_touched,
                      grad2d, touched, (float*)nullptr, (float*)nullptr, (float4*)nullptr,
                      (float*)nullptr, (float*)nullptr, adam);
    };
    switch (sh_degree) {
        case 0: return go(project_bwd_kernel<1, float, true>);
        case 1: return go(project_bwd_kernel<4, float, true>);
        case 2: return go(project_bwd_kernel<9, float, true>);
        default: return go(project_bwd_kernel<16, float, true>);
    }
}

}  // namespace gs
