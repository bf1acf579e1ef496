// gs_device.cuh -- device helpers shared by the libgs kernels (sm_103a).
//
// The projection chain, the tile spans and the per-pixel quadratic decide
// integers (radii, tile counts, pair lists, hit tests).  They are written
// with explicit round-to-nearest intrinsics in one fixed operation order so
// that no multiply-add is contracted and every result is reproducible bit for
// bit, as the hit test must be ("What the 3DGS Literature Left on the Table",
// Step 5: exact round-to-nearest quadratic evaluation).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace gs {

constexpr int kTile = 16;
constexpr float kTMin = 1e-4f;
constexpr float kAlphaMax = 0.99f;
constexpr float kNegHalfLog2e = -0.72134752044448170368f;  // -log2(e) / 2
constexpr float kPadUnit = 0.00390625f;                     // 2^-8 px
constexpr float kPadScale = 9.5367431640625e-07f;           // 2^-20
constexpr float kDiscPad = 4.76837158203125e-07f;           // 2^-21 (of tau)
// the sub-tile mask's approximate square root and reciprocal: a wider margin
constexpr float kMaskPadScale = 1.52587890625e-05f;         // 2^-16
constexpr float kMaskDiscPad = 1.9073486328125e-06f;        // 2^-19 (of tau)
constexpr int kRadiusMax = 1 << 30;
constexpr int kMaxChunks = 16;  // largest k of the chunking policy

__host__ __device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
__host__ __device__ __forceinline__ int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

// ---------------------------------------------------------------------------
// round-to-nearest fp32 arithmetic (never contracted)
// ---------------------------------------------------------------------------
__device__ __forceinline__ float rmul(float a, float b) { return __fmul_rn(a, b); }
__device__ __forceinline__ float radd(float a, float b) { return __fadd_rn(a, b); }
__device__ __forceinline__ float rsub(float a, float b) { return __fsub_rn(a, b); }
__device__ __forceinline__ float rdiv(float a, float b) { return __fdiv_rn(a, b); }
__device__ __forceinline__ float rsqrt_exact(float a) { return __fsqrt_rn(a); }
__device__ __forceinline__ float rfma(float a, float b, float c) { return __fmaf_rn(a, b, c); }
// min / max with the semantics of `x < y ? x : y` (no NaN special-casing)
__device__ __forceinline__ float smin(float x, float y) { return x < y ? x : y; }
__device__ __forceinline__ float smax(float x, float y) { return x > y ? x : y; }

// 2^x on the SFU (flush-to-zero); results are tested against the oracle's exp()
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Programmatic dependent launch: every kernel starts with this.  It waits
// until the kernel launched before it on the stream has completed and its
// writes are visible (immediately, when it was launched without the
// programmatic-serialisation attribute), then lets the next kernel on the
// stream begin launching while this one runs.
__device__ __forceinline__ void grid_dep_sync() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// 16-byte asynchronous global -> shared copies; complete for the calling
// thread after cp_async_wait<N> (all but the N most recent groups)
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    const unsigned sa = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ int to_int_clamped(float f, int lo, int hi) {
    if (!(f >= (float)lo)) return lo;
    if (f > (float)hi) return hi;
    return (int)f;
}

// ---------------------------------------------------------------------------
// splat record: three float4 per splat (48 bytes, 16-byte aligned)
//   r0 = (mux, muy, l11, l12)   r1 = (l22, tau, log2 o, rx)   r2 = (r, g, b, ry)
// The conic Lambda = Sigma'^-1 is carried by its Cholesky factor
// L = [[l11, l12], [0, l22]] (Lambda = L^T L), so that the quadratic
// q = (l11 dx + l12 dy)^2 + (l22 dy)^2 is a sum of non-negative terms and its
// fp32 evaluation stays well conditioned for thin splats far from the image.
// ---------------------------------------------------------------------------
struct Ellipse {
    float mux, muy, l11, l12, l22, tau, rx, ry;
};

__device__ __forceinline__ Ellipse ellipse_of(const float4& r0, const float4& r1, const float4& r2) {
    return Ellipse{r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.w, r2.w};
}

// ---------------------------------------------------------------------------
// exact row spans ("What the 3DGS Literature Left on the Table", Step 1 (b))
// ---------------------------------------------------------------------------
// The support ellipse q(d) <= tau has right boundary
//   x_r(dy) = (sqrt(tau - (l22 dy)^2) - l12 dy) / l11,
// concave in dy with its vertex at dy = -sqrt(tau) l12 / (l22 h),
// h = sqrt(l12^2 + l22^2); the left boundary is x_l(dy) = -x_r(-dy).  The
// fp32 evaluation is widened just enough that every pixel whose fp32 hit test
// passes lies in an emitted tile (u = 2^-24): the discriminant, whose
// absolute error of about 4 u tau moves the boundary by about sqrt(u) r near
// the tips, gets + 2^-21 tau before the root; the other roundings of the span
// and of the hit test are a few u of the extent, covered by
// pad = 2^-8 px + r 2^-20 on the extents and bands (the 2^-8 px for the
// rounding of mu' + x_r in pixel coordinates up to a 32768-pixel image).
__device__ __forceinline__ float xr_at(const Ellipse& s, float dy) {
    float t = rmul(s.l22, dy);
    float disc = rsub(s.tau, rmul(t, t));
    if (!(disc > 0.f)) disc = 0.f;
    disc = radd(disc, rmul(s.tau, kDiscPad));
    return rdiv(rsub(rsqrt_exact(disc), rmul(s.l12, dy)), s.l11);
}

__device__ __forceinline__ float vertex_dy(const Ellipse& s) {
    float h = rsqrt_exact(radd(rmul(s.l12, s.l12), rmul(s.l22, s.l22)));
    return -rdiv(rmul(rsqrt_exact(s.tau), s.l12), rmul(s.l22, h));
}

__device__ __forceinline__ float pad_of(float r) { return radd(kPadUnit, rmul(r, kPadScale)); }

// x-extent [*Xlo, *Xhi] of the padded support over the y band [y0, y1] (pixel
// coordinates, y1 already clipped to the image); false if the band misses it.
// dyv is vertex_dy(s), computed once per splat by the caller.
__device__ __forceinline__ bool band_extent(const Ellipse& s, float dyv, float y0, float y1,
                                            float* Xlo, float* Xhi) {
    float padx = pad_of(s.rx);
    float ryp = radd(s.ry, pad_of(s.ry));
    float lo = smax(rsub(y0, s.muy), -ryp);
    float hi = smin(rsub(y1, s.muy), ryp);
    if (!(lo <= hi)) return false;
    float dh = smin(smax(smin(smax(dyv, lo), hi), -s.ry), s.ry);
    float dl = smin(smax(smin(smax(dyv, -hi), -lo), -s.ry), s.ry);
    float xhi = radd(xr_at(s, dh), padx);
    float xlo_neg = radd(xr_at(s, dl), padx);
    *Xhi = radd(s.mux, xhi);
    *Xlo = rsub(s.mux, xlo_neg);
    return true;
}

// Rows [*ty0, *ty1) the padded support may cover.
__device__ __forceinline__ void row_range(const Ellipse& s, int nty, int* ty0, int* ty1) {
    float ryp = radd(s.ry, pad_of(s.ry));
    float f0 = ceilf(rmul(rsub(rsub(s.muy, ryp), 15.5f), 0.0625f));
    float f1 = radd(floorf(rmul(rsub(radd(s.muy, ryp), 0.5f), 0.0625f)), 1.0f);
    *ty0 = to_int_clamped(f0, 0, nty);
    *ty1 = to_int_clamped(f1, 0, nty);
}

// Tile columns [*tx0, *tx1) of row ty; false when empty.  A tile's region is
// the closed hull of its pixel centres, clipped to the W x H image.  dyv is
// vertex_dy(s).
__device__ __forceinline__ bool row_span(const Ellipse& s, float dyv, int ty, int W, int H, int ntx,
                                         int* tx0, int* tx1) {
    float y0 = radd((float)(16 * ty), 0.5f);
    float y1 = smin(radd((float)(16 * ty), 15.5f), rsub((float)H, 0.5f));
    float Xlo, Xhi;
    if (!band_extent(s, dyv, y0, y1, &Xlo, &Xhi)) return false;
    if (Xlo > rsub((float)W, 0.5f) || Xhi < 0.5f) return false;
    float f0 = ceilf(rmul(rsub(Xlo, 15.5f), 0.0625f));
    float f1 = radd(floorf(rmul(rsub(Xhi, 0.5f), 0.0625f)), 1.0f);
    *tx0 = to_int_clamped(f0, 0, ntx);
    *tx1 = to_int_clamped(f1, 0, ntx);
    return *tx0 < *tx1;
}

// ---------------------------------------------------------------------------
// per-pixel quadratic: q = fma(u1, u1, u2 u2), u1 = fma(l11, dx, l12 dy), u2 = l22 dy
// ---------------------------------------------------------------------------
__device__ __forceinline__ float quad_q(float l11, float l12, float l22, float dx, float dy,
                                        float* u1_out, float* u2_out) {
    const float u1 = rfma(l11, dx, rmul(l12, dy));
    const float u2 = rmul(l22, dy);
    *u1_out = u1;
    *u2_out = u2;
    return rfma(u1, u1, rmul(u2, u2));
}

// ---------------------------------------------------------------------------
// 8x4 sub-tile mask ("What the 3DGS Literature Left on the Table", Step 1 (c)):
// bit w set if the padded support meets the pixel-centre hull of the 8x4
// sub-tile of warp w (warp w covers columns 8 (w & 1) .. +7, rows 4 (w >> 1) .. +3
// of the tile).  It only has to be conservative (every hit pixel of a warp has
// its bit set), so it uses the SFU's approximate square root and reciprocal
// with wider margins than the spans (2^-19 tau on the discriminant, r 2^-16 on
// the extents): their few-ulp errors are well inside those.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float sqrt_approx(float x) {
    float y;
    asm("sqrt.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t subtile_mask(const Ellipse& s, int tx, int ty, int W, int H) {
    const float inv_l11 = rcp_approx(s.l11);
    const float h = sqrt_approx(fmaf(s.l12, s.l12, s.l22 * s.l22));
    const float dyv = -(sqrt_approx(s.tau) * s.l12) * rcp_approx(s.l22 * h);
    const float padx = fmaf(s.rx, kMaskPadScale, kPadUnit);
    const float ryp = s.ry + fmaf(s.ry, kMaskPadScale, kPadUnit);
    const float dpad = s.tau * kMaskDiscPad;
    const float xb = (float)(16 * tx);
    const float xl0 = xb + 0.5f, xl1 = xb + 7.5f;
    const float xr0 = xb + 8.5f;
    const float xr1 = fminf(xb + 15.5f, (float)W - 0.5f);
    const float ylim = (float)H - 0.5f;
    uint32_t m = 0;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const float y0 = (float)(16 * ty + 4 * r) + 0.5f;
        if (y0 > ylim) break;
        const float y1 = fminf(y0 + 3.f, ylim);
        const float lo = fmaxf(y0 - s.muy, -ryp), hi = fminf(y1 - s.muy, ryp);
        if (!(lo <= hi)) continue;
        const float dh = fminf(fmaxf(fminf(fmaxf(dyv, lo), hi), -s.ry), s.ry);
        const float dl = fminf(fmaxf(fminf(fmaxf(dyv, -hi), -lo), -s.ry), s.ry);
        const float th = s.l22 * dh, tl = s.l22 * dl;
        const float xh = (sqrt_approx(fmaxf(fmaf(-th, th, s.tau), 0.f) + dpad) - s.l12 * dh) * inv_l11;
        const float xl = (sqrt_approx(fmaxf(fmaf(-tl, tl, s.tau), 0.f) + dpad) - s.l12 * dl) * inv_l11;
        const float Xhi = s.mux + xh + padx, Xlo = s.mux - xl - padx;
        if (Xhi >= xl0 && Xlo <= xl1) m |= 1u << (2 * r);
        if (xr0 <= xr1 && Xhi >= xr0 && Xlo <= xr1) m |= 1u << (2 * r + 1);
    }
    return m;
}

}  // namespace gs
