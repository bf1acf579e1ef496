// gs_loss.cu -- the photometric training loss before the backward, fused into
// one pass per 32 x 32 pixel tile: L = (1 - lambda) mean |x - y| +
// lambda (1 - mean SSIM(x, y)) and dL/dx, for the rendered image x and the
// target y, both [H][W][3].
//
// The pages' Metal port ("perf: rasterizer and pipeline optimizations",
// Breakdown and Queue) runs this stage as loss_fwd_bwd and names its cost: five
// windowed moments per colour channel (mu_x, mu_y, E[x^2], E[y^2], E[xy]) kept
// as [H][W][15] intermediates that go to memory and back.  Here they never
// leave the SM.  The structural similarity is that of Wang et al. (2004) over
// an 11 x 11 Gaussian window with zero outside the image.  Its gradient w.r.t.
// x(p) gathers, over the pixels q whose window holds p, the derivatives of
// SSIM(q) by mu_x(q), E[x^2](q) and E[xy](q), each blurred by the same window:
//
//   dSSIM/dx(p) = (w * a)(p) + 2 x(p) (w * b)(p) + y(p) (w * c)(p)
//   a = dS/dmu_x = (2 mu_y (A2 - A1) - 2 mu_x S (B2 - B1)) / (B1 B2)
//   b = dS/dE[x^2] = -S B1 / (B1 B2),   c = dS/dE[xy] = 2 A1 / (B1 B2)
//
// with A1 = 2 mu_x mu_y + c1, A2 = 2 cov + c2, B1 = mu_x^2 + mu_y^2 + c1,
// B2 = var_x + var_y + c2 and a = b = c = 0 outside the image.
//
// One block per tile, one colour channel at a time.  It stages x and y over
// the tile plus a 10-pixel halo, blurs the five products along rows then
// columns (the window is separable), forms S, a, b and c on the tile plus a
// 5-pixel halo, blurs those along rows then columns, and writes dL/dx for its
// own pixels after the third channel.  Every 1D pass keeps a strip of outputs
// per thread in registers, so each staged value is read from shared memory
// once per strip instead of once per tap.  Row strides in shared memory are
// odd, so a warp walking down a column of rows hits 32 different banks.
//
// The sums of |x - y| and SSIM over each tile's own pixels go to a per-tile
// pair; a one-block kernel adds them in a fixed order (in double) and writes
// the loss.  The result is deterministic.

#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "gs_device.cuh"
#include "gs_internal.h"

namespace gs {
namespace {

constexpr int kLT = 32;                  // tile side (pixels)
constexpr int kLR = 5;                   // window radius: 11 taps
constexpr int kTaps = 2 * kLR + 1;
constexpr int kIn = kLT + 4 * kLR;       // 52: staged x, y (tile + 10-pixel halo)
constexpr int kMom = kLT + 2 * kLR;      // 42: moments and S, a, b, c (tile + 5)
constexpr int kInPitch = kIn + 1;        // 53
constexpr int kMomPitch = kMom + 1;      // 43
constexpr int kOutPitch = kLT + 1;       // 33
constexpr int kLossThreads = 256;

// strip lengths of the four 1D passes (outputs per thread)
constexpr int kH1 = 14;  // rows of x, y -> 3 strips of 14 columns (42)
constexpr int kV1 = 7;   // columns of the row sums -> 6 strips of 7 rows (42)
constexpr int kH2 = 8;   // rows of a, b, c -> 4 strips of 8 columns (32)
constexpr int kV2 = 4;   // columns -> 8 strips of 4 rows (32)
static_assert(kMom % kH1 == 0 && kMom % kV1 == 0 && kLT % kH2 == 0 && kLT % kV2 == 0, "strips");
static_assert(kIn * (kMom / kH1) <= kLossThreads && kMom * (kMom / kV1) <= kLossThreads &&
                  kMom * (kLT / kH2) <= kLossThreads && kLT * (kLT / kV2) <= kLossThreads,
              "one strip per thread in every pass");

// shared memory, in floats.  The moments of x and of y share a pass and sit in
// float2 pairs, summed with the packed FMA (two lanes of fp32 per instruction,
// each rounded as fmaf); so do SSIM's derivatives by mu_x and E[x^2]
constexpr int kXs = 0;                                // x: [kIn][kInPitch]
constexpr int kYs = kXs + kIn * kInPitch;             // y
constexpr int kRow1 = kYs + kIn * kInPitch;           // row sums of
constexpr int kRowM = kRow1;                          //   (x, y): float2 [kIn][kMomPitch]
constexpr int kRowE = kRowM + 2 * kIn * kMomPitch;    //   (x^2, y^2): float2 [kIn][kMomPitch]
constexpr int kRowC = kRowE + 2 * kIn * kMomPitch;    //   xy: [kIn][kMomPitch]
constexpr int kCoef = kRowC + kIn * kMomPitch;        // (a, b): float2 [kMom][kMomPitch]
constexpr int kCoefC = kCoef + 2 * kMom * kMomPitch;  // c: [kMom][kMomPitch]
constexpr int kRow2 = kRow1;                          // their row sums: (a, b) float2
constexpr int kRow2C = kRow2 + 2 * kMom * kOutPitch;  //   [kMom][kOutPitch], c
constexpr int kGrad = kCoefC + kMom * kMomPitch;      // dL/dx: [kLT][kLT][3]
constexpr int kRed = kGrad + kLT * kLT * 3;           // 2 x 8 warp partials
constexpr int kLossSmemFloats = kRed + 2 * (kLossThreads / 32);
static_assert(3 * kMom * kOutPitch <= 5 * kIn * kMomPitch, "second row sums fit the first's room");
static_assert(kRowM % 2 == 0 && kRowE % 2 == 0 && kCoef % 2 == 0 && kRow2 % 2 == 0,
              "float2 arrays on 8-byte boundaries");
constexpr size_t kLossSmem = sizeof(float) * kLossSmemFloats;

struct LossArgs {
    float g[kTaps];     // normalised window taps g(-5) .. g(5)
    float c1, c2;
    float l1w, ssw;     // (1 - lambda) / (3 H W), lambda / (3 H W)
};

// 4-byte asynchronous global -> shared copy; writes 0 instead when !valid (the
// source address is then not read)
__device__ __forceinline__ void cp_async4_zfill(float* smem, const float* gmem, bool valid) {
    const unsigned sa = (unsigned)__cvta_generic_to_shared(smem);
    const int n = valid ? 4 : 0;
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(sa), "l"(gmem), "r"(n)
                 : "memory");
}

__global__ void __launch_bounds__(kLossThreads, 2)
    loss_ssim_kernel(int W, int H, const float* __restrict__ img, const float* __restrict__ tgt,
                     LossArgs la, float* __restrict__ dimg, float2* __restrict__ part) {
    grid_dep_sync();
    extern __shared__ float sm[];
    float* xs = sm + kXs;
    float* ys = sm + kYs;
    float2* rowm = reinterpret_cast<float2*>(sm + kRowM);
    float2* rowe = reinterpret_cast<float2*>(sm + kRowE);
    float* rowc = sm + kRowC;
    float2* coef = reinterpret_cast<float2*>(sm + kCoef);
    float* coefc = sm + kCoefC;
    float2* row2 = reinterpret_cast<float2*>(sm + kRow2);
    float* row2c = sm + kRow2C;
    float* grad = sm + kGrad;
    // the window's taps as (g, g) pairs
    auto g2 = [&](int k) { return make_float2(la.g[k], la.g[k]); };
    const int tid = threadIdx.x;
    const int tx0 = blockIdx.x * kLT, ty0 = blockIdx.y * kLT;
    float l1_sum = 0.f, ssim_sum = 0.f;

    // stage channel ch of x and y over the tile and a 10-pixel halo (0 outside) as
    // asynchronous copies; channel ch + 1 is staged while channel ch's derivative
    // maps are summed, once nothing reads the staged values any more
    auto stage = [&](int ch) {
        for (int i = tid; i < kIn * kIn; i += kLossThreads) {
            const int r = i / kIn, c = i - r * kIn;
            const int gy = ty0 - 2 * kLR + r, gx = tx0 - 2 * kLR + c;
            const bool in = gy >= 0 && gy < H && gx >= 0 && gx < W;
            const int64_t o = in ? ((int64_t)gy * W + gx) * 3 + ch : 0;
            cp_async4_zfill(xs + r * kInPitch + c, img + o, in);
            cp_async4_zfill(ys + r * kInPitch + c, tgt + o, in);
        }
        cp_async_commit();
    };
    stage(0);

    for (int ch = 0; ch < 3; ++ch) {
        cp_async_wait<0>();
        __syncthreads();

        // along rows: x, y, x^2, y^2, xy summed with the window, 42 columns
        if (tid < kIn * (kMom / kH1)) {
            const int r = tid % kIn, s = tid / kIn;
            const float* xr = xs + r * kInPitch + s * kH1;
            const float* yr = ys + r * kInPitch + s * kH1;
            float2 am[kH1], ae[kH1];
            float ac[kH1];
#pragma unroll
            for (int j = 0; j < kH1; ++j) {
                am[j] = ae[j] = make_float2(0.f, 0.f);
                ac[j] = 0.f;
            }
#pragma unroll
            for (int i = 0; i < kH1 + 2 * kLR; ++i) {
                const float2 v = make_float2(xr[i], yr[i]);
                const float2 v2 = __fmul2_rn(v, v);
                const float vc = v.x * v.y;
#pragma unroll
                for (int j = 0; j < kH1; ++j) {
                    const int k = i - j;
                    if (k >= 0 && k < kTaps) {
                        am[j] = __ffma2_rn(g2(k), v, am[j]);
                        ae[j] = __ffma2_rn(g2(k), v2, ae[j]);
                        ac[j] = fmaf(la.g[k], vc, ac[j]);
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < kH1; ++j) {
                const int o = r * kMomPitch + s * kH1 + j;
                rowm[o] = am[j];
                rowe[o] = ae[j];
                rowc[o] = ac[j];
            }
        }
        __syncthreads();

        // along columns: the five moments on the tile + 5, then S, a, b, c
        if (tid < kMom * (kMom / kV1)) {
            const int c = tid % kMom, s = tid / kMom;
            float2 am[kV1], ae[kV1];
            float ac[kV1];
#pragma unroll
            for (int j = 0; j < kV1; ++j) {
                am[j] = ae[j] = make_float2(0.f, 0.f);
                ac[j] = 0.f;
            }
#pragma unroll
            for (int i = 0; i < kV1 + 2 * kLR; ++i) {
                const int o = (s * kV1 + i) * kMomPitch + c;
                const float2 vm = rowm[o], ve = rowe[o];
                const float vc = rowc[o];
#pragma unroll
                for (int j = 0; j < kV1; ++j) {
                    const int k = i - j;
                    if (k >= 0 && k < kTaps) {
                        am[j] = __ffma2_rn(g2(k), vm, am[j]);
                        ae[j] = __ffma2_rn(g2(k), ve, ae[j]);
                        ac[j] = fmaf(la.g[k], vc, ac[j]);
                    }
                }
            }
            const int gx = tx0 - kLR + c;
#pragma unroll
            for (int j = 0; j < kV1; ++j) {
                const int r = s * kV1 + j;
                const int gy = ty0 - kLR + r;
                float a = 0.f, b = 0.f, cc = 0.f;
                if (gy >= 0 && gy < H && gx >= 0 && gx < W) {
                    const float mx = am[j].x, my = am[j].y;
                    const float vx = ae[j].x - mx * mx, vy = ae[j].y - my * my;
                    const float cov = ac[j] - mx * my;
                    const float A1 = 2.f * mx * my + la.c1, A2 = 2.f * cov + la.c2;
                    const float B1 = mx * mx + my * my + la.c1, B2 = vx + vy + la.c2;
                    const float rD = rcp_approx(B1 * B2);  // ~1 ulp: far below the
                                                           // cancellation error of B2
                    const float S = A1 * A2 * rD;
                    a = (2.f * my * (A2 - A1) - 2.f * mx * S * (B2 - B1)) * rD;
                    b = -S * B1 * rD;
                    cc = 2.f * A1 * rD;
                    if (r >= kLR && r < kLR + kLT && c >= kLR && c < kLR + kLT) {
                        ssim_sum += S;
                        const int o = (r + kLR) * kInPitch + c + kLR;
                        l1_sum += fabsf(xs[o] - ys[o]);
                    }
                }
                coef[r * kMomPitch + c] = make_float2(a, b);
                coefc[r * kMomPitch + c] = cc;
            }
        }
        __syncthreads();
        if (ch < 2) stage(ch + 1);

        // along rows: a, b, c summed with the window, the tile's 32 columns
        if (tid < kMom * (kLT / kH2)) {
            const int r = tid % kMom, s = tid / kMom;
            float2 aab[kH2];
            float acc_c[kH2];
#pragma unroll
            for (int j = 0; j < kH2; ++j) {
                aab[j] = make_float2(0.f, 0.f);
                acc_c[j] = 0.f;
            }
#pragma unroll
            for (int i = 0; i < kH2 + 2 * kLR; ++i) {
                const int o = r * kMomPitch + s * kH2 + i;
                const float2 vab = coef[o];
                const float vc = coefc[o];
#pragma unroll
                for (int j = 0; j < kH2; ++j) {
                    const int k = i - j;
                    if (k >= 0 && k < kTaps) {
                        aab[j] = __ffma2_rn(g2(k), vab, aab[j]);
                        acc_c[j] = fmaf(la.g[k], vc, acc_c[j]);
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < kH2; ++j) {
                row2[r * kOutPitch + s * kH2 + j] = aab[j];
                row2c[r * kOutPitch + s * kH2 + j] = acc_c[j];
            }
        }
        __syncthreads();

        // along columns, then dL/dx of the tile's pixels for this channel
        {
            const int c = tid % kLT, s = tid / kLT;
            float2 aab[kV2];
            float acc_c[kV2];
#pragma unroll
            for (int j = 0; j < kV2; ++j) {
                aab[j] = make_float2(0.f, 0.f);
                acc_c[j] = 0.f;
            }
#pragma unroll
            for (int i = 0; i < kV2 + 2 * kLR; ++i) {
                const int o = (s * kV2 + i) * kOutPitch + c;
                const float2 vab = row2[o];
                const float vc = row2c[o];
#pragma unroll
                for (int j = 0; j < kV2; ++j) {
                    const int k = i - j;
                    if (k >= 0 && k < kTaps) {
                        aab[j] = __ffma2_rn(g2(k), vab, aab[j]);
                        acc_c[j] = fmaf(la.g[k], vc, acc_c[j]);
                    }
                }
            }
            // the pixel's own x and y (the staging room holds the next channel by now;
            // pixels outside the image are never written)
            float xv[kV2], yv[kV2];
#pragma unroll
            for (int j = 0; j < kV2; ++j) {
                const int gy = ty0 + s * kV2 + j, gx = tx0 + c;
                const bool in = gy < H && gx < W;
                const int64_t o = in ? ((int64_t)gy * W + gx) * 3 + ch : 0;
                xv[j] = in ? __ldg(img + o) : 0.f;
                yv[j] = in ? __ldg(tgt + o) : 0.f;
            }
#pragma unroll
            for (int j = 0; j < kV2; ++j) {
                const int r = s * kV2 + j;
                const float sg = xv[j] > yv[j] ? 1.f : (xv[j] < yv[j] ? -1.f : 0.f);
                const float ds = aab[j].x + 2.f * xv[j] * aab[j].y + yv[j] * acc_c[j];
                grad[(r * kLT + c) * 3 + ch] = la.l1w * sg - la.ssw * ds;
            }
        }
        __syncthreads();
    }

    // the tile's rows of dL/dx, three channels at once (coalesced)
    const int w = min(kLT, W - tx0);
    for (int i = tid; i < kLT * kLT * 3; i += kLossThreads) {
        const int r = i / (kLT * 3), k = i - r * (kLT * 3);
        if (ty0 + r < H && k < 3 * w)
            dimg[((int64_t)(ty0 + r) * W + tx0) * 3 + k] = grad[r * kLT * 3 + k];
    }

    // the tile's sums of |x - y| and SSIM
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        l1_sum += __shfl_xor_sync(0xffffffffu, l1_sum, off);
        ssim_sum += __shfl_xor_sync(0xffffffffu, ssim_sum, off);
    }
    float* red = sm + kRed;
    if ((tid & 31) == 0) {
        red[tid >> 5] = l1_sum;
        red[(kLossThreads >> 5) + (tid >> 5)] = ssim_sum;
    }
    __syncthreads();
    if (tid == 0) {
        float a = 0.f, b = 0.f;
        for (int k = 0; k < kLossThreads / 32; ++k) {
            a += red[k];
            b += red[(kLossThreads >> 5) + k];
        }
        part[blockIdx.y * gridDim.x + blockIdx.x] = make_float2(a, b);
    }
}

constexpr int kFinThreads = 256;

// out = (L, mean |x - y|, mean SSIM) from the per-tile sums, in double and a
// fixed order
__global__ void __launch_bounds__(kFinThreads)
    loss_finish_kernel(const float2* __restrict__ part, int n_part, double inv, double lambda,
                       float* __restrict__ out) {
    grid_dep_sync();
    __shared__ double s1[kFinThreads], s2[kFinThreads];
    double a = 0.0, b = 0.0;
    for (int i = threadIdx.x; i < n_part; i += kFinThreads) {
        const float2 p = part[i];
        a += (double)p.x;
        b += (double)p.y;
    }
    s1[threadIdx.x] = a;
    s2[threadIdx.x] = b;
    __syncthreads();
    for (int h = kFinThreads / 2; h > 0; h >>= 1) {
        if ((int)threadIdx.x < h) {
            s1[threadIdx.x] += s1[threadIdx.x + h];
            s2[threadIdx.x] += s2[threadIdx.x + h];
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        const double l1 = s1[0] * inv, ssim = s2[0] * inv;
        out[0] = (float)((1.0 - lambda) * l1 + lambda * (1.0 - ssim));
        out[1] = (float)l1;
        out[2] = (float)ssim;
    }
}

}  // namespace

int64_t loss_tiles(int W, int H) {
    return (int64_t)((W + kLT - 1) / kLT) * ((H + kLT - 1) / kLT);
}

cudaError_t launch_loss_l1_ssim(int W, int H, const float* img, const float* tgt, double lambda,
                                float c1, float c2, double sigma, float* dimg, float* loss_out,
                                void* ws, cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(loss_ssim_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kLossSmem);
    if (e != cudaSuccess) return e;
    LossArgs la{};
    double gs[kTaps], sum = 0.0;
    for (int k = -kLR; k <= kLR; ++k) {
        gs[k + kLR] = std::exp(-(double)(k * k) / (2.0 * sigma * sigma));
        sum += gs[k + kLR];
    }
    for (int k = 0; k < kTaps; ++k) la.g[k] = (float)(gs[k] / sum);
    la.c1 = c1;
    la.c2 = c2;
    const double inv = 1.0 / (3.0 * (double)W * (double)H);
    la.l1w = (float)((1.0 - lambda) * inv);
    la.ssw = (float)(lambda * inv);
    const dim3 grid((W + kLT - 1) / kLT, (H + kLT - 1) / kLT);
    float2* part = static_cast<float2*>(ws);
    e = launch(loss_ssim_kernel, grid, dim3(kLossThreads), kLossSmem, st, W, H, img,
                           tgt, la, dimg, part);
    if (e != cudaSuccess) return e;
    return launch(loss_finish_kernel, dim3(1), dim3(kFinThreads), 0, st,
                  static_cast<const float2*>(part), (int)(grid.x * grid.y), inv, lambda,
                  loss_out);
}

}  // namespace gs
