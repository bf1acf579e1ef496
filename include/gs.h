/*
 * gs.h -- C ABI of libgs, a tile-based differentiable 3D Gaussian splatting
 * rasterizer (forward and backward) for NVIDIA GB300 (sm_103a).
 *
 * The five calls below are the hot path, in the order a training step runs
 * them:
 *
 *   gs_project        3D Gaussians -> 2D splat records, depths, tile counts
 *   gs_bin_sort       splats -> (tile, depth, id)-ordered id lists, tile
 *                     ranges, heavy-tile-first (LPT) tile order
 *   gs_rasterize_fwd  front-to-back alpha blending per pixel
 *   gs_rasterize_bwd  per-pixel gradient recomputation -> nine screen-space
 *                     derivatives per splat
 *   gs_project_bwd    chain rule back to means, scales, quaternions,
 *                     opacities and SH coefficients
 *
 * Around them: gs_loss_l1_ssim (the L1 + SSIM loss between the forward and
 * the backward), gs_project_bwd_adam (the chain rule fused with one Adam
 * step), bfloat16-SH variants of the projection and its chain rule, and
 * gs_bin_sort_noalloc.
 *
 * Sources (page title, section / equation):
 *   [RY]  Ryu & Yoo, "Mitigating SM-Level Load Imbalance in 3D Gaussian
 *         Splatting on GPUs": Sec. 2.1 Eq. 1 (projection), Eq. 2 (alpha),
 *         Eq. 3 (blending, 1e-4 stop), Sec. 4.1 (LPT persistent kernel),
 *         Sec. 4.2 Eq. 4-5 (depth-wise chunking, saturation signalling),
 *         Sec. 4.3 (selective chunking), Sec. 4.4 Eq. 6 (per-frame policy).
 *   [K]   Kopanas, "What the 3DGS Literature Left on the Table": Step 1 (a)
 *         warp reduction of the nine gradients, (b) opacity-aware exact
 *         conic-tile spans, (c) sub-tile masks and the 48-byte splat record,
 *         (d) two-stage depth / tile radix sort, (e) gated SH and base-2
 *         exponentials; Step 2 (reduce-scatter); Step 3 (SH, 59 gradient
 *         floats per Gaussian); Step 5 (round-to-nearest quadratic).
 *
 * Conventions for every call
 *   - All array arguments are DEVICE pointers (CUDA global memory), fp32 or
 *     int32 unless stated, row-major and contiguous, 16-byte aligned.  The
 *     caller owns every buffer; the library allocates no device memory.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Work is
 *     enqueued on it and the call returns without waiting, except
 *     gs_bin_sort when `n_pairs_host` is non-NULL (one stream sync).
 *     gs_bin_sort forks part of its work onto two side streams the library
 *     keeps per device (created with four events on the first call there)
 *     and joins them back into `stream` before it returns, so its outputs are
 *     ordered on `stream` like every other call's.  Kernels are launched
 *     with programmatic stream serialisation: each may start launching
 *     while the previous kernel on the stream runs, and waits for that
 *     kernel's completion before touching memory.
 *   - Argument errors are detected synchronously on the host and returned
 *     as GS_ERR_INVALID_ARG before anything is enqueued.  A failed launch
 *     returns GS_ERR_CUDA.
 *   - Fixed method constants: 16x16 pixel tiles, alpha cutoff 1/255 (a
 *     splat reaches pixel offset d iff q(d) <= tau = 2 ln(255 o)), alpha
 *     clamp 0.99, transmittance stop 1e-4.  Pixel centres are at
 *     (x + 0.5, y + 0.5); the principal point (cx, cy) is in the same frame.
 *   - Activations are the caller's: scales > 0 and opacities in (0, 1) are
 *     passed activated; quaternions (w, x, y, z) are normalised inside and
 *     their gradient is taken w.r.t. the raw input.
 */
#ifndef GS_H
#define GS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GS_TILE 16
#define GS_ALPHA_MAX 0.99f
#define GS_T_MIN 1e-4f
#define GS_SPLAT_FLOATS 12 /* floats per splat record */
#define GS_GRAD2D_FLOATS 9 /* screen-space derivatives per splat */
#define GS_MAX_CHUNKS 16   /* largest k of the chunking policy */

typedef enum {
    GS_OK = 0,
    GS_ERR_INVALID_ARG = 1, /* bad pointer, size, alignment or setting */
    GS_ERR_CUDA = 2,        /* a CUDA runtime call or launch failed */
    GS_ERR_CAPACITY = 3,    /* the pair list does not fit: see gs_bin_sort */
    GS_ERR_TIMEOUT = 4,     /* a bounded device wait gave up (gs_bin_sort's radix sort;
                               reported when the call synchronises) */
    GS_ERR_WORKSPACE = 5    /* workspace smaller than the size query returned */
} gs_status;

/* Pinhole camera.  viewmat is the row-major 4x4 world->camera matrix (rows 0..2
 * used: rotation W and translation t_v); camera axes x right, y down, z forward.
 * Gaussians with camera depth t_z <= znear (> 0) are culled. */
typedef struct gs_camera {
    float viewmat[16];
    float fx, fy, cx, cy;
    int32_t width, height;
    float znear;
} gs_camera;

/* Scheduling of the blending kernels ([RY] Sec. 4.3-4.4).  These choose how the
 * work is split across CTAs; they never change results. */
typedef struct gs_settings {
    int32_t split_mode;  /* 0: per-frame policy (Eq. 6); 1: never split;
                            2: split the force_h heaviest tiles into force_k chunks */
    int32_t force_h;     /* split_mode 2: number of tiles to split (<= h_max) */
    int32_t force_k;     /* split_mode 2: chunks per split tile, 2..GS_MAX_CHUNKS */
    int32_t h_max;       /* most tiles that may be split; min(h_max, tiles) sizes the workspace */
    float policy_lambda; /* per-chunk overhead in Gaussian-equivalents (Eq. 6) */
    float policy_beta;   /* residual-imbalance penalty (Eq. 6) */
    float policy_eps;    /* split only if the estimate improves by this fraction */
} gs_settings;

/* Default settings: policy on, h_max 256, lambda 256, beta 0.05, eps 0.10. */
gs_settings gs_default_settings(void);

/* Human-readable name of a status code (static string). */
const char* gs_status_string(gs_status status);

/* Number of 16x16 tiles of a width x height image: ceil(w/16) * ceil(h/16). */
int64_t gs_num_tiles(int32_t width, int32_t height);

/*
 * gs_project -- [RY] Eq. 1; [K] Step 1 (b), (c), (e); Step 3.
 * Per Gaussian i: camera-space t = W m + t_v; projected centre mu' (pinhole);
 * Sigma = R(q) S S^T R(q)^T; Sigma' = J W Sigma W^T J^T with J the Jacobian of
 * the projection at t; conic (a, b, c) = inverse of Sigma' with
 * q(d) = a dx^2 + 2 b dx dy + c dy^2, carried by its Cholesky factor
 * (l11, l12, l22), a = l11^2, b = l11 l12, c = l12^2 + l22^2, taken from
 * Sigma' as l22 = 1/sqrt(Sigma'_yy), l11 = sqrt(Sigma'_yy / det Sigma'),
 * l12 = -(Sigma'_xy / Sigma'_yy) l11; tau = 2 ln(255 o) (fp32 rounding of the
 * exact value); support half-extents rx = sqrt(tau Sigma'_xx),
 * ry = sqrt(tau Sigma'_yy); the number of tiles whose pixel-centre hull meets
 * the support ellipse (exact row spans); colour c = sum_k Y_k(d) s_k over the
 * (sh_degree+1)^2 real SH basis functions at the unit view direction d (no
 * offset, no clamp), evaluated only for visible Gaussians.
 * The chain that decides integers (mu', conic, tau, extents, spans) is
 * evaluated in fp32 with one fixed operation order (round-to-nearest, no
 * contraction), so its results are reproducible bit for bit.
 *
 *   n              number of Gaussians (>= 0)
 *   sh_degree      0..3; K = (sh_degree + 1)^2 coefficients per channel
 *   means [n][3], scales [n][3] (> 0), quats [n][4] (w, x, y, z),
 *   opacities [n] (in (0, 1)), sh [n][K][3]
 * Outputs (visible = tiles_touched > 0; culled rows are all zero):
 *   splats [n][12]  mux, muy, l11, l12 | l22, tau, log2(o), rx | r, g, b, ry
 *   depths [n]      camera depth t_z
 *   radii [n][2]    ceil(rx), ceil(ry) (clamped to 2^30)
 *   tiles_touched [n]
 */
gs_status gs_project(const gs_camera* cam, int64_t n, int32_t sh_degree, const float* means,
                     const float* scales, const float* quats, const float* opacities,
                     const float* sh, float* splats, float* depths, int32_t* radii,
                     int32_t* tiles_touched, void* stream);

/* Workspace bytes gs_bin_sort needs for n Gaussians, a pair capacity and an
 * image size (an upper bound; 0 on invalid arguments). */
size_t gs_bin_sort_workspace_bytes(int64_t n, int64_t capacity, int32_t width, int32_t height);

/*
 * gs_bin_sort -- [K] Step 1 (b), (d); [RY] Sec. 4.1 (LPT ordering).
 * Per-tile buckets: every (tile, Gaussian) pair of the exact row spans is
 * counted in its tile's counter, a prefix scan of the counts lays the tiles
 * out, the pairs are scattered into their tiles' slices and every slice is
 * sorted by (depth, id).  For capacities of 8 Mi pairs and more the call
 * takes the two-stage radix sort instead ([K] Step 1 (d)): the visible
 * Gaussians sorted by depth, their pairs emitted in that order and sorted
 * stably by tile.  Either way the pair list is ordered by (tile, depth, id),
 * and the outputs are the same bit for bit.
 *
 *   splats, depths, tiles_touched   outputs of gs_project
 *   workspace       device scratch of >= gs_bin_sort_workspace_bytes(...)
 *   sorted_ids [capacity]     Gaussian id of every pair, in list order
 *   tile_ranges [n_tiles][2]  [start, end) of each tile in sorted_ids
 *   lpt_order [n_tiles]       tiles by descending pair count, ties by
 *                             ascending tile id (heavy tiles first)
 *   counts_device  optional device int64[2]: visible Gaussians M, pairs I
 *   n_pairs_host   optional host int64: if non-NULL the call synchronises
 *                  the stream and stores I; if I > capacity it returns
 *                  GS_ERR_CAPACITY (outputs are then invalid: retry with a
 *                  larger list).  With n_pairs_host NULL the call never
 *                  synchronises and the caller must ensure I <= capacity;
 *                  when I > capacity every tile range is empty and nothing
 *                  is written beyond capacity.
 */
gs_status gs_bin_sort(const gs_camera* cam, int64_t n, const float* splats, const float* depths,
                      const int32_t* tiles_touched, void* workspace, size_t workspace_bytes,
                      int32_t* sorted_ids, int64_t capacity, int32_t* tile_ranges,
                      int32_t* lpt_order, int64_t* counts_device, int64_t* n_pairs_host,
                      void* stream);

/* Workspace bytes the two rasterize calls share for an image size, the pair
 * list capacity given to gs_bin_sort and the settings (NULL = defaults). */
size_t gs_raster_workspace_bytes(int32_t width, int32_t height, int64_t capacity,
                                 const gs_settings* settings);

/*
 * gs_rasterize_fwd -- [RY] Eq. 2-5, Sec. 4.1-4.4; [K] Step 1 (c), Step 5, 6.
 * Per pixel, front to back over its tile's list: stop before a splat once
 * T < 1e-4; a splat is hit iff q <= tau, q = fma(u1, u1, u2 u2) with
 * u1 = fma(l11, dx, l12 dy), u2 = l22 dy, dx = (x + 0.5) - mux,
 * dy = (y + 0.5) - muy in fp32 round-to-nearest (a sum of non-negative terms,
 * well conditioned for thin splats); alpha = min(0.99, o exp(-q/2)); C += c alpha T;
 * T *= 1 - alpha.  A persistent kernel takes work from a queue in LPT order;
 * the heaviest tiles may be split into depth chunks whose partial results
 * are composed with Eq. 5 (replaying the chunk that holds a pixel's stop, so
 * the result is the sequential one).
 *
 *   settings        NULL = gs_default_settings()
 *   sorted_ids, capacity, tile_ranges, lpt_order   as given to / returned by
 *                   gs_bin_sort
 *   workspace       >= gs_raster_workspace_bytes(...); it carries state to
 *                   gs_rasterize_bwd and must not change between the calls
 *                   (split-tile state, and for every pair an 8-bit mask of the
 *                   warps that blended it: the backward skips the rest,
 *                   [K] Step 4.2)
 * Outputs:
 *   image [H][W][3], t_final [H][W] (final transmittance; no background),
 *   n_contrib [H][W] (blended splats), last_idx [H][W] (position in
 *   sorted_ids of the last blended splat, -1 if none)
 */
gs_status gs_rasterize_fwd(const gs_camera* cam, const gs_settings* settings, int64_t n,
                           const float* splats, const int32_t* sorted_ids, int64_t capacity,
                           const int32_t* tile_ranges, const int32_t* lpt_order, void* workspace,
                           size_t workspace_bytes, float* image, float* t_final,
                           int32_t* n_contrib, int32_t* last_idx, void* stream);

/*
 * gs_rasterize_bwd -- [K] Step 1 (a), (e); Step 2; Step 5.
 * Per pixel, back to front from last_idx, recovering T by division by
 * (1 - alpha): for each blended splat with transmittance T_k before it,
 * G = dL/dC and gT = dL/dT_final,
 *   dL/dc       = alpha T_k G
 *   dL/dalpha   = T_k (c . G) - (B_k . G) / (1 - alpha) - gT T_final / (1 - alpha)
 *   (B_k the colour blended behind the splat) and, unless the 0.99 clamp is
 *   active, dL/do = exp(-q/2) dL/dalpha, dL/dq = -(alpha/2) dL/dalpha,
 *   dL/dmu' = -2 [a dx + b dy, b dx + c dy] dL/dq,
 *   dL/d(a, b, c) = (dx^2, 2 dx dy, dy^2) dL/dq.
 * Each warp reduces the nine values over its pixels (reduce-scatter of warp
 * shuffles) before nine lanes add them atomically to grad2d.
 *
 *   splats .. workspace        as passed to gs_rasterize_fwd
 *   t_final, last_idx          outputs of gs_rasterize_fwd
 *   dL_dimage [H][W][3]
 *   dL_dt_final [H][W]         optional (NULL = 0)
 * Outputs (zeroed by the call first):
 *   grad2d [n][9]   mux, muy, a, b, c, opacity, r, g, b
 *   touched [n]     1 where a splat blended into some pixel of the image
 *                   (optional; its gradient may still be zero)
 */
gs_status gs_rasterize_bwd(const gs_camera* cam, const gs_settings* settings, int64_t n,
                           const float* splats, const int32_t* sorted_ids, int64_t capacity,
                           const int32_t* tile_ranges, const int32_t* lpt_order, void* workspace,
                           size_t workspace_bytes, const float* t_final, const int32_t* last_idx,
                           const float* dL_dimage, const float* dL_dt_final, float* grad2d,
                           uint8_t* touched, void* stream);

/*
 * gs_project_bwd -- chain rule of gs_project ([RY] Eq. 1; [K] Step 3).
 * From grad2d (the nine screen-space derivatives) to the 59 parameter
 * gradients per Gaussian: conic -> Sigma' -> (Sigma, J) -> (scales,
 * quaternion, t) -> means; colour -> SH coefficients and, through the view
 * direction, -> means.  Gaussians that are culled (tiles_touched == 0) or
 * untouched (touched == 0 when touched is given) get exact zeros; every row
 * of every output is written.
 *
 *   inputs as for gs_project, plus tiles_touched (from gs_project),
 *   grad2d [n][9] and touched [n] (optional) from gs_rasterize_bwd
 * Outputs: dmeans [n][3], dscales [n][3], dquats [n][4], dopacities [n],
 *   dsh [n][K][3]
 */
gs_status gs_project_bwd(const gs_camera* cam, int64_t n, int32_t sh_degree, const float* means,
                         const float* scales, const float* quats, const float* opacities,
                         const float* sh, const int32_t* tiles_touched, const float* grad2d,
                         const uint8_t* touched, float* dmeans, float* dscales, float* dquats,
                         float* dopacities, float* dsh, void* stream);

/*
 * gs_raster_stats -- diagnostics of the last gs_rasterize_fwd on a workspace.
 * Synchronises the stream and copies to host out[16]:
 *   out[0] h*  (tiles split)        out[1] k*  (chunks per split tile)
 *   out[2] K   (resident CTAs)      out[3] work items of the persistent kernel
 *   out[4] device error word (0 = none)
 *   per-frame tile load ("Mitigating SM-Level Load Imbalance...", Sec. 3.1):
 *   out[5] pairs of the heaviest tile   out[6] of the lightest non-empty tile
 *   out[7] pairs of all tiles           out[8] non-empty tiles
 *   256-splat batches of the forward (Sec. 4.2): out[9] blended by whole tiles,
 *   out[10] blended by depth chunks, out[11] left unread by chunks that saw
 *   the saturation flag, out[12] left unread by chunks whose pixels had all
 *   stopped, out[13] blended by chunks the composition discarded (every pixel
 *   had stopped before them)
 */
gs_status gs_raster_stats(const void* workspace, size_t workspace_bytes, int64_t* out,
                          void* stream);

/*
 * gs_project_sh16, gs_project_bwd_sh16 -- gs_project and gs_project_bwd with the
 * SH coefficients stored as bfloat16 ([K] Step 6: bfloat16 SH halves the bytes
 * the two calls read for them).  `sh` holds the raw 16-bit patterns (the upper
 * half of each fp32 value; widening is exact), same layout [n][K][3], 16-byte
 * aligned.  Everything else -- arguments, outputs (dsh is fp32), errors -- is as
 * for the fp32 calls; the arithmetic is fp32 on the widened values.
 */
gs_status gs_project_sh16(const gs_camera* cam, int64_t n, int32_t sh_degree, const float* means,
                          const float* scales, const float* quats, const float* opacities,
                          const uint16_t* sh, float* splats, float* depths, int32_t* radii,
                          int32_t* tiles_touched, void* stream);
gs_status gs_project_bwd_sh16(const gs_camera* cam, int64_t n, int32_t sh_degree,
                              const float* means, const float* scales, const float* quats,
                              const float* opacities, const uint16_t* sh,
                              const int32_t* tiles_touched, const float* grad2d,
                              const uint8_t* touched, float* dmeans, float* dscales,
                              float* dquats, float* dopacities, float* dsh, void* stream);

/*
 * gs_project_bwd_adam -- gs_project_bwd fused with one Adam step ("proj_sh_bwd_adam"
 * of the pages' Metal port: the chain rule's gradients are never written, the step
 * reads and writes the parameters and moments instead).  The parameters are the
 * RAW ones a training loop optimises -- means [n][3], log-scales [n][3],
 * quaternions [n][4] (w, x, y, z; not normalised), opacity logits [n], SH
 * [n][K][3] -- and are updated in place; the forward of the same step must have
 * been given scales = exp(log-scales) and opacities = sigmoid(logits).  Gradients
 * of the raw parameters: dL/dlog s = s dL/ds, dL/dlogit = o (1 - o) dL/do, the
 * rest as gs_project_bwd.  Every Gaussian takes the step (culled or untouched ones
 * with a zero gradient: their moments decay and their parameters still move).
 *
 *   Adam, per element:  m <- b1 m + (1 - b1) g;  v <- b2 v + (1 - b2) g^2;
 *                       p <- p - lr (m / (1 - b1^t)) / (sqrt(v / (1 - b2^t)) + eps)
 *   moments         device m[5], v[5], each of the layout of its parameter, in the
 *                   order above; updated in place
 *   adam            learning rates per group (SH band 0 = the first 3 values of a
 *                   row, bands 1-3 the rest), b1, b2 in [0, 1), eps > 0, step t >= 1
 *   scales_out      optional [n][3] (NULL = not written): exp(log-scales) after the
 *                   step, the next forward's scales
 *   opacities_out   optional [n]: sigmoid(logits) after the step
 */
typedef struct {
    float lr_means, lr_scales, lr_quats, lr_opacities, lr_sh0, lr_shN;
    float beta1, beta2, eps;
    int32_t step;
} gs_adam_settings;

typedef struct {
    float* m[5];
    float* v[5];
} gs_adam_moments;

gs_status gs_project_bwd_adam(const gs_camera* cam, int64_t n, int32_t sh_degree, float* means,
                              float* log_scales, float* quats, float* opacity_logits, float* sh,
                              const int32_t* tiles_touched, const float* grad2d,
                              const uint8_t* touched, const gs_adam_moments* moments,
                              const gs_adam_settings* adam, float* scales_out,
                              float* opacities_out, void* stream);

/*
 * gs_loss_l1_ssim -- the photometric loss of a training step and its gradient, the
 * step between gs_rasterize_fwd and gs_rasterize_bwd ("loss_fwd_bwd" of the pages'
 * Metal port, "perf: rasterizer and pipeline optimizations", Breakdown and Queue,
 * which keeps five windowed moments per colour channel; the formula is the usual
 * 3DGS objective, which the pages do not print):
 *
 *   L = (1 - lambda) mean |x - y| + lambda (1 - mean SSIM(x, y))
 *
 * over the width * height * 3 values of the rendered image x and the target y.
 * SSIM per pixel and channel is that of Wang et al. (2004):
 *   (2 mu_x mu_y + c1)(2 cov + c2) / ((mu_x^2 + mu_y^2 + c1)(var_x + var_y + c2)),
 * the means, variances and covariance taken over the 11 x 11 window centred on
 * the pixel with weights g(a) g(b), g(k) ~ exp(-k^2 / (2 sigma^2)) normalised
 * over k = -5..5, and pixels outside the image counting as zero.  The L1 term's
 * derivative is sign(x - y), 0 where x = y.
 *
 *   image, target   [height][width][3] (the layout gs_rasterize_fwd writes)
 *   settings        lambda in [0, 1] (3DGS uses 0.2); c1, c2 > 0 (0.01^2 and
 *                   0.03^2 for values in [0, 1]); sigma > 0 (1.5)
 *   dL_dimage       out [height][width][3], the gradient w.r.t. image (the input
 *                   gs_rasterize_bwd takes); must not overlap image or target
 *   loss_out        out, device float[3] = (L, mean |x - y|, mean SSIM)
 *   workspace       device scratch of gs_loss_workspace_bytes(width, height) bytes
 *
 * Two launches; deterministic (fixed summation order).  width, height >= 1.
 */
typedef struct {
    float lambda, c1, c2, sigma;
} gs_loss_settings;

size_t gs_loss_workspace_bytes(int32_t width, int32_t height);

gs_status gs_loss_l1_ssim(int32_t width, int32_t height, const float* image, const float* target,
                          const gs_loss_settings* settings, float* dL_dimage, float* loss_out,
                          void* workspace, size_t workspace_bytes, void* stream);

/*
 * gs_bin_sort_noalloc -- gs_bin_sort for callers that may not allocate device
 * memory.  The papers have no counterpart: it exists for hosts that own all
 * of the GPU's memory (a plugin inside an application with its own
 * allocator) or that cannot afford the synchronisation an allocation may
 * cause.  Arguments, outputs and results are those of gs_bin_sort, minus
 * the workspace: the scratch is one fixed 7 MiB device array inside this
 * library (held on every device the library is loaded on until the process
 * exits), so the call allocates nothing.
 *
 * Limits: n <= 65536 Gaussians, capacity <= 262144 pairs and at most 16384
 * tiles (2048 x 2048 pixels); larger sizes return GS_ERR_WORKSPACE before
 * anything is enqueued.  Use gs_bin_sort for more.
 *
 * Every call looks up the array's address with the calling thread's current
 * device; the first call on a device may load the library's device code
 * there, so make it before capturing the stream into a graph.  The array
 * keeps the previous call's contents (the sort clears what must start at
 * zero itself), and it is shared: calls whose GPU work overlaps (different
 * streams or host threads without ordering between them) race on it and
 * give undefined results.
 */
gs_status gs_bin_sort_noalloc(const gs_camera* cam, int64_t n, const float* splats,
                              const float* depths, const int32_t* tiles_touched,
                              int32_t* sorted_ids, int64_t capacity, int32_t* tile_ranges,
                              int32_t* lpt_order, int64_t* counts_device, int64_t* n_pairs_host,
                              void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GS_H */
