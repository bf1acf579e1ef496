// gs_api.cu -- the extern "C" entry points of libgs (see include/gs.h).
//
// Host side only: argument validation (synchronous, before anything is
// enqueued), workspace carving and kernel launches on the caller's stream.
// The library allocates no device memory.  gs_bin_sort keeps two side streams
// and four events per device, created on its first call there, for work that
// overlaps the main sequence and is joined back into the caller's stream.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/gs.h"
#include "gs_internal.h"
#include "gs_project_variants.h"

using namespace gs;

namespace {

constexpr int kDefaultHMax = 256;
constexpr int32_t kMaxImageSide = 1 << 15;
constexpr int64_t kMaxIds = (int64_t(1) << 31) - 1;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool finite_f(float x) { return std::isfinite(x); }

bool camera_ok(const gs_camera* cam) {
    if (!cam) return false;
    if (cam->width < 1 || cam->height < 1 || cam->width > kMaxImageSide ||
        cam->height > kMaxImageSide)
        return false;
    for (int i = 0; i < 16; ++i)
        if (!finite_f(cam->viewmat[i])) return false;
    if (!finite_f(cam->fx) || !finite_f(cam->fy) || !finite_f(cam->cx) || !finite_f(cam->cy))
        return false;
    if (!(cam->znear > 0.f) || !finite_f(cam->znear)) return false;
    return true;
}

constexpr int kMaxDevices = 64;
std::mutex g_side_mu;  // guards g_side and orders the enqueues that use it
SideStream g_side[kMaxDevices];
bool g_side_ready[kMaxDevices];

// The side stream of the current device; call with g_side_mu held.
cudaError_t side_stream(const SideStream** out) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!g_side_ready[dev]) {
        SideStream s{};
        err = cudaStreamCreateWithFlags(&s.stream, cudaStreamNonBlocking);
        if (err == cudaSuccess) err = cudaStreamCreateWithFlags(&s.stream2, cudaStreamNonBlocking);
        if (err != cudaSuccess) return err;
        err = cudaEventCreateWithFlags(&s.fork, cudaEventDisableTiming);
        if (err == cudaSuccess) err = cudaEventCreateWithFlags(&s.fork2, cudaEventDisableTiming);
        if (err == cudaSuccess) err = cudaEventCreateWithFlags(&s.join, cudaEventDisableTiming);
        if (err == cudaSuccess) err = cudaEventCreateWithFlags(&s.join2, cudaEventDisableTiming);
        if (err != cudaSuccess) {  // release what was made, so a retry starts clean
            for (cudaStream_t st : {s.stream, s.stream2})
                if (st) cudaStreamDestroy(st);
            for (cudaEvent_t ev : {s.fork, s.fork2, s.join, s.join2})
                if (ev) cudaEventDestroy(ev);
            return err;
        }
        g_side[dev] = s;
        g_side_ready[dev] = true;
    }
    *out = &g_side[dev];
    return cudaSuccess;
}

CamParams cam_params(const gs_camera* cam) {
    CamParams c{};
    for (int r = 0; r < 3; ++r)
        for (int k = 0; k < 4; ++k) c.V[4 * r + k] = cam->viewmat[4 * r + k];
    c.fx = cam->fx;
    c.fy = cam->fy;
    c.cx = cam->cx;
    c.cy = cam->cy;
    c.znear = cam->znear;
    c.W = cam->width;
    c.H = cam->height;
    c.ntx = (cam->width + GS_TILE - 1) / GS_TILE;
    c.nty = (cam->height + GS_TILE - 1) / GS_TILE;
    // camera centre c_w = -W^T t_v
    for (int j = 0; j < 3; ++j) {
        double acc = 0.0;
        for (int r = 0; r < 3; ++r) acc -= (double)cam->viewmat[4 * r + j] * cam->viewmat[4 * r + 3];
        c.cw[j] = (float)acc;
    }
    return c;
}

bool settings_ok(const gs_settings* s) {
    if (s->split_mode < 0 || s->split_mode > 2) return false;
    if (s->h_max < 1 || s->h_max > 65536) return false;
    if (s->split_mode == 2) {
        if (s->force_h < 0 || s->force_h > s->h_max) return false;
        if (s->force_h > 0 && (s->force_k < 2 || s->force_k > GS_MAX_CHUNKS)) return false;
    }
    if (!(s->policy_lambda >= 0.f) || !(s->policy_beta >= 0.f) || !finite_f(s->policy_lambda) ||
        !finite_f(s->policy_beta))
        return false;
    if (!(s->policy_eps >= 0.f && s->policy_eps < 1.f)) return false;
    return true;
}

RasterConfig raster_config(const gs_settings* s) {
    RasterConfig c{};
    c.split_mode = s->split_mode;
    c.force_h = s->force_h;
    c.force_k = s->force_k;
    c.h_max = s->h_max;
    c.lambda = s->policy_lambda;
    c.beta = s->policy_beta;
    c.eps = s->policy_eps;
    return c;
}

gs_status cuda_status(cudaError_t e) { return e == cudaSuccess ? GS_OK : GS_ERR_CUDA; }

}  // namespace

namespace gs {

bool camera_valid(const gs_camera* cam) { return camera_ok(cam); }

gs_status bin_sort_entry(const gs_camera* cam, int64_t n, const float* splats,
                         const float* depths, const int32_t* tiles_touched, void* workspace,
                         size_t workspace_bytes, int32_t* sorted_ids, int64_t capacity,
                         int32_t* tile_ranges, int32_t* lpt_order, int64_t* counts_device,
                         int64_t* n_pairs_host, void* stream, bool overlap) {
    if (!camera_ok(cam) || n < 0 || n > kMaxIds || capacity < 1 || capacity > kMaxIds)
        return GS_ERR_INVALID_ARG;
    if (n > 0) {
        const void* ptrs[] = {splats, depths, tiles_touched};
        for (const void* p : ptrs)
            if (!p || !aligned16(p)) return GS_ERR_INVALID_ARG;
    }
    const void* outs[] = {workspace, sorted_ids, tile_ranges, lpt_order};
    for (const void* p : outs)
        if (!p || !aligned16(p)) return GS_ERR_INVALID_ARG;
    if (counts_device && (reinterpret_cast<uintptr_t>(counts_device) & 7u)) return GS_ERR_INVALID_ARG;
    const int64_t nt = gs_num_tiles(cam->width, cam->height);
    cudaStream_t st = (cudaStream_t)stream;
    char* ws = static_cast<char*>(workspace);
    cudaError_t err;
    // long pair lists: the two-stage radix sort (no per-tile atomics); the choice
    // depends on the capacity alone, so the workspace query agrees with it
    const bool radix = capacity >= kRadixMinPairs;
    if (radix) {
        const RadixBinLayout R = radix_bin_layout(n, capacity, nt);
        if (workspace_bytes < R.total) return GS_ERR_WORKSPACE;
        err = run_bin_sort_radix(cam_params(cam), n, splats, depths, tiles_touched, ws, R,
                                 sorted_ids, capacity, tile_ranges, lpt_order, counts_device, st);
        if (err != cudaSuccess) return GS_ERR_CUDA;
        if (n_pairs_host) {
            const int64_t* counts = reinterpret_cast<const int64_t*>(ws + R.off_counts);
            int64_t host_counts[8] = {0};
            err = cudaMemcpyAsync(host_counts, counts, sizeof(host_counts), cudaMemcpyDeviceToHost, st);
            if (err != cudaSuccess) return GS_ERR_CUDA;
            err = cudaStreamSynchronize(st);
            if (err != cudaSuccess) return GS_ERR_CUDA;
            *n_pairs_host = host_counts[1];
            if (host_counts[kRadixErrWord] != 0) return GS_ERR_TIMEOUT;
            if (host_counts[1] > capacity) return GS_ERR_CAPACITY;
        }
        return GS_OK;
    }
    const BinSortLayout L = binsort_layout(n, capacity, nt);
    if (workspace_bytes < L.total) return GS_ERR_WORKSPACE;
    {
        // the whole sequence is enqueued under the lock, so that the join event
        // still marks this call's side work when the caller's stream waits on it
        std::unique_lock<std::mutex> lk(g_side_mu, std::defer_lock);
        const SideStream* side = nullptr;
        if (overlap) {
            lk.lock();
            err = side_stream(&side);
            if (err != cudaSuccess) return GS_ERR_CUDA;
        }
        err = run_bin_sort(cam_params(cam), n, splats, depths, tiles_touched, ws, L, sorted_ids,
                           capacity, tile_ranges, lpt_order, counts_device, st, side);
    }
    if (err != cudaSuccess) return GS_ERR_CUDA;
    const int64_t* counts = reinterpret_cast<const int64_t*>(ws + L.off_counts);
    if (n_pairs_host) {
        int64_t host_counts[2] = {0, 0};
        err = cudaMemcpyAsync(host_counts, counts, 2 * sizeof(int64_t), cudaMemcpyDeviceToHost, st);
        if (err != cudaSuccess) return GS_ERR_CUDA;
        err = cudaStreamSynchronize(st);
        if (err != cudaSuccess) return GS_ERR_CUDA;
        *n_pairs_host = host_counts[1];
        if (host_counts[1] > capacity) return GS_ERR_CAPACITY;
    }
    return GS_OK;
}

}  // namespace gs

extern "C" {

gs_settings gs_default_settings(void) {
    gs_settings s;
    s.split_mode = 0;
    s.force_h = 0;
    s.force_k = 4;
    s.h_max = kDefaultHMax;
    s.policy_lambda = 256.f;
    s.policy_beta = 0.05f;
    s.policy_eps = 0.10f;
    return s;
}

const char* gs_status_string(gs_status status) {
    switch (status) {
        case GS_OK: return "ok";
        case GS_ERR_INVALID_ARG: return "invalid argument";
        case GS_ERR_CUDA: return "CUDA error";
        case GS_ERR_CAPACITY: return "pair list capacity exceeded";
        case GS_ERR_TIMEOUT: return "device wait timed out";
        case GS_ERR_WORKSPACE: return "workspace too small";
        default: return "unknown status";
    }
}

int64_t gs_num_tiles(int32_t width, int32_t height) {
    if (width < 1 || height < 1) return 0;
    // in 64 bits: width + 15 overflows int32 for widths near INT32_MAX
    return (((int64_t)width + GS_TILE - 1) / GS_TILE) * (((int64_t)height + GS_TILE - 1) / GS_TILE);
}

gs_status gs_project(const gs_camera* cam, int64_t n, int32_t sh_degree, const float* means,
                     const float* scales, const float* quats, const float* opacities,
                     const float* sh, float* splats, float* depths, int32_t* radii,
                     int32_t* tiles_touched, void* stream) {
    if (!camera_ok(cam) || n < 0 || n > kMaxIds || sh_degree < 0 || sh_degree > 3)
        return GS_ERR_INVALID_ARG;
    if (n == 0) return GS_OK;
    const void* ptrs[] = {means, scales, quats, opacities, sh, splats, depths, radii, tiles_touched};
    for (const void* p : ptrs)
        if (!p || !aligned16(p)) return GS_ERR_INVALID_ARG;
    return cuda_status(launch_project(cam_params(cam), n, sh_degree, means, scales, quats,
                                      opacities, sh, splats, depths, radii, tiles_touched,
                                      (cudaStream_t)stream));
}

size_t gs_bin_sort_workspace_bytes(int64_t n, int64_t capacity, int32_t width, int32_t height) {
    if (n < 0 || n > kMaxIds || capacity < 1 || capacity > kMaxIds || width < 1 || height < 1 ||
        width > kMaxImageSide || height > kMaxImageSide)
        return 0;
    const int64_t nt = gs_num_tiles(width, height);
    return capacity >= kRadixMinPairs ? radix_bin_layout(n, capacity, nt).total
                                      : binsort_layout(n, capacity, nt).total;
}

gs_status gs_bin_sort(const gs_camera* cam, int64_t n, const float* splats, const float* depths,
                      const int32_t* tiles_touched, void* workspace, size_t workspace_bytes,
                      int32_t* sorted_ids, int64_t capacity, int32_t* tile_ranges,
                      int32_t* lpt_order, int64_t* counts_device, int64_t* n_pairs_host,
                      void* stream) {
    return gs::bin_sort_entry(cam, n, splats, depths, tiles_touched, workspace, workspace_bytes,
                              sorted_ids, capacity, tile_ranges, lpt_order, counts_device,
                              n_pairs_host, stream, true);
}


size_t gs_raster_workspace_bytes(int32_t width, int32_t height, int64_t capacity,
                                 const gs_settings* settings) {
    gs_settings s = settings ? *settings : gs_default_settings();
    if (width < 1 || height < 1 || capacity < 1 || capacity > kMaxIds || !settings_ok(&s)) return 0;
    return raster_layout(width, height, s.h_max, capacity).total;
}

gs_status gs_rasterize_fwd(const gs_camera* cam, const gs_settings* settings, int64_t n,
                           const float* splats, const int32_t* sorted_ids, int64_t capacity,
                           const int32_t* tile_ranges, const int32_t* lpt_order, void* workspace,
                           size_t workspace_bytes, float* image, float* t_final,
                           int32_t* n_contrib, int32_t* last_idx, void* stream) {
    gs_settings s = settings ? *settings : gs_default_settings();
    if (!camera_ok(cam) || !settings_ok(&s) || n < 0 || n > kMaxIds || capacity < 1 ||
        capacity > kMaxIds)
        return GS_ERR_INVALID_ARG;
    const void* ptrs[] = {sorted_ids, tile_ranges, lpt_order, workspace, image, t_final,
                          n_contrib, last_idx};
    for (const void* p : ptrs)
        if (!p || !aligned16(p)) return GS_ERR_INVALID_ARG;
    if (n > 0 && (!splats || !aligned16(splats))) return GS_ERR_INVALID_ARG;
    const RasterLayout L = raster_layout(cam->width, cam->height, s.h_max, capacity);
    if (workspace_bytes < L.total) return GS_ERR_WORKSPACE;
    return cuda_status(run_raster_fwd(cam_params(cam), raster_config(&s), splats, sorted_ids,
                                      tile_ranges, lpt_order, static_cast<char*>(workspace), L,
                                      image, t_final, n_contrib, last_idx, (cudaStream_t)stream));
}

gs_status gs_rasterize_bwd(const gs_camera* cam, const gs_settings* settings, int64_t n,
                           const float* splats, const int32_t* sorted_ids, int64_t capacity,
                           const int32_t* tile_ranges, const int32_t* lpt_order, void* workspace,
                           size_t workspace_bytes, const float* t_final, const int32_t* last_idx,
                           const float* dL_dimage, const float* dL_dt_final, float* grad2d,
                           uint8_t* touched, void* stream) {
    gs_settings s = settings ? *settings : gs_default_settings();
    if (!camera_ok(cam) || !settings_ok(&s) || n < 0 || n > kMaxIds || capacity < 1 ||
        capacity > kMaxIds)
        return GS_ERR_INVALID_ARG;
    const void* ptrs[] = {sorted_ids, tile_ranges, lpt_order, workspace, t_final, last_idx,
                          dL_dimage};
    for (const void* p : ptrs)
        if (!p || !aligned16(p)) return GS_ERR_INVALID_ARG;
    if (n > 0 && (!splats || !aligned16(splats) || !grad2d || !aligned16(grad2d)))
        return GS_ERR_INVALID_ARG;
    if (dL_dt_final && !aligned16(dL_dt_final)) return GS_ERR_INVALID_ARG;
    const RasterLayout L = raster_layout(cam->width, cam->height, s.h_max, capacity);
    if (workspace_bytes < L.total) return GS_ERR_WORKSPACE;
    return cuda_status(run_raster_bwd(cam_params(cam), raster_config(&s), n, splats, sorted_ids,
                                      tile_ranges, lpt_order, static_cast<char*>(workspace), L,
                                      t_final, last_idx, dL_dimage, dL_dt_final, grad2d, touched,
                                      (cudaStream_t)stream));
}

gs_status gs_project_sh16(const gs_camera* cam, int64_t n, int32_t sh_degree, const float* means,
                          const float* scales, const float* quats, const float* opacities,
                          const uint16_t* sh, float* splats, float* depths, int32_t* radii,
                          int32_t* tiles_touched, void* stream) {
    if (!camera_ok(cam) || n < 0 || n > kMaxIds || sh_degree < 0 || sh_degree > 3)
        return GS_ERR_INVALID_ARG;
    if (n == 0) return GS_OK;
    const void* ptrs[] = {means, scales, quats, opacities, sh, splats, depths, radii, tiles_touched};
    for (const void* p : ptrs)
        if (!p || !aligned16(p)) return GS_ERR_INVALID_ARG;
    return cuda_status(launch_project_sh16(cam_params(cam), n, sh_degree, means, scales, quats,
                                           opacities, sh, splats, depths, radii, tiles_touched,
                                           (cudaStream_t)stream));
}

gs_status gs_project_bwd_sh16(const gs_camera* cam, int64_t n, int32_t sh_degree,
                              const float* means, const float* scales, const float* quats,
                              const float* opacities, const uint16_t* sh,
                              const int32_t* tiles_touched, const float* grad2d,
                              const uint8_t* touched, float* dmeans, float* dscales,
                              float* dquats, float* dopacities, float* dsh, void* stream) {
    if (!camera_ok(cam) || n < 0 || n > kMaxIds || sh_degree < 0 || sh_degree > 3)
        return GS_ERR_INVALID_ARG;
    if (n == 0) return GS_OK;
    const void* ptrs[] = {means, scales, quats, sh, tiles_touched, grad2d,
                          dmeans, dscales, dquats, dopacities, dsh};
    for (const void* p : ptrs)
        if (!p || !aligned16(p)) return GS_ERR_INVALID_ARG;
    return cuda_status(launch_project_bwd_sh16(cam_params(cam), n, sh_degree, means, scales,
                                               quats, opacities, sh, tiles_touched, grad2d,
                                               touched, dmeans, dscales, dquats, dopacities, dsh,
                                               (cudaStream_t)stream));
}

gs_status gs_project_bwd_adam(const gs_camera* cam, int64_t n, int32_t sh_degree, float* means,
                              float* log_scales, float* quats, float* opacity_logits, float* sh,
                              const int32_t* tiles_touched, const float* grad2d,
                              const uint8_t* touched, const gs_adam_moments* moments,
                              const gs_adam_settings* adam, float* scales_out,
                              float* opacities_out, void* stream) {
    if (!camera_ok(cam) || n < 0 || n > kMaxIds || sh_degree < 0 || sh_degree > 3 || !moments ||
        !adam)
        return GS_ERR_INVALID_ARG;
    const float lrs[6] = {adam->lr_means, adam->lr_scales, adam->lr_quats, adam->lr_opacities,
                          adam->lr_sh0, adam->lr_shN};
    for (float lr : lrs)
        if (!finite_f(lr) || lr < 0.f) return GS_ERR_INVALID_ARG;
    if (!(adam->beta1 >= 0.f && adam->beta1 < 1.f) || !(adam->beta2 >= 0.f && adam->beta2 < 1.f) ||
        !(adam->eps > 0.f) || !finite_f(adam->eps) || adam->step < 1)
        return GS_ERR_INVALID_ARG;
    if (n == 0) return GS_OK;
    const void* ptrs[] = {means, log_scales, quats, opacity_logits, sh, tiles_touched, grad2d,
                          moments->m[0], moments->m[1], moments->m[2], moments->m[3], moments->m[4],
                          moments->v[0], moments->v[1], moments->v[2], moments->v[3], moments->v[4]};
    for (const void* p : ptrs)
        if (!p || !aligned16(p)) return GS_ERR_INVALID_ARG;
    AdamArgs a{};
    float* params[5] = {means, log_scales, quats, opacity_logits, sh};
    for (int k = 0; k < 5; ++k) {
        a.p[k] = params[k];
        a.m[k] = moments->m[k];
        a.v[k] = moments->v[k];
    }
    for (int k = 0; k < 6; ++k) a.lr[k] = lrs[k];
    a.b1 = adam->beta1;
    a.b2 = adam->beta2;
    a.eps = adam->eps;
    a.c1 = (float)(1.0 / (1.0 - std::pow((double)adam->beta1, (double)adam->step)));
    a.c2 = (float)(1.0 / (1.0 - std::pow((double)adam->beta2, (double)adam->step)));
    if ((scales_out && !aligned16(scales_out)) || (opacities_out && !aligned16(opacities_out)))
        return GS_ERR_INVALID_ARG;
    a.act_scales = scales_out;
    a.act_opacities = opacities_out;
    return cuda_status(launch_project_bwd_adam(cam_params(cam), n, sh_degree, tiles_touched,
                                               grad2d, touched, a, (cudaStream_t)stream));
}

gs_status gs_project_bwd(const gs_camera* cam, int64_t n, int32_t sh_degree, const float* means,
                         const float* scales, const float* quats, const float* opacities,
                         const float* sh, const int32_t* tiles_touched, const float* grad2d,
                         const uint8_t* touched, float* dmeans, float* dscales, float* dquats,
                         float* dopacities, float* dsh, void* stream) {
    if (!camera_ok(cam) || n < 0 || n > kMaxIds || sh_degree < 0 || sh_degree > 3)
        return GS_ERR_INVALID_ARG;
    if (n == 0) return GS_OK;
    const void* ptrs[] = {means, scales, quats, sh, tiles_touched, grad2d,
                          dmeans, dscales, dquats, dopacities, dsh};
    for (const void* p : ptrs)
        if (!p || !aligned16(p)) return GS_ERR_INVALID_ARG;
    return cuda_status(launch_project_bwd(cam_params(cam), n, sh_degree, means, scales, quats,
                                          opacities, sh, tiles_touched, grad2d, touched, dmeans,
                                          dscales, dquats, dopacities, dsh, (cudaStream_t)stream));
}

size_t gs_loss_workspace_bytes(int32_t width, int32_t height) {
    if (width < 1 || height < 1) return 0;
    return (size_t)loss_tiles(width, height) * 2 * sizeof(float);
}

gs_status gs_loss_l1_ssim(int32_t width, int32_t height, const float* image, const float* target,
                          const gs_loss_settings* settings, float* dL_dimage, float* loss_out,
                          void* workspace, size_t workspace_bytes, void* stream) {
    if (width < 1 || height < 1 || width > (1 << 20) || height > (1 << 20) || !settings)
        return GS_ERR_INVALID_ARG;
    const gs_loss_settings& ls = *settings;
    if (!(ls.lambda >= 0.f && ls.lambda <= 1.f) || !(ls.c1 > 0.f) || !finite_f(ls.c1) ||
        !(ls.c2 > 0.f) || !finite_f(ls.c2) || !(ls.sigma > 0.f) || !finite_f(ls.sigma))
        return GS_ERR_INVALID_ARG;
    const void* ptrs[] = {image, target, dL_dimage, loss_out, workspace};
    for (const void* p : ptrs)
        if (!p || !aligned16(p)) return GS_ERR_INVALID_ARG;
    const size_t bytes = (size_t)width * height * 3 * sizeof(float);
    const char* d = (const char*)dL_dimage;
    for (const void* p : {(const void*)image, (const void*)target}) {
        const char* q = (const char*)p;
        if (d < q + bytes && q < d + bytes) return GS_ERR_INVALID_ARG;
    }
    if (workspace_bytes < gs_loss_workspace_bytes(width, height)) return GS_ERR_WORKSPACE;
    return cuda_status(launch_loss_l1_ssim(width, height, image, target, ls.lambda, ls.c1, ls.c2,
                                           ls.sigma, dL_dimage, loss_out, workspace,
                                           (cudaStream_t)stream));
}

gs_status gs_raster_stats(const void* workspace, size_t workspace_bytes, int64_t* out,
                          void* stream) {
    if (!workspace || !out || workspace_bytes < kCtlWords * sizeof(int)) return GS_ERR_INVALID_ARG;
    int ctrl[kCtlWords];
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t err = cudaMemcpyAsync(ctrl, workspace, sizeof(ctrl), cudaMemcpyDeviceToHost, st);
    if (err == cudaSuccess) err = cudaStreamSynchronize(st);
    if (err != cudaSuccess) return GS_ERR_CUDA;
    for (int i = 0; i < 16; ++i) out[i] = 0;
    out[0] = ctrl[kCtlH];
    out[1] = ctrl[kCtlK];
    out[2] = ctrl[kCtlResident];
    out[3] = ctrl[kCtlItems];
    out[4] = ctrl[kCtlError];
    out[5] = ctrl[kCtlNMax];
    out[6] = ctrl[kCtlNMinNz];
    out[7] = ctrl[kCtlNTotal];
    out[8] = ctrl[kCtlNonEmpty];
    out[9] = ctrl[kCtlBatchTile];
    out[10] = ctrl[kCtlBatchChunk];
    out[11] = ctrl[kCtlSkipFlag];
    out[12] = ctrl[kCtlSkipDone];
    out[13] = ctrl[kCtlDiscard];
    return GS_OK;
}

}  // extern "C"
