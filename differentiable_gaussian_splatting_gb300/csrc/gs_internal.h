// gs_internal.h -- launch parameters and kernel-launch declarations shared by
// the libgs translation units (host and device side).  Not part of the C ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include <utility>

#include "../../include/gs.h"

namespace gs {

// Camera as the kernels see it: rows 0..2 of the view matrix, intrinsics,
// image and tile grid, and the camera centre in world space (for SH).
struct CamParams {
    float V[12];
    float fx, fy, cx, cy, znear;
    int W, H, ntx, nty;
    float cw[3];
};

// ---- projection (gs_project.cu) -------------------------------------------
cudaError_t launch_project(const CamParams& cam, int64_t n, int sh_degree, const float* means,
                           const float* scales, const float* quats, const float* opacities,
                           const float* sh, float* splats, float* depths, int32_t* radii,
                           int32_t* tiles_touched, cudaStream_t st);

cudaError_t launch_project_bwd(const CamParams& cam, int64_t n, int sh_degree, const float* means,
                               const float* scales, const float* quats, const float* opacities,
                               const float* sh, const int32_t* tiles_touched, const float* grad2d,
                               const uint8_t* touched, float* dmeans, float* dscales,
                               float* dquats, float* dopacities, float* dsh, cudaStream_t st);

// ---- binning + sort (gs_binsort.cu) ---------------------------------------
struct BinSortLayout {
    size_t total;
    size_t off_counts;   // int64[8]: M, I, min(I, capacity), raw pairs, medium / large tiles
    size_t off_raw;      // uint2[capacity]: raw (tile, Gaussian) pairs; later a merge buffer
    size_t off_keys;     // uint64[capacity]: the tiles' slices of (depth bits << 32 | id)
    size_t off_tcount;   // int32[n_tiles]: pairs per tile
    size_t off_cursor;   // uint64[n_tiles]: bucket cursors
    size_t off_lists;    // int32[2 n_tiles]: tiles sorted by a block, tiles sorted by merge rounds
    size_t off_lchunk;   // int32[n_tiles + 1]: chunk offsets of the long slices
    size_t off_lruns;    // uint64[n_tiles rounded up to 1024]: sorted runs of LPT keys
};
BinSortLayout binsort_layout(int64_t n, int64_t capacity, int64_t n_tiles);

// The two-stage radix sort (gs_binsort_radix.cu), taken for pair capacities of
// at least kRadixMinPairs; its counts words are M, I, min(I, capacity) and, at
// kRadixErrWord, a flag that a look-back wait gave up.
constexpr int64_t kRadixMinPairs = int64_t(8) << 20;
constexpr int kRadixErrWord = 4;
struct RadixBinLayout {
    size_t total;
    size_t off_counts;   // int64[8]
    size_t off_bsum;     // int64[nblk_n + 1] scan block sums
    size_t off_dkeys0, off_dkeys1, off_dvals0, off_dvals1;  // uint32 / int32 [n]
    size_t off_poff;     // int64[n + 1]: each visible Gaussian's first pair (by depth rank)
    size_t off_bstart;   // int64[emission blocks + 1]: each emission block's first Gaussian
    size_t off_pkeys0, off_pkeys1, off_pvals0, off_pvals1;  // [capacity]
    size_t off_hist;     // radix sort control: pass tickets, digit counts, look-back words
    size_t off_lruns;    // sorted runs of LPT keys
};
RadixBinLayout radix_bin_layout(int64_t n, int64_t capacity, int64_t n_tiles);
cudaError_t run_bin_sort_radix(const CamParams& cam, int64_t n, const float* splats,
                               const float* depths, const int32_t* tiles_touched, char* ws,
                               const RadixBinLayout& L, int32_t* sorted_ids, int64_t capacity,
                               int32_t* tile_ranges, int32_t* lpt_order, int64_t* counts_out,
                               cudaStream_t st);

// L1 + SSIM loss and its gradient (gs_loss.cu): per-tile partial sums in ws
// (loss_tiles(W, H) float2), loss_out = (L, mean |x - y|, mean SSIM)
int64_t loss_tiles(int W, int H);
cudaError_t launch_loss_l1_ssim(int W, int H, const float* img, const float* tgt, double lambda,
                                float c1, float c2, double sigma, float* dimg, float* loss_out,
                                void* ws, cudaStream_t st);

// LPT order of the tiles from their ranges (gs_binsort.cu); runs is scratch of
// lpt_runs_bytes(nt) bytes
size_t lpt_runs_bytes(int64_t nt);
cudaError_t launch_lpt(const int2* ranges, int64_t nt, uint64_t* runs, int32_t* lpt_order,
                       cudaStream_t st);

// Launch a kernel on st with programmatic stream serialisation: it may begin
// launching while the kernel before it on st still runs, and waits for that
// kernel's completion in its first statement (grid_dep_sync).  cluster > 1
// groups the blocks into thread-block clusters of that many blocks.
template <typename... P, typename... A>
inline cudaError_t launch_clustered(void (*kernel)(P...), unsigned cluster, dim3 grid, dim3 block,
                                    size_t smem, cudaStream_t st, A&&... args) {
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = cluster > 1 ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<A>(args)...);
}

template <typename... P, typename... A>
inline cudaError_t launch(void (*kernel)(P...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t st, A&&... args) {
    return launch_clustered(kernel, 1, grid, block, smem, st, std::forward<A>(args)...);
}

// A second stream with fork / join events: work that depends only on an
// earlier step runs on it beside the main sequence and is joined back.
struct SideStream {
    cudaStream_t stream, stream2;
    cudaEvent_t fork, fork2, join, join2;
};

// the camera checks every call makes (finite matrix and intrinsics, image
// sides 1..32768, znear > 0)
bool camera_valid(const gs_camera* cam);

// gs_bin_sort with its argument checks; overlap = false keeps every launch in
// order on the caller's stream and creates no side stream.
gs_status bin_sort_entry(const gs_camera* cam, int64_t n, const float* splats,
                         const float* depths, const int32_t* tiles_touched, void* workspace,
                         size_t workspace_bytes, int32_t* sorted_ids, int64_t capacity,
                         int32_t* tile_ranges, int32_t* lpt_order, int64_t* counts_device,
                         int64_t* n_pairs_host, void* stream, bool overlap);

// side may be null (everything in order on st)
cudaError_t run_bin_sort(const CamParams& cam, int64_t n, const float* splats, const float* depths,
                         const int32_t* tiles_touched, char* ws, const BinSortLayout& L,
                         int32_t* sorted_ids, int64_t capacity, int32_t* tile_ranges,
                         int32_t* lpt_order, int64_t* counts_out, cudaStream_t st,
                         const SideStream* side);

// ---- rasterization (gs_raster.cu) ------------------------------------------
struct RasterConfig {
    int split_mode, force_h, force_k, h_max;
    float lambda, beta, eps;
};

struct RasterLayout {
    size_t total;
    size_t off_ctrl;     // int32[16] control words
    size_t off_sat;      // int32[h_max] saturation flags
    size_t off_done;     // int32[h_max] finished-chunk counters
    size_t off_cbatch;   // int32[h_max][16]: batches each chunk blended
    size_t off_part_c;   // float4[h_max][16][256]: chunk partial (C.rgb, T)
    size_t off_part_n;   // int2[h_max][16][256]: chunk partial (n, last)
    size_t off_bwd;      // float4[h_max][16][256]: (T after chunk, colour behind chunk)
    size_t off_cmask;    // uint8[capacity]: warps that blended each pair
};
RasterLayout raster_layout(int W, int H, int h_max, int64_t capacity);

// control word indices
enum : int {
    kCtlQueueFwd = 0,
    kCtlQueueBwd = 1,
    kCtlH = 2,
    kCtlK = 3,
    kCtlItems = 4,
    kCtlResident = 5,
    kCtlError = 6,
    // per-frame tile load (the policy kernel): pairs of the heaviest tile, of the
    // lightest non-empty tile, of all tiles, and the number of non-empty tiles
    kCtlNMax = 7,
    kCtlNMinNz = 8,
    kCtlNTotal = 9,
    kCtlNonEmpty = 10,
    // 256-splat batches of the forward: blended by whole tiles, blended by depth
    // chunks, left unread by chunks that saw the saturation flag, left unread by
    // chunks whose own pixels had all stopped, and blended by chunks whose result
    // the composition discarded (every pixel had stopped before them)
    kCtlBatchTile = 11,
    kCtlBatchChunk = 12,
    kCtlSkipFlag = 13,
    kCtlSkipDone = 14,
    kCtlDiscard = 15,
    kCtlWords = 16
};

int raster_resident_ctas(int device);

cudaError_t run_raster_fwd(const CamParams& cam, const RasterConfig& cfg, const float* splats,
                           const int32_t* sorted_ids, const int32_t* tile_ranges,
                           const int32_t* lpt_order, char* ws, const RasterLayout& L, float* image,
                           float* t_final, int32_t* n_contrib, int32_t* last_idx, cudaStream_t st);

cudaError_t run_raster_bwd(const CamParams& cam, const RasterConfig& cfg, int64_t n,
                           const float* splats, const int32_t* sorted_ids,
                           const int32_t* tile_ranges, const int32_t* lpt_order, char* ws,
                           const RasterLayout& L, const float* t_final, const int32_t* last_idx,
                           const float* dL_dimage, const float* dL_dt, float* grad2d,
                           uint8_t* touched, cudaStream_t st);

}  // namespace gs
