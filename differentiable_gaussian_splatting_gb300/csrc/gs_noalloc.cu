// gs_noalloc.cu -- gs_bin_sort_noalloc: the tile binning and sort of
// gs_bin_sort for callers that cannot allocate device memory.
//
// Some callers are not allowed to allocate: a plugin that runs inside a host
// application whose memory manager owns all of the GPU's memory, or a frame
// loop that cannot afford the device-wide synchronisation cudaMalloc may
// cause.  They still pass their inputs and outputs; the sort's scratch lives
// here instead, in one statically sized device array that every GPU which
// loads this library holds until the process exits.
//
// Every call looks up the array's device address on the current device (a
// host-side lookup; the first one on a device may load the library's device
// code there, so make the first call on each device before any stream
// capture).  All calls share the array and it keeps the previous call's
// contents: the sort clears what must start at zero itself, and calls whose
// work overlaps on the GPU (other streams, other threads) race on it.
#include <cuda_runtime.h>

#include "../../include/gs.h"
#include "gs_internal.h"

namespace {

// The limits below need 6,619,648 bytes of scratch when all three are at
// their maximum (the layout grows with each of them); 7 MiB leaves a margin.
constexpr size_t kScratchBytes = size_t(7) << 20;  // 7 MiB
constexpr int64_t kMaxGaussians = int64_t(1) << 16;
constexpr int64_t kMaxCapacity = int64_t(1) << 18;
constexpr int64_t kMaxTiles = int64_t(1) << 14;

__device__ __align__(256) char g_scratch[kScratchBytes];

// Device address of g_scratch in the current device's context.  It is looked
// up on every call, not cached: a cached address would go stale if the
// context were destroyed and recreated (cudaDeviceReset) while the library
// stays loaded.
cudaError_t scratch_address(void** out) {
    void* p = nullptr;
    const cudaError_t err = cudaGetSymbolAddress(&p, g_scratch);
    if (err != cudaSuccess) return err;
    *out = p;
    return cudaSuccess;
}

}  // namespace

extern "C" gs_status gs_bin_sort_noalloc(const gs_camera* cam, int64_t n, const float* splats,
                                         const float* depths, const int32_t* tiles_touched,
                                         int32_t* sorted_ids, int64_t capacity,
                                         int32_t* tile_ranges, int32_t* lpt_order,
                                         int64_t* counts_device, int64_t* n_pairs_host,
                                         void* stream) {
    if (!gs::camera_valid(cam) || n < 0 || capacity < 1) return GS_ERR_INVALID_ARG;
    // sizes the fixed scratch cannot hold: a caller error, reported before any GPU work
    const int64_t nt = gs_num_tiles(cam->width, cam->height);
    if (n > kMaxGaussians || capacity > kMaxCapacity || nt > kMaxTiles) return GS_ERR_WORKSPACE;
    if (gs_bin_sort_workspace_bytes(n, capacity, cam->width, cam->height) > kScratchBytes)
        return GS_ERR_WORKSPACE;
    void* scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) return GS_ERR_CUDA;
    // in order on the caller's stream: no side stream or events are created here
    return gs::bin_sort_entry(cam, n, splats, depths, tiles_touched, scratch, kScratchBytes,
                              sorted_ids, capacity, tile_ranges, lpt_order, counts_device,
                              n_pairs_host, stream, false);
}
