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
// The first call on a device looks up the array's device address (with that
// device current) and caches it; make that first call before any stream
// capture.  All calls share the array and it keeps the previous call's
// contents: the sort clears what must start at zero itself, and calls whose
// work overlaps on the GPU (other streams, other threads) race on it.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/gs.h"
#include "gs_internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(6) << 20;  // 6 MiB
constexpr int64_t kMaxGaussians = int64_t(1) << 16;
constexpr int64_t kMaxCapacity = int64_t(1) << 18;
constexpr int64_t kMaxTiles = int64_t(1) << 14;

__device__ __align__(256) char g_scratch[kScratchBytes];

std::mutex g_mu;
void* g_addr[64];

// Device address of g_scratch on the current device (looked up once per device).
cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_addr[dev]) {
        void* p = nullptr;
        err = cudaGetSymbolAddress(&p, g_scratch);
        if (err != cudaSuccess) return err;
        g_addr[dev] = p;
    }
    *out = g_addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" gs_status gs_bin_sort_noalloc(const gs_camera* cam, int64_t n, const float* splats,
                                         const float* depths, const int32_t* tiles_touched,
                                         int32_t* sorted_ids, int64_t capacity,
                                         int32_t* tile_ranges, int32_t* lpt_order,
                                         int64_t* counts_device, int64_t* n_pairs_host,
                                         void* stream) {
    if (!cam || cam->width < 1 || cam->height < 1 || n < 0 || capacity < 1)
        return GS_ERR_INVALID_ARG;
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
