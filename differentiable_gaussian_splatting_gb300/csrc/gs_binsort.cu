// gs_binsort.cu -- tile binning and the two-stage radix sort.
//
// "What the 3DGS Literature Left on the Table" (Kopanas), Step 1 (b): each
// visible splat's tiles come from exact per-row spans of its support ellipse;
// Step 1 (d): the visible Gaussians are sorted once by a 32-bit depth key and
// the (tile, Gaussian) pairs, emitted in that depth order, are then sorted by
// a narrow tile key with a stable radix sort.  "Mitigating SM-Level Load
// Imbalance in 3D Gaussian Splatting on GPUs" (Ryu & Yoo), Sec. 4.1: the tile
// indices are radix-sorted by descending pair count (LPT order).
//
// Everything stays on the device: element counts that depend on the data
// (visible Gaussians M, pairs I) are read by the kernels from device memory,
// so the whole call can run without a host synchronisation.
//
// Radix sort: LSD, 8-bit digits, per pass three kernels -- per-block digit
// counts (upsweep), an exclusive scan of every digit's row of block counts
// (one block per digit), and a stable scatter in which each warp ranks its
// keys with __match_any_sync and each block combines its warps' counts.
#include <cuda_runtime.h>

#include <algorithm>

#include "gs_device.cuh"
#include "gs_internal.h"

namespace gs {

namespace {

constexpr int kRsBlock = 256;
constexpr int kRsIpt = 16;
constexpr int kRsTile = kRsBlock * kRsIpt;  // 4096 keys per block
constexpr int kRsWarps = kRsBlock / 32;
constexpr int kScanThreads = 1024;

__host__ __device__ inline int64_t nblk_of(int64_t n) { return (n + kRsTile - 1) / kRsTile; }

__device__ __forceinline__ int64_t count_of(const int64_t* n_dev, int64_t n_static) {
    return n_dev ? *n_dev : n_static;
}

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// exclusive scan of one value per thread over a block of kRsBlock threads
template <typename T>
__device__ __forceinline__ T block_exclusive_scan_256(T v, T* s_warp, T* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    T x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        T y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        T w = lane < kRsWarps ? s_warp[lane] : T(0);
#pragma unroll
        for (int o = 1; o < kRsWarps; o <<= 1) {
            T y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < kRsWarps) s_warp[lane] = w;  // inclusive warp prefix
    }
    __syncthreads();
    T warp_excl = warp > 0 ? s_warp[warp - 1] : T(0);
    *total = s_warp[kRsWarps - 1];
    __syncthreads();
    return warp_excl + x - v;
}

// ---------------------------------------------------------------------------
// radix sort kernels
// ---------------------------------------------------------------------------
// Look-back words: one per (block, digit), written once per pass.  Bits 63-62
// hold the state (0 not ready, 1 the block's own digit count, 2 the inclusive
// prefix over blocks 0..b), bits 61-56 the pass (1-based, so words left by an
// earlier pass of the same sort read as not ready) and bits 55-0 the count.
constexpr uint64_t kLbAgg = 1ull << 62;
constexpr uint64_t kLbPrefix = 2ull << 62;
constexpr uint64_t kLbCount = (1ull << 56) - 1;
constexpr int kMaxPasses = 4;
// polls of one look-back word before the block gives up and flags an error
constexpr int kSpinLimit = 1 << 22;
constexpr int kLbWindow = 8;

__device__ __forceinline__ bool lb_ready(uint64_t w, uint64_t epoch) {
    return (w >> 62) != 0 && (w & ~(kLbPrefix | kLbAgg | kLbCount)) == epoch;
}

__device__ __forceinline__ uint64_t ld_relaxed(const uint64_t* p) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed(uint64_t* p, uint64_t v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Digit counts of every pass in one read of the keys: ghist[pass][digit]
// (zeroed beforehand).  Equal digits within a warp round are aggregated with
// __match_any_sync, so near-constant high bytes do not serialise on one counter.
__global__ void __launch_bounds__(kRsBlock) rs_global_hist(const uint32_t* __restrict__ keys,
                                                           const int64_t* n_dev, int64_t n_static,
                                                           int passes,
                                                           uint32_t* __restrict__ ghist) {
    const int64_t n = count_of(n_dev, n_static);
    __shared__ uint32_t cnt[kMaxPasses][256];
    const int tid = threadIdx.x, lane = tid & 31;
#pragma unroll
    for (int p = 0; p < kMaxPasses; ++p) cnt[p][tid] = 0;
    __syncthreads();
    const int64_t stride = (int64_t)gridDim.x * kRsBlock;
    for (int64_t base = (int64_t)blockIdx.x * kRsBlock; base < n; base += stride) {
        const int64_t idx = base + tid;
        const bool valid = idx < n;
        const uint32_t k = valid ? __ldg(keys + idx) : 0u;
        for (int p = 0; p < passes; ++p) {
            const uint32_t d = (k >> (8 * p)) & 255u;
            const uint32_t peers = __match_any_sync(0xffffffffu, valid ? d : 256u + lane);
            if (valid && (peers & lanemask_lt()) == 0) atomicAdd(&cnt[p][d], __popc(peers));
        }
    }
    __syncthreads();
    for (int p = 0; p < passes; ++p)
        if (cnt[p][tid]) atomicAdd(ghist + p * 256 + tid, cnt[p][tid]);
}

// One pass of the stable LSD sort: blocks take consecutive 4096-key tiles in
// ticket order, rank their keys by digit (warps with __match_any_sync, then
// across warps), publish their digit counts, and add the counts of the tiles
// before them by looking back through the published words (decoupled
// look-back: a block only waits on tiles that started before it, so waits
// end).  Keys are staged in shared memory in block-sorted order so that each
// digit's run is written to global memory contiguously.
struct OnesweepSmem {
    uint32_t keys[kRsTile];
    int32_t vals[kRsTile];
    uint32_t wcnt[kRsWarps][256];
    uint32_t dstart[256];
    int64_t gbase[256];
    uint32_t warp_sums[kRsWarps];
    int ticket;
};

__global__ void __launch_bounds__(kRsBlock, 2) rs_onesweep(
    const uint32_t* __restrict__ keys_in, const int32_t* __restrict__ vals_in,
    uint32_t* __restrict__ keys_out, int32_t* __restrict__ vals_out, const int64_t* n_dev,
    int64_t n_static, int pass, const uint32_t* __restrict__ ghist, int* __restrict__ tickets,
    uint64_t* __restrict__ lookback, unsigned long long* __restrict__ err) {
    __shared__ OnesweepSmem S;
    const int64_t n = count_of(n_dev, n_static);
    const int64_t nblk = nblk_of(n);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int shift = 8 * pass;
    const uint64_t epoch = (uint64_t)(pass + 1) << 56;
    if (tid == 0) S.ticket = atomicAdd(tickets + pass, 1);
#pragma unroll
    for (int w = 0; w < kRsWarps; ++w) S.wcnt[w][tid] = 0;
    __syncthreads();
    const int64_t b = S.ticket;
    if (b >= nblk) return;

    // ---- load (each warp owns 512 consecutive keys) and rank within the warp
    const int64_t wbase = b * kRsTile + (int64_t)warp * (32 * kRsIpt);
    uint32_t k[kRsIpt];
    int32_t v[kRsIpt];
    uint32_t loc[kRsIpt];
#pragma unroll
    for (int r = 0; r < kRsIpt; ++r) {
        const int64_t idx = wbase + r * 32 + lane;
        const bool valid = idx < n;
        k[r] = valid ? __ldg(keys_in + idx) : 0xffffffffu;
        v[r] = valid ? __ldg(vals_in + idx) : 0;
    }
#pragma unroll
    for (int r = 0; r < kRsIpt; ++r) {
        const int64_t idx = wbase + r * 32 + lane;
        const bool valid = idx < n;
        const uint32_t d = (k[r] >> shift) & 255u;
        const uint32_t peers = __match_any_sync(0xffffffffu, valid ? d : 256u + lane);
        const uint32_t rank = __popc(peers & lanemask_lt());
        const uint32_t prev = S.wcnt[warp][d];
        loc[r] = prev + rank;
        __syncwarp();
        if (valid && rank == 0) S.wcnt[warp][d] = prev + __popc(peers);
        __syncwarp();
    }
    __syncthreads();

    // ---- per digit (thread = digit): warp prefixes, block count, publish
    const int d = tid;
    uint32_t cd = 0;
#pragma unroll
    for (int w = 0; w < kRsWarps; ++w) {
        const uint32_t c = S.wcnt[w][d];
        S.wcnt[w][d] = cd;
        cd += c;
    }
    uint64_t* my = lookback + b * 256 + d;
    st_relaxed(my, (b == 0 ? kLbPrefix : kLbAgg) | epoch | (uint64_t)cd);
    // block-local start of each digit's run
    uint32_t x = cd;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) S.warp_sums[warp] = x;
    // global start of each digit: exclusive scan of the pass's digit counts
    uint32_t gd = ghist[pass * 256 + d];
    uint32_t gx = gd;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, gx, o);
        if (lane >= o) gx += y;
    }
    __syncthreads();
    uint32_t wpre = 0;
#pragma unroll
    for (int w = 0; w < kRsWarps; ++w) wpre += w < warp ? S.warp_sums[w] : 0u;
    const uint32_t dstart = wpre + x - cd;
    S.dstart[d] = dstart;
    __syncthreads();
    if (lane == 31) S.warp_sums[warp] = gx;
    __syncthreads();
    uint64_t gpre = 0;
#pragma unroll
    for (int w = 0; w < kRsWarps; ++w) gpre += w < warp ? S.warp_sums[w] : 0u;
    const uint64_t gstart = gpre + gx - gd;

    // ---- look back over the earlier tiles for this digit, kLbWindow words in
    // flight at a time (nearest first), up to the first inclusive prefix
    uint64_t excl = 0;
    if (b > 0) {
        bool found = false;
        for (int64_t jb = b - 1; jb >= 0 && !found; jb -= kLbWindow) {
            uint64_t wv[kLbWindow];
#pragma unroll
            for (int i = 0; i < kLbWindow; ++i)
                wv[i] = jb - i >= 0 ? ld_relaxed(lookback + (jb - i) * 256 + d) : 0ull;
#pragma unroll
            for (int i = 0; i < kLbWindow; ++i) {
                if (found || jb - i < 0) break;
                const uint64_t* wp = lookback + (jb - i) * 256 + d;
                int spins = 0;
                while (!lb_ready(wv[i], epoch) && ++spins < kSpinLimit) wv[i] = ld_relaxed(wp);
                if (spins >= kSpinLimit) {
                    atomicOr(err, 1ull);  // the tile before never published: give up
                    found = true;
                    break;
                }
                excl += wv[i] & kLbCount;
                found = (wv[i] >> 62) == 2;
            }
        }
        st_relaxed(my, kLbPrefix | epoch | (excl + cd));
    }
    S.gbase[d] = (int64_t)(gstart + excl) - (int64_t)dstart;

    // ---- stage in block-sorted order, then write each digit run contiguously
#pragma unroll
    for (int r = 0; r < kRsIpt; ++r) {
        const int64_t idx = wbase + r * 32 + lane;
        if (idx < n) {
            const uint32_t dd = (k[r] >> shift) & 255u;
            const uint32_t li = S.dstart[dd] + S.wcnt[warp][dd] + loc[r];
            S.keys[li] = k[r];
            S.vals[li] = v[r];
        }
    }
    __syncthreads();
    const int cnt = (int)min64(kRsTile, n - b * kRsTile);
    for (int i = tid; i < cnt; i += kRsBlock) {
        const uint32_t key = S.keys[i];
        const int64_t pos = S.gbase[(key >> shift) & 255u] + i;
        keys_out[pos] = key;
        vals_out[pos] = S.vals[i];
    }
}

// Stable LSD radix sort of (keys, vals) on bits [0, bits), bits <= 32.  The
// count is read from n_dev (device) when given, else n_static; n_max bounds
// it.  Passes ping-pong between (k0, v0) and (k1, v1), starting from (k0, v0).
// The last pass writes its values to vf when given (a buffer distinct from v0,
// v1) and its keys to the scratch buffer the pass did not read; *kres / *vres
// return where the sorted keys and values are.  ctl is the sort's control
// region (rs_ctl_bytes(n_max)), cleared here; err collects give-up flags.
size_t rs_ctl_bytes(int64_t n_max) {
    return 16 + kMaxPasses * 256 * 4 + (size_t)std::max<int64_t>(1, nblk_of(n_max)) * 256 * 8;
}

cudaError_t radix_sort(uint32_t* k0, int32_t* v0, uint32_t* k1, int32_t* v1, int32_t* vf,
                       const int64_t* n_dev, int64_t n_static, int64_t n_max, int bits, char* ctl,
                       unsigned long long* err, cudaStream_t st, uint32_t** kres,
                       int32_t** vres) {
    const int passes = std::max(1, (bits + 7) / 8);
    const unsigned grid = (unsigned)std::max<int64_t>(1, nblk_of(n_max));
    int* tickets = reinterpret_cast<int*>(ctl);
    uint32_t* ghist = reinterpret_cast<uint32_t*>(ctl + 16);
    uint64_t* lookback = reinterpret_cast<uint64_t*>(ctl + 16 + kMaxPasses * 256 * 4);
    cudaError_t e = cudaMemsetAsync(ctl, 0, rs_ctl_bytes(n_max), st);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const unsigned hgrid = (unsigned)std::max<int64_t>(
        1, std::min<int64_t>((n_max + kRsBlock - 1) / kRsBlock, (int64_t)std::max(sms, 1)));
    rs_global_hist<<<hgrid, kRsBlock, 0, st>>>(k0, n_dev, n_static, passes, ghist);
    uint32_t* kin = k0;
    int32_t* vin = v0;
    for (int p = 0; p < passes; ++p) {
        const bool last = p == passes - 1;
        uint32_t* kout = kin == k0 ? k1 : k0;
        int32_t* vout = (last && vf) ? vf : (vin == v0 ? v1 : v0);
        rs_onesweep<<<grid, kRsBlock, 0, st>>>(kin, vin, kout, vout, n_dev, n_static, p, ghist,
                                               tickets, lookback, err);
        kin = kout;
        vin = vout;
    }
    if (kres) *kres = kin;
    if (vres) *vres = vin;
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// scans: per-block sums, a single-block scan of the sums, per-block writes
// ---------------------------------------------------------------------------
// exclusive scan in place of bsum[0 .. nb), nb = ceil(count / kRsTile);
// count = *count_dev (or count_static).  Writes the grand total to *total_out
// and min(total, cap) to *capped_out (if given).
__global__ void __launch_bounds__(kScanThreads) scan_block_sums(int64_t* __restrict__ bsum,
                                                                const int64_t* count_dev,
                                                                int64_t count_static,
                                                                int64_t* total_out,
                                                                int64_t cap, int64_t* capped_out) {
    const int64_t nb = nblk_of(count_of(count_dev, count_static));
    __shared__ int64_t s_part[kScanThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t per = (nb + kScanThreads - 1) / kScanThreads;
    const int64_t lo = min64(nb, per * tid), hi = min64(nb, lo + per);
    int64_t sum = 0;
    for (int64_t j = lo; j < hi; ++j) sum += bsum[j];
    int64_t x = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int64_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_part[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int64_t w = s_part[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int64_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        s_part[lane] = w;
    }
    __syncthreads();
    int64_t run = (warp > 0 ? s_part[warp - 1] : 0) + x - sum;
    for (int64_t j = lo; j < hi; ++j) {
        int64_t c = bsum[j];
        bsum[j] = run;
        run += c;
    }
    if (tid == kScanThreads - 1) {
        int64_t total = s_part[31];
        *total_out = total;
        if (capped_out) *capped_out = total < cap ? total : cap;
    }
}

// visible Gaussians: per-block counts
__global__ void __launch_bounds__(kRsBlock) vis_count(const int32_t* __restrict__ tiles_touched,
                                                      int64_t n, int64_t* __restrict__ bsum) {
    __shared__ int64_t s_warp[kRsWarps];
    const int64_t base = (int64_t)blockIdx.x * kRsTile;
    int64_t c = 0;
#pragma unroll 4
    for (int i = threadIdx.x; i < kRsTile; i += kRsBlock) {
        int64_t idx = base + i;
        if (idx < n && tiles_touched[idx] > 0) ++c;
    }
    int64_t total;
    block_exclusive_scan_256<int64_t>(c, s_warp, &total);
    if (threadIdx.x == 0) bsum[blockIdx.x] = total;
}

// visible Gaussians, in id order: (depth key, id).  Blocked: each thread owns 16
// consecutive items, so one block-wide scan of per-thread counts suffices.
__global__ void __launch_bounds__(kRsBlock) vis_write(const int32_t* __restrict__ tiles_touched,
                                                      const float* __restrict__ depths, int64_t n,
                                                      const int64_t* __restrict__ bsum,
                                                      uint32_t* __restrict__ keys,
                                                      int32_t* __restrict__ vals) {
    __shared__ int64_t s_warp[kRsWarps];
    const int64_t base = (int64_t)blockIdx.x * kRsTile + (int64_t)threadIdx.x * kRsIpt;
    bool vis[kRsIpt];
    int64_t c = 0;
#pragma unroll
    for (int r = 0; r < kRsIpt; ++r) {
        const int64_t idx = base + r;
        vis[r] = idx < n && tiles_touched[idx] > 0;
        c += vis[r];
    }
    int64_t total;
    int64_t pos = bsum[blockIdx.x] + block_exclusive_scan_256<int64_t>(c, s_warp, &total);
#pragma unroll
    for (int r = 0; r < kRsIpt; ++r) {
        if (vis[r]) {
            const int64_t idx = base + r;
            keys[pos] = __float_as_uint(depths[idx]);  // depth > znear > 0: bits are ordered
            vals[pos] = (int32_t)idx;
            ++pos;
        }
    }
}

// pairs per visible Gaussian in depth order: per-block sums
__global__ void __launch_bounds__(kRsBlock) pairs_count(const int32_t* __restrict__ order,
                                                        const int32_t* __restrict__ tiles_touched,
                                                        const int64_t* __restrict__ m_dev,
                                                        int64_t* __restrict__ bsum) {
    const int64_t m = *m_dev;
    if ((int64_t)blockIdx.x >= nblk_of(m)) return;
    __shared__ int64_t s_warp[kRsWarps];
    const int64_t base = (int64_t)blockIdx.x * kRsTile;
    int64_t c = 0;
#pragma unroll 4
    for (int i = threadIdx.x; i < kRsTile; i += kRsBlock) {
        int64_t j = base + i;
        if (j < m) c += tiles_touched[order[j]];
    }
    int64_t total;
    block_exclusive_scan_256<int64_t>(c, s_warp, &total);
    if (threadIdx.x == 0) bsum[blockIdx.x] = total;
}

__global__ void __launch_bounds__(kRsBlock) pairs_offsets(const int32_t* __restrict__ order,
                                                          const int32_t* __restrict__ tiles_touched,
                                                          const int64_t* __restrict__ m_dev,
                                                          const int64_t* __restrict__ bsum,
                                                          int64_t* __restrict__ poff) {
    const int64_t m = *m_dev;
    if ((int64_t)blockIdx.x >= nblk_of(m)) return;
    __shared__ int64_t s_warp[kRsWarps];
    const int64_t base = (int64_t)blockIdx.x * kRsTile + (int64_t)threadIdx.x * kRsIpt;
    int32_t c[kRsIpt];
    int64_t sum = 0;
#pragma unroll
    for (int r = 0; r < kRsIpt; ++r) {
        const int64_t j = base + r;
        c[r] = j < m ? tiles_touched[order[j]] : 0;
        sum += c[r];
    }
    int64_t total;
    int64_t pos = bsum[blockIdx.x] + block_exclusive_scan_256<int64_t>(sum, s_warp, &total);
#pragma unroll
    for (int r = 0; r < kRsIpt; ++r) {
        const int64_t j = base + r;
        if (j < m) poff[j] = pos;
        pos += c[r];
    }
}

// emit (tile, Gaussian) pairs in depth order from the exact row spans.  A warp
// takes 32 consecutive splats; small ones are emitted by their own lane, large
// ones (> kEmitLane tiles) by the whole warp, one tile row per lane.
constexpr int kEmitLane = 16;

__global__ void __launch_bounds__(256) emit_pairs(CamParams cam, const float4* __restrict__ splats,
                                                  const int32_t* __restrict__ order,
                                                  const int32_t* __restrict__ tiles_touched,
                                                  const int64_t* __restrict__ poff,
                                                  const int64_t* __restrict__ m_dev,
                                                  int64_t capacity, uint32_t* __restrict__ pkeys,
                                                  int32_t* __restrict__ pvals) {
    const int64_t m = *m_dev;
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t base = warp0 * 32; base < m; base += nwarps * 32) {
        const int64_t j = base + lane;
        const bool valid = j < m;
        int32_t g = 0;
        int64_t off = 0;
        Ellipse e{};
        int ty0 = 0, ty1 = 0;
        bool big = false;
        if (valid) {
            g = order[j];
            off = poff[j];
            const float4 r0 = __ldg(splats + 3 * (int64_t)g), r1 = __ldg(splats + 3 * (int64_t)g + 1),
                         r2 = __ldg(splats + 3 * (int64_t)g + 2);
            e = ellipse_of(r0, r1, r2);
            row_range(e, cam.nty, &ty0, &ty1);
            big = tiles_touched[g] > kEmitLane;
            if (!big) {
                const float dyv = vertex_dy(e);
                int tx0, tx1;
                for (int ty = ty0; ty < ty1; ++ty) {
                    if (!row_span(e, dyv, ty, cam.W, cam.H, cam.ntx, &tx0, &tx1)) continue;
                    const uint32_t rowkey = (uint32_t)ty * (uint32_t)cam.ntx;
                    for (int tx = tx0; tx < tx1; ++tx, ++off)
                        if (off < capacity) {
                            pkeys[off] = rowkey + (uint32_t)tx;
                            pvals[off] = g;
                        }
                }
            }
        }
        uint32_t todo = __ballot_sync(0xffffffffu, big);
        while (todo) {
            const int src = __ffs(todo) - 1;
            todo &= todo - 1;
            const unsigned F = 0xffffffffu;
            Ellipse eb;
            eb.mux = __shfl_sync(F, e.mux, src);
            eb.muy = __shfl_sync(F, e.muy, src);
            eb.l11 = __shfl_sync(F, e.l11, src);
            eb.l12 = __shfl_sync(F, e.l12, src);
            eb.l22 = __shfl_sync(F, e.l22, src);
            eb.tau = __shfl_sync(F, e.tau, src);
            eb.rx = __shfl_sync(F, e.rx, src);
            eb.ry = __shfl_sync(F, e.ry, src);
            const int32_t gb = __shfl_sync(F, g, src);
            const int b0 = __shfl_sync(F, ty0, src), b1 = __shfl_sync(F, ty1, src);
            int64_t ob = __shfl_sync(F, off, src);
            const float dyv = vertex_dy(eb);
            for (int rb = b0; rb < b1; rb += 32) {
                const int ty = rb + lane;
                int tx0 = 0, tx1 = 0;
                const bool has = ty < b1 && row_span(eb, dyv, ty, cam.W, cam.H, cam.ntx, &tx0, &tx1);
                const int cnt = has ? tx1 - tx0 : 0;
                int incl = cnt;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int y = __shfl_up_sync(F, incl, o);
                    if (lane >= o) incl += y;
                }
                int64_t o2 = ob + (incl - cnt);
                const uint32_t rowkey = (uint32_t)ty * (uint32_t)cam.ntx;
                for (int tx = tx0; tx < tx1; ++tx, ++o2)
                    if (o2 < capacity) {
                        pkeys[o2] = rowkey + (uint32_t)tx;
                        pvals[o2] = gb;
                    }
                ob += __shfl_sync(F, incl, 31);
            }
        }
    }
}

// tile ranges [start, end) from the sorted keys (ranges zeroed beforehand)
__global__ void tile_ranges_kernel(const uint32_t* __restrict__ keys, const int64_t* __restrict__ n_dev,
                                   int2* __restrict__ ranges) {
    const int64_t n = *n_dev;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const uint32_t t = keys[i];
        if (i == 0 || keys[i - 1] != t) ranges[t].x = (int)i;
        if (i == n - 1 || keys[i + 1] != t) ranges[t].y = (int)(i + 1);
    }
}

// empty tiles get [p, p) with p the end of the last non-empty tile before them
// (so that starts are the exclusive prefix sum of the counts); one block
__global__ void __launch_bounds__(kScanThreads) fill_empty_ranges(int2* __restrict__ ranges,
                                                                  int64_t nt) {
    __shared__ int s_part[kScanThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t per = (nt + kScanThreads - 1) / kScanThreads;
    const int64_t lo = min64(nt, per * tid), hi = min64(nt, lo + per);
    int m = 0;
    for (int64_t t = lo; t < hi; ++t) m = max(m, ranges[t].y);
    int x = m;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x = max(x, y);
    }
    if (lane == 31) s_part[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = s_part[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w = max(w, y);
        }
        s_part[lane] = w;
    }
    __syncthreads();
    // exclusive running max of the ends before this thread's segment
    int run = warp > 0 ? s_part[warp - 1] : 0;
    int prev_lane = __shfl_up_sync(0xffffffffu, x, 1);
    if (lane > 0) run = max(run, prev_lane);
    for (int64_t t = lo; t < hi; ++t) {
        int2 r = ranges[t];
        if (r.y == 0) {
            ranges[t] = make_int2(run, run);
        } else {
            run = max(run, r.y);
        }
    }
}

// LPT order ("Mitigating SM-Level Load Imbalance in 3D Gaussian Splatting on
// GPUs", Sec. 4.1): tiles by descending pair count, ties by ascending tile id,
// i.e. ascending unique 64-bit keys ((2^32 - 1 - count) << 32 | tile).  Runs of
// 1024 keys are sorted in shared memory (bitonic), then every key's rank is its
// position in its run plus, in every other run, the number of smaller keys.
constexpr int kLptRun = 1024;

__global__ void __launch_bounds__(kLptRun / 2) lpt_sort_runs(const int2* __restrict__ ranges,
                                                            int64_t nt, uint64_t* __restrict__ runs) {
    __shared__ uint64_t sk[kLptRun];
    const int tid = threadIdx.x;
    const int64_t base = (int64_t)blockIdx.x * kLptRun;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int i = tid + h * (kLptRun / 2);
        const int64_t t = base + i;
        uint64_t key = ~0ull;
        if (t < nt) {
            const int2 r = ranges[t];
            key = ((uint64_t)(0xffffffffu - (uint32_t)(r.y - r.x)) << 32) | (uint64_t)t;
        }
        sk[i] = key;
    }
    __syncthreads();
    for (int size = 2; size <= kLptRun; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const int i = 2 * tid - (tid & (stride - 1));  // lower index of this thread's pair
            const int jx = i + stride;
            const bool up = (i & size) == 0;
            const uint64_t a = sk[i], b = sk[jx];
            if ((a > b) == up) {
                sk[i] = b;
                sk[jx] = a;
            }
            __syncthreads();
        }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int i = tid + h * (kLptRun / 2);
        runs[base + i] = sk[i];
    }
}

__global__ void lpt_merge(const uint64_t* __restrict__ runs, int64_t nt, int32_t* __restrict__ lpt) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t nruns = (nt + kLptRun - 1) / kLptRun;
    if (i >= nruns * kLptRun) return;
    const uint64_t key = runs[i];
    if (key == ~0ull) return;  // padding
    const int64_t r = i / kLptRun;
    int64_t rank = i - r * kLptRun;
    for (int64_t r2 = 0; r2 < nruns; ++r2) {
        if (r2 == r) continue;
        const uint64_t* run = runs + r2 * kLptRun;
        int lo = 0, hi = kLptRun;  // number of keys < key
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (run[mid] < key) lo = mid + 1;
            else hi = mid;
        }
        rank += lo;
    }
    lpt[rank] = (int32_t)(key & 0xffffffffu);
}

size_t align_up(size_t x) { return (x + 255) & ~size_t(255); }

int bits_for(int64_t v) {
    int b = 0;
    while (b < 62 && (int64_t(1) << b) <= v) ++b;
    return std::max(b, 1);
}

}  // namespace

BinSortLayout binsort_layout(int64_t n, int64_t capacity, int64_t n_tiles) {
    BinSortLayout L{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t o = off;
        off = align_up(off + bytes);
        return o;
    };
    const int64_t nn = std::max<int64_t>(n, 1), cap = std::max<int64_t>(capacity, 1);
    const int64_t nt = std::max<int64_t>(n_tiles, 1);
    L.off_counts = take(4 * sizeof(int64_t));
    L.off_bsum = take((size_t)(nblk_of(nn) + 1) * sizeof(int64_t));
    L.off_dkeys0 = take((size_t)nn * 4);
    L.off_dkeys1 = take((size_t)nn * 4);
    L.off_dvals0 = take((size_t)nn * 4);
    L.off_dvals1 = take((size_t)nn * 4);
    L.off_poff = take((size_t)(nn + 1) * sizeof(int64_t));
    L.off_pkeys0 = take((size_t)cap * 4);
    L.off_pkeys1 = take((size_t)cap * 4);
    L.off_pvals0 = take((size_t)cap * 4);
    L.off_pvals1 = take((size_t)cap * 4);
    L.off_hist = take(rs_ctl_bytes(std::max(nn, cap)));
    L.off_lruns = take((size_t)((nt + kLptRun - 1) / kLptRun) * kLptRun * sizeof(uint64_t));
    L.total = off;
    return L;
}

cudaError_t run_bin_sort(const CamParams& cam, int64_t n, const float* splats, const float* depths,
                         const int32_t* tiles_touched, char* ws, const BinSortLayout& L,
                         int32_t* sorted_ids, int64_t capacity, int32_t* tile_ranges,
                         int32_t* lpt_order, cudaStream_t st) {
    auto* counts = reinterpret_cast<int64_t*>(ws + L.off_counts);
    auto* bsum = reinterpret_cast<int64_t*>(ws + L.off_bsum);
    auto* dk0 = reinterpret_cast<uint32_t*>(ws + L.off_dkeys0);
    auto* dk1 = reinterpret_cast<uint32_t*>(ws + L.off_dkeys1);
    auto* dv0 = reinterpret_cast<int32_t*>(ws + L.off_dvals0);
    auto* dv1 = reinterpret_cast<int32_t*>(ws + L.off_dvals1);
    auto* poff = reinterpret_cast<int64_t*>(ws + L.off_poff);
    auto* pk0 = reinterpret_cast<uint32_t*>(ws + L.off_pkeys0);
    auto* pk1 = reinterpret_cast<uint32_t*>(ws + L.off_pkeys1);
    auto* pv0 = reinterpret_cast<int32_t*>(ws + L.off_pvals0);
    auto* pv1 = reinterpret_cast<int32_t*>(ws + L.off_pvals1);
    char* rs_ctl = ws + L.off_hist;
    auto* sort_err = reinterpret_cast<unsigned long long*>(ws + L.off_counts + 3 * sizeof(int64_t));
    auto* lruns = reinterpret_cast<uint64_t*>(ws + L.off_lruns);
    const int64_t nt = (int64_t)cam.ntx * cam.nty;
    cudaError_t err;

    err = cudaMemsetAsync(counts, 0, 4 * sizeof(int64_t), st);
    if (err != cudaSuccess) return err;
    err = cudaMemsetAsync(tile_ranges, 0, (size_t)nt * 2 * sizeof(int32_t), st);
    if (err != cudaSuccess) return err;

    if (n > 0) {
        const unsigned nb = (unsigned)nblk_of(n);
        // 1. compact the visible Gaussians (id order) into (depth key, id)
        vis_count<<<nb, kRsBlock, 0, st>>>(tiles_touched, n, bsum);
        scan_block_sums<<<1, kScanThreads, 0, st>>>(bsum, nullptr, n, counts + 0, 0, nullptr);
        vis_write<<<nb, kRsBlock, 0, st>>>(tiles_touched, depths, n, bsum, dk0, dv0);
        // 2. stable depth sort of the M visible (31 significant key bits)
        uint32_t* dks = nullptr;
        int32_t* dvs = nullptr;
        err = radix_sort(dk0, dv0, dk1, dv1, nullptr, counts + 0, 0, n, 31, rs_ctl, sort_err, st, &dks,
                         &dvs);
        if (err != cudaSuccess) return err;
        // 3. pair offsets in depth order, I = total, min(I, capacity)
        pairs_count<<<nb, kRsBlock, 0, st>>>(dvs, tiles_touched, counts + 0, bsum);
        scan_block_sums<<<1, kScanThreads, 0, st>>>(bsum, counts + 0, 0, counts + 1, capacity,
                                                     counts + 2);
        pairs_offsets<<<nb, kRsBlock, 0, st>>>(dvs, tiles_touched, counts + 0, bsum, poff);
        // 4. emit pairs in depth order
        const unsigned eg = (unsigned)std::min<int64_t>((n + 255) / 256, 65535);
        emit_pairs<<<eg, 256, 0, st>>>(cam, reinterpret_cast<const float4*>(splats), dvs,
                                       tiles_touched, poff, counts + 0, capacity, pk0, pv0);
        // 5. stable sort by tile key; values land in sorted_ids
        uint32_t* pks = nullptr;
        err = radix_sort(pk0, pv0, pk1, pv1, sorted_ids, counts + 2, 0, capacity,
                         bits_for(nt - 1), rs_ctl, sort_err, st, &pks, nullptr);
        if (err != cudaSuccess) return err;
        // 6. tile ranges
        tile_ranges_kernel<<<1024, 256, 0, st>>>(pks, counts + 2, reinterpret_cast<int2*>(tile_ranges));
        fill_empty_ranges<<<1, kScanThreads, 0, st>>>(reinterpret_cast<int2*>(tile_ranges), nt);
    }
    // 7. LPT order: tiles by descending count, ties by tile id
    {
        const unsigned nruns = (unsigned)((nt + kLptRun - 1) / kLptRun);
        lpt_sort_runs<<<nruns, kLptRun / 2, 0, st>>>(reinterpret_cast<const int2*>(tile_ranges), nt,
                                                     lruns);
        lpt_merge<<<(unsigned)((nruns * (int64_t)kLptRun + 255) / 256), 256, 0, st>>>(lruns, nt,
                                                                                   lpt_order);
    }
    return cudaGetLastError();
}

}  // namespace gs
