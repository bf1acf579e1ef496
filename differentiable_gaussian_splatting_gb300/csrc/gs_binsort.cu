// gs_binsort.cu -- tile binning: per-tile buckets of (tile, Gaussian) pairs.
//
// "What the 3DGS Literature Left on the Table" (Kopanas), Step 1 (b): each
// visible splat's tiles come from exact per-row spans of its support ellipse,
// counted with per-tile counters and laid out by a device prefix scan; Step 1
// (d): each tile's list is ordered by depth (ties by Gaussian id).  "Mitigating
// SM-Level Load Imbalance in 3D Gaussian Splatting on GPUs" (Ryu & Yoo), Sec.
// 4.1: the tiles are ordered by descending pair count (LPT order).
//
// The pipeline (every count stays on the device, so the call needs no host
// synchronisation):
//   1. bucket_emit     one pass over the Gaussians: every (tile, Gaussian) pair
//                      of the exact row spans is appended to a raw list (each
//                      block reserves its slice with one atomic) and counted in
//                      its tile's counter
//   2. bucket_scan     exclusive scan of the tile counts -> tile ranges
//   3. bucket_scatter  stream the raw list into the tiles' slices as 64-bit keys
//                      (depth bits << 32 | id); depth > 0, so the key order is
//                      the (depth, id) order
//   4. slice sorts     up to 512 keys: one warp, in registers and shared memory
//                      (bucket_sort_small); up to 4096: one block in shared memory
//                      (bucket_sort_blocks); longer slices: a merge sort over the
//                      whole grid (long_plan, long_chunks, long_round), 4096-key
//                      chunks sorted in shared memory, then merge rounds whose
//                      4096-key output pieces are each merged by one block
//   5. LPT order of the tiles.
#include <cuda_runtime.h>

#include <algorithm>

#include <cooperative_groups.h>

#include "gs_device.cuh"
#include "gs_internal.h"

namespace gs {

namespace {

constexpr int kScanThreads = 1024;
constexpr int kEmitThreads = 256;
constexpr int kSortThreads = 256;
constexpr int kWarpSortMax = 512;  // keys one warp sorts (16 per lane)
constexpr int kBlockSortMax = 4096;  // keys one block sorts in shared memory
// Tile counters and cursors sit 64 bytes apart: atomics on different words of
// one 32-byte sector serialise in L2, and neighbouring tiles are hot together.
constexpr int kCountStride = 16;   // ints
constexpr int kCursorStride = 8;   // uint64

// counts words (int64): M, I, min(I, capacity), raw pairs appended, tiles of
// kWarpSortMax + 1 .. kBlockSortMax pairs, tiles of more
constexpr int kCountRaw = 3;
constexpr int kCountMedium = 4;
constexpr int kCountLarge = 5;
constexpr int kCountLongChunks = 6;  // chunks of kBlockSortMax keys in the long slices
constexpr int kCountLongest = 7;     // keys of the longest slice

// ---------------------------------------------------------------------------
// 0. the call's counters and the tile counters to zero
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) bin_zero(int64_t* __restrict__ counts,
                                                int* __restrict__ tile_count, int64_t nt) {
    grid_dep_sync();
    const int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i0 < 8) counts[i0] = 0;
    for (int64_t t = i0; t < nt; t += (int64_t)gridDim.x * blockDim.x) tile_count[t * kCountStride] = 0;
}

// ---------------------------------------------------------------------------
// 1. one pass over the Gaussians: raw (tile, Gaussian) pairs and tile counts
// ---------------------------------------------------------------------------
struct EmitShared {
    float e[8][kEmitThreads];      // Ellipse fields, structure of arrays
    float dyv[kEmitThreads];       // vertex_dy of each splat
    int ty0[kEmitThreads];         // first tile row
    int off[kEmitThreads + 1];     // exclusive prefix of row counts
    int poff[kEmitThreads];        // exclusive prefix of pair counts
    int pcur[kEmitThreads];        // pairs placed so far per Gaussian
    int wsum[kEmitThreads / 32];
    int wpair[kEmitThreads / 32];
    long long base;                // the block's slice of the raw list
};

__global__ void __launch_bounds__(kEmitThreads) bucket_emit(CamParams cam,
                                                            const float4* __restrict__ splats,
                                                            const int32_t* __restrict__ tiles_touched,
                                                            int64_t n, int64_t capacity,
                                                            int* __restrict__ tile_count,
                                                            uint2* __restrict__ raw,
                                                            int64_t* __restrict__ counts) {
    grid_dep_sync();
    __shared__ EmitShared S;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t g = (int64_t)blockIdx.x * kEmitThreads + tid;
    const int tt = g < n ? tiles_touched[g] : 0;
    const bool vis = tt > 0;
    int nrows = 0;
    if (vis) {
        const float4 r0 = __ldg(splats + 3 * g), r1 = __ldg(splats + 3 * g + 1),
                     r2 = __ldg(splats + 3 * g + 2);
        const Ellipse e = ellipse_of(r0, r1, r2);
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
        S.dyv[tid] = vertex_dy(e);
        S.ty0[tid] = ty0;
    }
    S.pcur[tid] = 0;
    // block scans of the row counts and the pair counts
    int ri = nrows, pi = tt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int rv = __shfl_up_sync(0xffffffffu, ri, o);
        const int pv = __shfl_up_sync(0xffffffffu, pi, o);
        if (lane >= o) {
            ri += rv;
            pi += pv;
        }
    }
    if (lane == 31) {
        S.wsum[warp] = ri;
        S.wpair[warp] = pi;
    }
    const int nvis = __syncthreads_count(vis);
    int rbase = 0, rtotal = 0, pbase = 0, ptotal = 0;
#pragma unroll
    for (int w = 0; w < kEmitThreads / 32; ++w) {
        const int rv = S.wsum[w], pv = S.wpair[w];
        rbase += w < warp ? rv : 0;
        rtotal += rv;
        pbase += w < warp ? pv : 0;
        ptotal += pv;
    }
    S.off[tid] = rbase + ri - nrows;
    S.poff[tid] = pbase + pi - tt;
    if (tid == 0) {
        S.off[kEmitThreads] = rtotal;
        S.base = ptotal ? (long long)atomicAdd(reinterpret_cast<unsigned long long*>(counts + kCountRaw),
                                               (unsigned long long)ptotal)
                        : 0ll;
        if (nvis) atomicAdd(reinterpret_cast<unsigned long long*>(counts), (unsigned long long)nvis);
    }
    __syncthreads();
    const long long base = S.base;
    const int64_t gbase = (int64_t)blockIdx.x * kEmitThreads;
    for (int r = tid; r < rtotal; r += kEmitThreads) {
        int lo = 0, hi = kEmitThreads;  // the last owner with off[owner] <= r
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (S.off[mid] <= r) lo = mid; else hi = mid;
        }
        const Ellipse e{S.e[0][lo], S.e[1][lo], S.e[2][lo], S.e[3][lo],
                        S.e[4][lo], S.e[5][lo], S.e[6][lo], S.e[7][lo]};
        const int ty = S.ty0[lo] + (r - S.off[lo]);
        int tx0, tx1;
        if (!row_span(e, S.dyv[lo], ty, cam.W, cam.H, cam.ntx, &tx0, &tx1)) continue;
        const int w = tx1 - tx0;
        const long long at = base + S.poff[lo] + atomicAdd(&S.pcur[lo], w);
        const int rowbase = ty * cam.ntx;
        const uint32_t gid = (uint32_t)(gbase + lo);
        for (int i = 0; i < w; ++i) {
            const int t = rowbase + tx0 + i;
            atomicAdd(tile_count + (int64_t)t * kCountStride, 1);
            if (at + i < capacity) raw[at + i] = make_uint2((uint32_t)t, gid);
        }
    }
}

// ---------------------------------------------------------------------------
// 2. one cluster: tile ranges from the exclusive scan of the counts, the bucket
// cursors, I and min(I, capacity).  When I > capacity the list cannot be
// built; every range is then empty, so nothing downstream reads it.
// ---------------------------------------------------------------------------
// exclusive block scan (kScanThreads threads) of two int64 per thread at once
__device__ __forceinline__ void scan_block2(int64_t& a, int64_t& b, int64_t* s_a, int64_t* s_b,
                                            int64_t* ta, int64_t* tb) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t a0 = a, b0 = b;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int64_t ya = __shfl_up_sync(0xffffffffu, a, o);
        const int64_t yb = __shfl_up_sync(0xffffffffu, b, o);
        if (lane >= o) {
            a += ya;
            b += yb;
        }
    }
    if (lane == 31) {
        s_a[warp] = a;
        s_b[warp] = b;
    }
    __syncthreads();
    if (warp == 0) {
        int64_t wa = s_a[lane], wb = s_b[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t ya = __shfl_up_sync(0xffffffffu, wa, o);
            const int64_t yb = __shfl_up_sync(0xffffffffu, wb, o);
            if (lane >= o) {
                wa += ya;
                wb += yb;
            }
        }
        s_a[lane] = wa;
        s_b[lane] = wb;
    }
    __syncthreads();
    a += (warp > 0 ? s_a[warp - 1] : 0) - a0;
    b += (warp > 0 ? s_b[warp - 1] : 0) - b0;
    *ta = s_a[31];
    *tb = s_b[31];
}

constexpr int kScanRegs = 8;  // tiles per thread held in registers (nt <= 8192)

__device__ __forceinline__ int size_class(int c) {
    return c > kBlockSortMax ? 2 : (c > kWarpSortMax ? 1 : 0);
}

// The scan runs on a cluster of kScanCluster blocks (one per SM), each over a
// contiguous share of the tiles; the blocks' totals are exchanged through
// distributed shared memory, so the strided counter reads and the range and
// start writes spread over kScanCluster SMs.
constexpr int kScanCluster = 8;

__global__ void __launch_bounds__(kScanThreads) bucket_scan(const int* __restrict__ tile_count,
                                                            int64_t nt, int64_t capacity,
                                                            int2* __restrict__ ranges,
                                                            unsigned long long* __restrict__ cursor,
                                                            int32_t* __restrict__ medium,
                                                            int32_t* __restrict__ large,
                                                            int64_t* __restrict__ counts,
                                                            int64_t* __restrict__ counts_out) {
    grid_dep_sync();
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    __shared__ int64_t s_a[kScanThreads / 32], s_b[kScanThreads / 32];
    __shared__ int64_t s_tot[2];  // this block's pair count and packed class counts
    __shared__ int64_t s_off[4];  // offsets from the lower blocks; totals of all
    const int tid = threadIdx.x, lane = tid & 31;
    const int rank = (int)cluster.block_rank();
    const int64_t share = (nt + kScanCluster - 1) / kScanCluster;
    const int64_t b0 = min64(nt, share * rank), b1 = min64(nt, b0 + share);
    const int64_t per = (b1 - b0 + kScanThreads - 1) / kScanThreads;
    // consecutive threads take consecutive tiles: step k covers tiles
    // b0 + k kScanThreads + tid.  A tile's size class is packed into one int64
    // (medium: low word, large: high word; both counts are below 2^32, as nt is)
    auto cls_of = [](int ct) -> int64_t {
        const int z = size_class(ct);
        return z == 1 ? 1ll : (z == 2 ? (1ll << 32) : 0ll);
    };
    const bool in_regs = per <= kScanRegs;
    int c[kScanRegs];
    int64_t tr = 0, tc = 0;  // this thread's pair count and packed class counts
    if (in_regs) {
#pragma unroll
        for (int k = 0; k < kScanRegs; ++k) {
            const int64_t t = b0 + (int64_t)k * kScanThreads + tid;
            c[k] = k < per && t < b1 ? tile_count[t * kCountStride] : 0;
            tr += c[k];
            tc += cls_of(c[k]);
        }
    } else {
        for (int64_t t = b0 + tid; t < b1; t += kScanThreads) {
            const int ct = tile_count[t * kCountStride];
            tr += ct;
            tc += cls_of(ct);
        }
    }
    int64_t blk_run, blk_cls;  // this block's totals
    scan_block2(tr, tc, s_a, s_b, &blk_run, &blk_cls);
    if (tid == 0) {
        s_tot[0] = blk_run;
        s_tot[1] = blk_cls;
    }
    cluster.sync();
    if (tid < 32) {
        int64_t a = 0, b = 0;
        if (lane < kScanCluster) {
            const int64_t* t = cluster.map_shared_rank(s_tot, lane);
            a = t[0];
            b = t[1];
        }
        int64_t ea = lane < rank ? a : 0, eb = lane < rank ? b : 0;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            ea += __shfl_xor_sync(0xffffffffu, ea, o);
            eb += __shfl_xor_sync(0xffffffffu, eb, o);
            a += __shfl_xor_sync(0xffffffffu, a, o);
            b += __shfl_xor_sync(0xffffffffu, b, o);
        }
        if (lane == 0) {
            s_off[0] = ea;
            s_off[1] = eb;
            s_off[2] = a;
            s_off[3] = b;
        }
    }
    __syncthreads();
    const int64_t total = s_off[2], tcls = s_off[3];
    const bool fits = total <= capacity;
    int64_t carry_run = s_off[0], carry_cls = s_off[1];  // pairs / classes before this step
    for (int64_t k = 0; k < per; ++k) {
        __syncthreads();  // s_a / s_b are free again
        const int64_t t = b0 + k * kScanThreads + tid;
        int ct = 0;
        if (in_regs) {
#pragma unroll
            for (int q = 0; q < kScanRegs; ++q)
                if (q == k) ct = c[q];
        } else if (t < b1) {
            ct = tile_count[t * kCountStride];
        }
        int64_t r = ct, q = cls_of(ct), sr, sq;
        scan_block2(r, q, s_a, s_b, &sr, &sq);
        r += carry_run;
        q += carry_cls;
        if (t < b1) {
            ranges[t] = fits ? make_int2((int)r, (int)(r + ct)) : make_int2(0, 0);
            cursor[t * kCursorStride] = (unsigned long long)r;
            const int z = size_class(ct);
            if (z == 1) medium[q & 0xffffffffll] = (int32_t)t;
            if (z == 2) large[q >> 32] = (int32_t)t;
        }
        carry_run += sr;
        carry_cls += sq;
    }
    if (rank == 0 && tid == 0) {
        counts[1] = total;
        counts[2] = fits ? total : capacity;
        counts[kCountMedium] = fits ? (tcls & 0xffffffffll) : 0;
        counts[kCountLarge] = fits ? (tcls >> 32) : 0;
        if (counts_out) {
            counts_out[0] = counts[0];  // M: complete, the span pass has finished
            counts_out[1] = total;
        }
    }
    cluster.sync();  // s_tot stays readable until every block has read it
}

// ---------------------------------------------------------------------------
// 3. raw pairs -> the tiles' slices as (depth bits << 32 | id)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) bucket_scatter(const uint2* __restrict__ raw,
                                                      const float* __restrict__ depths,
                                                      unsigned long long* __restrict__ cursor,
                                                      int64_t capacity, uint64_t* __restrict__ keys,
                                                      const int64_t* __restrict__ counts) {
    grid_dep_sync();
    constexpr int kIlp = 4;
    const int64_t m = min64(counts[kCountRaw], capacity);
    const int64_t step = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i0 < m; i0 += kIlp * step) {
        uint2 p[kIlp];
        uint32_t d[kIlp];
        unsigned long long pos[kIlp];
#pragma unroll
        for (int u = 0; u < kIlp; ++u) {
            const int64_t i = i0 + u * step;
            p[u] = i < m ? raw[i] : make_uint2(0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < kIlp; ++u)
            d[u] = i0 + u * step < m ? __float_as_uint(__ldg(depths + p[u].y)) : 0u;
#pragma unroll
        for (int u = 0; u < kIlp; ++u)
            pos[u] = i0 + u * step < m ? atomicAdd(cursor + (int64_t)p[u].x * kCursorStride, 1ull)
                                       : ~0ull;
#pragma unroll
        for (int u = 0; u < kIlp; ++u)
            if (pos[u] < (unsigned long long)capacity) keys[pos[u]] = ((uint64_t)d[u] << 32) | p[u].y;
    }
}

// ---------------------------------------------------------------------------
// 4. sorting the slices
// ---------------------------------------------------------------------------
// Shared-memory index of element i: one pad word after every 16 elements, so
// that lanes reading 16 consecutive elements each hit different banks.
__device__ __forceinline__ int sk_idx(int i) { return i + (i >> 4); }
__host__ __device__ constexpr int sk_len(int n) { return n + n / 16; }

// number of elements of run a among the first k of merge(a[0, na), b[0, nb))
// (keys are unique); a and b index through sk_idx from a0 / b0
__device__ __forceinline__ int merge_split_s(const uint64_t* s, int a0, int na, int b0, int nb,
                                             int k) {
    int lo = max(0, k - nb), hi = min(k, na);
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (s[sk_idx(a0 + mid)] < s[sk_idx(b0 + k - 1 - mid)]) lo = mid + 1;
        else hi = mid;
    }
    return lo;
}

// One warp sorts the 32 E keys at src[0, 32 E) (shared memory, sk_idx layout)
// ascending, using dst[0, 32 E) as scratch; returns the buffer holding the
// result.  Each lane sorts its E consecutive keys in registers (bitonic
// network), then five merge-path rounds double the sorted runs.
template <int E>
__device__ __forceinline__ uint64_t* warp_merge_sort(uint64_t* src, uint64_t* dst, int lane) {
    uint64_t a[E];
#pragma unroll
    for (int r = 0; r < E; ++r) a[r] = src[sk_idx(lane * E + r)];
#pragma unroll
    for (int size = 2; size <= E; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
#pragma unroll
            for (int r = 0; r < E; ++r) {
                const int q = r ^ stride;
                if (q <= r) continue;
                const bool up = (r & size) == 0;
                const uint64_t x = a[r], y = a[q];
                const bool sw = (x > y) == up;
                a[r] = sw ? y : x;
                a[q] = sw ? x : y;
            }
        }
    }
#pragma unroll
    for (int r = 0; r < E; ++r) src[sk_idx(lane * E + r)] = a[r];
    __syncwarp();
#pragma unroll
    for (int L = E; L < 32 * E; L <<= 1) {
        const int o0 = lane * E;          // this lane's first output
        const int p0 = (o0 / (2 * L)) * (2 * L);
        const int k = o0 - p0;
        int i = merge_split_s(src, p0, L, p0 + L, L, k), j = k - i;
#pragma unroll
        for (int r = 0; r < E; ++r) {
            const uint64_t va = i < L ? src[sk_idx(p0 + i)] : ~0ull;
            const uint64_t vb = j < L ? src[sk_idx(p0 + L + j)] : ~0ull;
            const bool ta = va < vb;
            dst[sk_idx(o0 + r)] = ta ? va : vb;
            i += ta;
            j += !ta;
        }
        __syncwarp();
        uint64_t* t = src;
        src = dst;
        dst = t;
    }
    return src;
}

template <int E>
__device__ __forceinline__ void warp_sort_tile(const uint64_t* __restrict__ keys, int64_t s, int cnt,
                                               uint64_t* b0, uint64_t* b1, int lane,
                                               int32_t* __restrict__ sorted_ids) {
#pragma unroll
    for (int r = 0; r < E; ++r) {
        const int e = r * 32 + lane;
        b0[sk_idx(e)] = e < cnt ? keys[s + e] : ~0ull;
    }
    __syncwarp();
    const uint64_t* out = warp_merge_sort<E>(b0, b1, lane);
#pragma unroll
    for (int r = 0; r < E; ++r) {
        const int e = r * 32 + lane;
        if (e < cnt) sorted_ids[s + e] = (int32_t)(uint32_t)out[sk_idx(e)];
    }
    __syncwarp();
}

// slices of 1 .. kWarpSortMax keys: one warp each
constexpr int kSmallWarps = 4;
__global__ void __launch_bounds__(32 * kSmallWarps, 6) bucket_sort_small(const int2* __restrict__ ranges,
                                                                      int64_t nt,
                                                                      const uint64_t* __restrict__ keys,
                                                                      int32_t* __restrict__ sorted_ids) {
    grid_dep_sync();
    __shared__ uint64_t sbuf[kSmallWarps][2][sk_len(kWarpSortMax)];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint64_t* b0 = sbuf[warp][0];
    uint64_t* b1 = sbuf[warp][1];
    const int64_t w0 = (int64_t)blockIdx.x * kSmallWarps + warp;
    const int64_t nw = (int64_t)gridDim.x * kSmallWarps;
    for (int64_t t = w0; t < nt; t += nw) {
        const int2 r = ranges[t];
        const int cnt = r.y - r.x;
        if (cnt == 1) {
            if (lane == 0) sorted_ids[r.x] = (int32_t)(uint32_t)keys[r.x];
        } else if (cnt > 1 && cnt <= 32) {
            warp_sort_tile<1>(keys, r.x, cnt, b0, b1, lane, sorted_ids);
        } else if (cnt > 32 && cnt <= 64) {
            warp_sort_tile<2>(keys, r.x, cnt, b0, b1, lane, sorted_ids);
        } else if (cnt > 64 && cnt <= 128) {
            warp_sort_tile<4>(keys, r.x, cnt, b0, b1, lane, sorted_ids);
        } else if (cnt > 128 && cnt <= 256) {
            warp_sort_tile<8>(keys, r.x, cnt, b0, b1, lane, sorted_ids);
        } else if (cnt > 256 && cnt <= kWarpSortMax) {
            warp_sort_tile<16>(keys, r.x, cnt, b0, b1, lane, sorted_ids);
        }
    }
}

// Block-wide merge-path rounds in shared memory: runs of length L0 .. P / 2 in
// src are merged pairwise until one run of P keys remains; returns its buffer.
__device__ __forceinline__ uint64_t* block_merge_rounds(uint64_t* src, uint64_t* dst, int L0, int P) {
    const int tid = threadIdx.x;
    const int per = P / kSortThreads;  // outputs per thread
    for (int L = L0; L < P; L <<= 1) {
        const int o0 = tid * per;
        const int p0 = (o0 / (2 * L)) * (2 * L);
        const int k = o0 - p0;
        int i = merge_split_s(src, p0, L, p0 + L, L, k), j = k - i;
        for (int q = 0; q < per; ++q) {
            const uint64_t va = i < L ? src[sk_idx(p0 + i)] : ~0ull;
            const uint64_t vb = j < L ? src[sk_idx(p0 + L + j)] : ~0ull;
            const bool ta = va < vb;
            dst[sk_idx(o0 + q)] = ta ? va : vb;
            i += ta;
            j += !ta;
        }
        __syncthreads();
        uint64_t* tmp = src;
        src = dst;
        dst = tmp;
    }
    return src;
}

// Sort P keys (P = 8 * 32 E, padded) in A: every warp sorts one chunk of 32 E
// (its result lands in B: five warp rounds), then block-wide rounds.
template <int E>
__device__ __forceinline__ uint64_t* block_sort_keys(uint64_t* A, uint64_t* B) {
    constexpr int kWarps = kSortThreads / 32;
    constexpr int C = 32 * E;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    static_assert(kWarps == 8, "eight warps");
    // chunk offsets are multiples of 16, so sk_idx is affine across them
    warp_merge_sort<E>(A + sk_idx(warp * C), B + sk_idx(warp * C), lane);
    __syncthreads();
    return block_merge_rounds(B, A, C, kWarps * C);
}

// One block sorts a slice of kWarpSortMax + 1 .. kBlockSortMax keys in shared
// memory (A, B: sk_len(kBlockSortMax) words each) and writes its ids.
__device__ __forceinline__ void sort_medium_slice(int2 r, const uint64_t* __restrict__ keys,
                                                  int32_t* __restrict__ sorted_ids, uint64_t* A,
                                                  uint64_t* B) {
    const int tid = threadIdx.x;
    const int cnt = r.y - r.x;
    int P = 2 * kWarpSortMax;
    while (P < cnt) P <<= 1;
    for (int e = tid; e < P; e += kSortThreads) A[sk_idx(e)] = e < cnt ? keys[r.x + e] : ~0ull;
    __syncthreads();
    const uint64_t* out = P == 1024 ? block_sort_keys<4>(A, B)
                          : P == 2048 ? block_sort_keys<8>(A, B)
                                      : block_sort_keys<16>(A, B);
    for (int e = tid; e < cnt; e += kSortThreads)
        sorted_ids[r.x + e] = (int32_t)(uint32_t)out[sk_idx(e)];
    __syncthreads();
}

// The medium slices (kWarpSortMax + 1 .. kBlockSortMax keys), one block each.
__global__ void __launch_bounds__(kSortThreads) bucket_sort_blocks(const int2* __restrict__ ranges,
                                                                   const int32_t* __restrict__ medium,
                                                                   const uint64_t* __restrict__ keys,
                                                                   int32_t* __restrict__ sorted_ids,
                                                                   const int64_t* __restrict__ counts) {
    grid_dep_sync();
    extern __shared__ uint64_t smem[];
    uint64_t* A = smem;                            // sk_len(kBlockSortMax)
    uint64_t* B = smem + sk_len(kBlockSortMax);    // sk_len(kBlockSortMax)
    const int64_t nm = counts[kCountMedium];
    for (int64_t m = blockIdx.x; m < nm; m += gridDim.x)
        sort_medium_slice(ranges[medium[m]], keys, sorted_ids, A, B);
}

// ---------------------------------------------------------------------------
// the long slices (more than kBlockSortMax keys): a merge sort over the whole
// grid.  Every slice is cut into chunks of kBlockSortMax keys, each chunk is
// sorted by one block in shared memory, and merge rounds double the sorted
// runs: in a round every kBlockSortMax-key piece of every slice's output is
// merged by one block from the two runs it falls between (the run split found
// by merge path in global memory, the piece merged in shared memory).  The
// round in which a slice becomes one run writes its ids.
// ---------------------------------------------------------------------------
constexpr int kLongChunk = kBlockSortMax;

// One block: chunk offsets of the long slices (exclusive prefix of their chunk
// counts, chunk_off[nl] = the total), the total and the longest slice.
__global__ void __launch_bounds__(kScanThreads) long_plan(const int2* __restrict__ ranges,
                                                          const int32_t* __restrict__ large,
                                                          int32_t* __restrict__ chunk_off,
                                                          int64_t* __restrict__ counts) {
    grid_dep_sync();
    __shared__ int64_t s_a[kScanThreads / 32], s_b[kScanThreads / 32];
    const int tid = threadIdx.x;
    const int64_t nl = counts[kCountLarge];
    int64_t carry = 0, longest = 0;
    for (int64_t b = 0; b < nl; b += kScanThreads) {
        const int64_t m = b + tid;
        int64_t ch = 0, len = 0;
        if (m < nl) {
            const int2 r = ranges[large[m]];
            len = r.y - r.x;
            ch = (len + kLongChunk - 1) / kLongChunk;
        }
        int64_t ex = ch, mx = len, tot, unused;
        scan_block2(ex, mx, s_a, s_b, &tot, &unused);
        if (m < nl) chunk_off[m] = (int32_t)(carry + ex);
        carry += tot;
        // the longest: a max over the block (mx was scanned as a sum; redo as a max)
        int64_t v = len;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
        __syncthreads();
        if ((tid & 31) == 0) s_a[tid >> 5] = v;
        __syncthreads();
        if (tid < 32) {
            int64_t w = s_a[tid];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) w = max(w, __shfl_xor_sync(0xffffffffu, w, o));
            if (tid == 0) s_b[0] = w;
        }
        __syncthreads();
        longest = max(longest, s_b[0]);
        __syncthreads();
    }
    if (tid == 0) {
        chunk_off[nl] = (int32_t)carry;
        counts[kCountLongChunks] = carry;
        counts[kCountLongest] = longest;
    }
}

// the long slice m holding global chunk c: chunk_off[m] <= c < chunk_off[m + 1]
__device__ __forceinline__ int64_t long_owner(const int32_t* __restrict__ chunk_off, int64_t nl,
                                              int64_t c) {
    int64_t lo = 0, hi = nl;  // chunk_off[lo] <= c < chunk_off[hi]
    while (hi - lo > 1) {
        const int64_t mid = (lo + hi) >> 1;
        if (chunk_off[mid] <= c) lo = mid; else hi = mid;
    }
    return lo;
}

__global__ void __launch_bounds__(kSortThreads) long_chunks(const int2* __restrict__ ranges,
                                                            const int32_t* __restrict__ large,
                                                            const int32_t* __restrict__ chunk_off,
                                                            uint64_t* __restrict__ keys,
                                                            const int64_t* __restrict__ counts) {
    grid_dep_sync();
    extern __shared__ uint64_t smem[];
    uint64_t* A = smem;
    uint64_t* B = smem + sk_len(kBlockSortMax);
    const int tid = threadIdx.x;
    const int64_t nl = counts[kCountLarge], T = counts[kCountLongChunks];
    for (int64_t c = blockIdx.x; c < T; c += gridDim.x) {
        const int64_t m = long_owner(chunk_off, nl, c);
        const int2 r = ranges[large[m]];
        const int64_t s = (int64_t)r.x + (c - chunk_off[m]) * kLongChunk;
        const int n = (int)min64(kLongChunk, (int64_t)r.y - s);
        for (int e = tid; e < kLongChunk; e += kSortThreads) A[sk_idx(e)] = e < n ? keys[s + e] : ~0ull;
        __syncthreads();
        const uint64_t* out = block_sort_keys<16>(A, B);
        for (int e = tid; e < n; e += kSortThreads) keys[s + e] = out[sk_idx(e)];
        __syncthreads();
    }
}

// Merge path in global memory by one warp: the number of elements of a[0, na)
// among the first k of merge(a, b) (keys are unique).  Each step tests 32
// evenly spaced candidates, so a search over 2^17 takes four steps.
__device__ __forceinline__ int64_t merge_split_warp(const uint64_t* __restrict__ a, int64_t na,
                                                    const uint64_t* __restrict__ b, int64_t nb,
                                                    int64_t k, int lane) {
    int64_t lo = max64(0, k - nb), hi = min64(k, na);  // the answer lies in [lo, hi]
    while (lo < hi) {
        const int64_t span = hi - lo;
        const int64_t step = (span + 31) / 32;
        const int64_t i = lo + (int64_t)lane * step;
        // true for i below the answer (a[i] precedes the (k - i)-th element of b)
        const bool p = i < hi && a[i] < b[k - 1 - i];
        const int t = __popc(__ballot_sync(0xffffffffu, p));
        if (step == 1) return lo + t;
        // samples 0 .. t-1 are below the answer, sample t (if any) is not
        const int64_t nlo = t > 0 ? lo + (int64_t)(t - 1) * step + 1 : lo;
        const int64_t nhi = min64(hi, lo + (int64_t)t * step);
        lo = nlo;
        hi = nhi;
    }
    return lo;
}

// One merge round of width w: the runs [p0, p0 + w) and [p0 + w, p0 + 2w) of
// every long slice still longer than w are merged from src into dst, or into
// the ids when the merged run is the whole slice.
__global__ void __launch_bounds__(kSortThreads) long_round(const int2* __restrict__ ranges,
                                                           const int32_t* __restrict__ large,
                                                           const int32_t* __restrict__ chunk_off,
                                                           const uint64_t* __restrict__ src,
                                                           uint64_t* __restrict__ dst,
                                                           int32_t* __restrict__ sorted_ids,
                                                           int64_t w,
                                                           const int64_t* __restrict__ counts) {
    grid_dep_sync();
    extern __shared__ uint64_t smem[];      // kLongChunk keys: the piece's inputs
    __shared__ int64_t s_split[2];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t nl = counts[kCountLarge], T = counts[kCountLongChunks];
    if (counts[kCountLongest] <= w) return;  // every slice is one run already
    constexpr int kPer = kLongChunk / kSortThreads;  // outputs per thread
    for (int64_t c = blockIdx.x; c < T; c += gridDim.x) {
        const int64_t m = long_owner(chunk_off, nl, c);
        const int2 r = ranges[large[m]];
        const int64_t n = (int64_t)r.y - r.x;
        if (n <= w) continue;  // this slice finished in an earlier round
        const int64_t o0 = (c - chunk_off[m]) * kLongChunk, o1 = min64(o0 + kLongChunk, n);
        const int64_t p0 = (o0 / (2 * w)) * (2 * w);
        const int64_t na = min64(w, n - p0), nb = min64(w, n - p0 - na);
        const bool last = 2 * w >= n;
        const uint64_t* a = src + r.x + p0;
        const uint64_t* b = a + na;
        if (warp < 2) {
            const int64_t k = (warp == 0 ? o0 : o1) - p0;
            const int64_t i = merge_split_warp(a, na, b, nb, k, lane);
            if (lane == 0) s_split[warp] = i;
        }
        __syncthreads();
        const int64_t i0 = s_split[0], i1 = s_split[1];
        const int64_t j0 = (o0 - p0) - i0, j1 = (o1 - p0) - i1;
        const int la = (int)(i1 - i0), lb = (int)(j1 - j0);
        for (int e = tid; e < la; e += kSortThreads) smem[e] = a[i0 + e];
        for (int e = tid; e < lb; e += kSortThreads) smem[la + e] = b[j0 + e];
        __syncthreads();
        // this thread's outputs [kPer tid, kPer tid + kPer) of the piece
        const int q0 = tid * kPer, q1 = min(q0 + kPer, la + lb);
        if (q0 < q1) {
            int lo = max(0, q0 - lb), hi = min(q0, la);
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (smem[mid] < smem[la + q0 - 1 - mid]) lo = mid + 1;
                else hi = mid;
            }
            int x = lo, y = q0 - lo;
            const int64_t out = r.x + o0;
            for (int q = q0; q < q1; ++q) {
                const uint64_t va = x < la ? smem[x] : ~0ull;
                const uint64_t vb = y < lb ? smem[la + y] : ~0ull;
                const bool ta = va < vb;
                const uint64_t v = ta ? va : vb;
                x += ta;
                y += !ta;
                if (last) sorted_ids[out + q] = (int32_t)(uint32_t)v;
                else dst[out + q] = v;
            }
        }
        __syncthreads();  // smem and s_split are reused by the next piece
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
    grid_dep_sync();
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

// rank of every key = its position in its run + the keys smaller than it in the
// other runs; the runs are searched in shared memory when they fit
constexpr int kLptSmemRuns = 6;
__global__ void __launch_bounds__(256) lpt_merge(const uint64_t* __restrict__ runs, int64_t nt,
                                                 int32_t* __restrict__ lpt) {
    grid_dep_sync();
    __shared__ uint64_t sr[kLptSmemRuns * kLptRun];
    const int64_t nruns = (nt + kLptRun - 1) / kLptRun;
    const bool in_smem = nruns <= kLptSmemRuns;
    if (in_smem) {
        for (int64_t e = threadIdx.x; e < nruns * kLptRun; e += blockDim.x) sr[e] = runs[e];
        __syncthreads();
    }
    const uint64_t* R = in_smem ? sr : runs;
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= nruns * kLptRun) return;
    const uint64_t key = R[i];
    if (key == ~0ull) return;  // padding
    const int64_t r = i / kLptRun;
    int64_t rank = i - r * kLptRun;
    for (int64_t r2 = 0; r2 < nruns; ++r2) {
        if (r2 == r) continue;
        const uint64_t* run = R + r2 * kLptRun;
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

}  // namespace

size_t lpt_runs_bytes(int64_t nt) {
    nt = std::max<int64_t>(nt, 1);
    return (size_t)((nt + kLptRun - 1) / kLptRun) * kLptRun * sizeof(uint64_t);
}

cudaError_t launch_lpt(const int2* ranges, int64_t nt, uint64_t* runs, int32_t* lpt_order,
                       cudaStream_t st) {
    const unsigned nruns = (unsigned)((nt + kLptRun - 1) / kLptRun);
    cudaError_t err = launch(lpt_sort_runs, nruns, kLptRun / 2, 0, st, ranges, nt, runs);
    if (err != cudaSuccess) return err;
    return launch(lpt_merge, (unsigned)((nruns * (int64_t)kLptRun + 255) / 256), 256, 0, st,
                  (const uint64_t*)runs, nt, lpt_order);
}

BinSortLayout binsort_layout(int64_t n, int64_t capacity, int64_t n_tiles) {
    BinSortLayout L{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t o = off;
        off = align_up(off + bytes);
        return o;
    };
    (void)n;
    const int64_t cap = std::max<int64_t>(capacity, 1);
    const int64_t nt = std::max<int64_t>(n_tiles, 1);
    L.off_counts = take(8 * sizeof(int64_t));
    L.off_raw = take((size_t)cap * sizeof(uint2));
    L.off_keys = take((size_t)cap * sizeof(uint64_t));
    L.off_tcount = take((size_t)nt * kCountStride * sizeof(int));
    L.off_cursor = take((size_t)nt * kCursorStride * sizeof(unsigned long long));
    L.off_lists = take((size_t)nt * 2 * sizeof(int32_t));
    L.off_lchunk = take((size_t)(nt + 1) * sizeof(int32_t));
    L.off_lruns = take(lpt_runs_bytes(nt));
    L.total = off;
    return L;
}

cudaError_t run_bin_sort(const CamParams& cam, int64_t n, const float* splats, const float* depths,
                         const int32_t* tiles_touched, char* ws, const BinSortLayout& L,
                         int32_t* sorted_ids, int64_t capacity, int32_t* tile_ranges,
                         int32_t* lpt_order, int64_t* counts_out, cudaStream_t st,
                         const SideStream* side) {
    auto* counts = reinterpret_cast<int64_t*>(ws + L.off_counts);
    auto* raw = reinterpret_cast<uint2*>(ws + L.off_raw);
    auto* keys = reinterpret_cast<uint64_t*>(ws + L.off_keys);
    auto* tcount = reinterpret_cast<int*>(ws + L.off_tcount);
    auto* cursor = reinterpret_cast<unsigned long long*>(ws + L.off_cursor);
    auto* medium = reinterpret_cast<int32_t*>(ws + L.off_lists);
    auto* lruns = reinterpret_cast<uint64_t*>(ws + L.off_lruns);
    const int64_t nt = (int64_t)cam.ntx * cam.nty;
    auto* large = medium + nt;
    auto* ranges = reinterpret_cast<int2*>(tile_ranges);
    cudaError_t err;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    sms = std::max(sms, 1);

    // 0. the counters start at zero
    err = launch(bin_zero, (unsigned)std::min<int64_t>((nt + 255) / 256, 4 * (int64_t)sms), 256, 0,
                 st, counts, tcount, nt);
    if (err != cudaSuccess) return err;
    // 1.-2. pairs and tile counts; tile ranges
    if (n > 0) {
        err = launch(bucket_emit, (unsigned)((n + kEmitThreads - 1) / kEmitThreads), kEmitThreads, 0,
                     st, cam, reinterpret_cast<const float4*>(splats), tiles_touched, n, capacity,
                     tcount, raw, counts);
        if (err != cudaSuccess) return err;
    }
    err = launch_clustered(bucket_scan, kScanCluster, kScanCluster, kScanThreads, 0, st,
                           (const int*)tcount, nt, capacity, ranges, cursor, medium, large, counts,
                           counts_out);
    if (err != cudaSuccess) return err;
    // 5. LPT order (tiles by descending count, ties by tile id) needs only the
    // ranges: on the side stream, when given, it runs beside steps 3 and 4
    cudaStream_t ls = st;
    if (side) {
        err = cudaEventRecord(side->fork, st);
        if (err != cudaSuccess) return err;
        err = cudaStreamWaitEvent(side->stream, side->fork, 0);
        if (err != cudaSuccess) return err;
        ls = side->stream;
    }
    err = launch_lpt(ranges, nt, lruns, lpt_order, ls);
    if (err != cudaSuccess) return err;
    if (n > 0) {
        // 3. the pairs into their tiles' slices
        const unsigned grid = (unsigned)std::max<int64_t>(
            1, std::min<int64_t>((capacity + 255) / 256, 8 * (int64_t)sms));
        err = launch(bucket_scatter, grid, 256, 0, st, (const uint2*)raw, depths, cursor, capacity,
                     keys, (const int64_t*)counts);
        if (err != cudaSuccess) return err;
        // 4. the short slices on st; the medium and long ones (other tiles, other
        // parts of the key and id lists) beside them on the side stream
        cudaStream_t ms = st;
        if (side) {
            err = cudaEventRecord(side->fork2, st);
            if (err != cudaSuccess) return err;
            err = cudaStreamWaitEvent(side->stream, side->fork2, 0);
            if (err != cudaSuccess) return err;
            ms = side->stream;
        }
        const unsigned sg = (unsigned)std::max<int64_t>(
            1, std::min<int64_t>((nt + kSmallWarps - 1) / kSmallWarps, 16 * (int64_t)sms));
        err = launch(bucket_sort_small, sg, 32 * kSmallWarps, 0, st, (const int2*)ranges, nt,
                     (const uint64_t*)keys, sorted_ids);
        if (err != cudaSuccess) return err;
        const size_t sbytes = 2 * sk_len(kBlockSortMax) * sizeof(uint64_t);
        err = cudaFuncSetAttribute(bucket_sort_blocks, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)sbytes);
        if (err != cudaSuccess) return err;
        const unsigned mg = (unsigned)std::max<int64_t>(1, std::min<int64_t>(nt, 3 * (int64_t)sms));
        err = launch(bucket_sort_blocks, mg, kSortThreads, sbytes, ms, (const int2*)ranges,
                     (const int32_t*)medium, (const uint64_t*)keys, sorted_ids,
                     (const int64_t*)counts);
        if (err != cudaSuccess) return err;
        // the long slices: chunk sorts, then merge rounds between the key list and
        // the raw list (free again) -- on a second side stream when given.  A tile
        // holds at most one pair per Gaussian, so min(n, capacity) bounds a slice
        // and fixes the number of rounds; rounds past the longest slice return at once.
        cudaStream_t gs = side ? side->stream2 : st;
        if (side) {
            err = cudaStreamWaitEvent(gs, side->fork2, 0);
            if (err != cudaSuccess) return err;
        }
        auto* chunk_off = reinterpret_cast<int32_t*>(ws + L.off_lchunk);
        err = launch(long_plan, 1, kScanThreads, 0, gs, (const int2*)ranges, (const int32_t*)large,
                     chunk_off, counts);
        if (err != cudaSuccess) return err;
        err = cudaFuncSetAttribute(long_chunks, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)sbytes);
        if (err != cudaSuccess) return err;
        err = launch(long_chunks, (unsigned)(3 * sms), kSortThreads, sbytes, gs, (const int2*)ranges,
                     (const int32_t*)large, (const int32_t*)chunk_off, keys, (const int64_t*)counts);
        if (err != cudaSuccess) return err;
        const int64_t bound = std::min<int64_t>(n, capacity);
        const size_t rbytes = (size_t)kLongChunk * sizeof(uint64_t);
        uint64_t* bufs[2] = {keys, reinterpret_cast<uint64_t*>(raw)};
        int r = 0;
        for (int64_t w = kLongChunk; w < bound; w *= 2, ++r) {
            err = launch(long_round, (unsigned)(6 * sms), kSortThreads, rbytes, gs,
                         (const int2*)ranges, (const int32_t*)large, (const int32_t*)chunk_off,
                         (const uint64_t*)bufs[r & 1], bufs[(r & 1) ^ 1], sorted_ids, w,
                         (const int64_t*)counts);
            if (err != cudaSuccess) return err;
        }
        if (side) {
            err = cudaEventRecord(side->join2, gs);
            if (err != cudaSuccess) return err;
            err = cudaStreamWaitEvent(st, side->join2, 0);
            if (err != cudaSuccess) return err;
        }
    }
    if (side) {
        // the LPT order and the medium and long slices are done
        err = cudaEventRecord(side->join, side->stream);
        if (err != cudaSuccess) return err;
        err = cudaStreamWaitEvent(st, side->join, 0);
        if (err != cudaSuccess) return err;
    }
    return cudaSuccess;
}

}  // namespace gs
