// gs_binsort_radix.cu -- tile binning for long pair lists: the two-stage
// radix sort.
//
// "What the 3DGS Literature Left on the Table" (Kopanas), Step 1 (b), (d): the
// visible Gaussians are sorted once by a 32-bit depth key, their (tile,
// Gaussian) pairs are emitted in that depth order from the exact row spans, and
// the pairs are then sorted by the tile key with a stable LSD radix sort, so the
// list is ordered by (tile, depth, id).  "Mitigating SM-Level Load Imbalance in
// 3D Gaussian Splatting on GPUs" (Ryu & Yoo), Sec. 4.1: LPT order of the tiles.
//
// gs_bin_sort takes this path when the pair capacity is large (millions of
// pairs): every pass is then a stream over the keys at memory speed, where the
// per-tile buckets of gs_binsort.cu contend on the counters of dense tiles.
// Same outputs, bit for bit.
//
// Radix sort: LSD, 8-bit digits, one kernel per pass; the digit counts of every
// pass are taken by the kernel that writes the keys (the visible-Gaussian
// compaction, the pair emission).  Blocks take 4096-key tiles in ticket order,
// rank keys within warps from one ballot per digit bit (eight, or fewer in a
// last pass whose higher bits are zero in every key) and one shared atomic per
// digit and warp, publish their digit counts and add those of earlier tiles by
// decoupled look-back (every wait is bounded and sets a give-up flag).
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

// One pass of the stable LSD sort: blocks take consecutive 4096-key tiles in
// ticket order, rank their keys by digit (within warps from ballots, then
// across warps), publish their digit counts, and add the counts of the tiles
// before them by looking back through the published words (decoupled
// look-back: a block only waits on tiles that started before it, so waits
// end).  Keys are staged in shared memory in block-sorted order so that each
// digit's run is written to global memory contiguously.  NB is the number of
// the pass's digit bits that keys can set (keys are below 2^bits): the others
// are zero in every key and need no ballot.
struct OnesweepSmem {
    uint32_t keys[kRsTile];
    int32_t vals[kRsTile];
    uint32_t wcnt[kRsWarps][256];
    uint32_t dstart[256];
    int64_t gbase[256];
    uint32_t warp_sums[kRsWarps];
    int ticket;
};

template <int NB>
__global__ void __launch_bounds__(kRsBlock, 4) rs_onesweep(
    const uint32_t* __restrict__ keys_in, const int32_t* __restrict__ vals_in,
    uint32_t* __restrict__ keys_out, int32_t* __restrict__ vals_out, const int64_t* n_dev,
    int64_t n_static, int pass, const uint32_t* __restrict__ ghist, int* __restrict__ tickets,
    uint64_t* __restrict__ lookback, unsigned long long* __restrict__ err) {
    grid_dep_sync();
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
    // The lanes holding the same digit come from NB ballots; the lowest of them
    // adds their number to the warp's count of that digit and hands the old count
    // to the others.  Items are ranked in order r = 0, 1, ...: the leaders of
    // item r may be other lanes than those of item r - 1, and __syncwarp() orders
    // the two items' shared-memory updates among the warp's lanes (the CUDA
    // programming guide's memory-ordering guarantee of __syncwarp), so item r's
    // offsets follow item r - 1's and the ranking is stable.
    const uint32_t lt = lanemask_lt();
#pragma unroll
    for (int r = 0; r < kRsIpt; ++r) {
        const int64_t idx = wbase + r * 32 + lane;
        const bool valid = idx < n;
        const uint32_t d = (k[r] >> shift) & 255u;
        uint32_t peers = __ballot_sync(0xffffffffu, valid);
#pragma unroll
        for (int bit = 0; bit < NB; ++bit) {
            const uint32_t m = __ballot_sync(0xffffffffu, (d >> bit) & 1u);
            peers &= ((d >> bit) & 1u) ? m : ~m;
        }
        if (!valid) peers = 1u << lane;
        const int leader = __ffs(peers) - 1;
        uint32_t old = 0;
        if (valid && leader == lane) old = atomicAdd(&S.wcnt[warp][d], (uint32_t)__popc(peers));
        loc[r] = __shfl_sync(0xffffffffu, old, leader) + __popc(peers & lt);
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

    // ---- stage in block-sorted order (before the look-back: the keys' registers
    // are free while it waits)
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

    // ---- look back over the earlier tiles for this digit, kLbWindow words in
    // flight at a time (nearest first), up to the first inclusive prefix (8, 16
    // and 32 words measured alike on 29.7M keys: the walk is not what bounds
    // the pass)
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

    // ---- write each digit run contiguously
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
// return where the sorted keys and values are.  ghist holds the digit counts of
// every pass ([pass][digit], taken when the keys were written).  ctl is the
// sort's control region (rs_ctl_bytes(n_max)), cleared here; err collects
// give-up flags.
size_t rs_ctl_bytes(int64_t n_max) {
    return 16 + kMaxPasses * 256 * 4 + (size_t)std::max<int64_t>(1, nblk_of(n_max)) * 256 * 8;
}

cudaError_t radix_sort(uint32_t* k0, int32_t* v0, uint32_t* k1, int32_t* v1, int32_t* vf,
                       const int64_t* n_dev, int64_t n_static, int64_t n_max, int bits, char* ctl,
                       const uint32_t* ghist_given, unsigned long long* err, cudaStream_t st,
                       uint32_t** kres, int32_t** vres) {
    const int passes = std::max(1, (bits + 7) / 8);
    const unsigned grid = (unsigned)std::max<int64_t>(1, nblk_of(n_max));
    int* tickets = reinterpret_cast<int*>(ctl);
    const uint32_t* ghist = ghist_given;  // taken by the kernel that wrote the keys
    uint64_t* lookback = reinterpret_cast<uint64_t*>(ctl + 16 + kMaxPasses * 256 * 4);
    cudaError_t e = cudaMemsetAsync(ctl, 0, rs_ctl_bytes(n_max), st);
    if (e != cudaSuccess) return e;
    uint32_t* kin = k0;
    int32_t* vin = v0;
    for (int p = 0; p < passes; ++p) {
        const bool last = p == passes - 1;
        uint32_t* kout = kin == k0 ? k1 : k0;
        int32_t* vout = (last && vf) ? vf : (vin == v0 ? v1 : v0);
        const int nb = std::min(8, bits - 8 * p);
        auto go = [&](auto kernel) {
            return launch(kernel, grid, kRsBlock, 0, st, (const uint32_t*)kin, (const int32_t*)vin,
                          kout, vout, n_dev, n_static, p, ghist, tickets, lookback, err);
        };
        switch (nb) {
            case 1: e = go(rs_onesweep<1>); break;
            case 2: e = go(rs_onesweep<2>); break;
            case 3: e = go(rs_onesweep<3>); break;
            case 4: e = go(rs_onesweep<4>); break;
            case 5: e = go(rs_onesweep<5>); break;
            case 6: e = go(rs_onesweep<6>); break;
            case 7: e = go(rs_onesweep<7>); break;
            default: e = go(rs_onesweep<8>); break;
        }
        if (e != cudaSuccess) return e;
        kin = kout;
        vin = vout;
    }
    if (kres) *kres = kin;
    if (vres) *vres = vin;
    return cudaSuccess;
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
    grid_dep_sync();
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
    grid_dep_sync();
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

// visible Gaussians, in id order: (depth key, id).  Warp w of a block owns its
// 512 consecutive ids in 16 sweeps of 32 (lane l takes id 32 r + l of sweep r),
// so loads and stores are coalesced; a ballot per sweep ranks the visible ones,
// and one scan of the 8 warps' counts places each warp's run.
__global__ void __launch_bounds__(kRsBlock) vis_write(const int32_t* __restrict__ tiles_touched,
                                                      const float* __restrict__ depths, int64_t n,
                                                      const int64_t* __restrict__ bsum,
                                                      uint32_t* __restrict__ keys,
                                                      int32_t* __restrict__ vals,
                                                      uint32_t* __restrict__ dhist) {
    grid_dep_sync();
    __shared__ int s_cnt[kRsWarps];
    __shared__ uint32_t hist[kMaxPasses][256];
#pragma unroll
    for (int p = 0; p < kMaxPasses; ++p) hist[p][threadIdx.x] = 0;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t wbase = (int64_t)blockIdx.x * kRsTile + (int64_t)warp * (32 * kRsIpt);
    uint32_t m[kRsIpt];
    int cnt = 0;
#pragma unroll
    for (int r = 0; r < kRsIpt; ++r) {
        const int64_t idx = wbase + 32 * r + lane;
        m[r] = __ballot_sync(0xffffffffu, idx < n && tiles_touched[idx] > 0);
        cnt += __popc(m[r]);
    }
    if (lane == 0) s_cnt[warp] = cnt;
    __syncthreads();
    int64_t pos = bsum[blockIdx.x];
#pragma unroll
    for (int w = 0; w < kRsWarps; ++w) pos += w < warp ? s_cnt[w] : 0;
    const uint32_t lt = lanemask_lt();
#pragma unroll
    for (int r = 0; r < kRsIpt; ++r) {
        if ((m[r] >> lane) & 1u) {
            const int64_t idx = wbase + 32 * r + lane;
            const int64_t at = pos + __popc(m[r] & lt);
            const uint32_t k = __float_as_uint(depths[idx]);  // depth > znear > 0: bits are ordered
            keys[at] = k;
            vals[at] = (int32_t)idx;
#pragma unroll
            for (int p = 0; p < kMaxPasses; ++p) atomicAdd(&hist[p][(k >> (8 * p)) & 255u], 1u);
        }
        pos += __popc(m[r]);
    }
    __syncthreads();
#pragma unroll
    for (int p = 0; p < kMaxPasses; ++p)
        if (hist[p][threadIdx.x]) atomicAdd(dhist + p * 256 + threadIdx.x, hist[p][threadIdx.x]);
}

// pairs per visible Gaussian in depth order: per-block sums
__global__ void __launch_bounds__(kRsBlock) pairs_count(const int32_t* __restrict__ order,
                                                        const int32_t* __restrict__ tiles_touched,
                                                        const int64_t* __restrict__ m_dev,
                                                        int64_t* __restrict__ bsum) {
    grid_dep_sync();
    const int64_t m = *m_dev;
    if ((int64_t)blockIdx.x >= nblk_of(m)) return;
    __shared__ int64_t s_warp[kRsWarps];
    const int64_t base = (int64_t)blockIdx.x * kRsTile;
    int64_t c = 0;
    // all of a thread's count gathers in flight at once
#pragma unroll
    for (int i = threadIdx.x; i < kRsTile; i += kRsBlock) {
        int64_t j = base + i;
        if (j < m) c += tiles_touched[order[j]];
    }
    int64_t total;
    block_exclusive_scan_256<int64_t>(c, s_warp, &total);
    if (threadIdx.x == 0) bsum[blockIdx.x] = total;
}

// Output pairs per block of the emission: the blocks split the depth-ordered pair
// list into equal contiguous pieces.
constexpr int kEmitPairs = 2048;

// poffd[j] = first pair of the depth-rank-j visible Gaussian (poffd[m] = I), and
// bstart[k] = the depth rank of the Gaussian holding pair k kEmitPairs, for the
// nbs emission blocks that exist (pairs past the capacity get no block).
__global__ void __launch_bounds__(kRsBlock) pairs_offsets(const int32_t* __restrict__ order,
                                                          const int32_t* __restrict__ tiles_touched,
                                                          const int64_t* __restrict__ m_dev,
                                                          const int64_t* __restrict__ bsum,
                                                          int64_t* __restrict__ poffd,
                                                          int64_t* __restrict__ bstart,
                                                          int64_t nbs) {
    grid_dep_sync();
    const int64_t m = *m_dev;
    if ((int64_t)blockIdx.x >= nblk_of(m)) return;
    __shared__ int64_t s_warp[kRsWarps];
    const int64_t base = (int64_t)blockIdx.x * kRsTile + (int64_t)threadIdx.x * kRsIpt;
    int32_t c[kRsIpt];
    int64_t sum = 0;
    int32_t g[kRsIpt];
#pragma unroll
    for (int r = 0; r < kRsIpt; ++r) {
        const int64_t j = base + r;
        g[r] = j < m ? order[j] : 0;
        c[r] = j < m ? tiles_touched[g[r]] : 0;
        sum += c[r];
    }
    int64_t total;
    int64_t pos = bsum[blockIdx.x] + block_exclusive_scan_256<int64_t>(sum, s_warp, &total);
#pragma unroll
    for (int r = 0; r < kRsIpt; ++r) {
        const int64_t j = base + r;
        if (j < m) {
            poffd[j] = pos;
            // the emission blocks whose first pair this Gaussian holds
            for (int64_t k = (pos + kEmitPairs - 1) / kEmitPairs;
                 k < nbs && k * kEmitPairs < pos + c[r]; ++k)
                bstart[k] = j;
            if (j == m - 1) poffd[m] = pos + c[r];
        }
        pos += c[r];
    }
}

// emit (tile, Gaussian) pairs into their depth-order places from the exact row
// spans.  Block k writes the pairs [k kEmitPairs, (k + 1) kEmitPairs) of the
// depth-ordered list: the Gaussians that hold them (from bstart, in depth order,
// kEmitThreads at a time), their tile rows spread evenly over the block's threads
// (a scan of the row counts and a search for each row's owner).  A Gaussian's
// pairs are numbered row by row, tiles left to right; a row's place in that
// numbering is the running sum of the earlier rows' span widths (a block scan per
// batch of rows), so a Gaussian split between blocks is cut at the same pair by
// both.  The block's piece is staged in shared memory and written out coalesced;
// every block gets the same number of pairs, however large or small its splats.
// The digit counts of the tile sort's passes are counted here.
constexpr int kEmitThreads = 256;
struct EmitRows {
    uint32_t okey[kEmitPairs];   // the block's piece of the pair list
    int32_t oval[kEmitPairs];
    float e[8][kEmitThreads];    // Ellipse fields, structure of arrays
    float dyv[kEmitThreads];
    int ty0[kEmitThreads];
    int off[kEmitThreads + 1];   // exclusive prefix of row counts
    int64_t pb[kEmitThreads];    // the Gaussian's first pair
    int64_t gp[kEmitThreads];    // running width sum at the Gaussian's first row
    int32_t gid[kEmitThreads];
    int wsum[kEmitThreads / 32];
    int64_t wsum64[kEmitThreads / 32];
    uint32_t hist[kMaxPasses][256];
    int diff0[257];              // pass 0 digit counts as a circular difference array
    uint32_t base0;              // + whole cycles of 256 consecutive tiles
};

// Digit counts of the tile keys [a, a + w) (consecutive tiles of one row) for
// every pass, by ranges instead of per key: pass 0 (the low byte) through the
// circular difference array, higher passes per digit the range overlaps.
__device__ __forceinline__ void count_tile_range(EmitRows& S, uint32_t a, int w, int passes) {
    atomicAdd(&S.base0, (uint32_t)(w >> 8));
    const int r = w & 255, s0 = (int)(a & 255u);
    if (r > 0) {
        atomicAdd(&S.diff0[s0], 1);
        if (s0 + r <= 256) {
            atomicSub(&S.diff0[s0 + r], 1);
        } else {
            atomicSub(&S.diff0[256], 1);
            atomicAdd(&S.diff0[0], 1);
            atomicSub(&S.diff0[s0 + r - 256], 1);
        }
    }
    const uint64_t b = (uint64_t)a + (uint64_t)w;  // one past the last key
    for (int p = 1; p < passes; ++p) {
        const int sh = 8 * p;
        const uint64_t lo = (uint64_t)a >> sh, hi = (b - 1) >> sh;
        for (uint64_t h = lo; h <= hi; ++h) {
            const uint64_t c0 = max((uint64_t)a, h << sh), c1 = min(b, (h + 1) << sh);
            atomicAdd(&S.hist[p][h & 255u], (uint32_t)(c1 - c0));
        }
    }
}

__global__ void __launch_bounds__(kEmitThreads) emit_pairs(
    CamParams cam, const float4* __restrict__ splats, const int32_t* __restrict__ order,
    const int64_t* __restrict__ poffd, const int64_t* __restrict__ bstart,
    const int64_t* __restrict__ counts, uint32_t* __restrict__ pkeys, int32_t* __restrict__ pvals,
    int passes, uint32_t* __restrict__ thist) {
    grid_dep_sync();
    __shared__ EmitRows S;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t m = counts[0], icap = counts[2];  // visible Gaussians, min(I, capacity)
    const int64_t lo = (int64_t)blockIdx.x * kEmitPairs;
    if (lo >= icap) return;
    const int64_t hi = min64(lo + kEmitPairs, icap);
#pragma unroll
    for (int p = 0; p < kMaxPasses; ++p) S.hist[p][tid] = 0;
    S.diff0[tid] = 0;
    if (tid == 0) {
        S.diff0[256] = 0;
        S.base0 = 0;
    }
    // the Gaussians holding pairs [lo, hi), kEmitThreads at a time in depth order
    for (int64_t jc = bstart[blockIdx.x];; jc += kEmitThreads) {
        const int64_t j = jc + tid;
        int nrows = 0;
        if (j < m && poffd[j] < hi) {
            const int32_t g = order[j];
            const float4 r0 = __ldg(splats + 3 * (int64_t)g), r1 = __ldg(splats + 3 * (int64_t)g + 1),
                         r2 = __ldg(splats + 3 * (int64_t)g + 2);
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
            S.pb[tid] = poffd[j];
            S.gid[tid] = g;
        }
        // block scan of the row counts
        int ri = nrows;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int rv = __shfl_up_sync(0xffffffffu, ri, o);
            if (lane >= o) ri += rv;
        }
        if (lane == 31) S.wsum[warp] = ri;
        __syncthreads();
        int rbase = 0, rtotal = 0;
#pragma unroll
        for (int w = 0; w < kEmitThreads / 32; ++w) {
            const int rv = S.wsum[w];
            rbase += w < warp ? rv : 0;
            rtotal += rv;
        }
        S.off[tid] = rbase + ri - nrows;
        if (tid == 0) S.off[kEmitThreads] = rtotal;
        __syncthreads();
        // rows in batches of kEmitThreads; carry = the span widths of earlier batches
        int64_t carry = 0;
        for (int r0 = 0; r0 < rtotal; r0 += kEmitThreads) {
            const int r = r0 + tid;
            int owner = 0, w = 0;
            uint32_t a = 0;
            if (r < rtotal) {
                int l = 0, h = kEmitThreads;  // the last owner with off[owner] <= r
                while (h - l > 1) {
                    const int mid = (l + h) >> 1;
                    if (S.off[mid] <= r) l = mid; else h = mid;
                }
                owner = l;
                const Ellipse e{S.e[0][l], S.e[1][l], S.e[2][l], S.e[3][l],
                                S.e[4][l], S.e[5][l], S.e[6][l], S.e[7][l]};
                const int ty = S.ty0[l] + (r - S.off[l]);
                int tx0, tx1;
                if (row_span(e, S.dyv[l], ty, cam.W, cam.H, cam.ntx, &tx0, &tx1)) {
                    w = tx1 - tx0;
                    a = (uint32_t)ty * (uint32_t)cam.ntx + (uint32_t)tx0;
                }
            }
            // exclusive block scan of the widths
            int x = w;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            if (lane == 31) S.wsum[warp] = x;
            __syncthreads();
            int wpre = 0, wtot = 0;
#pragma unroll
            for (int q = 0; q < kEmitThreads / 32; ++q) {
                const int v = S.wsum[q];
                wpre += q < warp ? v : 0;
                wtot += v;
            }
            const int64_t run = carry + wpre + x - w;  // width sum before this row
            if (r < rtotal && r == S.off[owner]) S.gp[owner] = run;
            __syncthreads();
            if (w > 0) {
                const int64_t pos = S.pb[owner] + (run - S.gp[owner]);  // its first pair
                const int64_t s0 = max64(pos, lo), s1 = min64(pos + w, hi);
                if (s0 < s1) {
                    const uint32_t a0 = a + (uint32_t)(s0 - pos);
                    const int32_t gid = S.gid[owner];
                    count_tile_range(S, a0, (int)(s1 - s0), passes);
                    for (int64_t q = s0; q < s1; ++q) {
                        S.okey[q - lo] = a0 + (uint32_t)(q - s0);
                        S.oval[q - lo] = gid;
                    }
                }
            }
            carry += wtot;
            __syncthreads();  // wsum and gp are rewritten by the next batch
        }
        const int64_t jn = jc + kEmitThreads;
        if (!(jn < m && poffd[jn] < hi)) break;
    }
    __syncthreads();
    for (int i = tid; i < (int)(hi - lo); i += kEmitThreads) {
        pkeys[lo + i] = S.okey[i];
        pvals[lo + i] = S.oval[i];
    }
    // pass 0: the running sum of the difference array, plus the whole cycles
    {
        int x = S.diff0[tid];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) S.wsum[warp] = x;
        __syncthreads();
        int pre = 0;
#pragma unroll
        for (int w = 0; w < kEmitThreads / 32; ++w) pre += w < warp ? S.wsum[w] : 0;
        S.hist[0][tid] = S.base0 + (uint32_t)(pre + x);
    }
    __syncthreads();
    for (int p = 0; p < passes; ++p)
        if (S.hist[p][tid]) atomicAdd(thist + p * 256 + tid, S.hist[p][tid]);
}

// tile ranges [start, end) from the sorted keys (ranges zeroed beforehand);
// none when the pair list did not fit (counts[1] > capacity)
// Each thread takes four consecutive sorted keys with one 16-byte load (the key
// buffer starts on a 16-byte boundary) and their two neighbours; the grid covers
// the capacity in a few strides, so each thread has one or two loads in flight
// rather than a long chain of dependent strides.
__global__ void __launch_bounds__(256) tile_ranges_kernel(const uint32_t* __restrict__ keys,
                                                          const int64_t* __restrict__ counts,
                                                          int64_t capacity,
                                                          int2* __restrict__ ranges) {
    grid_dep_sync();
    if (counts[1] > capacity) return;
    const int64_t n = counts[2];
    const int64_t ng = (n + 3) / 4;
    for (int64_t gi = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; gi < ng;
         gi += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i0 = 4 * gi;
        uint32_t k[4];
        if (i0 + 4 <= n) {
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(keys) + gi);
            k[0] = v.x;
            k[1] = v.y;
            k[2] = v.z;
            k[3] = v.w;
        } else {
#pragma unroll
            for (int r = 0; r < 4; ++r) k[r] = i0 + r < n ? keys[i0 + r] : 0u;
        }
        const uint32_t prev = i0 > 0 ? keys[i0 - 1] : 0u;
        const uint32_t next = i0 + 4 < n ? keys[i0 + 4] : 0u;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int64_t i = i0 + r;
            if (i >= n) break;
            const bool first = i == 0 || (r == 0 ? prev : k[r - 1]) != k[r];
            const bool last = i == n - 1 || (r == 3 ? next : k[r + 1]) != k[r];
            if (first) ranges[k[r]].x = (int)i;
            if (last) ranges[k[r]].y = (int)(i + 1);
        }
    }
}

// empty tiles get [p, p) with p the end of the last non-empty tile before them
// (so that starts are the exclusive prefix sum of the counts); one block
__global__ void __launch_bounds__(kScanThreads) fill_empty_ranges(int2* __restrict__ ranges,
                                                                  int64_t nt,
                                                                  const int64_t* __restrict__ counts,
                                                                  int64_t* __restrict__ counts_out) {
    grid_dep_sync();
    if (threadIdx.x == 0 && counts_out) {
        counts_out[0] = counts[0];
        counts_out[1] = counts[1];
    }
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


size_t align_up(size_t x) { return (x + 255) & ~size_t(255); }

int bits_for(int64_t v) {
    int b = 0;
    while (b < 62 && (int64_t(1) << b) <= v) ++b;
    return std::max(b, 1);
}


}  // namespace

RadixBinLayout radix_bin_layout(int64_t n, int64_t capacity, int64_t n_tiles) {
    RadixBinLayout L{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t o = off;
        off = align_up(off + bytes);
        return o;
    };
    const int64_t nn = std::max<int64_t>(n, 1), cap = std::max<int64_t>(capacity, 1);
    const int64_t nt = std::max<int64_t>(n_tiles, 1);
    L.off_counts = take(8 * sizeof(int64_t) + 2 * kMaxPasses * 256 * sizeof(uint32_t));
    L.off_bsum = take((size_t)(nblk_of(nn) + 1) * sizeof(int64_t));
    L.off_dkeys0 = take((size_t)nn * 4);
    L.off_dkeys1 = take((size_t)nn * 4);
    L.off_dvals0 = take((size_t)nn * 4);
    L.off_dvals1 = take((size_t)nn * 4);
    L.off_poff = take((size_t)(nn + 1) * sizeof(int64_t));
    L.off_bstart = take((size_t)((cap + kEmitPairs - 1) / kEmitPairs + 1) * sizeof(int64_t));
    L.off_pkeys0 = take((size_t)cap * 4);
    L.off_pkeys1 = take((size_t)cap * 4);
    L.off_pvals0 = take((size_t)cap * 4);
    L.off_pvals1 = take((size_t)cap * 4);
    L.off_hist = take(rs_ctl_bytes(std::max(nn, cap)));
    L.off_lruns = take(lpt_runs_bytes(nt));
    L.total = off;
    return L;
}

cudaError_t run_bin_sort_radix(const CamParams& cam, int64_t n, const float* splats,
                               const float* depths, const int32_t* tiles_touched, char* ws,
                               const RadixBinLayout& L, int32_t* sorted_ids, int64_t capacity,
                               int32_t* tile_ranges, int32_t* lpt_order, int64_t* counts_out,
                               cudaStream_t st) {
    auto* counts = reinterpret_cast<int64_t*>(ws + L.off_counts);
    auto* bsum = reinterpret_cast<int64_t*>(ws + L.off_bsum);
    auto* dk0 = reinterpret_cast<uint32_t*>(ws + L.off_dkeys0);
    auto* dk1 = reinterpret_cast<uint32_t*>(ws + L.off_dkeys1);
    auto* dv0 = reinterpret_cast<int32_t*>(ws + L.off_dvals0);
    auto* dv1 = reinterpret_cast<int32_t*>(ws + L.off_dvals1);
    auto* poff = reinterpret_cast<int64_t*>(ws + L.off_poff);
    auto* bstart = reinterpret_cast<int64_t*>(ws + L.off_bstart);
    const int64_t nbs = (capacity + kEmitPairs - 1) / kEmitPairs;  // emission blocks
    auto* pk0 = reinterpret_cast<uint32_t*>(ws + L.off_pkeys0);
    auto* pk1 = reinterpret_cast<uint32_t*>(ws + L.off_pkeys1);
    auto* pv0 = reinterpret_cast<int32_t*>(ws + L.off_pvals0);
    auto* pv1 = reinterpret_cast<int32_t*>(ws + L.off_pvals1);
    char* rs_ctl = ws + L.off_hist;
    auto* sort_err = reinterpret_cast<unsigned long long*>(counts + kRadixErrWord);
    auto* lruns = reinterpret_cast<uint64_t*>(ws + L.off_lruns);
    const int64_t nt = (int64_t)cam.ntx * cam.nty;
    auto* ranges = reinterpret_cast<int2*>(tile_ranges);
    cudaError_t err;

    // counts, then the digit counts of the depth sort and of the tile sort
    auto* dhist = reinterpret_cast<uint32_t*>(counts + 8);
    auto* thist = dhist + kMaxPasses * 256;
    err = cudaMemsetAsync(counts, 0, 8 * sizeof(int64_t) + 2 * kMaxPasses * 256 * sizeof(uint32_t),
                          st);
    if (err != cudaSuccess) return err;
    err = cudaMemsetAsync(tile_ranges, 0, (size_t)nt * 2 * sizeof(int32_t), st);
    if (err != cudaSuccess) return err;

    if (n > 0) {
        const unsigned nb = (unsigned)nblk_of(n);
        // 1. compact the visible Gaussians (id order) into (depth key, id)
        err = launch(vis_count, nb, kRsBlock, 0, st, tiles_touched, n, bsum);
        if (err != cudaSuccess) return err;
        err = launch(scan_block_sums, 1, kScanThreads, 0, st, bsum, (const int64_t*)nullptr, n,
                     counts + 0, (int64_t)0, (int64_t*)nullptr);
        if (err != cudaSuccess) return err;
        err = launch(vis_write, nb, kRsBlock, 0, st, tiles_touched, depths, n, (const int64_t*)bsum,
                     dk0, dv0, dhist);
        if (err != cudaSuccess) return err;
        // 2. stable depth sort of the M visible (31 significant key bits)
        uint32_t* dks = nullptr;
        int32_t* dvs = nullptr;
        err = radix_sort(dk0, dv0, dk1, dv1, nullptr, counts + 0, 0, n, 31, rs_ctl, dhist, sort_err,
                         st, &dks, &dvs);
        if (err != cudaSuccess) return err;
        // 3. pair offsets in depth order, I = total, min(I, capacity)
        err = launch(pairs_count, nb, kRsBlock, 0, st, (const int32_t*)dvs, tiles_touched,
                     (const int64_t*)(counts + 0), bsum);
        if (err != cudaSuccess) return err;
        err = launch(scan_block_sums, 1, kScanThreads, 0, st, bsum, (const int64_t*)(counts + 0),
                     (int64_t)0, counts + 1, capacity, counts + 2);
        if (err != cudaSuccess) return err;
        err = launch(pairs_offsets, nb, kRsBlock, 0, st, (const int32_t*)dvs, tiles_touched,
                     (const int64_t*)(counts + 0), (const int64_t*)bsum, poff, bstart, nbs);
        if (err != cudaSuccess) return err;
        // 4. emit pairs in depth order
        const int tbits = bits_for(nt - 1);
        err = launch(emit_pairs, (unsigned)std::max<int64_t>(1, nbs), kEmitThreads, 0, st, cam,
                     reinterpret_cast<const float4*>(splats), (const int32_t*)dvs,
                     (const int64_t*)poff, (const int64_t*)bstart, (const int64_t*)counts, pk0,
                     pv0, (tbits + 7) / 8, thist);
        if (err != cudaSuccess) return err;
        // 5. stable sort by tile key; values land in sorted_ids
        uint32_t* pks = nullptr;
        err = radix_sort(pk0, pv0, pk1, pv1, sorted_ids, counts + 2, 0, capacity, tbits, rs_ctl,
                         thist, sort_err, st, &pks, nullptr);
        if (err != cudaSuccess) return err;
        // 6. tile ranges
        int dev = 0, sms = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        const unsigned rg = (unsigned)std::max<int64_t>(
            1, std::min<int64_t>((capacity + 1023) / 1024, 64 * (int64_t)std::max(sms, 1)));
        err = launch(tile_ranges_kernel, rg, 256, 0, st, (const uint32_t*)pks,
                     (const int64_t*)counts, capacity, ranges);
        if (err != cudaSuccess) return err;
    }
    err = launch(fill_empty_ranges, 1, kScanThreads, 0, st, ranges, nt, (const int64_t*)counts,
                 counts_out);
    if (err != cudaSuccess) return err;
    // 7. LPT order: tiles by descending count, ties by tile id
    return launch_lpt(ranges, nt, lruns, lpt_order, st);
}

}  // namespace gs

// ---------------------------------------------------------------------------
// Test hook (not part of the C ABI in gs.h): makes the look-back's bounded wait
// run out with the unmodified one-sweep kernel.  One pass over n keys (n >
// 4096, so that there are at least two 4096-key tiles) runs with the pass's
// ticket counter set to 1 before the launch: the block that draws ticket 1
// waits on tile 0's published counts, which no block writes, gives up after
// its poll limit and sets the give-up flag; every access stays inside the
// buffers.  ws must hold gs_test_lookback_timeout_ws_bytes(n) bytes; keys_out
// and vals_out receive meaningless values.  Returns GS_ERR_TIMEOUT when the
// flag was set (the status gs_bin_sort returns then), GS_OK if not.
// ---------------------------------------------------------------------------
namespace {
size_t lookback_test_ws_layout(int64_t n, size_t* off_ghist, size_t* off_err) {
    const size_t ctl = gs::rs_ctl_bytes(n);
    *off_ghist = (ctl + 255) & ~size_t(255);
    *off_err = *off_ghist + 4 * 256 * sizeof(uint32_t);
    return *off_err + 256;
}
}  // namespace

extern "C" size_t gs_test_lookback_timeout_ws_bytes(int64_t n) {
    size_t a, b;
    return n > 0 ? lookback_test_ws_layout(n, &a, &b) : 0;
}

extern "C" gs_status gs_test_lookback_timeout(const uint32_t* keys_in, const int32_t* vals_in,
                                              uint32_t* keys_out, int32_t* vals_out, int64_t n,
                                              void* ws, size_t ws_bytes, void* stream) {
    using namespace gs;
    if (!keys_in || !vals_in || !keys_out || !vals_out || !ws || n <= kRsTile || n > (1 << 24))
        return GS_ERR_INVALID_ARG;
    size_t off_ghist, off_err;
    if (ws_bytes < lookback_test_ws_layout(n, &off_ghist, &off_err)) return GS_ERR_WORKSPACE;
    cudaStream_t st = (cudaStream_t)stream;
    char* w = static_cast<char*>(ws);
    if (cudaMemsetAsync(w, 0, ws_bytes, st) != cudaSuccess) return GS_ERR_CUDA;
    // ticket counter of pass 0 (the first int of the control region) := 1
    if (cudaMemsetAsync(w, 1, 1, st) != cudaSuccess) return GS_ERR_CUDA;
    int* tickets = reinterpret_cast<int*>(w);
    uint64_t* lookback = reinterpret_cast<uint64_t*>(w + 16 + kMaxPasses * 256 * 4);
    auto* ghist = reinterpret_cast<const uint32_t*>(w + off_ghist);
    auto* err = reinterpret_cast<unsigned long long*>(w + off_err);
    const unsigned grid = (unsigned)nblk_of(n);
    if (launch(rs_onesweep<8>, grid, kRsBlock, 0, st, keys_in, vals_in, keys_out, vals_out,
               (const int64_t*)nullptr, n, 0, ghist, tickets, lookback, err) != cudaSuccess)
        return GS_ERR_CUDA;
    unsigned long long flag = 0;
    if (cudaMemcpyAsync(&flag, err, sizeof(flag), cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return GS_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return GS_ERR_CUDA;
    return flag ? GS_ERR_TIMEOUT : GS_OK;
}
