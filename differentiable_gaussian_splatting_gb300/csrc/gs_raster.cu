// gs_raster.cu -- per-tile alpha blending (forward) and its gradient (backward).
//
// Forward ("Mitigating SM-Level Load Imbalance in 3D Gaussian Splatting on
// GPUs", Ryu & Yoo): Eq. 2-3 per pixel; Sec. 4.1 a persistent kernel of K
// resident CTAs takes work from a queue in LPT order (one atomicAdd per fetch);
// Sec. 4.2 the heaviest tiles are split into k depth-contiguous chunks that
// blend from unit transmittance, signal saturation through a per-tile
// atomicMin flag that later chunks check once per 256-splat batch, and are
// composed with Eq. 5; Sec. 4.3-4.4 the per-frame policy of Eq. 6 picks how
// many tiles to split and how deeply.  Chunk items and whole-tile items share
// one queue (heavy chunks first), which is the fused form of the selective
// chunking; the CTA that finishes a split tile's last chunk composes it.
// Composition replays, for a pixel, the chunk in which the sequential blend
// would stop, so the result equals the sequential definition.
//
// Per tile ("What the 3DGS Literature Left on the Table", Kopanas): 256
// threads, 8 warps of 8x4 pixels; batches of 256 splat records (three float4
// each) are staged in shared memory with an 8-bit sub-tile mask per splat;
// each warp walks the splats of its sub-tile with __ballot_sync / __ffs (Step
// 1 (c)); misses are predicated to alpha = 0 (Step 5); the quadratic is
// evaluated with round-to-nearest operations so forward and backward agree
// bit for bit on every hit (Step 5); opacity is folded into the base-2
// exponent (Step 6.3).
//
// Backward (Kopanas, Step 1 (a), Step 2): back to front from each pixel's
// last blended splat, T recovered by division by (1 - alpha); the nine
// per-splat derivatives of a warp are summed by a halving reduce-scatter of
// 12 shuffles, after which nine lanes add them atomically.
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <mutex>

#include "gs_device.cuh"
#include "gs_internal.h"

namespace gs {

namespace {

constexpr int kThreads = 256;
constexpr int kBatch = 256;
constexpr int kPolicyThreads = 1024;

struct RasterArgs {
    int W, H, ntx, nty;
    const float4* splats;
    const int32_t* ids;
    const int2* ranges;
    const int32_t* lpt;
    int* ctrl;
    int* sat;
    int* done;
    int* cbatch;
    float4* part_c;
    int2* part_n;
    float4* bstate;
    uint8_t* cmask;  // per pair: warps that blended it (forward writes, backward reads)
    // forward outputs
    float* image;
    float* t_final;
    int32_t* n_contrib;
    int32_t* last_idx;
    // backward inputs / outputs
    const float* t_final_in;
    const int32_t* last_in;
    const float* dimg;
    const float* dT;
    float* grad2d;
    uint8_t* touched;
};

__device__ __forceinline__ int64_t chunk_lo(int64_t s, int64_t len, int p, int k) {
    return s + (len * p) / k;
}

// pixel of thread tid inside its tile: warp w covers the 8x4 sub-tile
// (8 (w & 1), 4 (w >> 1)); lane l is pixel (l & 7, l >> 3) of it
__device__ __forceinline__ void tile_pixel(int tid, int* lx, int* ly) {
    const int w = tid >> 5, l = tid & 31;
    *lx = ((w & 1) << 3) + (l & 7);
    *ly = ((w >> 1) << 2) + (l >> 3);
}

struct WorkItem {
    int tile;
    int slot;   // split-tile index (0..h-1), -1 for a whole tile
    int chunk;  // chunk index p
    int k;
    int64_t s, e;
};

__device__ __forceinline__ WorkItem decode_item(const RasterArgs& A, int item, int h, int k) {
    WorkItem it;
    if (item < h * k) {
        it.slot = item / k;
        it.chunk = item - it.slot * k;
        it.k = k;
        it.tile = A.lpt[it.slot];
        const int2 r = A.ranges[it.tile];
        const int64_t len = (int64_t)r.y - r.x;
        it.s = chunk_lo(r.x, len, it.chunk, k);
        it.e = chunk_lo(r.x, len, it.chunk + 1, k);
    } else {
        it.slot = -1;
        it.chunk = 0;
        it.k = 1;
        it.tile = A.lpt[h + (item - h * k)];
        const int2 r = A.ranges[it.tile];
        it.s = r.x;
        it.e = r.y;
    }
    return it;
}

struct PixelState {
    float T, cr, cg, cb;
    int n, last;
    bool done;
};

struct Smem {
    float4 r0[kBatch];
    float4 r1[kBatch];
    float4 r2[kBatch];
    uint8_t mask[kBatch];
    uint32_t cm[8 * (kBatch / 32)];  // [warp][32-splat chunk] blended bits
    int item;
    int flag;
};

// Batches of one blend_range call (block-uniform): blended, and left unread
// because an earlier chunk saturated the tile or because every pixel had stopped.
struct BatchCount {
    int blended, skip_flag, skip_done;
};

// Front-to-back blend of list positions [s, e) for the calling thread's pixel.
// All threads of the CTA must call it.  When sat_slot >= 0 the chunk stops
// early once sat[sat_slot] < chunk (an earlier chunk saturated the tile).
// With write_cmask, every position's 8-bit mask of the warps that blended it
// is stored in A.cmask ("What the 3DGS Literature Left on the Table", Step 4.2).
// Returns true if it stopped on the saturation signal.
__device__ __forceinline__ bool blend_range(const RasterArgs& A, Smem& S, int tx, int ty, float px, float py,
                            int64_t s, int64_t e, PixelState& st, int sat_slot, int chunk,
                            bool write_cmask, BatchCount& bc) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    bc = BatchCount{0, 0, 0};
    // A pixel blends while its running T is at least 1e-4 (T only falls, so that is
    // the stop rule); a pixel that takes no part (outside the image, already
    // stopped, or not being replayed) runs with T = 0 and gets its T back at the end.
    const bool frozen = st.done;
    float T = frozen ? 0.f : st.T;
    bool on_flag = false;
    for (int64_t bs = s; bs < e; bs += kBatch) {
        if (tid == 0)
            S.flag = (sat_slot >= 0 && chunk > 0) ? (*(volatile int*)(A.sat + sat_slot) < chunk) : 0;
        const int live = __syncthreads_or(T >= kTMin);
        const int left = (int)((e - bs + kBatch - 1) / kBatch);
        if (!live) {
            bc.skip_done = left;
            break;
        }
        if (S.flag) {
            bc.skip_flag = left;
            on_flag = true;
            break;
        }
        ++bc.blended;
        const int64_t j = bs + tid;
        if (tid < 8 * (kBatch / 32)) S.cm[tid] = 0u;
        if (j < e) {
            const int32_t g = __ldg(A.ids + j);
            const float4 r0 = __ldg(A.splats + 3 * (int64_t)g);
            const float4 r1 = __ldg(A.splats + 3 * (int64_t)g + 1);
            const float4 r2 = __ldg(A.splats + 3 * (int64_t)g + 2);
            S.r0[tid] = r0;
            S.r1[tid] = r1;
            S.r2[tid] = r2;
            S.mask[tid] = (uint8_t)subtile_mask(ellipse_of(r0, r1, r2), tx, ty, A.W, A.H);
        } else {
            S.mask[tid] = 0;
        }
        __syncthreads();
        const int nb = (int)min64(kBatch, e - bs);
        const int pos0 = (int)bs;  // list positions fit in 32 bits (capacity < 2^31)
        for (int c = 0; c < nb; c += 32) {
            if (__ballot_sync(0xffffffffu, T >= kTMin) == 0) break;
            const int jj = c + lane;
            const uint32_t bit = jj < nb ? (S.mask[jj] >> warp) & 1u : 0u;
            uint32_t work = __ballot_sync(0xffffffffu, bit);
            uint32_t blended = 0u;  // this lane's blended splats of the chunk
            while (work) {
                const int q = __ffs(work) - 1;
                work &= work - 1;
                const int idx = c + q;
                const float4 r0 = S.r0[idx], r1 = S.r1[idx], r2 = S.r2[idx];
                const float dx = rsub(px, r0.x), dy = rsub(py, r0.y);
                float u1, u2;
                const float qv = quad_q(r0.z, r0.w, r1.x, dx, dy, &u1, &u2);
                const bool hit = (qv <= r1.y) && (T >= kTMin);
                float alpha = fminf(ex2_approx(fmaf(qv, kNegHalfLog2e, r1.z)), kAlphaMax);
                alpha = hit ? alpha : 0.f;
                const float w = alpha * T;
                st.cr = fmaf(w, r2.x, st.cr);
                st.cg = fmaf(w, r2.y, st.cg);
                st.cb = fmaf(w, r2.z, st.cb);
                T = T - w;  // T (1 - alpha), as one subtraction of the blend weight
                // branch-free bookkeeping (no reconvergence point in the loop)
                blended |= (hit ? 1u : 0u) << q;
            }
            // the chunk's hits, in order: their count, and the last one
            st.n += __popc(blended);
            st.last = blended ? pos0 + c + 31 - __clz(blended) : st.last;
            if (write_cmask) {
                blended = __reduce_or_sync(0xffffffffu, blended);
                if (lane == 0) S.cm[warp * (kBatch / 32) + (c >> 5)] = blended;
            }
        }
        __syncthreads();
        if (write_cmask && j < e) {
            uint32_t m = 0;
#pragma unroll
            for (int w = 0; w < 8; ++w) m |= ((S.cm[w * (kBatch / 32) + (tid >> 5)] >> lane) & 1u) << w;
            A.cmask[j] = (uint8_t)m;
        }
    }
    if (!frozen) {
        st.T = T;
        st.done = T < kTMin;
    }
    return on_flag;
}

// ---------------------------------------------------------------------------
// per-frame chunking policy (Ryu & Yoo, Eq. 6), one cluster of kPolicyCluster
// blocks: every block sums the tile counts, block r evaluates the candidates
// c = r mod kPolicyCluster (the float64 arithmetic spread over as many SMs),
// and block 0 takes the least of the blocks' best through distributed shared
// memory and writes the choice
// ---------------------------------------------------------------------------
constexpr int kPolicyCluster = 8;

__device__ __forceinline__ bool key_less(uint64_t ca, int ia, uint64_t cb, int ib) {
    return ca < cb || (ca == cb && ia < ib);
}

__global__ void __launch_bounds__(kPolicyThreads) policy_kernel(const int32_t* __restrict__ lpt,
                                                                const int2* __restrict__ ranges,
                                                                int nt, int K, RasterConfig cfg,
                                                                int* ctrl, int* sat, int* done) {
    grid_dep_sync();
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    __shared__ long long s_tot[kPolicyThreads / 32];
    __shared__ uint64_t s_best;  // this block's least (cost, candidate)
    __shared__ int s_best_cand;
    __shared__ uint64_t s_cost[kPolicyThreads / 32];
    __shared__ int s_cand[kPolicyThreads / 32];
    __shared__ int s_hk[2];
    __shared__ int s_nz[kPolicyThreads / 32], s_nmin[kPolicyThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    auto count_at = [&](int j) -> double {
        if (j >= nt) return 0.0;
        const int2 r = ranges[lpt[j]];
        return (double)(r.y - r.x);
    };
    // the loads that do not depend on N_total are issued before its reduction:
    // N_1 and N_{h+1} of this thread's first candidate
    const int hm = cfg.split_mode == 0 ? min(nt, cfg.h_max) : 0;
    const double N1 = count_at(0);
    const int cand0 = rank + kPolicyCluster * tid;
    const double n_first = cand0 < hm * 4 ? count_at(1 + (cand0 >> 2)) : 0.0;
    // N_total: an integer sum (exactly the double sum of the counts, all below 2^53);
    // beside it the lightest non-empty tile and the number of non-empty tiles
    long long part = 0;
    int nz = 0, nmin = INT_MAX;
    for (int t = tid; t < nt; t += kPolicyThreads) {
        const int2 r = ranges[t];
        const int c = r.y - r.x;
        part += (long long)c;
        if (c > 0) {
            ++nz;
            nmin = min(nmin, c);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        part += __shfl_xor_sync(0xffffffffu, part, o);
        nz += __shfl_xor_sync(0xffffffffu, nz, o);
        nmin = min(nmin, __shfl_xor_sync(0xffffffffu, nmin, o));
    }
    if (lane == 0) {
        s_tot[warp] = part;
        s_nz[warp] = nz;
        s_nmin[warp] = nmin;
    }
    __syncthreads();
    long long itot = 0;
    int inz = 0, imin = INT_MAX;
#pragma unroll
    for (int w = 0; w < kPolicyThreads / 32; ++w) {
        itot += s_tot[w];
        inz += s_nz[w];
        imin = min(imin, s_nmin[w]);
    }
    const double tot = (double)itot;
    // Eq. 6 multiplied by K > 0 (same minimiser, no division), in round-to-nearest
    // double with no contraction: K T(h, k) = max(N_total + lambda h k, K l) + beta K l,
    // l = max(N_1 / k, N_{h+1}); N_1 / k is an exact scaling by a power of two
    const double lam = cfg.lambda, beta = cfg.beta, Kd = (double)K;
    const double KN1 = __dmul_rn(Kd, N1);
    const double base = __dadd_rn(fmax(tot, KN1), __dmul_rn(beta, KN1));
    int bh = 0, bk = 1;
    if (cfg.split_mode == 2) {
        bh = min(min(cfg.force_h, cfg.h_max), nt);
        bk = bh > 0 ? cfg.force_k : 1;
    } else if (cfg.split_mode == 0) {
        // candidate c = 4 (h - 1) + i, k = 2^(i + 1): increasing c is increasing (h, k), so
        // the lexicographic minimum of (cost, h, k) is that of (cost, c).  Costs are
        // non-negative, so their bit patterns order as unsigned integers.
        uint64_t best = ~0ull;
        int cand_best = INT_MAX;
        for (int cand = cand0; cand < hm * 4; cand += kPolicyCluster * kPolicyThreads) {
            const int h = 1 + (cand >> 2);
            const int k = 2 << (cand & 3);
            // 1 / k = 2^-((cand & 3) + 1), built from its exponent bits (exact, no division)
            const double inv_k = __longlong_as_double((long long)(1022 - (cand & 3)) << 52);
            const double l = fmax(__dmul_rn(N1, inv_k), cand == cand0 ? n_first : count_at(h));
            const double Kl = __dmul_rn(Kd, l);
            const double work = __dadd_rn(tot, __dmul_rn(__dmul_rn(lam, (double)h), (double)k));
            const double cost = __dadd_rn(fmax(work, Kl), __dmul_rn(beta, Kl));
            const uint64_t cb = (uint64_t)__double_as_longlong(cost);
            if (key_less(cb, cand, best, cand_best)) {
                best = cb;
                cand_best = cand;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const uint64_t oc = __shfl_xor_sync(0xffffffffu, best, o);
            const int oi = __shfl_xor_sync(0xffffffffu, cand_best, o);
            if (key_less(oc, oi, best, cand_best)) {
                best = oc;
                cand_best = oi;
            }
        }
        if (lane == 0) {
            s_cost[warp] = best;
            s_cand[warp] = cand_best;
        }
        __syncthreads();
        if (warp == 0) {
            best = s_cost[lane];
            cand_best = s_cand[lane];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const uint64_t oc = __shfl_xor_sync(0xffffffffu, best, o);
                const int oi = __shfl_xor_sync(0xffffffffu, cand_best, o);
                if (key_less(oc, oi, best, cand_best)) {
                    best = oc;
                    cand_best = oi;
                }
            }
            if (lane == 0) {
                s_best = best;
                s_best_cand = cand_best;
            }
        }
        cluster.sync();
        if (rank == 0 && warp == 0) {
            best = ~0ull;
            cand_best = INT_MAX;
            if (lane < kPolicyCluster) {
                best = *cluster.map_shared_rank(&s_best, lane);
                cand_best = *cluster.map_shared_rank(&s_best_cand, lane);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const uint64_t oc = __shfl_xor_sync(0xffffffffu, best, o);
                const int oi = __shfl_xor_sync(0xffffffffu, cand_best, o);
                if (key_less(oc, oi, best, cand_best)) {
                    best = oc;
                    cand_best = oi;
                }
            }
            if (lane == 0) {
                int h_best = 0, k_best = 1;
                // a split must cost strictly less than no split (h = 0 wins ties) ...
                const double bc = __longlong_as_double((long long)best);
                if (cand_best != INT_MAX && bc < base) {
                    h_best = 1 + (cand_best >> 2);
                    k_best = 2 << (cand_best & 3);
                    // ... and save at least eps of it
                    if (!(bc <= __dmul_rn(__dsub_rn(1.0, (double)cfg.eps), base))) {
                        h_best = 0;
                        k_best = 1;
                    }
                }
                s_hk[0] = h_best;
                s_hk[1] = k_best;
            }
        }
        // the other blocks' shared memory stays readable until block 0 has read it
        cluster.sync();
        __syncthreads();
        bh = s_hk[0];
        bk = s_hk[1];
    }
    if (rank != 0) return;
    for (int j = tid; j < bh; j += kPolicyThreads) {
        sat[j] = INT_MAX;
        done[j] = 0;
    }
    if (tid == 0) {
        ctrl[kCtlH] = bh;
        ctrl[kCtlK] = bk;
        ctrl[kCtlItems] = bh * bk + (nt - bh);
        ctrl[kCtlResident] = K;
        ctrl[kCtlQueueFwd] = 0;
        ctrl[kCtlQueueBwd] = 0;
        ctrl[kCtlError] = 0;
        ctrl[kCtlNMax] = (int)N1;
        ctrl[kCtlNMinNz] = inz > 0 ? imin : 0;
        ctrl[kCtlNTotal] = (int)itot;  // pair counts stay below 2^31
        ctrl[kCtlNonEmpty] = inz;
        for (int w = kCtlBatchTile; w <= kCtlDiscard; ++w) ctrl[w] = 0;
    }
}

// ---------------------------------------------------------------------------
// forward: persistent kernel over whole tiles and depth chunks
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 5) raster_fwd_kernel(RasterArgs A) {
    grid_dep_sync();
    __shared__ Smem S;
    const int tid = threadIdx.x;
    const int h = A.ctrl[kCtlH], k = A.ctrl[kCtlK], nitems = A.ctrl[kCtlItems];
    int lx, ly;
    tile_pixel(tid, &lx, &ly);
    while (true) {
        if (tid == 0) S.item = atomicAdd(A.ctrl + kCtlQueueFwd, 1);
        __syncthreads();
        const int item = S.item;
        __syncthreads();
        if (item >= nitems) break;
        const WorkItem it = decode_item(A, item, h, k);
        const int tx = it.tile % A.ntx, ty = it.tile / A.ntx;
        const int x = tx * kTile + lx, y = ty * kTile + ly;
        const bool inside = x < A.W && y < A.H;
        const float px = (float)x + 0.5f, py = (float)y + 0.5f;
        PixelState st{1.f, 0.f, 0.f, 0.f, 0, -1, !inside};
        BatchCount bc;
        if (it.slot < 0) {
            blend_range(A, S, tx, ty, px, py, it.s, it.e, st, -1, 0, true, bc);
            if (tid == 0) atomicAdd(A.ctrl + kCtlBatchTile, bc.blended);
            if (inside) {
                const int64_t p = (int64_t)y * A.W + x;
                A.image[3 * p] = st.cr;
                A.image[3 * p + 1] = st.cg;
                A.image[3 * p + 2] = st.cb;
                A.t_final[p] = st.T;
                A.n_contrib[p] = st.n;
                A.last_idx[p] = st.last;
            }
            continue;
        }
        // ---- a depth chunk of a split tile: blend from T = 1 ----
        blend_range(A, S, tx, ty, px, py, it.s, it.e, st, it.slot, it.chunk, true, bc);
        if (tid == 0) {
            A.cbatch[it.slot * kMaxChunks + it.chunk] = bc.blended;
            atomicAdd(A.ctrl + kCtlBatchChunk, bc.blended);
            atomicAdd(A.ctrl + kCtlSkipFlag, bc.skip_flag);
            atomicAdd(A.ctrl + kCtlSkipDone, bc.skip_done);
        }
        const int64_t pidx = ((int64_t)it.slot * kMaxChunks + it.chunk) * kThreads + tid;
        A.part_c[pidx] = make_float4(st.cr, st.cg, st.cb, st.T);
        A.part_n[pidx] = make_int2(st.n, st.last);
        const int saturated = __syncthreads_and(st.done);
        if (tid == 0 && saturated) atomicMin(A.sat + it.slot, it.chunk);
        __threadfence();
        __syncthreads();
        if (tid == 0) S.flag = (atomicAdd(A.done + it.slot, 1) == it.k - 1);
        __syncthreads();
        if (!S.flag) continue;
        __threadfence();
        // ---- last chunk of this tile to finish: compose the chunks (Eq. 5) ----
        PixelState acc{1.f, 0.f, 0.f, 0.f, 0, -1, !inside};
        const int2 rr = A.ranges[it.tile];
        const int64_t len = (int64_t)rr.y - rr.x;
        int discard = 0;
        for (int p = 0; p < it.k; ++p) {
            const int64_t slotp = ((int64_t)it.slot * kMaxChunks + p) * kThreads + tid;
            // every pixel stopped before chunk p: its blended batches were wasted
            if (__syncthreads_and(acc.done)) discard += __ldcg(A.cbatch + it.slot * kMaxChunks + p);
            const float Tb = acc.T;
            const float cr0 = acc.cr, cg0 = acc.cg, cb0 = acc.cb;
            bool replay = false;
            if (!acc.done) {
                const float4 pc = __ldcg(A.part_c + slotp);
                const int2 pn = __ldcg(A.part_n + slotp);
                const float Tn = acc.T * pc.w;
                if (pc.w >= kTMin && Tn >= kTMin) {
                    // no stop can fall inside the chunk: T is monotone
                    acc.cr = fmaf(acc.T, pc.x, acc.cr);
                    acc.cg = fmaf(acc.T, pc.y, acc.cg);
                    acc.cb = fmaf(acc.T, pc.z, acc.cb);
                    acc.T = Tn;
                    acc.n += pn.x;
                    if (pn.x > 0) acc.last = pn.y;
                } else {
                    replay = true;
                }
            }
            if (__syncthreads_or(replay)) {
                // replay chunk p sequentially from the running state for the
                // pixels whose stop lies in it
                PixelState rs = acc;
                rs.done = !replay;
                BatchCount rc;
                blend_range(A, S, tx, ty, px, py, chunk_lo(rr.x, len, p, it.k),
                            chunk_lo(rr.x, len, p + 1, it.k), rs, -1, 0, false, rc);
                if (replay) {
                    acc = rs;
                    acc.done = rs.T < kTMin;
                }
            }
            // state for the backward of chunk p: T after the chunk, colour it added
            A.bstate[slotp] = make_float4(acc.T, acc.cr - cr0, acc.cg - cg0, acc.cb - cb0);
            (void)Tb;
        }
        if (tid == 0 && discard) atomicAdd(A.ctrl + kCtlDiscard, discard);
        // colour added by chunks q > p ("colour behind" chunk p)
        {
            float br = 0.f, bg = 0.f, bb = 0.f;
            for (int p = it.k - 1; p >= 0; --p) {
                const int64_t slotp = ((int64_t)it.slot * kMaxChunks + p) * kThreads + tid;
                float4 v = A.bstate[slotp];
                const float ir = v.y, ig = v.z, ib = v.w;
                A.bstate[slotp] = make_float4(v.x, br, bg, bb);
                br += ir;
                bg += ig;
                bb += ib;
            }
        }
        if (inside) {
            const int64_t p = (int64_t)y * A.W + x;
            A.image[3 * p] = acc.cr;
            A.image[3 * p + 1] = acc.cg;
            A.image[3 * p + 2] = acc.cb;
            A.t_final[p] = acc.T;
            A.n_contrib[p] = acc.n;
            A.last_idx[p] = acc.last;
        }
    }
}

// ---------------------------------------------------------------------------
// backward
// ---------------------------------------------------------------------------
// Two splats' column moments summed over the warp ("What the 3DGS Literature
// Left on the Table", Step 2 and Step 6.4).  Every lane holds, per splat, six
// values of its two pixels: the log-alpha derivative sums m = g0 + g1,
// sy = g0 dy0 + g1 dy1, syy = g0 dy0^2 + g1 dy1^2 and the colour terms
// w0 G0 + w1 G1 (r, g, b).  Lanes l, l ^ 8, l ^ 16, l ^ 24 share a pixel
// column, hence dx:
//   xor 16  lanes 0-15 keep splat a, lanes 16-31 splat b (6 shuffles);
//   xor 8   each column's four lanes summed; geometry (m, sy, syy) stays on
//           the lanes with bit 3 clear, colour on the others (3 shuffles);
//           the geometry lanes form the column's dx-weighted terms once per
//           column instead of per pixel: dx^2 m, dx sy and, with the splat's
//           conic factor, the mean derivatives l11 s and l12 s + l22^2 sy,
//           s = l11 dx m + l12 sy the column's sum of g u1;
//   xor 4, 2, 1  the columns summed (3 + 2 + 1 shuffles).
// Afterwards lane l holds, for the splat of its half, the quantity
// moment_of_lane(l & 15).  15 shuffles for two splats.
__device__ __forceinline__ float reduce_moments2(const float a[6], const float b[6], float dxa,
                                                 float dxb, float l11, float l12, float l22,
                                                 int lane) {
    const unsigned F = 0xffffffffu;
    const bool lo16 = !(lane & 16);
    float k[6];
#pragma unroll
    for (int i = 0; i < 6; ++i) {
        const float r = __shfl_xor_sync(F, lo16 ? b[i] : a[i], 16);
        k[i] = (lo16 ? a[i] : b[i]) + r;
    }
    const bool lo8 = !(lane & 8);
    float v[6];
#pragma unroll
    for (int i = 0; i < 3; ++i) {
        const float r = __shfl_xor_sync(F, lo8 ? k[3 + i] : k[i], 8);
        v[i] = (lo8 ? k[i] : k[3 + i]) + r;
    }
    // geometry lanes: (m, d/dmuy, syy, d/dmux, dx^2 m, dx sy) of the column, with
    // sum g u1 = l11 dx m + l12 sy (u1 = l11 dx + l12 dy); colour lanes: (r, g, b, unused)
    const float dx = lo16 ? dxa : dxb;
    const float dxm = dx * v[0];
    const float su1 = fmaf(l11, dxm, l12 * v[1]);
    v[3] = l11 * su1;
    v[4] = dx * dxm;
    v[5] = dx * v[1];
    // (slot 1 holds green on the colour lanes)
    v[1] = lo8 ? fmaf(l12, su1, l22 * (l22 * v[1])) : v[1];
    const bool lo4 = !(lane & 4);
    float w[3];
#pragma unroll
    for (int i = 0; i < 3; ++i) {
        const float r = __shfl_xor_sync(F, lo4 ? v[3 + i] : v[i], 4);
        w[i] = (lo4 ? v[i] : v[3 + i]) + r;
    }
    const bool lo2 = !(lane & 2);
    const float r0 = __shfl_xor_sync(F, lo2 ? w[2] : w[0], 2);
    const float x0 = (lo2 ? w[0] : w[2]) + r0;
    const float r1 = __shfl_xor_sync(F, lo2 ? 0.f : w[1], 2);
    const float x1 = (lo2 ? w[1] : 0.f) + r1;
    const bool lo1 = !(lane & 1);
    const float r = __shfl_xor_sync(F, lo1 ? x1 : x0, 1);
    return (lo1 ? x0 : x1) + r;
}

// What lane l (0..15 within its half) holds after reduce_moments2, as the
// grad2d component it feeds (mux, muy, a, b, c, opacity, r, g, b), or -1:
//   0: sum g           -> opacity (times 1 / o)
//   1: d/dmuy
//   2: sum g dy^2      -> c (times -1/2)
//   4: d/dmux
//   5: sum g dx^2      -> a (times -1/2)
//   6: sum g dx dy     -> b (times -1)
//   8, 9, 10: sum w G  -> r, g, b
__device__ __forceinline__ int moment_comp_of_lane(int l) {
    switch (l) {
        case 0: return 5;
        case 1: return 1;
        case 2: return 4;
        case 4: return 0;
        case 5: return 2;
        case 6: return 3;
        case 8: return 6;
        case 9: return 7;
        case 10: return 8;
        default: return -1;
    }
}

__device__ __forceinline__ float moment_scale(int l) {
    return (l == 2 || l == 5) ? -0.5f : (l == 6 ? -1.f : 1.f);
}

// ---------------------------------------------------------------------------
// The backward kernel ("What the 3DGS Literature Left on the Table", Step 6.1,
// 6.2): every warp owns one 8 x 8 quadrant of a tile, two vertically adjacent
// pixels per lane (lane l: column l & 7, rows 2 (l >> 3) and 2 (l >> 3) + 1),
// and walks the tile's list back to front on its own -- no block barrier --
// from its last blended splat, staging in a private 32-splat slice only the
// splats the forward's contributor mask marks for its quadrant.
// ---------------------------------------------------------------------------
constexpr int kBwdWarps = 4;
constexpr int kBwdThreads = 32 * kBwdWarps;

struct BwdSlice {
    float4 r0[32], r1[32], r2[32];
    int32_t gid[32];
};

// Start staging list positions [cs, cs + n) for a quadrant into slice B: the
// splats whose contributor mask has a bit of qmask.  Returns the warp's work
// mask (bit q: position cs + q is staged); the copies complete at the next
// cp_async_wait that covers this group.
__device__ __forceinline__ uint32_t stage_slice(const RasterArgs& A, BwdSlice& B, int64_t cs, int n,
                                                uint32_t qmask, int lane) {
    const bool bit = lane < n && (A.cmask[cs + lane] & qmask) != 0;
    if (bit) {
        const int32_t g = __ldg(A.ids + cs + lane);
        const float4* src = A.splats + 3 * (int64_t)g;
        cp_async16(&B.r0[lane], src);
        cp_async16(&B.r1[lane], src + 1);
        cp_async16(&B.r2[lane], src + 2);
        B.gid[lane] = g;
        if (A.touched) A.touched[g] = 1;  // it blended into some pixel
    }
    cp_async_commit();
    return __ballot_sync(0xffffffffu, bit);
}

// forward thread of tile pixel (lx, ly): the forward's warps cover 8 x 4 pixels
__device__ __forceinline__ int fwd_thread(int lx, int ly) {
    return 32 * ((lx >> 3) + 2 * (ly >> 2)) + (lx & 7) + 8 * (ly & 3);
}

// the back-to-front state of one pixel; accg is the colour behind (dotted
// with dL/dC) plus dL/dT_final * T_final, the two always appear summed
struct BwdPixel {
    float T, accg, Gr, Gg, Gb;
};

// One row of one splat: recovers the transmittance in front of the splat,
// updates the colour behind it; gives the pixel's log-alpha derivative gs (zero
// when it did not blend the splat or the clamp was active) and its blend weight.
__device__ __forceinline__ void row_step(const float4& r0, const float4& r1, const float4& r2,
                                         float dx, float dy, bool in_range, BwdPixel& P,
                                         float* gs, float* wgt) {
    float u1, u2;
    const float qv = quad_q(r0.z, r0.w, r1.x, dx, dy, &u1, &u2);
    const bool act = (qv <= r1.y) && in_range;
    float alpha = fminf(ex2_approx(fmaf(qv, kNegHalfLog2e, r1.z)), kAlphaMax);
    alpha = act ? alpha : 0.f;
    // alpha = 0 gives inv = 1 exactly, so T is unchanged without a select
    const float inv = __fdividef(1.f, 1.f - alpha);
    const float Tb = P.T * inv;
    const float w = alpha * Tb;
    const float cG = r2.x * P.Gr + r2.y * P.Gg + r2.z * P.Gb;
    const float dalpha = Tb * cG - P.accg * inv;
    P.accg = fmaf(cG, w, P.accg);
    // zero when the pixel did not blend (alpha = 0) or the clamp was active
    *gs = alpha < kAlphaMax ? alpha * dalpha : 0.f;
    *wgt = w;
    P.T = Tb;
}

// One splat for the lane's two pixels: its six moments (reduce_moments2) in v
// and its dx.  The conic and mean
// derivatives are formed from the moments inside the reduction: with the
// evaluated quadratic's conic a = l11^2, b = l11 l12, c = l12^2 + l22^2,
// dL/dmux = l11 (l11 sum g dx + l12 sum g dy) and
// dL/dmuy = l12 (l11 sum g dx + l12 sum g dy) + l22^2 sum g dy.
__device__ __forceinline__ void splat_moments2(const BwdSlice& S, int q, float px, float py0,
                                               float py1, int rel0, int rel1, BwdPixel& P0,
                                               BwdPixel& P1, float v[6], float* dx_out) {
    const float4 r0 = S.r0[q], r1 = S.r1[q], r2 = S.r2[q];
    const float dx = rsub(px, r0.x);
    const float dy0 = rsub(py0, r0.y), dy1 = rsub(py1, r0.y);
    float g0, g1, w0, w1;
    row_step(r0, r1, r2, dx, dy0, q <= rel0, P0, &g0, &w0);
    row_step(r0, r1, r2, dx, dy1, q <= rel1, P1, &g1, &w1);
    const float gdy0 = g0 * dy0, gdy1 = g1 * dy1;
    v[0] = g0 + g1;
    v[1] = gdy0 + gdy1;
    v[2] = fmaf(gdy1, dy1, gdy0 * dy0);
    v[3] = fmaf(w1, P1.Gr, w0 * P0.Gr);
    v[4] = fmaf(w1, P1.Gg, w0 * P0.Gg);
    v[5] = fmaf(w1, P1.Gb, w0 * P0.Gb);
    *dx_out = dx;
}

__device__ __forceinline__ void load_bwd_pixel(const RasterArgs& A, const WorkItem& it, int x, int y,
                                               int lx, int ly, BwdPixel& P, int& last) {
    P = BwdPixel{1.f, 0.f, 0.f, 0.f, 0.f};
    last = -1;
    if (x >= A.W || y >= A.H) return;
    const int64_t p = (int64_t)y * A.W + x;
    last = A.last_in[p];
    const float Tfin = A.t_final_in[p];
    P.Gr = A.dimg[3 * p];
    P.Gg = A.dimg[3 * p + 1];
    P.Gb = A.dimg[3 * p + 2];
    P.accg = A.dT ? A.dT[p] * Tfin : 0.f;
    if (it.slot < 0) {
        P.T = Tfin;
    } else {
        const int64_t slotp =
            ((int64_t)it.slot * kMaxChunks + it.chunk) * kThreads + fwd_thread(lx, ly);
        const float4 b = A.bstate[slotp];
        P.T = b.x;
        P.accg += b.y * P.Gr + b.z * P.Gg + b.w * P.Gb;
    }
}

// The accumulators of the backward to zero: grad2d (nf floats, 16-byte
// aligned), the touched flags (n bytes, any alignment; may be null) and the
// work-queue counter.
__global__ void __launch_bounds__(256) bwd_zero(float* __restrict__ grad2d, int64_t nf,
                                                uint8_t* __restrict__ touched, int64_t n,
                                                int* __restrict__ queue) {
    grid_dep_sync();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t n4 = nf / 4;
    float4* g4 = reinterpret_cast<float4*>(grad2d);
    for (int64_t i = i0; i < n4; i += stride) g4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int64_t i = 4 * n4 + i0; i < nf; i += stride) grad2d[i] = 0.f;
    if (touched) {
        // bytes up to the first 16-byte boundary, 16-byte words, the tail
        const int64_t head = min64(n, (int64_t)((16u - (reinterpret_cast<uintptr_t>(touched) & 15u)) & 15u));
        const int64_t n16 = (n - head) / 16;
        uint4* t16 = reinterpret_cast<uint4*>(touched + head);
        if (i0 < head) touched[i0] = 0;
        for (int64_t i = i0; i < n16; i += stride) t16[i] = make_uint4(0u, 0u, 0u, 0u);
        for (int64_t i = head + 16 * n16 + i0; i < n; i += stride) touched[i] = 0;
    }
    if (i0 == 0) *queue = 0;
}

__global__ void __launch_bounds__(kBwdThreads, 6) raster_bwd_kernel(RasterArgs A) {
    grid_dep_sync();
    __shared__ BwdSlice SL[kBwdWarps][2];  // double-buffered per warp
    const unsigned F = 0xffffffffu;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int h = A.ctrl[kCtlH], k = A.ctrl[kCtlK], nitems = A.ctrl[kCtlItems];
    const int nunits = 4 * nitems;  // (work item, quadrant)
    // the writing lanes (reduce_moments2): their component, constant factor and role
    const int sl = lane & 15;
    const int my_comp = moment_comp_of_lane(sl);
    const float my_scale = moment_scale(sl);
    const bool is_opac = sl == 0;
    const bool first = lane < 16;
    const int col = lane & 7, rp = lane >> 3;
    while (true) {
        int unit = 0;
        if (lane == 0) unit = atomicAdd(A.ctrl + kCtlQueueBwd, 1);
        unit = __shfl_sync(F, unit, 0);
        if (unit >= nunits) break;
        const int quad = unit & 3;
        const WorkItem it = decode_item(A, unit >> 2, h, k);
        const int tx = it.tile % A.ntx, ty = it.tile / A.ntx;
        const int lx = 8 * (quad & 1) + col, ly0 = 8 * (quad >> 1) + 2 * rp;
        const int x = tx * kTile + lx, y0 = ty * kTile + ly0;
        const float px = (float)x + 0.5f, py0 = (float)y0 + 0.5f, py1 = (float)(y0 + 1) + 0.5f;
        BwdPixel P0, P1;
        int last0, last1;
        load_bwd_pixel(A, it, x, y0, lx, ly0, P0, last0);
        load_bwd_pixel(A, it, x, y0 + 1, lx, ly0 + 1, P1, last1);
        // the quadrant's two forward sub-tiles (8 x 4 each) in the contributor mask
        const int w0 = (quad & 1) + 4 * (quad >> 1);
        const uint32_t qmask = (1u << w0) | (1u << (w0 + 2));
        int wlast = max((int)min64((int64_t)last0, it.e - 1), (int)min64((int64_t)last1, it.e - 1));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) wlast = max(wlast, __shfl_xor_sync(F, wlast, o));
        if ((int64_t)wlast + 1 <= it.s) continue;
        // 32-position slices back to front; the next slice is staged while
        // the current one is processed
        int cur = 0;
        int64_t cs = max64(it.s, (int64_t)wlast + 1 - 32);
        uint32_t work = stage_slice(A, SL[warp][0], cs, (int)((int64_t)wlast + 1 - cs), qmask, lane);
        while (true) {
            const bool more = cs > it.s;
            int64_t cs2 = 0;
            uint32_t work2 = 0;
            if (more) {
                cs2 = max64(it.s, cs - 32);
                work2 = stage_slice(A, SL[warp][cur ^ 1], cs2, (int)(cs - cs2), qmask, lane);
                cp_async_wait<1>();
            } else {
                cp_async_wait<0>();
            }
            __syncwarp();
            const BwdSlice& S = SL[warp][cur];
            // list positions fit in 32 bits (the pair capacity is below 2^31)
            const int rel0 = last0 - (int)cs, rel1 = last1 - (int)cs;
            while (work) {
                // splats two at a time, back to front: q1 behind q2.  Every staged
                // splat was blended by some pixel of the quadrant (its contributor
                // bit), so its sums are written without asking which lanes took part;
                // where none did (a split tile's chunk blended it past a pixel's
                // global stop) they are zero and adding them changes nothing.
                const int q1 = 31 - __clz(work);
                work &= ~(1u << q1);
                float va[6], dxa;
                splat_moments2(S, q1, px, py0, py1, rel0, rel1, P0, P1, va, &dxa);
                float sum;
                int q;
                bool wr;
                if (work) {
                    const int q2 = 31 - __clz(work);
                    work &= ~(1u << q2);
                    float vb[6], dxb;
                    splat_moments2(S, q2, px, py0, py1, rel0, rel1, P0, P1, vb, &dxb);
                    q = first ? q1 : q2;
                    wr = true;
                    const float4 r0 = S.r0[q];
                    sum = reduce_moments2(va, vb, dxa, dxb, r0.z, r0.w, S.r1[q].x, lane);
                } else {
                    // a lone last splat: paired with zeros
                    const float vz[6] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                    q = q1;
                    wr = first;
                    const float4 r0 = S.r0[q];
                    sum = reduce_moments2(va, vz, dxa, 0.f, r0.z, r0.w, S.r1[q].x, lane);
                }
                // every lane forms its write; only the atomic is predicated.  The
                // opacity lane divides o back out, o = 2^log2(o)
                const float f = is_opac ? ex2_approx(-S.r1[q].z) : my_scale;
                float* dst = A.grad2d + 9 * (int64_t)S.gid[q] + my_comp;
                if (my_comp >= 0 && wr) atomicAdd(dst, sum * f);
            }
            __syncwarp();  // the slice is restaged two steps later
            if (!more) break;
            cs = cs2;
            work = work2;
            cur ^= 1;
        }
    }
}

int g_resident[64][2];
std::mutex g_mu;

}  // namespace

int raster_resident_ctas(int device) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (device < 0 || device >= 64) return 0;
    if (g_resident[device][0] == 0) {
        int sms = 0, per = 0;
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, raster_fwd_kernel, kThreads, 0);
        g_resident[device][0] = std::max(1, sms * std::max(per, 1));
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, raster_bwd_kernel, kBwdThreads, 0);
        g_resident[device][1] = std::max(1, sms * std::max(per, 1));
    }
    return g_resident[device][0];
}

static int resident_bwd(int device) {
    raster_resident_ctas(device);
    std::lock_guard<std::mutex> lk(g_mu);
    return g_resident[device][1];
}

RasterLayout raster_layout(int W, int H, int h_max, int64_t capacity) {
    RasterLayout L{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t o = off;
        off = (off + bytes + 255) & ~size_t(255);
        return o;
    };
    // at most min(h_max, tiles) tiles are split (the policy's candidates)
    const int64_t nt = (((int64_t)W + kTile - 1) / kTile) * (((int64_t)H + kTile - 1) / kTile);
    const size_t hm = (size_t)std::max<int64_t>(std::min<int64_t>(h_max, nt), 1);
    const size_t px = hm * kMaxChunks * kThreads;
    L.off_ctrl = take(kCtlWords * sizeof(int));
    L.off_sat = take(hm * sizeof(int));
    L.off_done = take(hm * sizeof(int));
    L.off_cbatch = take(hm * kMaxChunks * sizeof(int));
    L.off_part_c = take(px * sizeof(float4));
    L.off_part_n = take(px * sizeof(int2));
    L.off_bwd = take(px * sizeof(float4));
    L.off_cmask = take((size_t)max64(capacity, 1));
    L.total = off;
    return L;
}

static RasterArgs make_args(const CamParams& cam, const float* splats, const int32_t* ids,
                            const int32_t* ranges, const int32_t* lpt, char* ws,
                            const RasterLayout& L) {
    RasterArgs A{};
    A.W = cam.W;
    A.H = cam.H;
    A.ntx = cam.ntx;
    A.nty = cam.nty;
    A.splats = reinterpret_cast<const float4*>(splats);
    A.ids = ids;
    A.ranges = reinterpret_cast<const int2*>(ranges);
    A.lpt = lpt;
    A.ctrl = reinterpret_cast<int*>(ws + L.off_ctrl);
    A.sat = reinterpret_cast<int*>(ws + L.off_sat);
    A.done = reinterpret_cast<int*>(ws + L.off_done);
    A.cbatch = reinterpret_cast<int*>(ws + L.off_cbatch);
    A.part_c = reinterpret_cast<float4*>(ws + L.off_part_c);
    A.part_n = reinterpret_cast<int2*>(ws + L.off_part_n);
    A.bstate = reinterpret_cast<float4*>(ws + L.off_bwd);
    A.cmask = reinterpret_cast<uint8_t*>(ws + L.off_cmask);
    return A;
}

cudaError_t run_raster_fwd(const CamParams& cam, const RasterConfig& cfg, const float* splats,
                           const int32_t* sorted_ids, const int32_t* tile_ranges,
                           const int32_t* lpt_order, char* ws, const RasterLayout& L, float* image,
                           float* t_final, int32_t* n_contrib, int32_t* last_idx, cudaStream_t st) {
    int dev = 0;
    cudaGetDevice(&dev);
    const int K = raster_resident_ctas(dev);
    RasterArgs A = make_args(cam, splats, sorted_ids, tile_ranges, lpt_order, ws, L);
    A.image = image;
    A.t_final = t_final;
    A.n_contrib = n_contrib;
    A.last_idx = last_idx;
    const int nt = cam.ntx * cam.nty;
    cudaError_t err = launch_clustered(policy_kernel, kPolicyCluster, kPolicyCluster,
                                       kPolicyThreads, 0, st, lpt_order,
                             (const int2*)A.ranges, nt, K, cfg, A.ctrl, A.sat, A.done);
    if (err != cudaSuccess) return err;
    return launch(raster_fwd_kernel, K, kThreads, 0, st, A);
}

cudaError_t run_raster_bwd(const CamParams& cam, const RasterConfig& cfg, int64_t n,
                           const float* splats, const int32_t* sorted_ids,
                           const int32_t* tile_ranges, const int32_t* lpt_order, char* ws,
                           const RasterLayout& L, const float* t_final, const int32_t* last_idx,
                           const float* dL_dimage, const float* dL_dt, float* grad2d,
                           uint8_t* touched, cudaStream_t st) {
    (void)cfg;
    int dev = 0;
    cudaGetDevice(&dev);
    const int K = resident_bwd(dev);
    RasterArgs A = make_args(cam, splats, sorted_ids, tile_ranges, lpt_order, ws, L);
    A.t_final_in = t_final;
    A.last_in = last_idx;
    A.dimg = dL_dimage;
    A.dT = dL_dt;
    A.grad2d = grad2d;
    A.touched = touched;
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t nf = n * 9;
    const int64_t zb = std::max<int64_t>(1, std::min<int64_t>((nf / 4 + 255) / 256,
                                                               8 * (int64_t)std::max(sms, 1)));
    cudaError_t err = launch(bwd_zero, (unsigned)zb, 256, 0, st, grad2d, nf, touched, n,
                             A.ctrl + kCtlQueueBwd);
    if (err != cudaSuccess) return err;
    return launch(raster_bwd_kernel, K, kBwdThreads, 0, st, A);
}

}  // namespace gs
