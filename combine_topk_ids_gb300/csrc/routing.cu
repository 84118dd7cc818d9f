// Routing kernels of moe_dispatch: per-expert / per-destination histograms, block prefix
// sums, and deterministic slot assignment in ascending (token, pick) order.
//
// Operation (Mooncake EP guide, "Buffer.dispatch(...)": topk_idx with -1 for masked picks,
// the local-expert-major packed layout with packed_recv_count / packed_recv_layout_range;
// FlashInfer "MoE-EP implementation & usage", section 3 "Algorithm / layout contracts":
// EXPERT_MAJOR rows pre-assigned to experts, RANK_MAJOR rows grouped by source rank,
// FLAT token-major, received topk_idx LOCAL with -1 for non-local picks).
//
// Three launches, no atomics deciding any position:
//   route_count   one block per (logical rank, token chunk): shared-memory histogram of the
//                 chunk's expert ids (and of the destination ranks of its tokens)
//   route_scan    one block: per expert / destination an exclusive scan over the chunks,
//                 split at logical-rank boundaries (layout ranges, RANK_MAJOR rows), then
//                 the expert offsets and the GEMM m-block prefix
//   route_assign  one block per chunk: every warp owns a contiguous run of picks, counts its
//                 run, takes an exclusive prefix over the block's warps, and then ranks its
//                 picks 32 at a time with __match_any_sync / __ballot_sync.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr unsigned kFull = 0xffffffffu;

struct RouteArgs {
    const void *ids;
    int ids64;
    const float *topk_w;
    const int32_t *active;          // EP rank-health mask [W] (NULL: all ranks active)
    int T, W, Tr, E, k, Le, layout, tb, nbpr, nb;
    int zero_status;                // the single-CTA kernel clears the status word first
    int32_t *sched;                 // and the GEMMs' tile counters (NULL: none)
    int64_t cap;
    int32_t *status, *counts, *offsets, *mprefix, *mprefix2, *pick_pos, *pick_src, *slot, *layout_range;
    int32_t *blk_hist, *blk_base;   // [E][nb]
    int32_t *recv_row, *recv_count, *num_recv, *recv_src, *recv_topk_idx;
    int32_t *blk_dhist, *blk_dbase; // [W][nb]
    float *recv_topk_w;
};

// Bit r set iff logical rank r is active (Mooncake EP active_ranks: 0 = failed rank).
// Read once per block into shared memory by the caller.
__device__ __forceinline__ unsigned long long load_active_mask(const RouteArgs &a) {
    unsigned long long m = 0;
    for (int r = 0; r < a.W; ++r)
        if (!a.active || a.active[r] != 0) m |= 1ull << r;
    return m;
}

// Expert id of pick i: [0, E) valid, -1 masked, -2 outside [-1, E), -3 dropped because its
// expert's rank or its token's source rank is inactive.
__device__ __forceinline__ int load_id(const RouteArgs &a, int64_t i, unsigned long long act) {
    long long v = a.ids64 ? reinterpret_cast<const long long *>(a.ids)[i]
                          : (long long)reinterpret_cast<const int *>(a.ids)[i];
    if (v == -1) return -1;
    if (v < -1 || v >= a.E) return -2;
    const int src = ((int)i / a.k) / a.Tr;   // picks fit in int32 (checked on the host)
    if (!((act >> ((int)v / a.Le)) & 1ull) || !((act >> src) & 1ull)) return -3;
    return (int)v;
}

// Bit d set iff token t has a valid pick on destination rank d.
__device__ __forceinline__ unsigned long long dest_mask(const RouteArgs &a, int t,
                                                        unsigned long long act) {
    unsigned long long m = 0;
    for (int j = 0; j < a.k; ++j) {
        int e = load_id(a, (int64_t)t * a.k + j, act);
        if (e >= 0) m |= 1ull << (e / a.Le);
    }
    return m;
}

// Tokens [t0, t1) of routing block b: chunk (b % nbpr) of logical rank b / nbpr.
__device__ __forceinline__ void block_tokens(const RouteArgs &a, int b, int &t0, int &t1) {
    int r = b / a.nbpr;
    t0 = r * a.Tr + (b % a.nbpr) * a.tb;
    t1 = min(min(t0 + a.tb, (r + 1) * a.Tr), a.T);
    if (t0 > t1) t0 = t1;
}

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

__device__ __forceinline__ int warp_incl_scan(int v) {
    int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int n = __shfl_up_sync(kFull, v, o);
        if (lane >= o) v += n;
    }
    return v;
}

__global__ void __launch_bounds__(kRouteThreads) route_count_kernel(RouteArgs a) {
    pdl_begin();   // after the previous kernel in the stream (programmatic launch)
    extern __shared__ int sm[];
    int *hist = sm;          // [E]
    int *dhist = sm + a.E;   // [W]
    __shared__ unsigned long long s_act;
    if (threadIdx.x == 0) s_act = load_active_mask(a);
    for (int i = threadIdx.x; i < a.E + a.W; i += blockDim.x) sm[i] = 0;
    __syncthreads();
    const unsigned long long act = s_act;
    int t0, t1;
    block_tokens(a, blockIdx.x, t0, t1);
    bool bad = false, inactive = false;
    for (int64_t i = (int64_t)t0 * a.k + threadIdx.x; i < (int64_t)t1 * a.k; i += blockDim.x) {
        int e = load_id(a, i, act);
        if (e >= 0) atomicAdd(&hist[e], 1);   // counts only; positions come later
        else if (e == -2) bad = true;
        else if (e == -3) inactive = true;
    }
    if (a.layout != MOE_LAYOUT_EXPERT_MAJOR) {
        for (int t = t0 + threadIdx.x; t < t1; t += blockDim.x) {
            unsigned long long m = dest_mask(a, t, act);
            while (m) {
                int d = __ffsll((long long)m) - 1;
                m &= m - 1;
                atomicAdd(&dhist[d], 1);
            }
        }
    }
    if (bad) atomicOr(a.status, MOE_STATUS_BAD_EXPERT_ID);
    if (inactive) atomicOr(a.status, MOE_STATUS_INACTIVE_RANK);
    __syncthreads();
    for (int e = threadIdx.x; e < a.E; e += blockDim.x)
        a.blk_hist[(int64_t)e * a.nb + blockIdx.x] = hist[e];
    if (a.layout != MOE_LAYOUT_EXPERT_MAJOR)
        for (int d = threadIdx.x; d < a.W; d += blockDim.x)
            a.blk_dhist[(int64_t)d * a.nb + blockIdx.x] = dhist[d];
}

// Exclusive scan of one row hist[0..nb) (blocks grouped by logical rank, nbpr per rank)
// into base[], warp-cooperative, in one pass over the row.  RANK_MAJOR destinations restart
// each source rank at row s*Tr.  on_rank(s, begin, count) is then called by lane s % 32 for
// every rank s (begin/count of the plain, non-restarted scan).  Returns the row total.
template <typename RankFn>
__device__ __forceinline__ int scan_row(const RouteArgs &a, const int32_t *hist, int32_t *base,
                                        bool restart_per_rank, RankFn on_rank) {
    const int lane = threadIdx.x & 31;
    int run = 0;
    // 256 chunks per round: all eight loads are issued before the first scan step
    for (int b00 = 0; b00 < a.nb; b00 += 256) {
        int v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int b = b00 + 32 * i + lane;
            v[i] = b < a.nb ? hist[b] : 0;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int b = b00 + 32 * i + lane;
            const int incl = warp_incl_scan(v[i]);
            if (b < a.nb) base[b] = run + incl - v[i];
            run += __shfl_sync(kFull, incl, 31);
        }
    }
    __syncwarp();
    // per-rank begin (= exclusive prefix at the rank's first block) and count
    int first[2] = {0, 0};   // ranks lane and lane + 32 (W <= 64)
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const int r = lane + 32 * q;
        if (r < a.W) {
            const int beg = base[r * a.nbpr];
            const int end = r + 1 < a.W ? base[(r + 1) * a.nbpr] : run;
            first[q] = beg;
            on_rank(r, beg, end - beg);
        }
    }
    if (restart_per_rank) {
        __syncwarp();
        for (int b0 = 0; b0 < a.nb; b0 += 32) {
            const int b = b0 + lane;
            const int r = (b < a.nb ? b : 0) / a.nbpr;
            const int f0 = __shfl_sync(kFull, first[0], r & 31);
            const int f1 = __shfl_sync(kFull, first[1], r & 31);
            if (b < a.nb) base[b] = r * a.Tr + base[b] - (r < 32 ? f0 : f1);
        }
        __syncwarp();
    }
    return run;
}

__global__ void __launch_bounds__(1024) route_scan_kernel(RouteArgs a) {
    pdl_begin();   // after the previous kernel in the stream (programmatic launch)
    __shared__ int wsum[3][32];
    __shared__ int carry[3];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    const bool em = a.layout == MOE_LAYOUT_EXPERT_MAJOR;
    // (1) per expert: chunk bases, layout ranges, counts (EM clamps to the region size)
    for (int e = warp; e < a.E; e += nwarps) {
        int total = scan_row(a, a.blk_hist + (int64_t)e * a.nb, a.blk_base + (int64_t)e * a.nb,
                             false, [&](int s, int begin, int cnt) {
                                 int64_t lim = em ? a.cap : (int64_t)1 << 40;
                                 int64_t b = begin < lim ? begin : lim;
                                 int64_t kept = lim - begin;
                                 kept = kept < 0 ? 0 : (kept > cnt ? cnt : kept);
                                 a.layout_range[((int64_t)e * a.W + s) * 2 + 0] = (int)b;
                                 a.layout_range[((int64_t)e * a.W + s) * 2 + 1] = (int)kept;
                             });
        if (lane == 0) a.counts[e] = (em && total > a.cap) ? (int)a.cap : total;
    }
    // (1b) per destination rank (RANK_MAJOR / FLAT): chunk row bases and received counts
    if (!em) {
        for (int d = warp; d < a.W; d += nwarps) {
            int total = scan_row(a, a.blk_dhist + (int64_t)d * a.nb, a.blk_dbase + (int64_t)d * a.nb,
                                 a.layout == MOE_LAYOUT_RANK_MAJOR, [&](int s, int, int cnt) {
                                     a.recv_count[d * a.W + s] = cnt;
                                 });
            if (lane == 0) a.num_recv[d] = total;
        }
    }
    __syncthreads();
    // (2) expert offsets and the prefixes of GEMM row blocks (128-row tiles of one SM,
    //     256-row tiles of an SM pair) over experts
    if (threadIdx.x == 0) carry[0] = carry[1] = carry[2] = 0;
    __syncthreads();
    for (int e0 = 0; e0 < a.E; e0 += blockDim.x) {
        int e = e0 + threadIdx.x;
        int v[3];
        v[0] = e < a.E ? a.counts[e] : 0;
        v[1] = (v[0] + kTileM - 1) / kTileM;
        v[2] = (v[0] + 2 * kTileM - 1) / (2 * kTileM);
        int inc[3];
#pragma unroll
        for (int q = 0; q < 3; ++q) inc[q] = warp_incl_scan(v[q]);
        if (lane == 31)
            for (int q = 0; q < 3; ++q) wsum[q][warp] = inc[q];
        __syncthreads();
        if (warp == 0) {
#pragma unroll
            for (int q = 0; q < 3; ++q) {
                int w = lane < nwarps ? wsum[q][lane] : 0;
                wsum[q][lane] = warp_incl_scan(w) - w;
            }
        }
        __syncthreads();
        if (e < a.E) {
            a.offsets[e] = carry[0] + wsum[0][warp] + inc[0] - v[0];
            a.mprefix[e] = carry[1] + wsum[1][warp] + inc[1] - v[1];
            a.mprefix2[e] = carry[2] + wsum[2][warp] + inc[2] - v[2];
        }
        __syncthreads();
        if (threadIdx.x == blockDim.x - 1)
            for (int q = 0; q < 3; ++q) carry[q] += wsum[q][warp] + inc[q];
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        a.offsets[a.E] = carry[0];
        a.mprefix[a.E] = carry[1];
        a.mprefix2[a.E] = carry[2];
    }
}

__global__ void __launch_bounds__(kRouteThreads) route_assign_kernel(RouteArgs a) {
    pdl_begin();   // after the previous kernel in the stream (programmatic launch)
    extern __shared__ int sm[];
    int *cur = sm;                          // [warps][E] running position inside expert
    int *dcur = sm + kRouteWarps * a.E;     // [warps][W] running row inside destination
    __shared__ unsigned long long s_act;
    if (threadIdx.x == 0) s_act = load_active_mask(a);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, b = blockIdx.x;
    const bool em = a.layout == MOE_LAYOUT_EXPERT_MAJOR;
    for (int i = threadIdx.x; i < kRouteWarps * (a.E + a.W); i += blockDim.x) sm[i] = 0;
    int t0, t1;
    block_tokens(a, b, t0, t1);
    // this warp's contiguous run of picks [wp0, wp1) and tokens [wt0, wt1)
    const int64_t p0 = (int64_t)t0 * a.k, np = (int64_t)(t1 - t0) * a.k;
    const int64_t ppw = (np + kRouteWarps * 32 - 1) / (kRouteWarps * 32) * 32;
    const int64_t wp0 = min(p0 + warp * ppw, p0 + np), wp1 = min(wp0 + ppw, p0 + np);
    const int tpw = ((t1 - t0) + kRouteWarps * 32 - 1) / (kRouteWarps * 32) * 32;
    const int wt0 = min(t0 + warp * tpw, t1), wt1 = min(wt0 + tpw, t1);
    __syncthreads();
    const unsigned long long act = s_act;
    // pass 1: per-warp counts
    for (int64_t i0 = wp0; i0 < wp1; i0 += 32) {
        int64_t i = i0 + lane;
        int e = i < wp1 ? load_id(a, i, act) : -1;
        int key = e >= 0 ? e : -1;
        unsigned peers = __match_any_sync(kFull, key);
        if (key >= 0 && lane == __ffs(peers) - 1) cur[warp * a.E + key] += __popc(peers);
        __syncwarp();
    }
    if (!em) {
        for (int tt = wt0; tt < wt1; tt += 32) {
            int t = tt + lane;
            unsigned long long m = t < wt1 ? dest_mask(a, t, act) : 0ull;
            for (int d = 0; d < a.W; ++d) {
                unsigned bal = __ballot_sync(kFull, (m >> d) & 1ull);
                if (lane == 0) dcur[warp * a.W + d] += __popc(bal);
            }
            __syncwarp();
        }
    }
    __syncthreads();
    // exclusive prefix over the block's warps, on top of the chunk's base
    for (int e = threadIdx.x; e < a.E; e += blockDim.x) {
        int run = a.blk_base[(int64_t)e * a.nb + b];
        for (int w = 0; w < kRouteWarps; ++w) {
            int c = cur[w * a.E + e];
            cur[w * a.E + e] = run;
            run += c;
        }
    }
    if (!em) {
        for (int d = threadIdx.x; d < a.W; d += blockDim.x) {
            int run = a.blk_dbase[(int64_t)d * a.nb + b];
            for (int w = 0; w < kRouteWarps; ++w) {
                int c = dcur[w * a.W + d];
                dcur[w * a.W + d] = run;
                run += c;
            }
        }
    }
    __syncthreads();
    // pass 2: ranks of the picks
    bool overflow = false;
    for (int64_t i0 = wp0; i0 < wp1; i0 += 32) {
        int64_t i = i0 + lane;
        int e = i < wp1 ? load_id(a, i, act) : -1;
        int key = e >= 0 ? e : -1;
        unsigned peers = __match_any_sync(kFull, key);
        int pos = key >= 0 ? cur[warp * a.E + key] + __popc(peers & lanemask_lt()) : 0;
        __syncwarp();
        if (key >= 0 && lane == __ffs(peers) - 1) cur[warp * a.E + key] += __popc(peers);
        __syncwarp();
        if (i < wp1) {
            int pp = -1, sl = -1;
            if (key >= 0) {
                if (pos < a.counts[key]) {   // EM counts are clamped to the region's rows
                    pp = a.offsets[key] + pos;
                    sl = (int)((int64_t)key * a.cap + pos);
                    a.pick_src[pp] = (int)i;
                } else {
                    overflow = true;
                }
            }
            a.pick_pos[i] = pp;
            if (em) a.slot[i] = sl;
        }
    }
    if (overflow) atomicOr(a.status, MOE_STATUS_EM_OVERFLOW);
    if (em) return;
    // pass 2 for destinations: rows, source tokens, local ids and weights
    for (int tt = wt0; tt < wt1; tt += 32) {
        int t = tt + lane;
        bool valid = t < wt1;
        unsigned long long m = valid ? dest_mask(a, t, act) : 0ull;
        for (int d = 0; d < a.W; ++d) {
            bool has = (m >> d) & 1ull;
            unsigned bal = __ballot_sync(kFull, has);
            int row = dcur[warp * a.W + d] + __popc(bal & lanemask_lt());
            __syncwarp();
            if (lane == 0) dcur[warp * a.W + d] += __popc(bal);
            __syncwarp();
            if (!valid) continue;
            if (!has) {
                a.recv_row[(int64_t)t * a.W + d] = -1;
                continue;
            }
            a.recv_row[(int64_t)t * a.W + d] = row;
            int64_t o = (int64_t)d * a.cap + row;
            a.recv_src[o] = t;
            for (int j = 0; j < a.k; ++j) {   // non-local until a local pick claims it below
                a.recv_topk_idx[o * a.k + j] = -1;
                a.recv_topk_w[o * a.k + j] = 0.0f;
            }
        }
    }
    __syncthreads();   // this block's receive rows exist; now place its local picks in them
    for (int64_t i = p0 + threadIdx.x; i < p0 + np; i += blockDim.x) {
        const int e = load_id(a, i, act);
        if (e < 0) continue;
        const int t = (int)i / a.k, j = (int)i - t * a.k, d = e / a.Le;
        const int64_t o = (int64_t)d * a.cap + a.recv_row[(int64_t)t * a.W + d];
        a.recv_topk_idx[o * a.k + j] = e - d * a.Le;
        a.recv_topk_w[o * a.k + j] = a.topk_w[i];
    }
}


// ---------------------------------------------------------------------------------------
// Small batches: the three steps above in one CTA of 32 warps, everything in shared memory
// (one launch instead of three; decode-sized batches are launch-latency bound).  Same
// deterministic scheme: each warp owns a contiguous run of picks (and of tokens), counts
// it, takes an exclusive prefix over the warps, then ranks its run 32 at a time.  Per
// (expert, source rank) and (destination, source rank) counts come from shared-memory
// atomics (counts only).  RANK_MAJOR rows are derived from the token's rank among all
// tokens received by the destination minus those of earlier source ranks.
constexpr int kFusedThreads = 1024;
constexpr int kFusedWarps = kFusedThreads / 32;

// Exclusive scan of three values per thread across a 1024-thread block.
__device__ __forceinline__ void block_excl_scan3(const int (&v)[3], int (&ex)[3], int (*wsum)[32]) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int inc[3];
#pragma unroll
    for (int q = 0; q < 3; ++q) inc[q] = warp_incl_scan(v[q]);
    if (lane == 31)
        for (int q = 0; q < 3; ++q) wsum[q][warp] = inc[q];
    __syncthreads();
    if (warp == 0) {
#pragma unroll
        for (int q = 0; q < 3; ++q) {
            int w = wsum[q][lane];
            wsum[q][lane] = warp_incl_scan(w) - w;
        }
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < 3; ++q) ex[q] = wsum[q][warp] + inc[q] - v[q];
}

__global__ void __launch_bounds__(kFusedThreads) route_fused_kernel(RouteArgs a) {
    pdl_begin();   // after the previous kernel in the stream (programmatic launch)
    extern __shared__ int sm[];
    __shared__ int wsum[3][32];
    const int E = a.E, W = a.W;
    int *cur = sm;                          // [warps][E]
    int *dcur = cur + kFusedWarps * E;      // [warps][W]
    int *ew = dcur + kFusedWarps * W;       // [E][W]  kept picks per (expert, source rank)
    int *dw = ew + E * W;                   // [W][W]  tokens per (destination, source rank)
    int *off = dw + W * W;                  // [E]     expert offsets
    int *cnt = off + E;                     // [E]     kept counts
    __shared__ unsigned long long s_act;
    if (threadIdx.x == 0) {
        s_act = load_active_mask(a);
        if (a.zero_status) {
            *a.status = 0;   // before the barrier below, so before any bit is set
            if (a.sched)
                for (int i = 0; i < 4; ++i) a.sched[i] = 0;
        }
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const bool em = a.layout == MOE_LAYOUT_EXPERT_MAJOR;
    const int total_sm = kFusedWarps * (E + W) + E * W + W * W + 2 * E;
    for (int i = threadIdx.x; i < total_sm; i += blockDim.x) sm[i] = 0;
    const int64_t P = (int64_t)a.T * a.k;
    const int64_t ppw = (P + kFusedWarps * 32 - 1) / (kFusedWarps * 32) * 32;
    const int64_t wp0 = min(warp * ppw, P), wp1 = min(wp0 + ppw, P);
    const int tpw = (a.T + kFusedWarps * 32 - 1) / (kFusedWarps * 32) * 32;
    const int wt0 = min(warp * tpw, a.T), wt1 = min(wt0 + tpw, a.T);
    __syncthreads();
    const unsigned long long act = s_act;
    // pass 1: counts
    bool bad = false, inactive = false;
    for (int64_t i0 = wp0; i0 < wp1; i0 += 32) {
        int64_t i = i0 + lane;
        int e = i < wp1 ? load_id(a, i, act) : -1;
        if (e == -2) bad = true;
        if (e == -3) inactive = true;
        int key = e >= 0 ? e : -1;
        unsigned peers = __match_any_sync(kFull, key);
        if (key >= 0 && lane == __ffs(peers) - 1) cur[warp * E + key] += __popc(peers);
        __syncwarp();
    }
    if (bad) atomicOr(a.status, MOE_STATUS_BAD_EXPERT_ID);
    if (inactive) atomicOr(a.status, MOE_STATUS_INACTIVE_RANK);
    if (!em) {
        for (int tt = wt0; tt < wt1; tt += 32) {
            int t = tt + lane;
            unsigned long long m = t < wt1 ? dest_mask(a, t, act) : 0ull;
            for (int d = 0; d < W; ++d) {
                bool has = (m >> d) & 1ull;
                unsigned bal = __ballot_sync(kFull, has);
                if (lane == 0) dcur[warp * W + d] += __popc(bal);
                if (has) atomicAdd(&dw[d * W + t / a.Tr], 1);
            }
            __syncwarp();
        }
    }
    __syncthreads();
    // per expert: exclusive prefix over warps; kept count (EM clamps to the region)
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int run = 0;
        for (int w = 0; w < kFusedWarps; ++w) {
            int c = cur[w * E + e];
            cur[w * E + e] = run;
            run += c;
        }
        int kept = (em && run > a.cap) ? (int)a.cap : run;
        cnt[e] = kept;
        a.counts[e] = kept;
    }
    // per destination: exclusive prefix over warps (rank among all tokens it receives),
    // received counts per source rank, and their exclusive prefix over source ranks
    if (!em) {
        for (int d = threadIdx.x; d < W; d += blockDim.x) {
            int run = 0;
            for (int w = 0; w < kFusedWarps; ++w) {
                int c = dcur[w * W + d];
                dcur[w * W + d] = run;
                run += c;
            }
            a.num_recv[d] = run;
            int b = 0;
            for (int s2 = 0; s2 < W; ++s2) {
                int c = dw[d * W + s2];
                a.recv_count[d * W + s2] = c;
                dw[d * W + s2] = b;
                b += c;
            }
        }
    }
    __syncthreads();
    // expert offsets and the 128 / 256-row block prefixes (E <= blockDim.x here)
    {
        int e = threadIdx.x;
        int v[3], ex[3];
        v[0] = e < E ? cnt[e] : 0;
        v[1] = (v[0] + kTileM - 1) / kTileM;
        v[2] = (v[0] + 2 * kTileM - 1) / (2 * kTileM);
        block_excl_scan3(v, ex, wsum);
        if (e < E) {
            off[e] = ex[0];
            a.offsets[e] = ex[0];
            a.mprefix[e] = ex[1];
            a.mprefix2[e] = ex[2];
        }
        if (threadIdx.x == blockDim.x - 1) {
            a.offsets[E] = ex[0] + v[0];
            a.mprefix[E] = ex[1] + v[1];
            a.mprefix2[E] = ex[2] + v[2];
        }
    }
    __syncthreads();
    // pass 2: positions of the picks
    bool overflow = false;
    for (int64_t i0 = wp0; i0 < wp1; i0 += 32) {
        int64_t i = i0 + lane;
        int e = i < wp1 ? load_id(a, i, act) : -1;
        int key = e >= 0 ? e : -1;
        unsigned peers = __match_any_sync(kFull, key);
        int pos = key >= 0 ? cur[warp * E + key] + __popc(peers & lanemask_lt()) : 0;
        __syncwarp();
        if (key >= 0 && lane == __ffs(peers) - 1) cur[warp * E + key] += __popc(peers);
        __syncwarp();
        if (i < wp1) {
            int pp = -1, sl = -1;
            if (key >= 0) {
                if (pos < cnt[key]) {
                    pp = off[key] + pos;
                    sl = (int)((int64_t)key * a.cap + pos);
                    a.pick_src[pp] = (int)i;
                    atomicAdd(&ew[key * W + (int)(i / a.k) / a.Tr], 1);
                } else {
                    overflow = true;
                }
            }
            a.pick_pos[i] = pp;
            if (em) a.slot[i] = sl;
        }
    }
    if (overflow) atomicOr(a.status, MOE_STATUS_EM_OVERFLOW);
    // layout ranges of the kept picks
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int b = 0;
        for (int r = 0; r < W; ++r) {
            int c = ew[e * W + r];
            a.layout_range[((int64_t)e * W + r) * 2 + 0] = b;
            a.layout_range[((int64_t)e * W + r) * 2 + 1] = c;
            b += c;
        }
    }
    if (em) return;
    // destinations: rows, source tokens, local ids and weights
    for (int tt = wt0; tt < wt1; tt += 32) {
        int t = tt + lane;
        bool valid = t < wt1;
        unsigned long long m = valid ? dest_mask(a, t, act) : 0ull;
        for (int d = 0; d < W; ++d) {
            bool has = (m >> d) & 1ull;
            unsigned bal = __ballot_sync(kFull, has);
            int flat = dcur[warp * W + d] + __popc(bal & lanemask_lt());
            __syncwarp();
            if (lane == 0) dcur[warp * W + d] += __popc(bal);
            __syncwarp();
            if (!valid) continue;
            if (!has) {
                a.recv_row[(int64_t)t * W + d] = -1;
                continue;
            }
            const int s2 = t / a.Tr;
            const int row = a.layout == MOE_LAYOUT_RANK_MAJOR ? s2 * a.Tr + flat - dw[d * W + s2] : flat;
            a.recv_row[(int64_t)t * W + d] = row;
            int64_t o = (int64_t)d * a.cap + row;
            a.recv_src[o] = t;
            for (int j = 0; j < a.k; ++j) {   // non-local until a local pick claims it below
                a.recv_topk_idx[o * a.k + j] = -1;
                a.recv_topk_w[o * a.k + j] = 0.0f;
            }
        }
    }
    __syncthreads();   // every receive row exists; now place the local picks in them
    for (int64_t i = threadIdx.x; i < P; i += blockDim.x) {
        const int e = load_id(a, i, act);
        if (e < 0) continue;
        const int t = (int)i / a.k, j = (int)i - t * a.k, d = e / a.Le;
        const int64_t o = (int64_t)d * a.cap + a.recv_row[(int64_t)t * W + d];
        a.recv_topk_idx[o * a.k + j] = e - d * a.Le;
        a.recv_topk_w[o * a.k + j] = a.topk_w[i];
    }
}

}  // namespace

#ifndef MOE_FUSED_ROUTING_MAX_PICKS
#define MOE_FUSED_ROUTING_MAX_PICKS 3072
#endif
// The single-CTA path wins for small batches over few experts (one launch instead of
// three: 9-12 vs 14-15 us for 128-2048 picks) and loses for larger ones (44.6 vs 15.9 us
// on 16384 picks over 16 experts; 82 vs 36 us with 256 experts, where its per-expert work
// runs on one SM), so it is kept for at most 3072 picks and E <= 64.
int routing_launches(const Plan &p) {
    return (p.P <= MOE_FUSED_ROUTING_MAX_PICKS && p.E <= 64 && p.E * p.W <= 4096) ? 1 : 3;
}

cudaError_t launch_routing(const Routing &r, const void *ids, int ids64, const float *topk_w,
                           const int32_t *active, cudaStream_t s) {
    const Plan &p = *r.p;
    RouteArgs a;
    a.ids = ids;
    a.ids64 = ids64;
    a.topk_w = topk_w;
    a.active = active;
    a.T = (int)p.T; a.W = (int)p.W; a.Tr = (int)p.Tr; a.E = (int)p.E; a.k = (int)p.k;
    a.Le = (int)(p.E / p.W);
    a.layout = p.layout;
    a.tb = p.tb; a.nbpr = p.nbpr; a.nb = p.nb;
    a.cap = p.cap;
    a.status = r.status; a.counts = r.counts; a.offsets = r.offsets; a.mprefix = r.mprefix;
    a.mprefix2 = r.mprefix2;
    a.pick_pos = r.pick_pos; a.pick_src = r.pick_src; a.slot = r.slot;
    a.layout_range = r.layout_range; a.blk_hist = r.blk_hist; a.blk_base = r.blk_base;
    a.recv_row = r.recv_row; a.recv_count = r.recv_count; a.num_recv = r.num_recv;
    a.recv_src = r.recv_src; a.recv_topk_idx = r.recv_topk_idx; a.recv_topk_w = r.recv_topk_w;
    a.blk_dhist = r.blk_dhist; a.blk_dbase = r.blk_dbase;
    a.zero_status = 0;
    a.sched = r.sched;

    // one fused CTA for small batches with few experts (bounded shared memory); it clears
    // the status word itself (one launch less in a latency-bound step)
    if (routing_launches(p) == 1) {
        a.zero_status = 1;
        const size_t smf = (size_t)(kFusedWarps * (a.E + a.W) + a.E * a.W + a.W * a.W + 2 * a.E) *
                           sizeof(int);
        if (smf > 48 * 1024) {
            cudaError_t e = cudaFuncSetAttribute(route_fused_kernel,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smf);
            if (e != cudaSuccess) return e;
        }
        return launch_pdl(route_fused_kernel, dim3(1), dim3(kFusedThreads), smf, s, a);
    }

    // several blocks may raise status bits: clear the word before the first of them runs
    // (the GEMMs' tile counters follow the status word when there is a workspace)
    if (cudaMemsetAsync(a.status, 0, (r.sched ? 5 : 1) * sizeof(int32_t), s) != cudaSuccess)
        return cudaGetLastError();
    size_t sm1 = (size_t)(a.E + a.W) * sizeof(int);
    cudaError_t e = launch_pdl(route_count_kernel, dim3(a.nb), dim3(kRouteThreads), sm1, s, a);
    if (e != cudaSuccess) return e;
    e = launch_pdl(route_scan_kernel, dim3(1), dim3(1024), 0, s, a);
    if (e != cudaSuccess) return e;
    size_t sm3 = (size_t)kRouteWarps * (a.E + a.W) * sizeof(int);
    if (sm3 > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(route_assign_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm3);
        if (e != cudaSuccess) return e;
    }
    return launch_pdl(route_assign_kernel, dim3(a.nb), dim3(kRouteThreads), sm3, s, a);
}

}  // namespace moe
