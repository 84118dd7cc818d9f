// Data-movement kernels of the layer: the dispatch row scatter, the RANK_MAJOR / FLAT
// pick gather and weighted local-pick reduction, the combine gather-reduce, and the
// one-time gate/up interleave of w1.  All are HBM-bound copies or reductions: one warp per
// (row, column chunk), 16-byte vector loads and stores, several loads in flight per lane.
//
// Sources: Mooncake EP guide, "Buffer.dispatch(...)" / "Buffer.combine(...)" (send each
// token row to the owners of its experts; return expert outputs by routing weight to the
// token's owner) and FlashInfer "MoE-EP implementation & usage", section 3 "Algorithm /
// layout contracts" (EXPERT_MAJOR reweights per token on combine; RANK_MAJOR / FLAT mask
// non-local picks to weight 0 and sum without weights across ranks).
#include <cuda_bf16.h>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kWarpsPerBlock = kCopyThreads / 32;

__device__ __forceinline__ uint4 ld_nc_v4(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ float4 ld_nc_f4(const float *p) {
    float4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}

// ---------------------------------------------------------------- dispatch row scatter
// x[t] is read once and written to each of its receive rows
// (EM: the slot of every kept pick; RM/FLAT: the row in every destination that got it).
// Rows are split into chunks of 32 lanes x kCopyU 16-byte vectors (1024 bf16 or 512 fp32
// columns); one warp handles one (row, chunk) so that even a 1024-token batch keeps
// thousands of warps and many loads in flight.
constexpr int kCopyU = 4;

struct CopyArgs {
    const uint16_t *x;
    uint16_t *recv;
    const int32_t *slot, *recv_row;
    int T, k, W, H, layout, nchunk;
    int64_t cap;
};

__global__ void __launch_bounds__(kCopyThreads) dispatch_copy_kernel(CopyArgs a) {
    __shared__ int64_t dst[kWarpsPerBlock][MOE_MAX_WORLD > MOE_MAX_TOPK ? MOE_MAX_WORLD : MOE_MAX_TOPK];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t gw = (int64_t)blockIdx.x * kWarpsPerBlock + warp;   // (token, chunk)
    const int64_t t = gw / a.nchunk;
    const int chunk = (int)(gw - t * a.nchunk);
    if (t >= a.T) return;
    const bool em = a.layout == MOE_LAYOUT_EXPERT_MAJOR;
    const int n = em ? a.k : a.W;
    int nd = 0;
    for (int q0 = 0; q0 < n; q0 += 32) {
        int q = q0 + lane;
        int64_t row = -1;
        if (q < n) {
            if (em) {
                row = a.slot[t * a.k + q];
            } else {
                int r = a.recv_row[t * a.W + q];
                row = r >= 0 ? (int64_t)q * a.cap + r : -1;
            }
        }
        unsigned bal = __ballot_sync(0xffffffffu, row >= 0);
        if (row >= 0) dst[warp][nd + __popc(bal & ((1u << lane) - 1u))] = row;
        nd += __popc(bal);
    }
    __syncwarp();
    const int nv = a.H / 8;   // uint4 per row
    const int c0 = chunk * 32 * kCopyU + lane;
    const uint4 *src = reinterpret_cast<const uint4 *>(a.x + t * a.H);
    uint4 v[kCopyU];
#pragma unroll
    for (int u = 0; u < kCopyU; ++u)
        if (c0 + 32 * u < nv) v[u] = ld_nc_v4(src + c0 + 32 * u);
    for (int d = 0; d < nd; ++d) {
        uint4 *o = reinterpret_cast<uint4 *>(a.recv + dst[warp][d] * a.H);
#pragma unroll
        for (int u = 0; u < kCopyU; ++u)
            if (c0 + 32 * u < nv) o[c0 + 32 * u] = v[u];
    }
}

// -------------------------------------------- RANK_MAJOR / FLAT: gather rows of the picks
// apick[p] = recv row of pick p (destination d = e / Le, row recv_row[t, d]), so the first
// GEMM reads the expert-grouped rows contiguously.
struct GatherArgs {
    const uint16_t *recv;
    uint16_t *apick;
    const int32_t *offsets, *pick_src, *recv_row;
    int E, Le, k, W, H, nchunk;
    int64_t P, cap;
};

__device__ __forceinline__ int expert_of_pick(const int32_t *offsets, int E, int p) {
    int lo = 0, hi = E - 1;   // largest e with offsets[e] <= p
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (offsets[mid] <= p) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

__global__ void __launch_bounds__(kCopyThreads) gather_picks_kernel(GatherArgs a) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t gw = (int64_t)blockIdx.x * kWarpsPerBlock + warp;   // (pick, chunk)
    const int64_t p = gw / a.nchunk;
    const int chunk = (int)(gw - p * a.nchunk);
    if (p >= a.P || p >= a.offsets[a.E]) return;
    const int e = expert_of_pick(a.offsets, a.E, (int)p);
    const int i = a.pick_src[p];
    const int t = i / a.k, d = e / a.Le;
    const int64_t row = (int64_t)d * a.cap + a.recv_row[(int64_t)t * a.W + d];
    const uint4 *src = reinterpret_cast<const uint4 *>(a.recv + row * a.H);
    uint4 *dst = reinterpret_cast<uint4 *>(a.apick + p * a.H);
    const int nv = a.H / 8;
    const int c0 = chunk * 32 * kCopyU + lane;
    uint4 v[kCopyU];
#pragma unroll
    for (int u = 0; u < kCopyU; ++u)
        if (c0 + 32 * u < nv) v[u] = ld_nc_v4(src + c0 + 32 * u);
#pragma unroll
    for (int u = 0; u < kCopyU; ++u)
        if (c0 + 32 * u < nv) dst[c0 + 32 * u] = v[u];
}

// ------------------------- RANK_MAJOR / FLAT: weighted reduction over a row's local picks
// expert_out[d*cap + r] = sum_j (ascending) recv_topk_w[d, r, j] * y(pick (t, j)) over the
// local picks j (recv_topk_idx >= 0); the others are masked to weight 0 (skipped).
struct ReduceArgs {
    const float *ypick;
    float *out;
    const int32_t *recv_count, *num_recv, *recv_src, *recv_topk_idx, *pick_pos;
    const float *recv_topk_w;
    int W, Tr, k, H, layout, nchunk;
    int64_t cap;
};

__global__ void __launch_bounds__(kCopyThreads) reduce_ranks_kernel(ReduceArgs a) {
    __shared__ int64_t src[kWarpsPerBlock][MOE_MAX_TOPK];
    __shared__ float wt[kWarpsPerBlock][MOE_MAX_TOPK];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t gw = (int64_t)blockIdx.x * kWarpsPerBlock + warp;   // (row, chunk)
    const int64_t gr = gw / a.nchunk;                                 // d*cap + r
    const int chunk = (int)(gw - gr * a.nchunk);
    if (gr >= (int64_t)a.W * a.cap) return;
    const int d = (int)(gr / a.cap);
    const int r = (int)(gr % a.cap);
    bool used = a.layout == MOE_LAYOUT_RANK_MAJOR
                    ? (r % a.Tr) < a.recv_count[d * a.W + r / a.Tr]
                    : r < a.num_recv[d];
    if (!used) return;
    const int t = a.recv_src[gr];
    int n = 0;
    {
        int j = lane;
        int64_t s = -1;
        float w = 0.f;
        if (j < a.k && a.recv_topk_idx[gr * a.k + j] >= 0) {
            s = a.pick_pos[(int64_t)t * a.k + j];
            w = a.recv_topk_w[gr * a.k + j];
        }
        unsigned bal = __ballot_sync(0xffffffffu, s >= 0);
        if (s >= 0) {
            int q = __popc(bal & ((1u << lane) - 1u));
            src[warp][q] = s;
            wt[warp][q] = w;
        }
        n = __popc(bal);
    }
    __syncwarp();
    const int nv = a.H / 4;
    const int c0 = chunk * 32 * kCopyU + lane;
    float4 acc[kCopyU];
#pragma unroll
    for (int u = 0; u < kCopyU; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int q = 0; q < n; ++q) {
        const float *row = a.ypick + src[warp][q] * a.H;
        const float w = wt[warp][q];
        float4 y[kCopyU];
#pragma unroll
        for (int u = 0; u < kCopyU; ++u)
            if (c0 + 32 * u < nv) y[u] = ld_nc_f4(row + 4 * (c0 + 32 * u));
#pragma unroll
        for (int u = 0; u < kCopyU; ++u) {
            acc[u].x = fmaf(w, y[u].x, acc[u].x);
            acc[u].y = fmaf(w, y[u].y, acc[u].y);
            acc[u].z = fmaf(w, y[u].z, acc[u].z);
            acc[u].w = fmaf(w, y[u].w, acc[u].w);
        }
    }
    float4 *o = reinterpret_cast<float4 *>(a.out + gr * a.H);
#pragma unroll
    for (int u = 0; u < kCopyU; ++u)
        if (c0 + 32 * u < nv) o[c0 + 32 * u] = acc[u];
}

// ----------------------------------------------------------------------------- combine
// EM:      out[t] = bf16( sum_j w[t, j] * expert_out[slot[t, j]] ), kept picks, ascending j
// RM/FLAT: out[t] = bf16( sum_d expert_out[d*cap + recv_row[t, d]] ), ascending d
struct CombineArgs {
    const float *eo;
    const float *topk_w;
    const int32_t *slot, *recv_row;
    uint16_t *out;
    int T, k, W, H, layout, nchunk;
    int64_t cap;
};

__global__ void __launch_bounds__(kCopyThreads) combine_kernel(CombineArgs a) {
    __shared__ int64_t src[kWarpsPerBlock][MOE_MAX_WORLD > MOE_MAX_TOPK ? MOE_MAX_WORLD : MOE_MAX_TOPK];
    __shared__ float wt[kWarpsPerBlock][MOE_MAX_WORLD > MOE_MAX_TOPK ? MOE_MAX_WORLD : MOE_MAX_TOPK];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t gw = (int64_t)blockIdx.x * kWarpsPerBlock + warp;   // (token, chunk)
    const int64_t t = gw / a.nchunk;
    const int chunk = (int)(gw - t * a.nchunk);
    if (t >= a.T) return;
    const bool em = a.layout == MOE_LAYOUT_EXPERT_MAJOR;
    const int n = em ? a.k : a.W;
    int ns = 0;
    for (int q0 = 0; q0 < n; q0 += 32) {
        int q = q0 + lane;
        int64_t row = -1;
        float w = 1.f;
        if (q < n) {
            if (em) {
                row = a.slot[t * a.k + q];
                w = a.topk_w[t * a.k + q];
            } else {
                int r = a.recv_row[t * a.W + q];
                row = r >= 0 ? (int64_t)q * a.cap + r : -1;
            }
        }
        unsigned bal = __ballot_sync(0xffffffffu, row >= 0);
        if (row >= 0) {
            int i = ns + __popc(bal & ((1u << lane) - 1u));
            src[warp][i] = row;
            wt[warp][i] = w;
        }
        ns += __popc(bal);
    }
    __syncwarp();
    const int nv = a.H / 4;   // float4 per row
    const int c0 = chunk * 32 * kCopyU + lane;
    float4 acc[kCopyU];
#pragma unroll
    for (int u = 0; u < kCopyU; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int q = 0; q < ns; ++q) {
        const float *row = a.eo + src[warp][q] * a.H;
        const float w = wt[warp][q];
        float4 y[kCopyU];
#pragma unroll
        for (int u = 0; u < kCopyU; ++u)
            if (c0 + 32 * u < nv) y[u] = ld_nc_f4(row + 4 * (c0 + 32 * u));
#pragma unroll
        for (int u = 0; u < kCopyU; ++u) {
            if (em) {
                acc[u].x = fmaf(w, y[u].x, acc[u].x);
                acc[u].y = fmaf(w, y[u].y, acc[u].y);
                acc[u].z = fmaf(w, y[u].z, acc[u].z);
                acc[u].w = fmaf(w, y[u].w, acc[u].w);
            } else {
                acc[u].x += y[u].x;
                acc[u].y += y[u].y;
                acc[u].z += y[u].z;
                acc[u].w += y[u].w;
            }
        }
    }
    uint2 *o = reinterpret_cast<uint2 *>(a.out + t * a.H);
#pragma unroll
    for (int u = 0; u < kCopyU; ++u) {
        if (c0 + 32 * u >= nv) continue;
        __nv_bfloat162 lo = __floats2bfloat162_rn(acc[u].x, acc[u].y);
        __nv_bfloat162 hi = __floats2bfloat162_rn(acc[u].z, acc[u].w);
        uint2 v;
        v.x = *reinterpret_cast<uint32_t *>(&lo);
        v.y = *reinterpret_cast<uint32_t *>(&hi);
        o[c0 + 32 * u] = v;
    }
}

// ------------------------------------------------------------ w1 gate/up interleave
// w1p row (e, 256*b + q) = w1 row (e, 128*b + q) for q < 128 (gate), and
// w1 row (e, I + 128*b + q - 128) for q >= 128 (up).
__global__ void __launch_bounds__(kCopyThreads) prepare_w1_kernel(const uint16_t *w1, uint16_t *w1p,
                                                                  int64_t rows, int I, int H) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t rp = (int64_t)blockIdx.x * kWarpsPerBlock + warp;
    if (rp >= rows) return;
    const int64_t e = rp / (2 * I);
    const int local = (int)(rp % (2 * I));
    const int b = local / 256, q = local % 256;
    const int src_local = q < 128 ? b * 128 + q : I + b * 128 + (q - 128);
    const uint4 *s = reinterpret_cast<const uint4 *>(w1 + (e * 2 * I + src_local) * (int64_t)H);
    uint4 *d = reinterpret_cast<uint4 *>(w1p + rp * (int64_t)H);
    for (int c = lane; c < H / 8; c += 32) d[c] = ld_nc_v4(s + c);
}

inline unsigned blocks_for(int64_t warps) {
    return (unsigned)((warps + kWarpsPerBlock - 1) / kWarpsPerBlock);
}

}  // namespace

cudaError_t launch_dispatch_copy(const Routing &r, const uint16_t *x, cudaStream_t s) {
    const Plan &p = *r.p;
    if (p.T == 0) return cudaSuccess;
    const int nchunk = (int)((p.H / 8 + 32 * kCopyU - 1) / (32 * kCopyU));
    CopyArgs a{x, r.recv_x, r.slot, r.recv_row, (int)p.T, (int)p.k, (int)p.W, (int)p.H,
               p.layout, nchunk, p.cap};
    dispatch_copy_kernel<<<blocks_for(p.T * nchunk), kCopyThreads, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_gather_picks(const Routing &r, cudaStream_t s) {
    const Plan &p = *r.p;
    if (p.P == 0) return cudaSuccess;
    const int nchunk = (int)((p.H / 8 + 32 * kCopyU - 1) / (32 * kCopyU));
    GatherArgs a{r.recv_x, r.apick, r.offsets, r.pick_src, r.recv_row,
                 (int)p.E, (int)(p.E / p.W), (int)p.k, (int)p.W, (int)p.H, nchunk, p.P, p.cap};
    gather_picks_kernel<<<blocks_for(p.P * nchunk), kCopyThreads, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_reduce_ranks(const Routing &r, float *expert_out, cudaStream_t s) {
    const Plan &p = *r.p;
    if (p.T == 0) return cudaSuccess;
    const int nchunk = (int)((p.H / 4 + 32 * kCopyU - 1) / (32 * kCopyU));
    ReduceArgs a{r.ypick, expert_out, r.recv_count, r.num_recv, r.recv_src, r.recv_topk_idx,
                 r.pick_pos, r.recv_topk_w, (int)p.W, (int)p.Tr, (int)p.k, (int)p.H, p.layout,
                 nchunk, p.cap};
    reduce_ranks_kernel<<<blocks_for(p.W * p.cap * nchunk), kCopyThreads, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_combine(const Routing &r, const float *expert_out, const float *topk_w,
                           uint16_t *out, cudaStream_t s) {
    const Plan &p = *r.p;
    if (p.T == 0) return cudaSuccess;
    const int nchunk = (int)((p.H / 4 + 32 * kCopyU - 1) / (32 * kCopyU));
    CombineArgs a{expert_out, topk_w, r.slot, r.recv_row, out, (int)p.T, (int)p.k, (int)p.W,
                  (int)p.H, p.layout, nchunk, p.cap};
    combine_kernel<<<blocks_for(p.T * nchunk), kCopyThreads, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_prepare_w1(const moe_geom &g, const uint16_t *w1, uint16_t *w1p,
                              cudaStream_t s) {
    int64_t rows = (int64_t)g.num_experts * 2 * g.intermediate;
    prepare_w1_kernel<<<blocks_for(rows), kCopyThreads, 0, s>>>(w1, w1p, rows, g.intermediate,
                                                               g.hidden);
    return cudaGetLastError();
}

}  // namespace moe
