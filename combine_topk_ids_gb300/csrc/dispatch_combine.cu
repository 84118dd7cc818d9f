// Data-movement kernels of the layer: the dispatch row scatter (bf16, or quantised to FP8
// on the way; for RANK_MAJOR / FLAT it also writes the rows in pick-list order for the
// first GEMM), the RANK_MAJOR / FLAT weighted local-pick reduction, the combine
// gather-reduce, and the one-time weight preparations (gate/up interleave of w1,
// FP8 block quantisation).  All are HBM-bound copies or reductions: one warp per
// (row, column chunk), 16-byte vector loads and stores, several loads in flight per lane.
//
// Sources: Mooncake EP guide, "Buffer.dispatch(...)" / "Buffer.combine(...)" (send each
// token row to the owners of its experts; return expert outputs by routing weight to the
// token's owner) and FlashInfer "MoE-EP implementation & usage", section 3 "Algorithm /
// layout contracts" (EXPERT_MAJOR reweights per token on combine; RANK_MAJOR / FLAT mask
// non-local picks to weight 0 and sum without weights across ranks).
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <atomic>

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

__device__ __forceinline__ uint2 ld_nc_v2(const void *p) {
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Four consecutive elements (index elem, a multiple of 4) of a float32 or bf16 row as fp32.
template <bool BF16>
__device__ __forceinline__ float4 ld_row4(const void *base, int64_t elem) {
    if (BF16) {
        const uint2 v = ld_nc_v2(reinterpret_cast<const uint16_t *>(base) + elem);
        return make_float4(bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y));
    }
    return ld_nc_f4(reinterpret_cast<const float *>(base) + elem);
}

// ---------------------------------------------------------------- dispatch row scatter
// x[t] is read once and written to each of its receive rows (EM: the slot of every kept
// pick; RM/FLAT: the row in every destination that got it, and the pick-ordered row of
// every kept pick, apick[pick_pos[t, j]], which the first GEMM reads contiguously per
// expert).  Rows are split into chunks of 32 lanes x kCopyU 16-byte vectors (1024 bf16 or
// 512 fp32 columns); one warp handles one (row, chunk) so that even a 1024-token batch
// keeps thousands of warps and many loads in flight.
constexpr int kCopyU = 4;
constexpr int kMaxDst = MOE_MAX_WORLD + MOE_MAX_TOPK;   // receive rows + pick rows of a token

struct CopyArgs {
    const uint16_t *x;
    uint16_t *recv;
    uint16_t *apick;   // RM/FLAT: [P, H] rows in pick-list order
    const int32_t *slot, *recv_row, *pick_pos;
    // RM/FLAT: received local ids and weights (read), the per-pick direct rows (written)
    const int32_t *recv_topk_idx;
    const float *recv_topk_w;
    int32_t *direct_row;
    float *direct_w;
    int T, k, W, H, layout, nchunk;
    int64_t cap;
};

// RM/FLAT: for every kept pick of token t, direct_row[p] = the received row d*cap + r
// when the pick is the only local pick of that row (its expert_out row is then
// weight * y, written by the second GEMM), else -1; direct_w[p] = its weight.  One warp
// (lane j = pick j) per token.
__device__ __forceinline__ void mark_direct_picks(const CopyArgs &a, int64_t t, int lane) {
    for (int d = 0; d < a.W; ++d) {
        const int r = a.recv_row[t * a.W + d];
        if (r < 0) continue;
        const int64_t gr = (int64_t)d * a.cap + r;
        const bool local = lane < a.k && a.recv_topk_idx[gr * a.k + lane] >= 0;
        const unsigned bal = __ballot_sync(0xffffffffu, local);
        if (!local) continue;
        const int p = a.pick_pos[t * a.k + lane];
        if (p < 0) continue;
        const bool single = __popc(bal) == 1;
        a.direct_row[p] = single ? (int32_t)gr : -1;
        if (single) a.direct_w[p] = a.recv_topk_w[gr * a.k + lane];
    }
}

// Appends to list[n..] the row indices of token t's destinations that pass `pick`: lanes
// scan q in [0, count), row_of(q) < 0 means none.  Returns the new length.
template <typename RowOf>
__device__ __forceinline__ int collect_rows(int64_t *list, int n, int count, int lane, RowOf row_of) {
    for (int q0 = 0; q0 < count; q0 += 32) {
        const int q = q0 + lane;
        const int64_t row = q < count ? row_of(q) : -1;
        const unsigned bal = __ballot_sync(0xffffffffu, row >= 0);
        if (row >= 0) list[n + __popc(bal & ((1u << lane) - 1u))] = row;
        n += __popc(bal);
    }
    return n;
}

__global__ void __launch_bounds__(kCopyThreads) dispatch_copy_kernel(CopyArgs a) {
    pdl_begin();   // after the previous kernel in the stream (programmatic launch)
    __shared__ int64_t dst[kWarpsPerBlock][kMaxDst];   // element offset of each target row
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t gw = (int64_t)blockIdx.x * kWarpsPerBlock + warp;   // (token, chunk)
    const int64_t t = gw / a.nchunk;
    const int chunk = (int)(gw - t * a.nchunk);
    if (t >= a.T) return;
    int nd;
    int np = 0;   // the last np entries are rows of apick
    if (a.layout == MOE_LAYOUT_EXPERT_MAJOR) {
        nd = collect_rows(dst[warp], 0, a.k, lane, [&](int q) -> int64_t {
            const int s = a.slot[t * a.k + q];
            return s >= 0 ? (int64_t)s * a.H : -1;
        });
    } else {
        nd = collect_rows(dst[warp], 0, a.W, lane, [&](int q) -> int64_t {
            const int r = a.recv_row[t * a.W + q];
            return r >= 0 ? ((int64_t)q * a.cap + r) * a.H : -1;
        });
        const int n0 = nd;
        nd = collect_rows(dst[warp], nd, a.k, lane, [&](int q) -> int64_t {
            const int p = a.pick_pos[t * a.k + q];
            return p >= 0 ? (int64_t)p * a.H : -1;
        });
        np = nd - n0;
        if (chunk == 0 && a.direct_row) mark_direct_picks(a, t, lane);
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
        uint4 *o = reinterpret_cast<uint4 *>((d < nd - np ? a.recv : a.apick) + dst[warp][d]);
#pragma unroll
        for (int u = 0; u < kCopyU; ++u)
            if (c0 + 32 * u < nv) o[c0 + 32 * u] = v[u];
    }
}

// ------------------------- RANK_MAJOR / FLAT: weighted reduction over a row's local picks
// expert_out[d*cap + r] = sum_j (ascending) recv_topk_w[d, r, j] * y(pick (t, j)) over the
// local picks j (recv_topk_idx >= 0); the others are masked to weight 0 (skipped).
struct ReduceArgs {
    const void *ypick;   // float32 or bf16 rows (the kernel's BF16 parameter)
    void *out;
    int skip_single;     // rows with one local pick were written by the second GEMM
    const int32_t *recv_count, *num_recv, *recv_src, *recv_topk_idx, *pick_pos;
    const float *recv_topk_w;
    int W, Tr, k, H, layout, nchunk;
    int64_t cap;
};

// G consecutive elements (16 bytes: 4 float32 or 8 bf16) of a row as fp32, and back.
template <bool BF16>
__device__ __forceinline__ void ld_group(const void *base, int64_t elem, float (&f)[BF16 ? 8 : 4]) {
    if (BF16) {
        const uint4 v = ld_nc_v4(reinterpret_cast<const uint16_t *>(base) + elem);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = bf16_lo(w[i]);
            f[2 * i + 1] = bf16_hi(w[i]);
        }
    } else {
        const float4 v = ld_nc_f4(reinterpret_cast<const float *>(base) + elem);
        f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
    }
}

template <bool BF16>
__device__ __forceinline__ void st_group(void *base, int64_t elem, const float (&f)[BF16 ? 8 : 4]) {
    if (BF16) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 b = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
            w[i] = *reinterpret_cast<uint32_t *>(&b);
        }
        *reinterpret_cast<uint4 *>(reinterpret_cast<uint16_t *>(base) + elem) = make_uint4(w[0], w[1], w[2], w[3]);
    } else {
        *reinterpret_cast<float4 *>(reinterpret_cast<float *>(base) + elem) = make_float4(f[0], f[1], f[2], f[3]);
    }
}

template <bool BF16>
__global__ void __launch_bounds__(kCopyThreads, 3) reduce_ranks_kernel(ReduceArgs a) {
    pdl_begin();   // after the previous kernel in the stream (programmatic launch)
    constexpr int G = BF16 ? 8 : 4;   // elements per 16-byte group
    constexpr int U = BF16 ? 2 : 4;   // groups per lane and pick in flight (<= 85 registers)
    __shared__ int64_t src[kWarpsPerBlock][MOE_MAX_TOPK];
    __shared__ float wt[kWarpsPerBlock][MOE_MAX_TOPK];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t rows = (int64_t)a.W * a.cap;
    const int64_t nwarps = (int64_t)gridDim.x * kWarpsPerBlock;
    const int ng = a.H / G;   // groups per row
    // grid-stride over received rows d*cap + r, one warp per row: a row's routing is read
    // once, unused rows and rows the second GEMM already wrote cost a few loads
    for (int64_t gr = (int64_t)blockIdx.x * kWarpsPerBlock + warp; gr < rows; gr += nwarps) {
        const int d = (int)(gr / a.cap);
        const int r = (int)(gr - (int64_t)d * a.cap);
        const bool used = a.layout == MOE_LAYOUT_RANK_MAJOR
                              ? (r % a.Tr) < a.recv_count[d * a.W + r / a.Tr]
                              : r < a.num_recv[d];
        if (!used) continue;   // warp-uniform
        const int t = a.recv_src[gr];
        int64_t s = -1;
        float w = 0.f;
        if (lane < a.k && a.recv_topk_idx[gr * a.k + lane] >= 0) {
            s = a.pick_pos[(int64_t)t * a.k + lane];
            w = a.recv_topk_w[gr * a.k + lane];
        }
        const unsigned bal = __ballot_sync(0xffffffffu, s >= 0);
        const int n = __popc(bal);
        if (n == 1 && a.skip_single) continue;   // warp-uniform
        __syncwarp();   // the previous row's readers are done with src / wt
        if (s >= 0) {
            const int q = __popc(bal & ((1u << lane) - 1u));
            src[warp][q] = s;
            wt[warp][q] = w;
        }
        __syncwarp();
        for (int g0 = lane; g0 < ng; g0 += 32 * U) {
            float acc[U][G];
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
                for (int i = 0; i < G; ++i) acc[u][i] = 0.f;
            // two picks' rows in flight at a time; the sum stays in ascending pick order
            for (int q = 0; q < n; q += 2) {
                const bool two = q + 1 < n;
                const int64_t row0 = src[warp][q] * a.H;
                const int64_t row1 = two ? src[warp][q + 1] * a.H : row0;
                float y0[U][G], y1[U][G];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int g = g0 + 32 * u;
                    if (g < ng) {
                        ld_group<BF16>(a.ypick, row0 + (int64_t)G * g, y0[u]);
                        if (two) ld_group<BF16>(a.ypick, row1 + (int64_t)G * g, y1[u]);
                    }
                }
                const float w0 = wt[warp][q];
#pragma unroll
                for (int u = 0; u < U; ++u)
#pragma unroll
                    for (int i = 0; i < G; ++i) acc[u][i] = fmaf(w0, y0[u][i], acc[u][i]);
                if (two) {
                    const float w1 = wt[warp][q + 1];
#pragma unroll
                    for (int u = 0; u < U; ++u)
#pragma unroll
                        for (int i = 0; i < G; ++i) acc[u][i] = fmaf(w1, y1[u][i], acc[u][i]);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int g = g0 + 32 * u;
                if (g < ng) st_group<BF16>(a.out, gr * a.H + (int64_t)G * g, acc[u]);
            }
        }
    }
}

// ----------------------------------------------------------------------------- combine
// EM:      out[t] = bf16( sum_j w[t, j] * expert_out[slot[t, j]] ), kept picks, ascending j
// RM/FLAT: out[t] = bf16( sum_d expert_out[d*cap + recv_row[t, d]] ), ascending d
struct CombineArgs {
    const void *eo;      // float32 or bf16 rows (the kernel's BF16 parameter)
    const float *topk_w;
    const int32_t *slot, *recv_row;
    uint16_t *out;
    int T, k, W, H, layout, nchunk;
    int64_t cap;
};

template <bool BF16>
__global__ void __launch_bounds__(kCopyThreads) combine_kernel(CombineArgs a) {
    pdl_begin();   // after the previous kernel in the stream (programmatic launch)
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
        const int64_t row = src[warp][q] * a.H;
        const float w = wt[warp][q];
        float4 y[kCopyU];
#pragma unroll
        for (int u = 0; u < kCopyU; ++u)
            if (c0 + 32 * u < nv) y[u] = ld_row4<BF16>(a.eo, row + 4 * (c0 + 32 * u));
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

// RANK_MAJOR / FLAT combine that also forms the local-pick sums of received rows with
// several local picks, in place of the rank reduction: for token t and each destination d
// (ascending) that received it, row r, the term is expert_out[d*cap + r] when the row has
// one local pick (the second GEMM wrote it), else the fmaf chain over its local picks j
// ascending of recv_topk_w * y_j (y_j: the pick's second-GEMM row), rounded as the
// reduction stores it (bf16 rows: to bf16); out[t] = bf16(sum of the terms).  These are the
// reduction's and combine_kernel's operations in the same order, so the output is the
// same bit for bit; expert_out's multi-pick rows are left unwritten.
struct FusedCombineArgs {
    const void *eo, *ypick;   // float32 or bf16 rows (the kernel's BF16 parameter)
    const int32_t *recv_row, *recv_topk_idx, *pick_pos;
    const float *recv_topk_w;
    uint16_t *out;
    int T, k, W, H, nchunk;
    int64_t cap;
};

template <bool BF16>
__global__ void __launch_bounds__(kCopyThreads) combine_fused_kernel(FusedCombineArgs a) {
    pdl_begin();   // after the previous kernel in the stream (programmatic launch)
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t gw = (int64_t)blockIdx.x * kWarpsPerBlock + warp;   // (token, chunk)
    const int64_t t = gw / a.nchunk;
    const int chunk = (int)(gw - t * a.nchunk);
    if (t >= a.T) return;
    const int nv = a.H / 4;   // float4 per row
    const int c0 = chunk * 32 * kCopyU + lane;
    float4 acc[kCopyU];
#pragma unroll
    for (int u = 0; u < kCopyU; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int d = 0; d < a.W; ++d) {
        const int r = a.recv_row[t * a.W + d];   // the same for every lane
        if (r < 0) continue;
        const int64_t gr = (int64_t)d * a.cap + r;
        int64_t p = -1;   // lane j: pick j's position in the pick list if it is local to d
        float w = 0.f;
        if (lane < a.k && a.recv_topk_idx[gr * a.k + lane] >= 0) {
            p = a.pick_pos[t * a.k + lane];
            w = a.recv_topk_w[gr * a.k + lane];
        }
        unsigned bal = __ballot_sync(0xffffffffu, p >= 0);
        float4 sd[kCopyU];
        if (__popc(bal) == 1) {
#pragma unroll
            for (int u = 0; u < kCopyU; ++u)
                if (c0 + 32 * u < nv) sd[u] = ld_row4<BF16>(a.eo, gr * a.H + 4 * (c0 + 32 * u));
        } else {
#pragma unroll
            for (int u = 0; u < kCopyU; ++u) sd[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            while (bal) {
                const int j = __ffs(bal) - 1;
                bal &= bal - 1;
                const int64_t pj = __shfl_sync(0xffffffffu, p, j);
                const float wj = __shfl_sync(0xffffffffu, w, j);
                float4 y[kCopyU];
#pragma unroll
                for (int u = 0; u < kCopyU; ++u)
                    if (c0 + 32 * u < nv) y[u] = ld_row4<BF16>(a.ypick, pj * a.H + 4 * (c0 + 32 * u));
#pragma unroll
                for (int u = 0; u < kCopyU; ++u) {
                    sd[u].x = fmaf(wj, y[u].x, sd[u].x);
                    sd[u].y = fmaf(wj, y[u].y, sd[u].y);
                    sd[u].z = fmaf(wj, y[u].z, sd[u].z);
                    sd[u].w = fmaf(wj, y[u].w, sd[u].w);
                }
            }
            if (BF16) {   // the reduction stores bf16 rows
#pragma unroll
                for (int u = 0; u < kCopyU; ++u)
                    sd[u] = make_float4(__bfloat162float(__float2bfloat16_rn(sd[u].x)),
                                        __bfloat162float(__float2bfloat16_rn(sd[u].y)),
                                        __bfloat162float(__float2bfloat16_rn(sd[u].z)),
                                        __bfloat162float(__float2bfloat16_rn(sd[u].w)));
            }
        }
#pragma unroll
        for (int u = 0; u < kCopyU; ++u) {
            acc[u].x += sd[u].x;
            acc[u].y += sd[u].y;
            acc[u].z += sd[u].z;
            acc[u].w += sd[u].w;
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

// ------------------------------------------------------------------------------- FP8
// Quantisation rule of a block with largest magnitude amax (float32, IEEE rounding):
// a = max(amax, 2^-100), scale = a / 448, inv = 448 / a, code = e4m3_rne_satfinite(v * inv).
__device__ __forceinline__ void fp8_scale(float amax, float &scale, float &inv) {
    const float a = fmaxf(amax, 0x1p-100f);
    scale = __fdiv_rn(a, 448.0f);
    inv = __fdiv_rn(448.0f, a);
}

// Four e4m3 codes (round to nearest even, saturating) of v0..v3 * inv; v0 in the lowest byte.
__device__ __forceinline__ uint32_t e4m3x4(float v0, float v1, float v2, float v3, float inv) {
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(__fmul_rn(v0, inv), __fmul_rn(v1, inv)),
                                                 __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(__fmul_rn(v2, inv), __fmul_rn(v3, inv)),
                                                 __NV_SATFINITE, __NV_E4M3);
    return lo | (hi << 16);
}

// FP8 dispatch: like dispatch_copy_kernel, but each 128-column block of x[t] is quantised
// once (16 lanes x 8 columns: the half-warp reduces amax) and the e4m3 codes plus the
// block scale are written to every receive row of the token (and for RM/FLAT to its
// pick-ordered rows).
struct QuantCopyArgs {
    const uint16_t *x;
    uint8_t *recv;          // [nrecv, H] codes
    float *recv_scales;     // [H/128][nrecv]
    uint8_t *apick;         // RM/FLAT: [P, H] codes in pick-list order
    float *apick_scales;    // RM/FLAT: [H/128][P]
    const int32_t *slot, *recv_row, *pick_pos;
    int T, k, W, H, layout, nchunk;
    int64_t cap, nrecv, P;
};

__global__ void __launch_bounds__(kCopyThreads) dispatch_quant_kernel(QuantCopyArgs a) {
    pdl_begin();   // after the previous kernel in the stream (programmatic launch)
    __shared__ int64_t dst[kWarpsPerBlock][kMaxDst];   // row index of each target row
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t gw = (int64_t)blockIdx.x * kWarpsPerBlock + warp;   // (token, chunk)
    const int64_t t = gw / a.nchunk;
    const int chunk = (int)(gw - t * a.nchunk);
    if (t >= a.T) return;
    int nd;
    int np = 0;   // the last np entries are rows of apick
    if (a.layout == MOE_LAYOUT_EXPERT_MAJOR) {
        nd = collect_rows(dst[warp], 0, a.k, lane, [&](int q) -> int64_t { return a.slot[t * a.k + q]; });
    } else {
        nd = collect_rows(dst[warp], 0, a.W, lane, [&](int q) -> int64_t {
            const int r = a.recv_row[t * a.W + q];
            return r >= 0 ? (int64_t)q * a.cap + r : -1;
        });
        const int n0 = nd;
        nd = collect_rows(dst[warp], nd, a.k, lane, [&](int q) -> int64_t { return a.pick_pos[t * a.k + q]; });
        np = nd - n0;
    }
    __syncwarp();
    const int nv = a.H / 8;   // 8-column vectors per row; a 128-column block is 16 of them
    const int c0 = chunk * 32 * kCopyU + lane;
    const uint4 *src = reinterpret_cast<const uint4 *>(a.x + t * a.H);
    uint2 q[kCopyU];
    float sc[kCopyU];
#pragma unroll
    for (int u = 0; u < kCopyU; ++u) {
        const int c = c0 + 32 * u;
        // c < nv is the same for the 16 lanes of a block (H is a multiple of 128)
        const uint4 v = c < nv ? ld_nc_v4(src + c) : make_uint4(0, 0, 0, 0);
        float f[8] = {bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y),
                      bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w)};
        float m = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(f[i]));
#pragma unroll
        for (int o = 8; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float inv;
        fp8_scale(m, sc[u], inv);
        q[u].x = e4m3x4(f[0], f[1], f[2], f[3], inv);
        q[u].y = e4m3x4(f[4], f[5], f[6], f[7], inv);
    }
    for (int d = 0; d < nd; ++d) {
        const int64_t row = dst[warp][d];
        const bool pick = d >= nd - np;
        uint2 *o = reinterpret_cast<uint2 *>((pick ? a.apick : a.recv) + row * a.H);
        float *so = (pick ? a.apick_scales : a.recv_scales) + row;
        const int64_t sstride = pick ? a.P : a.nrecv;
#pragma unroll
        for (int u = 0; u < kCopyU; ++u) {
            const int c = c0 + 32 * u;
            if (c < nv) {
                o[c] = q[u];
                if ((lane & 15) == 0) so[(int64_t)(c >> 4) * sstride] = sc[u];
            }
        }
    }
}

// 128x128-block quantisation of bf16 weights [E, R, C]: one CTA per block, thread
// (r, h) = (tid / 2, tid % 2) owns 64 columns of block row r.  With w1_inter = I > 0 the
// output row blocks are the gate/up interleave of moe_prepare_weights (gate block j ->
// 2j, up block j -> 2j + 1); scales [E, R/128, C/128] follow the same block order.
__global__ void __launch_bounds__(256) quantize_blocks_kernel(const uint16_t *w, uint8_t *q, float *sc,
                                                              int64_t R, int64_t C, int64_t w1_inter) {
    __shared__ float red[8];
    const int64_t RB = R / 128, CB = C / 128;
    const int64_t bid = blockIdx.x;
    const int64_t e = bid / (RB * CB);
    const int64_t rem = bid - e * RB * CB;
    const int64_t rb = rem / CB, cb = rem - (rem / CB) * CB;
    const int r = threadIdx.x >> 1, h = threadIdx.x & 1;
    const uint4 *src = reinterpret_cast<const uint4 *>(w + (e * R + rb * 128 + r) * C + cb * 128 + h * 64);
    float f[64];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint4 v = ld_nc_v4(src + i);
        f[8 * i + 0] = bf16_lo(v.x); f[8 * i + 1] = bf16_hi(v.x);
        f[8 * i + 2] = bf16_lo(v.y); f[8 * i + 3] = bf16_hi(v.y);
        f[8 * i + 4] = bf16_lo(v.z); f[8 * i + 5] = bf16_hi(v.z);
        f[8 * i + 6] = bf16_lo(v.w); f[8 * i + 7] = bf16_hi(v.w);
    }
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < 64; ++i) m = fmaxf(m, fabsf(f[i]));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    m = red[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) m = fmaxf(m, red[i]);
    float scale, inv;
    fp8_scale(m, scale, inv);
    int64_t orb = rb;
    if (w1_inter > 0) {
        const int64_t IB = w1_inter / 128;
        orb = rb < IB ? 2 * rb : 2 * (rb - IB) + 1;
    }
    uint4 *dst = reinterpret_cast<uint4 *>(q + (e * R + orb * 128 + r) * C + cb * 128 + h * 64);
#pragma unroll
    for (int i = 0; i < 4; ++i)
        dst[i] = make_uint4(e4m3x4(f[16 * i + 0], f[16 * i + 1], f[16 * i + 2], f[16 * i + 3], inv),
                            e4m3x4(f[16 * i + 4], f[16 * i + 5], f[16 * i + 6], f[16 * i + 7], inv),
                            e4m3x4(f[16 * i + 8], f[16 * i + 9], f[16 * i + 10], f[16 * i + 11], inv),
                            e4m3x4(f[16 * i + 12], f[16 * i + 13], f[16 * i + 14], f[16 * i + 15], inv));
    if (threadIdx.x == 0) sc[(e * RB + orb) * CB + cb] = scale;
}

// Gate/up interleave of FP8 w1 codes [E, 2I, H] (row permutation of prepare_w1_kernel)
// and of its block scales [E, 2I/128, H/128].
__global__ void __launch_bounds__(kCopyThreads) prepare_w1_fp8_kernel(const uint8_t *w1, const float *s1,
                                                                      uint8_t *w1p, float *s1p,
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
    for (int c = lane; c < H / 16; c += 32) d[c] = ld_nc_v4(s + c);
    if (local % 128 == 0) {   // first row of a 128-row block: move the block's scales
        const int CB = H / 128;
        const float *ss = s1 + (e * (2 * I / 128) + src_local / 128) * CB;
        float *ds = s1p + (e * (2 * I / 128) + local / 128) * CB;
        for (int c = lane; c < CB; c += 32) ds[c] = ss[c];
    }
}

inline unsigned blocks_for(int64_t warps) {
    return (unsigned)((warps + kWarpsPerBlock - 1) / kWarpsPerBlock);
}

}  // namespace

cudaError_t launch_dispatch_copy(const Routing &r, const uint16_t *x, cudaStream_t s) {
    const Plan &p = *r.p;
    if (p.T == 0) return cudaSuccess;
    const int nchunk = (int)((p.H / 8 + 32 * kCopyU - 1) / (32 * kCopyU));
    CopyArgs a{x, r.recv_x, r.apick, r.slot, r.recv_row, r.pick_pos, r.recv_topk_idx, r.recv_topk_w,
               r.direct_row, r.direct_w, (int)p.T, (int)p.k, (int)p.W, (int)p.H, p.layout, nchunk, p.cap};
    return launch_pdl(dispatch_copy_kernel, dim3(blocks_for(p.T * nchunk)), dim3(kCopyThreads), 0, s, a);
}

cudaError_t launch_combine_fused(const Routing &r, const void *expert_out, uint16_t *out, cudaStream_t s) {
    const Plan &p = *r.p;
    if (p.T == 0) return cudaSuccess;
    const int nchunk = (int)((p.H / 4 + 32 * kCopyU - 1) / (32 * kCopyU));
    FusedCombineArgs a{expert_out, r.ypick, r.recv_row, r.recv_topk_idx, r.pick_pos, r.recv_topk_w, out,
                       (int)p.T, (int)p.k, (int)p.W, (int)p.H, nchunk, p.cap};
    if (p.eo_bf16)
        return launch_pdl(combine_fused_kernel<true>, dim3(blocks_for(p.T * nchunk)), dim3(kCopyThreads), 0, s, a);
    return launch_pdl(combine_fused_kernel<false>, dim3(blocks_for(p.T * nchunk)), dim3(kCopyThreads), 0, s, a);
}

cudaError_t launch_reduce_ranks(const Routing &r, void *expert_out, bool skip_single, cudaStream_t s) {
    const Plan &p = *r.p;
    if (p.T == 0) return cudaSuccess;
    const int nchunk = (int)((p.H / 4 + 32 * kCopyU - 1) / (32 * kCopyU));
    ReduceArgs a{r.ypick, expert_out, skip_single ? 1 : 0, r.recv_count, r.num_recv, r.recv_src, r.recv_topk_idx,
                 r.pick_pos, r.recv_topk_w, (int)p.W, (int)p.Tr, (int)p.k, (int)p.H, p.layout,
                 nchunk, p.cap};
    // grid-stride over rows: no more blocks than can be resident at once, so that no block
    // starts its rows after the others have finished theirs
    // (the kernels' occupancy depends on the architecture only; cached once per variant)
    static std::atomic<int> resident[2] = {{0}, {0}};
    const int bi = p.eo_bf16 ? 1 : 0;
    int per_sm = resident[bi].load(std::memory_order_relaxed);
    if (per_sm == 0) {
        int nb = 0;
        const cudaError_t e = p.eo_bf16
            ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, reduce_ranks_kernel<true>, kCopyThreads, 0)
            : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, reduce_ranks_kernel<false>, kCopyThreads, 0);
        if (e != cudaSuccess) return e;
        per_sm = nb > 0 ? nb : 1;
        resident[bi].store(per_sm, std::memory_order_relaxed);
    }
    int64_t blocks = blocks_for(p.W * p.cap);
    if (blocks > (int64_t)num_sms() * per_sm) blocks = (int64_t)num_sms() * per_sm;
    if (p.eo_bf16) return launch_pdl(reduce_ranks_kernel<true>, dim3((unsigned)blocks), dim3(kCopyThreads), 0, s, a);
    return launch_pdl(reduce_ranks_kernel<false>, dim3((unsigned)blocks), dim3(kCopyThreads), 0, s, a);
}

cudaError_t launch_combine(const Routing &r, const void *expert_out, const float *topk_w,
                           uint16_t *out, cudaStream_t s) {
    const Plan &p = *r.p;
    if (p.T == 0) return cudaSuccess;
    const int nchunk = (int)((p.H / 4 + 32 * kCopyU - 1) / (32 * kCopyU));
    CombineArgs a{expert_out, topk_w, r.slot, r.recv_row, out, (int)p.T, (int)p.k, (int)p.W,
                  (int)p.H, p.layout, nchunk, p.cap};
    if (p.eo_bf16) return launch_pdl(combine_kernel<true>, dim3(blocks_for(p.T * nchunk)), dim3(kCopyThreads), 0, s, a);
    return launch_pdl(combine_kernel<false>, dim3(blocks_for(p.T * nchunk)), dim3(kCopyThreads), 0, s, a);
}

cudaError_t launch_prepare_w1(const moe_geom &g, const uint16_t *w1, uint16_t *w1p,
                              cudaStream_t s) {
    int64_t rows = (int64_t)g.num_experts * 2 * g.intermediate;
    prepare_w1_kernel<<<blocks_for(rows), kCopyThreads, 0, s>>>(w1, w1p, rows, g.intermediate,
                                                               g.hidden);
    return cudaGetLastError();
}

cudaError_t launch_dispatch_quant(const Routing &r, const uint16_t *x, cudaStream_t s) {
    const Plan &p = *r.p;
    if (p.T == 0) return cudaSuccess;
    const int nchunk = (int)((p.H / 8 + 32 * kCopyU - 1) / (32 * kCopyU));
    QuantCopyArgs a{x, reinterpret_cast<uint8_t *>(r.recv_x), r.recv_scales, reinterpret_cast<uint8_t *>(r.apick),
                    r.apick_scales, r.slot, r.recv_row, r.pick_pos, (int)p.T, (int)p.k, (int)p.W, (int)p.H,
                    p.layout, nchunk, p.cap, p.nrecv, p.P};
    return launch_pdl(dispatch_quant_kernel, dim3(blocks_for(p.T * nchunk)), dim3(kCopyThreads), 0, s, a);
}

cudaError_t launch_quantize_weights_fp8(const uint16_t *w, int64_t E, int64_t rows, int64_t cols,
                                        int64_t w1_inter, uint8_t *q, float *sc, cudaStream_t s) {
    const int64_t blocks = E * (rows / 128) * (cols / 128);
    if (blocks == 0) return cudaSuccess;
    if (blocks >= ((int64_t)1 << 31)) return cudaErrorInvalidValue;
    quantize_blocks_kernel<<<(unsigned)blocks, 256, 0, s>>>(w, q, sc, rows, cols, w1_inter);
    return cudaGetLastError();
}

cudaError_t launch_prepare_w1_fp8(const moe_geom &g, const uint8_t *w1q, const float *w1s,
                                  uint8_t *w1qp, float *w1sp, cudaStream_t s) {
    int64_t rows = (int64_t)g.num_experts * 2 * g.intermediate;
    prepare_w1_fp8_kernel<<<blocks_for(rows), kCopyThreads, 0, s>>>(w1q, w1s, w1qp, w1sp, rows,
                                                                   g.intermediate, g.hidden);
    return cudaGetLastError();
}

}  // namespace moe
