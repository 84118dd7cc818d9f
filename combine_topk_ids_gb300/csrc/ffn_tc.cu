// Grouped SwiGLU expert FFN on 5th-generation tensor cores (tcgen05, sm_103a).
//
// Operation (FlashInfer "MoE-EP implementation & usage", section 2 "Call stack": a pure
// per-expert grouped GEMM with no routing; section 4 step 1: w1 [E, 2I, H], w2 [E, H, I]):
// for every expert e and each of its n_e rows x,
//     GEMM1   h   = x W1[e]^T            [n_e, 2I], fp32 accumulate in tensor memory
//     SwiGLU  act = silu(h[:, :I]) * h[:, I:]   fp32 (fused into GEMM1's epilogue), stored
//                   as bf16 (round to nearest even), or with MOE_ACT_BF16_PAIR as a pair of
//                   bf16 arrays act_hi = bf16(act), act_lo = bf16(act - act_hi)
//     GEMM2   y   = act W2[e]^T, or act_hi W2[e]^T + act_lo W2[e]^T   [n_e, H], fp32
// The pair carries act to about 16 significant bits (GEMM2 then runs two MMAs per k-step).
//
// One persistent kernel per GEMM, one CTA per SM, 384 threads:
//   warp 0      TMA producer: 128x64 A tile(s) + 256x64 B tile per stage (SWIZZLE_128B),
//               a 192 KB mbarrier ring: 4 stages of 48 KB (128-row tiles), 3 of 64 KB
//               (256-row tiles, or the bf16-pair A operand), 6 of 32 KB (two-SM tiles)
//   warp 1      MMA issuer (one thread): tcgen05.mma.cta_group::1.kind::f16, M=128 (M=64
//               for 128 rows of a tile that hold at most 64), N=256, K=16, bf16 x bf16 ->
//               fp32 into one of two 256-column TMEM accumulators, tcgen05.commit frees
//               smem stages and hands tiles over
//   warp 2      TMEM allocator (512 columns)
//   warps 4-11  epilogue, two warps per TMEM lane quarter, each on half of the tile's
//               columns: tcgen05.ld 32x32b rows -> registers -> SwiGLU / fp32 or bf16
//               -> (GEMM2) a 4 KB shared-memory buffer per warp -> whole 128-byte row
//               segments in global memory, overlapped with the next tile's mainloop
//               (double-buffered accumulator)
// Tiles: per expert ceil(n_e/128) m-blocks x (N/256) n-blocks, enumerated expert by expert,
// n-block-major with the m-blocks of one weight tile adjacent (they run on neighbouring
// SMs at the same time and share the weight tile through L2).  Experts with no rows issue
// no tiles and read no weights.  CTAs take tiles round-robin, except the one-CTA 256-row
// tiles, which are handed out in order from a device counter (so that the tiles in flight
// stay a contiguous window when an expert's last, short tile takes one MMA per k-step
// instead of two).  Every mbarrier wait is bounded: on timeout the kernel sets
// MOE_STATUS_TIMEOUT, drains and frees its tensor memory, and returns.
#include <cuda.h>
#include <cuda_bf16.h>

#include "tc_common.cuh"

namespace moe {
namespace {

constexpr int BM = 128, BN = 256, BK = 64;   // BN: widest n-tile (GEMM2 may use 128)
constexpr int A_BYTES = BM * BK * 2;            // 16 KB
constexpr int B_BYTES = BN * BK * 2;            // 32 KB
constexpr int THREADS = 384;                    // 4 control warps + 8 epilogue warps
constexpr int EPI_WARPS = 8;
constexpr int TMEM_COLS = 2 * BN;               // two fp32 accumulators of 128 x 256
constexpr int kStageRowsBytes = 32 * 128;       // one epilogue warp's 32 rows x 128 B

// Pipeline shape.  HILO: the A operand is a bf16 pair (two A tiles per stage).  PAIR: a
// cluster of two CTAs on two SMs computes a 256-row tile with tcgen05.mma.cta_group::2;
// each CTA stages its own 128 rows of A and half of the B tile.  TALL: one CTA computes a
// 256-row tile as two M = 128 MMAs that share each staged B tile (a third fewer operand
// bytes per FLOP than 128-row tiles); the two 128 x 256 accumulators fill the tensor
// memory, so there is one accumulator buffer instead of two.
template <bool HILO, bool PAIR, bool TALL> struct Pipe {
    static_assert(!(TALL && (PAIR || HILO)), "TALL tiles take a single bf16 A operand on one SM");
    static constexpr int kATiles = HILO ? 2 : 1;
    static constexpr int kABytes = TALL ? 2 * A_BYTES : A_BYTES;       // one A tile
    static constexpr int kBBytes = PAIR ? B_BYTES / 2 : B_BYTES;
    static constexpr int kStageBytes = kATiles * kABytes + kBBytes;     // 32..64 KB
    static constexpr int kStages = (192 * 1024) / kStageBytes;          // 3..6
    static constexpr int kSmemBytes =
        kStages * kStageBytes + 1024 /*align*/ + 256 /*barriers*/ + EPI_WARPS * kStageRowsBytes /*epilogue*/;
    static constexpr int kMRows = (PAIR || TALL) ? 2 * BM : BM;         // rows of one tile
    static constexpr int kAccBufs = TALL ? 1 : 2;                       // accumulator buffers
};

// Instruction descriptor of tcgen05.mma kind::f16: D fp32 (bits 4-5 = 1), A bf16
// (bits 7-9 = 1), B bf16 (bits 10-12 = 1), both K-major (bits 15/16 = 0),
// N >> 3 at bits 17-22, M >> 4 at bits 24-28.
__host__ __device__ constexpr uint32_t make_idesc(int m, int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(m >> 4) << 24);
}

struct FfnArgs {
    const int32_t *counts, *offsets;
    const int32_t *mprefix;   // prefix over experts of ceil(rows / tile rows)
    int E;
    int bn;        // n-tile width: 256 or 128
    int nb;        // n-blocks per expert (N / bn)
    int kb;        // k-blocks (K / BK)
    int a_mode;    // 0: A row = e*a_cap + m; 1: A row = offsets[e] + m
    int64_t a_cap;
    int64_t b_rows;   // rows of B per expert (N)
    int mode;      // 0: SwiGLU epilogue -> act as a bf16 (hi, lo) pair; 1: fp32 store
    int out_bf16;  // mode 1: store the rows as bf16 (round to nearest even) instead
    void *out;     // mode 0: act_hi; mode 1: fp32 rows
    void *out2;    // mode 0: act_lo (NULL: single bf16 activation)
    int64_t out_ld;   // elements per output row
    int out_mode;  // 0: row = e*out_cap + m; 1: row = offsets[e] + m
    int64_t out_cap;
    // mode 1, out_mode 1 (RANK_MAJOR / FLAT per-pick rows), or NULL: a pick p with
    // direct_row[p] >= 0 is the only local pick of its received row, so the row
    // direct_row[p] of out_direct gets direct_w[p] * y (the local-pick sum) instead of
    // out getting y
    const int32_t *direct_row;
    const float *direct_w;
    void *out_direct;
    int32_t *status;
    // TALL tiles in dynamic order (NULL: the static order): sched[0] counts the tiles
    // handed out after each CTA's first one, sched[1] the CTAs that finished; both are zero
    // when the kernel starts, and the last CTA to finish zeroes them again
    int32_t *sched;
};
constexpr int kRing = 4;   // tiles in flight from the producer to the MMA and epilogue warps
// 128 rows of a tile that hold at most 64 (in an expert's last block) take M = 64 MMAs on
// one SM: a 128-row tile, or either half of a one-CTA 256-row tile.  An M = 64 accumulator
// holds row r in tensor-memory lane 32 * (r / 16) + r % 16: each epilogue warp's lane
// quarter carries 16 rows in its first 16 lanes.  (The two-SM tiles keep M = 256.)
constexpr bool kM64Tails = true;
constexpr int kM64Rows = 64;

// --- two-SM (cluster of two CTAs) variants
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t num_clusters_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}
// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}
// TMA load into this CTA's shared memory, completing on an mbarrier of either CTA of the pair.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                                 uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar_cluster)
        : "memory");
}
__device__ __forceinline__ void mma_bf16_pair(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                              uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
// Arrive once on the mbarrier at `bar` in both CTAs of the pair when this thread's
// earlier tcgen05 operations complete.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(bar),
        "h"((uint16_t)3)
        : "memory");
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

// Store 32 rows x 128 bytes held one row per lane (w = lane's row) to global rows
// gbase + r * row_bytes, r < nvalid, as full 128-byte segments: the rows pass through this
// warp's 4 KB shared-memory buffer (16-byte chunk q of row r at chunk q ^ (r & 7), so that
// neither the row-per-lane writes nor the segment-per-8-lanes reads conflict on banks),
// then each store instruction writes four whole rows' 128-byte segments.
// With dbase set, row r goes to dbase + drow_r * row_bytes instead when the drow of lane r
// is >= 0.
__device__ __forceinline__ void warp_store_rows(uint32_t stg, const uint32_t (&w)[32], char *gbase,
                                                int64_t row_bytes, int nvalid, int lane,
                                                int64_t drow = -1, char *dbase = nullptr) {
    const uint32_t mine = stg + (uint32_t)lane * 128u;
#pragma unroll
    for (int q = 0; q < 8; ++q)
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(mine + (uint32_t)((q ^ (lane & 7)) << 4)),
                     "r"(w[4 * q]), "r"(w[4 * q + 1]), "r"(w[4 * q + 2]), "r"(w[4 * q + 3])
                     : "memory");
    __syncwarp();
    const int ch = lane & 7;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int r = (lane >> 3) + 4 * i;
        uint4 v;
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                     : "r"(stg + (uint32_t)r * 128u + (uint32_t)((ch ^ (r & 7)) << 4))
                     : "memory");
        char *dst = gbase + (int64_t)r * row_bytes;
        if (dbase) {
            const int64_t dr = __shfl_sync(0xffffffffu, drow, r);
            if (dr >= 0) dst = dbase + dr * row_bytes;
        }
        if (r < nvalid) *reinterpret_cast<uint4 *>(dst + ch * 16) = v;
    }
    __syncwarp();   // the buffer is reused by the next call
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&b);
}

// silu(g) * u of the SwiGLU epilogue.  TALL tiles drain both accumulators before the
// next tile's MMAs can start (nothing overlaps their epilogue), so they take the fast
// reciprocal divide (within 2 ulp of the IEEE quotient); the other tiles' epilogue runs
// under the next mainloop and keeps the IEEE divide.
template <bool FAST> __device__ __forceinline__ float silu_act(float g, float u) {
    return FAST ? silu_mul_fast(g, u) : silu_mul(g, u);
}

// Tile index -> (expert, m-block, n-block).  Experts are laid out by the m-block prefix:
// expert e owns tiles [mprefix[e]*nb, mprefix[e+1]*nb); inside, n-block-major.
__device__ __forceinline__ void decode_tile(const FfnArgs &a, int tile, int &e, int &mb, int &nbk) {
    const int q = tile / a.nb;
    int lo = 0, hi = a.E - 1;   // largest e with mprefix[e] <= q
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (__ldg(a.mprefix + mid) <= q) lo = mid;
        else hi = mid - 1;
    }
    e = lo;
    const int m0 = __ldg(a.mprefix + e);
    const int mt = __ldg(a.mprefix + e + 1) - m0;
    const int local = tile - m0 * a.nb;
    nbk = local / mt;
    mb = local - nbk * mt;
}

template <bool HILO, bool PAIR, bool TALL>
__global__ void __launch_bounds__(THREADS, 1)
    ffn_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
                    const __grid_constant__ CUtensorMap tmB, FfnArgs a) {
    using P = Pipe<HILO, PAIR, TALL>;
    constexpr int STAGES = P::kStages;
    // the set-up below touches no global memory; pdl_wait() follows it
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t *sA = smem;                                     // [STAGES][kATiles] A tiles
    uint8_t *sB = smem + STAGES * P::kATiles * P::kABytes;  // [STAGES] B tiles (or halves)
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + STAGES * P::kStageBytes);
    // bars: full[STAGES], empty[STAGES], tfull[2], tempty[2], then (dynamic tile order)
    // rfull[kRing], rempty[kRing]; then the TMEM address, the abort flag, the ring's tiles
    // and the rows of their row blocks
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * STAGES + 4 + 2 * kRing);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    volatile int *ring_tile = reinterpret_cast<volatile int *>(tmem_slot + 2);
    volatile int *ring_rows = ring_tile + kRing;
    const bool dyn = TALL && a.sched != nullptr;
    const uint32_t rfull0 = smem_u32(bars + 2 * STAGES + 4), rempty0 = rfull0 + 8 * kRing;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + STAGES);
    const uint32_t tfull0 = smem_u32(bars + 2 * STAGES), tempty0 = smem_u32(bars + 2 * STAGES + 2);
    // PAIR: rank 0 (the leader) issues the MMAs for both CTAs and owns the barriers they
    // wait on; rank 1 stages rows 128..255 of A and the second half of B.
    const uint32_t rank = PAIR ? cluster_ctarank() : 0;
    const bool leader = rank == 0;
    const int first_tile = PAIR ? (int)cluster_id_x() : (int)blockIdx.x;
    const int tile_step = PAIR ? (int)num_clusters_x() : (int)gridDim.x;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(tfull0 + 8 * s, 1);
            mbar_init(tempty0 + 8 * s, PAIR ? 2 * EPI_WARPS : EPI_WARPS);   // one arrival per epilogue warp
        }
        for (int s = 0; s < kRing; ++s) {
            mbar_init(rfull0 + 8 * s, 1);                 // the producer publishes a tile
            mbar_init(rempty0 + 8 * s, 1 + EPI_WARPS);    // the MMA thread and every epilogue warp took it
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
        if (HILO || dyn)
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA2)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
    }
    if (warp == 2) {
        if (PAIR) {
            asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                             smem_u32(tmem_slot)),
                         "r"(TMEM_COLS)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
        } else {
            asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                             smem_u32(tmem_slot)),
                         "r"(TMEM_COLS)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        }
    }
    tc_fence_before();
    __syncthreads();
    if (PAIR) cluster_sync();   // the peer's barriers exist before anyone signals them
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    pdl_wait();   // the previous kernel in the stream has completed: its outputs are visible
    const int total = __ldg(a.mprefix + a.E) * a.nb;

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------------------- TMA producer
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        const int b_rows_cta = PAIR ? a.bn / 2 : a.bn;
        const uint32_t tx_cta = (uint32_t)(P::kATiles * P::kABytes + b_rows_cta * BK * 2);
        const uint32_t tx = PAIR ? 2 * tx_cta : tx_cta;   // the leader's barrier sees both CTAs
        int seq = 0;
        for (int tile = first_tile; ok;) {
            bool short_tile = false;
            int e = 0, mb = 0, nbk = 0, rows = 0;
            if (tile < total) {
                decode_tile(a, tile, e, mb, nbk);
                // a tile whose rows end in its first 128 loads only those, through the
                // 128-row box of tmA2, and the MMA issuer skips the second half
                rows = __ldg(a.counts + e) - mb * P::kMRows;
                short_tile = dyn && rows <= BM;
            }
            if (dyn) {   // publish the tile (or the end) to the MMA and epilogue warps
                const int slot = seq & (kRing - 1);
                if (!mbar_wait(rempty0 + 8 * slot, ((seq / kRing) & 1) ^ 1, abort_flag, a.status)) break;
                ring_tile[slot] = tile < total ? tile : -1;
                ring_rows[slot] = rows;
                mbar_arrive(rfull0 + 8 * slot);
                ++seq;
            }
            if (tile >= total) break;
            const int64_t arow = (a.a_mode == 0 ? (int64_t)e * a.a_cap : (int64_t)__ldg(a.offsets + e)) +
                                 (int64_t)mb * P::kMRows + (int64_t)rank * BM;
            const int64_t brow = (int64_t)e * a.b_rows + (int64_t)nbk * a.bn + (int64_t)rank * b_rows_cta;
            for (int kb = 0; kb < a.kb; ++kb) {
                if (!mbar_wait(empty0 + 8 * stage, phase ^ 1, abort_flag, a.status)) { ok = false; break; }
                const uint32_t fb = full0 + 8 * stage;
                uint8_t *sa = sA + stage * P::kATiles * P::kABytes;
                const uint32_t sb = smem_u32(sB + stage * P::kBBytes);
                if (PAIR) {
                    if (leader) mbar_expect_tx(fb, tx);
                    const uint32_t fbl = map_to_rank(fb, 0);
                    tma_load_2d_pair(smem_u32(sa), &tmA, kb * BK, (int)arow, fbl);
                    if (HILO) tma_load_2d_pair(smem_u32(sa + A_BYTES), &tmA2, kb * BK, (int)arow, fbl);
                    tma_load_2d_pair(sb, &tmB, kb * BK, (int)brow, fbl);
                } else if (short_tile) {
                    mbar_expect_tx(fb, (uint32_t)(A_BYTES + a.bn * BK * 2));
                    tma_load_2d(smem_u32(sa), &tmA2, kb * BK, (int)arow, fb);
                    tma_load_2d(sb, &tmB, kb * BK, (int)brow, fb);
                } else {
                    mbar_expect_tx(fb, tx);
                    tma_load_2d(smem_u32(sa), &tmA, kb * BK, (int)arow, fb);
                    if (HILO) tma_load_2d(smem_u32(sa + A_BYTES), &tmA2, kb * BK, (int)arow, fb);
                    tma_load_2d(sb, &tmB, kb * BK, (int)brow, fb);
                }
                if (++stage == STAGES) { stage = 0; phase ^= 1; }
            }
            // dynamic order: a CTA takes its next tile from a device counter once it has
            // queued this one's loads, so tiles start in increasing order, the tiles in flight
            // stay a contiguous window and the m-blocks that share a weight tile run at the
            // same time even when some tiles are shorter than others
            tile = dyn ? (int)gridDim.x + atomicAdd(a.sched, 1) : tile + tile_step;
        }
    } else if (warp == 1 && lane == 0 && leader) {
        // ---------------------------------------------------------------- MMA issuer
        int stage = 0;
        uint32_t phase = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        bool ok = true;
        const uint32_t idesc_full = make_idesc(TALL ? BM : P::kMRows, a.bn);
        const uint32_t idesc_m64 = make_idesc(kM64Rows, a.bn);
        int seq = 0;
        for (int tile = first_tile; ok; tile += tile_step) {
            bool second_half = TALL;   // TALL: rows 128..255 of the tile hold data
            bool m64 = false, m64_2 = false;   // M = 64 for the first / the second 128 rows
            if (dyn) {
                const int slot = seq & (kRing - 1);
                if (!mbar_wait(rfull0 + 8 * slot, (seq / kRing) & 1, abort_flag, a.status)) break;
                tile = ring_tile[slot];
                const int rows = ring_rows[slot];
                second_half = rows > BM;
                m64 = kM64Tails && rows <= kM64Rows;
                m64_2 = kM64Tails && rows - BM <= kM64Rows;
                mbar_arrive(rempty0 + 8 * slot);
                ++seq;
                if (tile < 0) break;
            } else if (tile >= total) {
                break;
            } else if (kM64Tails && !PAIR && !TALL) {
                int e, mb, nbk;
                decode_tile(a, tile, e, mb, nbk);
                m64 = __ldg(a.counts + e) - mb * P::kMRows <= kM64Rows;
            }
            const uint32_t idesc = m64 ? idesc_m64 : idesc_full;
            const uint32_t idesc2 = m64_2 ? idesc_m64 : idesc_full;
            if (!mbar_wait(tempty0 + 8 * acc, acc_phase ^ 1, abort_flag, a.status)) break;
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
            for (int kb = 0; kb < a.kb; ++kb) {
                if (!mbar_wait(full0 + 8 * stage, phase, abort_flag, a.status)) { ok = false; break; }
                tc_fence_after();
                const uint32_t a0 = smem_u32(sA + stage * P::kATiles * P::kABytes);
                const uint32_t b0 = smem_u32(sB + stage * P::kBBytes);
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk) {
                    const uint64_t bd = sw128_desc(b0 + kk * 32);
                    const uint64_t ad = sw128_desc(a0 + kk * 32);
                    const uint32_t accum = (kb | kk) != 0 ? 1u : 0u;
                    if (PAIR) {
                        mma_bf16_pair(d_tmem, ad, bd, idesc, accum);
                        if (HILO) mma_bf16_pair(d_tmem, sw128_desc(a0 + A_BYTES + kk * 32), bd, idesc, 1u);
                    } else {
                        mma_bf16(d_tmem, ad, bd, idesc, accum);
                        if (HILO) mma_bf16(d_tmem, sw128_desc(a0 + A_BYTES + kk * 32), bd, idesc, 1u);
                        // rows 128..255 of the tile: the second 16 KB of the A tile, the
                        // second accumulator
                        if (TALL && second_half)
                            mma_bf16(d_tmem + BN, sw128_desc(a0 + A_BYTES + kk * 32), bd, idesc2, accum);
                    }
                }
                // the stage is reusable (in both CTAs) once these MMAs finish
                if (PAIR) mma_commit_pair(empty0 + 8 * stage);
                else mma_commit(empty0 + 8 * stage);
                if (++stage == STAGES) { stage = 0; phase ^= 1; }
            }
            if (!ok) break;
            if (PAIR) mma_commit_pair(tfull0 + 8 * acc);   // accumulators ready in both CTAs
            else mma_commit(tfull0 + 8 * acc);
            if (++acc == P::kAccBufs) { acc = 0; acc_phase ^= 1; }
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------------ epilogue
        // Warp quad reads TMEM lanes 32*quad .. +31 (rows of the tile; lane i holds row
        // 32*quad + i).  GEMM2 rows go through the warp's shared-memory buffer and leave as
        // whole 128-byte row segments (32 fp32 or 64 bf16 columns at a time); GEMM1's
        // SwiGLU activation is stored from registers (staging it measured slower).
        // Warps 4-7 and 8-11 read the same TMEM lane quarters (warp % 4) and split the
        // tile's columns in halves.
        const int quad = warp & 3;
        const int chalf = (warp - 4) >> 2;   // 0: first half of the columns, 1: second
        const uint32_t stg = smem_u32(smem + STAGES * P::kStageBytes + 256) + (uint32_t)((warp - 4) * kStageRowsBytes);
        int acc = 0;
        uint32_t acc_phase = 0;
        int seq = 0;
        for (int tile = first_tile;; tile += tile_step) {
            if (dyn) {
                const int slot = seq & (kRing - 1);
                if (!mbar_wait(rfull0 + 8 * slot, (seq / kRing) & 1, abort_flag, a.status)) break;
                tile = ring_tile[slot];
                __syncwarp();
                if (lane == 0) mbar_arrive(rempty0 + 8 * slot);
                ++seq;
                if (tile < 0) break;
            } else if (tile >= total) {
                break;
            }
            int e, mb, nbk;
            decode_tile(a, tile, e, mb, nbk);
            const int count = __ldg(a.counts + e);
            // the MMA issuer's choice: M = 64 for 128 rows of the tile that hold at most 64
            const int blk_rows = count - mb * P::kMRows;
            const bool m64_ok = kM64Tails && !PAIR && (dyn || !TALL);
            const int64_t obase = a.out_mode == 0 ? (int64_t)e * a.out_cap : (int64_t)__ldg(a.offsets + e);
            if (!mbar_wait(tfull0 + 8 * acc, acc_phase, abort_flag, a.status)) break;
            tc_fence_after();
            // TALL tiles hold rows 0..127 in the first accumulator and 128..255 in the second
#pragma unroll 1
            for (int half = 0; half < (TALL ? 2 : 1); ++half) {
            // first row of this warp: PAIR tiles split rows by CTA, TALL tiles by accumulator
            const int rq = m64_ok && blk_rows - half * BM <= kM64Rows ? 16 : 32;   // rows per epilogue warp
            const int m0 = mb * P::kMRows + (int)rank * BM + half * BM + quad * rq;
            const int nvalid = min(rq, count - m0);   // rows this warp stores (its lanes 0 .. nvalid-1)
            const int64_t orow0 = obase + m0;
            const uint32_t tbase = tmem_base + (uint32_t)((acc + half) * BN) + ((uint32_t)(quad * 32) << 16);
            if (nvalid <= 0) {
                // every row of this warp is padding: nothing to store
            } else if (a.mode == 0) {
                // columns [0,128) gate, [128,256) up of act columns nbk*128 .. +128, stored
                // straight from registers (64 bytes of a row per lane and round)
                const int64_t o0 = (orow0 + lane) * a.out_ld + (int64_t)nbk * (BN / 2);
                __nv_bfloat16 *out_hi = reinterpret_cast<__nv_bfloat16 *>(a.out) + o0;
                __nv_bfloat16 *out_lo = a.out2 ? reinterpret_cast<__nv_bfloat16 *>(a.out2) + o0 : nullptr;
#pragma unroll 1
                for (int c = chalf * (BN / 4); c < (chalf + 1) * (BN / 4); c += 32) {
                    uint32_t g[32], u[32];
                    tmem_ld32(tbase + c, g);
                    tmem_ld32(tbase + BN / 2 + c, u);
                    tmem_wait_ld();
                    if (lane < nvalid) {
                        uint4 *oh = reinterpret_cast<uint4 *>(out_hi + c);
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            uint32_t wh[4], wl[4];
#pragma unroll
                            for (int h = 0; h < 4; ++h) {
                                const int i = v * 8 + h * 2;
                                const float a0 = silu_act<TALL>(__uint_as_float(g[i]), __uint_as_float(u[i]));
                                const float a1 = silu_act<TALL>(__uint_as_float(g[i + 1]), __uint_as_float(u[i + 1]));
                                __nv_bfloat162 hi = __floats2bfloat162_rn(a0, a1);
                                wh[h] = *reinterpret_cast<uint32_t *>(&hi);
                                wl[h] = pack_bf16x2(a0 - __low2float(hi), a1 - __high2float(hi));
                            }
                            oh[v] = make_uint4(wh[0], wh[1], wh[2], wh[3]);
                            if (out_lo) reinterpret_cast<uint4 *>(out_lo + c)[v] = make_uint4(wl[0], wl[1], wl[2], wl[3]);
                        }
                    }
                }
            } else {
                // the direct row of this lane's pick (RANK_MAJOR / FLAT), or -1
                int64_t drow = -1;
                float dw = 0.f;
                if (a.direct_row && lane < nvalid) {
                    drow = __ldg(a.direct_row + orow0 + lane);
                    if (drow >= 0) dw = __ldg(a.direct_w + orow0 + lane);
                }
                const int esz = a.out_bf16 ? 2 : 4;
                char *out = reinterpret_cast<char *>(a.out) + (orow0 * a.out_ld + (int64_t)nbk * a.bn) * esz;
                char *dout = a.direct_row ? reinterpret_cast<char *>(a.out_direct) + (int64_t)nbk * a.bn * esz
                                          : nullptr;
                if (a.out_bf16) {
#pragma unroll 1
                    for (int c = chalf * (a.bn / 2); c < (chalf + 1) * (a.bn / 2); c += 64) {
                        uint32_t w[32];
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            uint32_t v[32];
                            tmem_ld32(tbase + c + 32 * h, v);
                            tmem_wait_ld();
                            if (drow >= 0) {
                                // the same roundings as the local-pick reduction of a
                                // one-pick row: bf16(y), then bf16(w * y)
#pragma unroll
                                for (int i = 0; i < 32; ++i)
                                    v[i] = __float_as_uint(__fmaf_rn(
                                        dw, __bfloat162float(__float2bfloat16_rn(__uint_as_float(v[i]))), 0.0f));
                            }
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                w[16 * h + i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
                        }
                        warp_store_rows(stg, w, out + (int64_t)c * 2, a.out_ld * 2, nvalid, lane, drow,
                                        dout ? dout + (int64_t)c * 2 : nullptr);
                    }
                } else {
#pragma unroll 1
                    for (int c = chalf * (a.bn / 2); c < (chalf + 1) * (a.bn / 2); c += 32) {
                        uint32_t v[32];
                        tmem_ld32(tbase + c, v);
                        tmem_wait_ld();
                        if (drow >= 0) {
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                v[i] = __float_as_uint(__fmaf_rn(dw, __uint_as_float(v[i]), 0.0f));
                        }
                        warp_store_rows(stg, v, out + (int64_t)c * 4, a.out_ld * 4, nvalid, lane, drow,
                                        dout ? dout + (int64_t)c * 4 : nullptr);
                    }
                }
            }
            }   // half
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {   // this warp is done with the accumulator
                if (PAIR) mbar_arrive_cluster(map_to_rank(tempty0 + 8 * acc, 0));
                else mbar_arrive(tempty0 + 8 * acc);
            }
            if (++acc == P::kAccBufs) { acc = 0; acc_phase ^= 1; }
        }
    }

    __syncthreads();
    if (PAIR) cluster_sync();   // no signal from the peer can still be on its way here
    if (dyn && threadIdx.x == 0) {
        // every tile this CTA took was taken before the barrier above; the last CTA to get
        // here zeroes the counters for the next launch
        __threadfence();
        if (atomicAdd(a.sched + 1, 1) == (int)gridDim.x - 1) {
            a.sched[0] = 0;
            a.sched[1] = 0;
        }
    }
    if (*abort_flag) {
        // Give in-flight TMA copies and MMAs time to land before the memory is released.
        unsigned long long t0 = globaltimer();
        while (globaltimer() - t0 < 1000000ull) {}
    }
    if (warp == 2) {
        tc_fence_after();
        if (PAIR)
            asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                         "r"(TMEM_COLS)
                         : "memory");
        else
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                         "r"(TMEM_COLS)
                         : "memory");
    }
}

// bf16 [rows, cols] map with a box of box_rows x 64 columns (see make_map_2d).
bool make_map(CUtensorMap *m, const void *base, int64_t rows, int64_t cols, int box_rows) {
    return make_map_2d(m, base, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, rows, cols, box_rows);
}

template <bool HILO, bool PAIR, bool TALL = false>
int launch_gemm(const CUtensorMap &ma, const CUtensorMap &ma2, const CUtensorMap &mb,
                const FfnArgs &args, int64_t max_tiles, cudaStream_t s) {
    if (max_tiles <= 0) return MOE_OK;
    constexpr int smem = Pipe<HILO, PAIR, TALL>::kSmemBytes;
    auto kernel = ffn_gemm_kernel<HILO, PAIR, TALL>;
    // kernel attributes are set per device (with that device current), once each
    struct PerDevice {
        std::once_flag once;
        cudaError_t attr_err = cudaSuccess;
        int max_clusters = 0;
    };
    static PerDevice per_device[64];
    const int dev = device_ordinal();
    if (dev < 0) return MOE_ERR_CUDA;
    PerDevice &pd = per_device[dev];
    cudaError_t &attr_err = pd.attr_err;
    int &max_clusters = pd.max_clusters;
    std::call_once(pd.once, [&] {
        attr_err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (attr_err == cudaSuccess && PAIR) {
            attr_err = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 0);
            cudaLaunchConfig_t q = {};
            cudaLaunchAttribute at[1];
            at[0].id = cudaLaunchAttributeClusterDimension;
            at[0].val.clusterDim.x = 2;
            at[0].val.clusterDim.y = 1;
            at[0].val.clusterDim.z = 1;
            q.gridDim = dim3(2 * (num_sms() / 2), 1, 1);
            q.blockDim = dim3(THREADS, 1, 1);
            q.dynamicSmemBytes = smem;
            q.attrs = at;
            q.numAttrs = 1;
            if (attr_err == cudaSuccess)
                attr_err = cudaOccupancyMaxActiveClusters(&max_clusters, kernel, &q);
        }
    });
    if (attr_err != cudaSuccess) return MOE_ERR_CUDA;
    if (!PAIR) {
        int grid = num_sms();
        if ((int64_t)grid > max_tiles) grid = (int)max_tiles;
        return launch_pdl(kernel, dim3(grid), dim3(THREADS), smem, s, ma, ma2, mb, args) == cudaSuccess
                   ? MOE_OK
                   : MOE_ERR_CUDA;
    }
    // persistent clusters of two CTAs: never more than can be resident at once
    int clusters = max_clusters > 0 ? max_clusters : num_sms() / 2;
    if ((int64_t)clusters > max_tiles) clusters = (int)max_tiles;
    if (clusters < 1) return MOE_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(2 * clusters, 1, 1);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kernel, ma, ma2, mb, args) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// Two-SM tiles (256 rows per tile).  Measured on GB300 (same box, same build, A/B): the
// cta_group::2 MMA spends ~24% more tensor-pipe cycles per FLOP than two cta_group::1
// MMAs here, and halving the per-SM B tile only pays that back on small per-expert GEMMs
// (K <= 2048 and N <= 2048: ragged 16384-token workload, GEMM1 -6%, GEMM2 -3%); on the
// Mixtral-like (K 4096 / 14336) and DeepSeek-like prefill (K 7168) shapes it was 2-30%
// slower.  It also needs many rows per expert, or most of a 256-row tile is padding.
// Decided from the geometry alone (the counts live on the device).
bool use_pair(const Plan &p, int64_t K, int64_t N) {
    return p.P >= 192 * p.E && K <= 2048 && N <= 2048;
}

// One-CTA 256-row tiles: for experts with four 128-row blocks or more on average and a
// long K loop (>= 4096), which amortises the unoverlapped epilogue.  Measured on GB300
// (A/B, same build): DeepSeek-like prefill GEMM1 (K 7168, ~1024 rows per expert) -10%
// clock for clock; on the Mixtral-like decode (~256 rows per expert, three of eight
// experts a few rows over 256) GEMM1 +9% and GEMM2 +50%, since a 256-row block holding
// a few tail rows streams the whole weight tile again and nothing hides its epilogue.  At
// K = 2048 instead of two-SM or 128-row tiles: ragged 16384-token GEMM1 +5% (bf16-pair
// activation) / -1.5% (single bf16), DeepSeek-like prefill single-bf16 GEMM2 +1.4%.
bool use_tall(const Plan &p, int64_t K) { return p.P >= 512 * p.E && K >= 4096; }

// upper bound of the row blocks over all experts: sum ceil(n_e/rows) <= P/rows + E
int64_t max_mblocks(const Plan &p, int rows) { return p.P / rows + p.E; }

FfnArgs base_args(const Routing &r, bool pair) {
    const Plan &p = *r.p;
    FfnArgs g{};
    g.counts = r.counts; g.offsets = r.offsets; g.mprefix = pair ? r.mprefix2 : r.mprefix;
    g.E = (int)p.E;
    g.status = r.status;
    return g;
}

}  // namespace

int launch_gemm1(const Routing &r, const uint16_t *w1p, cudaStream_t s) {
    const Plan &p = *r.p;
    if (p.P == 0) return MOE_OK;
    const bool em = p.layout == MOE_LAYOUT_EXPERT_MAJOR;
    const bool pair = use_pair(p, p.H, 2 * p.I);
    const bool tall = !pair && use_tall(p, p.H);
    CUtensorMap mA, mA2, mB;
    const void *a1 = em ? (const void *)r.recv_x : (const void *)r.apick;
    const int64_t a1_rows = em ? p.E * p.cap : p.P;
    if (!make_map(&mA, a1, a1_rows, p.H, tall ? 2 * BM : BM) ||
        (tall && !make_map(&mA2, a1, a1_rows, p.H, BM)) ||   // short tail tiles of TALL
        !make_map(&mB, w1p, p.E * 2 * p.I, p.H, pair ? BN / 2 : BN))
        return MOE_ERR_CUDA;
    FfnArgs g = base_args(r, pair || tall);
    g.bn = BN; g.nb = (int)(2 * p.I / BN); g.kb = (int)(p.H / BK);
    g.a_mode = em ? 0 : 1; g.a_cap = p.cap; g.b_rows = 2 * p.I;
    g.mode = 0; g.out = r.act; g.out2 = p.act_pair ? r.act_lo : nullptr; g.out_ld = p.I; g.out_mode = 1;
    g.out_cap = 0;
    if (pair) return launch_gemm<false, true>(mA, mA, mB, g, max_mblocks(p, 2 * BM) * g.nb, s);
    if (tall) {
        g.sched = r.sched;
        return launch_gemm<false, false, true>(mA, mA2, mB, g, max_mblocks(p, 2 * BM) * g.nb, s);
    }
    return launch_gemm<false, false>(mA, mA, mB, g, max_mblocks(p, BM) * g.nb, s);
}

int launch_gemm2(const Routing &r, const uint16_t *w2, void *expert_out, cudaStream_t s) {
    const Plan &p = *r.p;
    if (p.P == 0) return MOE_OK;
    const bool em = p.layout == MOE_LAYOUT_EXPERT_MAJOR;
    const bool pair = use_pair(p, p.I, p.H);
    const bool tall = !pair && !p.act_pair && use_tall(p, p.I);
    const int bn = (p.H % 256 == 0) ? 256 : 128;
    CUtensorMap mA, mA2, mB;
    if (!make_map(&mA, r.act, p.P, p.I, tall ? 2 * BM : BM) ||
        (p.act_pair && !make_map(&mA2, r.act_lo, p.P, p.I, BM)) ||
        (tall && !make_map(&mA2, r.act, p.P, p.I, BM)) ||   // short tail tiles of TALL
        !make_map(&mB, w2, p.E * p.H, p.I, pair ? bn / 2 : bn))
        return MOE_ERR_CUDA;
    FfnArgs g = base_args(r, pair || tall);
    g.bn = bn; g.nb = (int)(p.H / bn); g.kb = (int)(p.I / BK);
    g.a_mode = 1; g.a_cap = 0; g.b_rows = p.H; g.mode = 1; g.out_ld = p.H; g.out_bf16 = p.eo_bf16;
    if (em) { g.out = expert_out; g.out_mode = 0; g.out_cap = p.cap; }
    else {
        g.out = r.ypick; g.out_mode = 1; g.out_cap = 0;
        g.direct_row = r.direct_row; g.direct_w = r.direct_w; g.out_direct = expert_out;
    }
    if (p.act_pair) {
        if (pair) return launch_gemm<true, true>(mA, mA2, mB, g, max_mblocks(p, 2 * BM) * g.nb, s);
        return launch_gemm<true, false>(mA, mA2, mB, g, max_mblocks(p, BM) * g.nb, s);
    }
    if (pair) return launch_gemm<false, true>(mA, mA, mB, g, max_mblocks(p, 2 * BM) * g.nb, s);
    if (tall) {
        g.sched = r.sched + 2;
        return launch_gemm<false, false, true>(mA, mA2, mB, g, max_mblocks(p, 2 * BM) * g.nb, s);
    }
    return launch_gemm<false, false>(mA, mA, mB, g, max_mblocks(p, BM) * g.nb, s);
}

}  // namespace moe
