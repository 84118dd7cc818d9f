// FP8 grouped SwiGLU expert FFN on 5th-generation tensor cores (tcgen05.mma kind::f8f6f4).
//
// Operation (Mooncake EP guide, "Buffer.dispatch(...)": with use_fp8 the received rows are
// FP8 data plus scales; FlashInfer "MoE-EP implementation & usage", section 2 "Call
// stack": a pure per-expert grouped GEMM; section 4 step 1: w1 [E, 2I, H], w2 [E, H, I]),
// on e4m3 rows with one float32 scale per 128 columns and e4m3 weights with one scale per
// 128 x 128 block:
//     GEMM1   h   = sum over k-blocks kb of  sa[row, kb] * sw1[n-block, kb] * (xq . w1q)_kb
//     SwiGLU  act = silu(h[:, :I]) * h[:, I:]                                 fp32
//             act -> e4m3 codes + one scale per 128 columns (the second GEMM's A operand)
//     GEMM2   y   = sum over kb of  sa_act[row, kb] * sw2[n-block, kb] * (aq . w2q)_kb   fp32
// A k-block is 128 columns, the block size of every scale, so each k-block's product sum
// (four K=32 MMAs, exact e4m3 products accumulated in fp32 in tensor memory) is scaled as a
// whole and added to an fp32 register accumulator: the "promotion" of the partial sum.
//
// One persistent kernel per GEMM, one CTA per SM, 384 threads:
//   warp 0      TMA producer: 128 x 128 B A tile + up to 256 x 128 B B tile per stage
//               (SWIZZLE_128B, the same byte layout as the bf16 kernel's 64-column tiles),
//               3-stage mbarrier ring
//   warp 1      MMA issuer: per k-block four tcgen05.mma.cta_group::1.kind::f8f6f4 (M=128,
//               N=256 or 128, K=32) into one of two 256-column TMEM partial-sum buffers
//   warp 2      TMEM allocator (512 columns)
//   warps 2-3   epilogue writers: take each finished tile from a shared-memory staging
//               buffer (GEMM1: the SwiGLU activation and per-half-row maxima, quantised one
//               thread per row into e4m3 codes + scale; GEMM2: fp32 or bf16 rows, stored in
//               two 128-column halves as coalesced rows)
//   warps 4-11  promotion: warp w reads TMEM lanes 32*(w%4).., warps 4-7 and 8-11 split the
//               columns; per k-block they load the partial sums (tcgen05.ld), multiply by
//               row scale x weight-block scale and add into registers (packed fp32x2 FMAs),
//               then release the buffer; after the last k-block they stage the tile
// The tile order, bounded waits and abort path are those of the bf16 kernel (ffn_tc.cu).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "tc_common.cuh"

namespace moe {
namespace {

constexpr int F_BM = 128;                       // rows per tile
constexpr int F_BN = 256;                       // n-tile width (GEMM2 uses 128 when H % 256 != 0)
constexpr int F_BK = 128;                       // k elements (bytes) per stage
constexpr int F_A_BYTES = F_BM * F_BK;          // 16 KB
constexpr int F_B_BYTES = F_BN * F_BK;          // 32 KB
constexpr int F_STAGE = F_A_BYTES + F_B_BYTES;  // 48 KB
constexpr int F_THREADS = 384;
constexpr int F_EPI_WARPS = 8;
constexpr int F_TMEM_COLS = 512;                // two 128 x 256 fp32 partial-sum buffers
// Register split (setmaxnreg): the control warpgroup (warps 0-3) gives registers to the two
// promotion warpgroups, which hold a 128-float accumulator plus a 64-column load per thread.
// The shares must add up to the launch's total, F_THREADS x F_LAUNCH_REGS (checked on the
// host against the compiled register count before the first launch).
constexpr int F_LAUNCH_REGS = 168;
constexpr int F_REGS_CTRL = 56;
constexpr int F_REGS_EPI = 224;
static_assert(128 * F_REGS_CTRL + 256 * F_REGS_EPI <= F_THREADS * F_LAUNCH_REGS, "register split");

// Shared memory: the TMA ring, 256 B of barriers and a 128 x 128 fp32 staging buffer,
// through which the promotion warps hand a finished tile to warps 2-3 so that the next
// tile's promotion does not wait for the epilogue.  GEMM1 stages the tile's activation
// (plus the two half-row maxima of each row) and warps 2-3 quantise and store it; GEMM2
// stages the 256-column fp32 tile in two 128-column halves and warps 2-3 store each half
// as coalesced rows.
template <int MODE> struct F8Smem {
    static constexpr int kStages = 3;
    static constexpr int kActBytes = F_BM * 128 * 4;
    static constexpr int kBytes = kStages * F_STAGE + 1024 /*align*/ + 256 + kActBytes + (MODE == 0 ? 1024 : 0);
};

// Instruction descriptor of tcgen05.mma kind::f8f6f4: D fp32 (bits 4-5 = 1), A and B
// e4m3 (format 0 in bits 7-9 and 10-12), both K-major (bits 15/16 = 0), N >> 3 at bits
// 17-22, M >> 4 at bits 24-28.
__host__ __device__ constexpr uint32_t make_idesc_f8(int m, int n) {
    return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

struct F8Args {
    const int32_t *counts, *offsets;
    const int32_t *mprefix;   // prefix over experts of ceil(rows / 128)
    int E;
    int bn;                   // n-tile width: 256 or 128
    int nb;                   // n-blocks per expert (N / bn)
    int kb;                   // k-blocks (K / 128)
    int a_mode;               // 0: A row = e*a_cap + m; 1: A row = offsets[e] + m
    int64_t a_cap;
    const float *a_scale;     // [K/128][a_scale_ld]: scale of A row r, k-block kb
    int64_t a_scale_ld;
    int64_t b_rows;           // rows of B per expert (N)
    const float *b_scale;     // [E][N/128][K/128]
    int mode;                 // 0: SwiGLU -> e4m3 act + scales; 1: fp32 rows
    int out_bf16;             // mode 1: rows stored as bf16 (round to nearest even)
    void *out;                // mode 0: act codes [P, I]; mode 1: fp32 rows
    float *out_scale;         // mode 0: act scales [I/128][out_scale_ld]
    int64_t out_scale_ld;
    int64_t out_ld;           // elements per output row
    int out_mode;             // 0: row = e*out_cap + m; 1: row = offsets[e] + m
    int64_t out_cap;
    int32_t *status;
};

__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void decode_tile_f8(const F8Args &a, int tile, int &e, int &mb, int &nbk) {
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

__device__ __forceinline__ void fp8_scale_dev(float amax, float &scale, float &inv) {
    const float a = fmaxf(amax, 0x1p-100f);
    scale = __fdiv_rn(a, 448.0f);
    inv = __fdiv_rn(448.0f, a);
}

__device__ __forceinline__ uint32_t e4m3x4_dev(float v0, float v1, float v2, float v3, float inv) {
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(__fmul_rn(v0, inv), __fmul_rn(v1, inv)),
                                                 __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(__fmul_rn(v2, inv), __fmul_rn(v3, inv)),
                                                 __NV_SATFINITE, __NV_E4M3);
    return lo | (hi << 16);
}

// acc[base/2 + i] += c * partial[col + 2i, col + 2i + 1], i < 32, for this warp's 32 TMEM
// lanes: one tensor-memory load round trip per 64 columns, packed fp32x2 FMAs (half the
// issue slots of scalar FMAs, which otherwise bound the promotion)
template <int BASE>
__device__ __forceinline__ void promote64(float2 (&acc)[64], uint32_t taddr, float c) {
    uint32_t v[64];
    tmem_ld64(taddr, v);
    tmem_wait_ld();
    const float2 cc = make_float2(c, c);
#pragma unroll
    for (int i = 0; i < 32; ++i)
        acc[BASE / 2 + i] = __ffma2_rn(make_float2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])),
                                       cc, acc[BASE / 2 + i]);
}

template <int MODE>
__global__ void __launch_bounds__(F_THREADS, 1)
    ffn_gemm_fp8_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        F8Args a) {
    constexpr int F_STAGES = F8Smem<MODE>::kStages;
    // the set-up below touches no global memory; pdl_wait() follows it
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t *sA = smem;                          // [STAGES] A tiles
    uint8_t *sB = smem + F_STAGES * F_A_BYTES;   // [STAGES] B tiles
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + F_STAGES * F_STAGE);
    // bars: full[STAGES], empty[STAGES], pfull[2], pempty[2], afull[2], aempty[2] (one pair
    // per staged half: GEMM1 uses pair 0 for the whole tile)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * F_STAGES + 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    // staging [128 rows][32 chunks of 4 floats], chunk q of row r stored at slot q ^ (r % 32)
    // (conflict-free row writes by lane = row and row reads by lane = q)
    float4 *act_s = reinterpret_cast<float4 *>(smem + F_STAGES * F_STAGE + 256);
    float *amax_s = reinterpret_cast<float *>(smem + F_STAGES * F_STAGE + 256 + F8Smem<MODE>::kActBytes);  // [2][128]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + F_STAGES);
    const uint32_t pfull0 = smem_u32(bars + 2 * F_STAGES), pempty0 = smem_u32(bars + 2 * F_STAGES + 2);
    const uint32_t afull0 = smem_u32(bars + 2 * F_STAGES + 4), aempty0 = smem_u32(bars + 2 * F_STAGES + 6);
    const uint32_t afull = afull0, aempty = aempty0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < F_STAGES; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(pfull0 + 8 * s, 1);
            mbar_init(pempty0 + 8 * s, F_EPI_WARPS);   // one arrival per promotion warp
        }
        for (int h = 0; h < 2; ++h) {
            // staged by the promotion warps (GEMM1: all eight; GEMM2: the four of the half)
            mbar_init(afull0 + 8 * h, MODE == 0 ? F_EPI_WARPS : F_EPI_WARPS / 2);
            mbar_init(aempty0 + 8 * h, 2);   // consumed by warps 2, 3
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
    }
    if (warp == 2) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(F_TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    pdl_wait();   // the previous kernel in the stream has completed: its outputs are visible
    const int total = __ldg(a.mprefix + a.E) * a.nb;
    // GEMM2 stages 256-column tiles of at least three k-blocks: then a promotion warp that
    // stages a half is never two phases of that half's barrier ahead of the storing warps
    // (the MMA of its tile's last k-block waited for every warp's promotion of an earlier
    // k-block of the same tile).  Otherwise the promotion warps store their rows directly.
    const bool staged = MODE == 0 || (a.bn == 256 && a.kb >= 3);
    if (warp < 4) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(F_REGS_CTRL));
        if (warp == 0 && lane == 0) {
            // ------------------------------------------------------------- TMA producer
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            const uint32_t tx = (uint32_t)(F_A_BYTES + a.bn * F_BK);
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
                int e, mb, nbk;
                decode_tile_f8(a, tile, e, mb, nbk);
                const int64_t arow = (a.a_mode == 0 ? (int64_t)e * a.a_cap : (int64_t)__ldg(a.offsets + e)) +
                                     (int64_t)mb * F_BM;
                const int64_t brow = (int64_t)e * a.b_rows + (int64_t)nbk * a.bn;
                for (int kb = 0; kb < a.kb; ++kb) {
                    if (!mbar_wait(empty0 + 8 * stage, phase ^ 1, abort_flag, a.status)) { ok = false; break; }
                    const uint32_t fb = full0 + 8 * stage;
                    mbar_expect_tx(fb, tx);
                    tma_load_2d(smem_u32(sA + stage * F_A_BYTES), &tmA, kb * F_BK, (int)arow, fb);
                    tma_load_2d(smem_u32(sB + stage * F_B_BYTES), &tmB, kb * F_BK, (int)brow, fb);
                    if (++stage == F_STAGES) { stage = 0; phase ^= 1; }
                }
            }
        } else if (warp == 1 && lane == 0) {
            // ---------------------------------------------------------------- MMA issuer
            int stage = 0;
            uint32_t phase = 0;
            uint32_t it = 0;   // k-blocks issued so far (partial-sum buffer it & 1)
            bool ok = true;
            const uint32_t idesc = make_idesc_f8(F_BM, a.bn);
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
                for (int kb = 0; kb < a.kb; ++kb, ++it) {
                    const uint32_t pb = it & 1, pph = (it >> 1) & 1;
                    if (!mbar_wait(pempty0 + 8 * pb, pph ^ 1, abort_flag, a.status)) { ok = false; break; }
                    tc_fence_after();
                    if (!mbar_wait(full0 + 8 * stage, phase, abort_flag, a.status)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + pb * (uint32_t)F_BN;
                    const uint32_t a0 = smem_u32(sA + stage * F_A_BYTES);
                    const uint32_t b0 = smem_u32(sB + stage * F_B_BYTES);
#pragma unroll
                    for (int kk = 0; kk < F_BK / 32; ++kk)
                        mma_f8(d_tmem, sw128_desc(a0 + kk * 32), sw128_desc(b0 + kk * 32), idesc, kk != 0 ? 1u : 0u);
                    mma_commit(empty0 + 8 * stage);   // the stage is reusable once these finish
                    mma_commit(pfull0 + 8 * pb);      // the partial sum is ready
                    if (++stage == F_STAGES) { stage = 0; phase ^= 1; }
                }
            }
        } else if (MODE == 0 && (warp == 2 || warp == 3)) {
            // ------------------------------------------- activation quantisation (GEMM1)
            // Thread t (0..63) owns rows t and t + 64: the row's amax is the larger of the
            // two half-row maxima the promotion warps staged, the scale is computed once per
            // row, and the 128 codes go out as eight 16-byte stores.
            const int qt = threadIdx.x - 64;
            int ntile = 0;
            for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++ntile) {
                int e, mb, nbk;
                decode_tile_f8(a, tile, e, mb, nbk);
                const int m0 = mb * F_BM;
                const int valid = min(F_BM, __ldg(a.counts + e) - m0);
                const int64_t obase = (int64_t)__ldg(a.offsets + e) + m0;   // act rows: pick list
                if (!mbar_wait(afull, (uint32_t)ntile & 1, abort_flag, a.status)) break;
                for (int r = qt; r < valid; r += 64) {
                    float scale, inv;
                    fp8_scale_dev(fmaxf(amax_s[r], amax_s[F_BM + r]), scale, inv);
                    uint4 *o = reinterpret_cast<uint4 *>(reinterpret_cast<uint8_t *>(a.out) + (obase + r) * a.out_ld +
                                                         (int64_t)nbk * 128);
#pragma unroll 2
                    for (int c = 0; c < 8; ++c) {   // 16 columns: chunks 4c .. 4c + 3
                        uint32_t w[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const float4 v = act_s[r * 32 + ((4 * c + j) ^ (r & 31))];
                            w[j] = e4m3x4_dev(v.x, v.y, v.z, v.w, inv);
                        }
                        o[c] = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                    a.out_scale[(int64_t)nbk * a.out_scale_ld + obase + r] = scale;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(aempty);
            }
        } else if (MODE == 1 && staged && (warp == 2 || warp == 3)) {
            // --------------------------------------------------- fp32 tile store (GEMM2)
            // Per half of the tile: one row per warp at a time (warp 2 even rows, warp 3
            // odd); lane l holds columns 4l..4l+3 of the half, so a row leaves as one
            // coalesced 512-byte store.
            int ntile = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++ntile) {
                int e, mb, nbk;
                decode_tile_f8(a, tile, e, mb, nbk);
                const int m0 = mb * F_BM;
                const int valid = min(F_BM, __ldg(a.counts + e) - m0);
                const int64_t obase =
                    (a.out_mode == 0 ? (int64_t)e * a.out_cap : (int64_t)__ldg(a.offsets + e)) + m0;
                for (int h = 0; h < 2; ++h) {
                    if (!mbar_wait(afull0 + 8 * h, (uint32_t)ntile & 1, abort_flag, a.status)) { ok = false; break; }
                    const int64_t col = (int64_t)nbk * a.bn + 128 * h + 4 * lane;
                    if (a.out_bf16) {
                        __nv_bfloat16 *out = reinterpret_cast<__nv_bfloat16 *>(a.out) + col;
#pragma unroll 4
                        for (int r = warp - 2; r < valid; r += 2) {
                            const float4 v = act_s[r * 32 + (lane ^ (r & 31))];
                            __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
                            *reinterpret_cast<uint2 *>(out + (obase + r) * a.out_ld) =
                                make_uint2(*reinterpret_cast<uint32_t *>(&lo), *reinterpret_cast<uint32_t *>(&hi));
                        }
                    } else {
                        float *out = reinterpret_cast<float *>(a.out) + col;
#pragma unroll 4
                        for (int r = warp - 2; r < valid; r += 2)
                            *reinterpret_cast<float4 *>(out + (obase + r) * a.out_ld) = act_s[r * 32 + (lane ^ (r & 31))];
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(aempty0 + 8 * h);
                }
            }
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(F_REGS_EPI));
        // -------------------------------------------------------- promotion + epilogue
        const int quad = warp & 3;                  // TMEM lanes 32*quad .. 32*quad+31
        const int half = (warp - 4) >> 2;           // which columns of the tile
        const int row = quad * 32 + lane;           // row inside the tile
        // columns of this thread: GEMM1 gate [64h, 64h+64) and up [128+64h, ...);
        // GEMM2 [h*bn/2, (h+1)*bn/2)
        const int ncol = MODE == 0 ? 64 : a.bn / 2;
        uint32_t it = 0;
        int ntile = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++ntile) {
            int e, mb, nbk;
            decode_tile_f8(a, tile, e, mb, nbk);
            const int m0 = mb * F_BM;
            const bool live = row < __ldg(a.counts + e) - m0;
            const int64_t arow = (a.a_mode == 0 ? (int64_t)e * a.a_cap : (int64_t)__ldg(a.offsets + e)) +
                                 (int64_t)m0 + row;
            const int bblocks = (int)(a.b_rows / 128);
            const int blk0 = MODE == 0 ? 2 * nbk : (a.bn == 256 ? 2 * nbk + half : nbk);
            const float *sb0p = a.b_scale + ((int64_t)e * bblocks + blk0) * a.kb;
            const float *sb1p = sb0p + a.kb;   // GEMM1: the up block (2 * nbk + 1)
            float2 acc[64];   // columns 2i, 2i + 1
#pragma unroll
            for (int i = 0; i < 64; ++i) acc[i] = make_float2(0.f, 0.f);
            // Scales of the next four k-blocks, shifted along a register queue (a k-block's
            // row scales are 4 * a_scale_ld bytes apart: after the L2 flush each one is a DRAM
            // round trip, longer than one k-block of promotion)
            auto ld_sa = [&](int kb) {
                return kb < a.kb && live ? __ldg(a.a_scale + (int64_t)kb * a.a_scale_ld + arow) : 0.f;
            };
            auto ld_sb = [&](const float *p, int kb) { return kb < a.kb ? __ldg(p + kb) : 0.f; };
            float sa0 = ld_sa(0), sa1 = ld_sa(1), sa2 = ld_sa(2), sa3 = ld_sa(3);
            float sg0 = ld_sb(sb0p, 0), sg1 = ld_sb(sb0p, 1), sg2 = ld_sb(sb0p, 2), sg3 = ld_sb(sb0p, 3);
            float su0 = 0.f, su1 = 0.f, su2 = 0.f, su3 = 0.f;
            if (MODE == 0) {
                su0 = ld_sb(sb1p, 0); su1 = ld_sb(sb1p, 1); su2 = ld_sb(sb1p, 2); su3 = ld_sb(sb1p, 3);
            }
            for (int kb = 0; kb < a.kb; ++kb, ++it) {
                const float c0 = sa0 * sg0, c1 = sa0 * su0;
                sa0 = sa1; sa1 = sa2; sa2 = sa3; sa3 = ld_sa(kb + 4);
                sg0 = sg1; sg1 = sg2; sg2 = sg3; sg3 = ld_sb(sb0p, kb + 4);
                if (MODE == 0) { su0 = su1; su1 = su2; su2 = su3; su3 = ld_sb(sb1p, kb + 4); }
                const uint32_t pb = it & 1, pph = (it >> 1) & 1;
                if (!mbar_wait(pfull0 + 8 * pb, pph, abort_flag, a.status)) { ok = false; break; }
                tc_fence_after();
                const uint32_t tb = tmem_base + pb * (uint32_t)F_BN + ((uint32_t)(quad * 32) << 16);
                if (MODE == 0) {
                    promote64<0>(acc, tb + 64 * half, c0);         // gate columns
                    promote64<64>(acc, tb + 128 + 64 * half, c1);  // up columns
                } else {
                    const uint32_t t0 = tb + (uint32_t)(ncol * half);
                    promote64<0>(acc, t0, c0);
                    if (ncol == 128) promote64<64>(acc, t0 + 64, c0);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(pempty0 + 8 * pb);   // buffer free for k-block it + 2
            }
            if (!ok) break;
            const int64_t orow = (a.out_mode == 0 ? (int64_t)e * a.out_cap : (int64_t)__ldg(a.offsets + e)) +
                                 (int64_t)m0 + row;
            if (MODE == 0) {
                // act = silu(gate) * up (gate columns in acc[0, 32), up in acc[32, 64)),
                // staged for the quantising warps once they are done with the previous tile
                if (!mbar_wait(aempty, ((uint32_t)ntile & 1) ^ 1, abort_flag, a.status)) break;
                float amax = 0.f;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float2 g0 = acc[2 * j], g1 = acc[2 * j + 1];
                    const float2 u0 = acc[32 + 2 * j], u1 = acc[32 + 2 * j + 1];
                    const float4 v = make_float4(silu_mul_fast(g0.x, u0.x), silu_mul_fast(g0.y, u0.y),
                                                 silu_mul_fast(g1.x, u1.x), silu_mul_fast(g1.y, u1.y));
                    amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
                    act_s[row * 32 + ((16 * half + j) ^ (row & 31))] = v;
                }
                amax_s[half * F_BM + row] = amax;
                __syncwarp();
                if (lane == 0) mbar_arrive(afull);
            } else if (staged) {
                // fp32 rows, staged half by half: half 0 once the storing warps are done with
                // half 1 of the previous tile, half 1 once they are done with this tile's half 0
                const uint32_t wait_bar = half == 0 ? aempty0 + 8 : aempty0;
                const uint32_t wait_par = half == 0 ? (((uint32_t)ntile & 1) ^ 1) : ((uint32_t)ntile & 1);
                if (!mbar_wait(wait_bar, wait_par, abort_flag, a.status)) break;
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    act_s[row * 32 + (j ^ (row & 31))] =
                        make_float4(acc[2 * j].x, acc[2 * j].y, acc[2 * j + 1].x, acc[2 * j + 1].y);
                __syncwarp();
                if (lane == 0) mbar_arrive(afull0 + 8 * half);
            } else if (live && a.out_bf16) {
                // direct row stores: ncol = 64 (128-column tiles) or 128 columns per thread
                uint4 *o = reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(a.out) + orow * a.out_ld +
                                                     (int64_t)nbk * a.bn + half * ncol);
                auto pk = [](float2 v) {
                    __nv_bfloat162 b = __floats2bfloat162_rn(v.x, v.y);
                    return *reinterpret_cast<uint32_t *>(&b);
                };
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    o[q] = make_uint4(pk(acc[4 * q]), pk(acc[4 * q + 1]), pk(acc[4 * q + 2]), pk(acc[4 * q + 3]));
                if (ncol == 128) {
#pragma unroll
                    for (int q = 8; q < 16; ++q)
                        o[q] = make_uint4(pk(acc[4 * q]), pk(acc[4 * q + 1]), pk(acc[4 * q + 2]), pk(acc[4 * q + 3]));
                }
            } else if (live) {
                float4 *o = reinterpret_cast<float4 *>(reinterpret_cast<float *>(a.out) + orow * a.out_ld +
                                                       (int64_t)nbk * a.bn + half * ncol);
#pragma unroll
                for (int q = 0; q < 16; ++q)
                    o[q] = make_float4(acc[2 * q].x, acc[2 * q].y, acc[2 * q + 1].x, acc[2 * q + 1].y);
                if (ncol == 128) {
#pragma unroll
                    for (int q = 16; q < 32; ++q)
                        o[q] = make_float4(acc[2 * q].x, acc[2 * q].y, acc[2 * q + 1].x, acc[2 * q + 1].y);
                }
            }
        }
    }

    __syncthreads();
    if (*abort_flag) {
        // Give in-flight TMA copies and MMAs time to land before the memory is released.
        unsigned long long t0 = globaltimer();
        while (globaltimer() - t0 < 1000000ull) {}
    }
    if (warp == 2) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(F_TMEM_COLS)
                     : "memory");
    }
}

template <int MODE>
int launch_gemm_fp8(const CUtensorMap &ma, const CUtensorMap &mb, const F8Args &args, int64_t max_tiles,
                    cudaStream_t s) {
    if (max_tiles <= 0) return MOE_OK;
    auto kernel = ffn_gemm_fp8_kernel<MODE>;
    constexpr int smem = F8Smem<MODE>::kBytes;
    // kernel attributes are set per device (with that device current), once each
    struct PerDevice {
        std::once_flag once;
        cudaError_t attr_err = cudaSuccess;
    };
    static PerDevice per_device[64];
    const int dev = device_ordinal();
    if (dev < 0) return MOE_ERR_CUDA;
    PerDevice &pd = per_device[dev];
    cudaError_t &attr_err = pd.attr_err;
    std::call_once(pd.once, [&] {
        attr_err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        // setmaxnreg.inc waits until the registers it asks for are free in the CTA's launch
        // allocation: never launch a build whose register count makes the split too large
        cudaFuncAttributes fa{};
        if (attr_err == cudaSuccess) attr_err = cudaFuncGetAttributes(&fa, kernel);
        if (attr_err == cudaSuccess && fa.numRegs * F_THREADS < 128 * F_REGS_CTRL + 256 * F_REGS_EPI)
            attr_err = cudaErrorInvalidConfiguration;
    });
    if (attr_err != cudaSuccess) return MOE_ERR_CUDA;
    int grid = num_sms();
    if ((int64_t)grid > max_tiles) grid = (int)max_tiles;
    return launch_pdl(kernel, dim3(grid), dim3(F_THREADS), smem, s, ma, mb, args) == cudaSuccess ? MOE_OK
                                                                                            : MOE_ERR_CUDA;
}

bool make_map_u8(CUtensorMap *m, const void *base, int64_t rows, int64_t cols, int box_rows) {
    return make_map_2d(m, base, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, rows, cols, box_rows);
}

F8Args base_args_f8(const Routing &r) {
    const Plan &p = *r.p;
    F8Args g{};
    g.counts = r.counts; g.offsets = r.offsets; g.mprefix = r.mprefix;
    g.E = (int)p.E;
    g.status = r.status;
    return g;
}

}  // namespace

int launch_gemm1_fp8(const Routing &r, const uint8_t *w1qp, const float *w1sp, cudaStream_t s) {
    const Plan &p = *r.p;
    if (p.P == 0) return MOE_OK;
    const bool em = p.layout == MOE_LAYOUT_EXPERT_MAJOR;
    CUtensorMap mA, mB;
    const void *a1 = em ? (const void *)r.recv_x : (const void *)r.apick;
    const int64_t a1_rows = em ? p.E * p.cap : p.P;
    if (!make_map_u8(&mA, a1, a1_rows, p.H, F_BM) || !make_map_u8(&mB, w1qp, p.E * 2 * p.I, p.H, F_BN))
        return MOE_ERR_CUDA;
    F8Args g = base_args_f8(r);
    g.bn = F_BN; g.nb = (int)(2 * p.I / F_BN); g.kb = (int)(p.H / F_BK);
    g.a_mode = em ? 0 : 1; g.a_cap = p.cap;
    g.a_scale = em ? r.recv_scales : r.apick_scales; g.a_scale_ld = em ? p.nrecv : p.P;
    g.b_rows = 2 * p.I; g.b_scale = w1sp;
    g.mode = 0; g.out = r.act; g.out_scale = r.act_scales; g.out_scale_ld = p.P;
    g.out_ld = p.I; g.out_mode = 1; g.out_cap = 0;
    return launch_gemm_fp8<0>(mA, mB, g, (p.P / F_BM + p.E) * g.nb, s);
}

int launch_gemm2_fp8(const Routing &r, const uint8_t *w2q, const float *w2s, void *expert_out,
                     cudaStream_t s) {
    const Plan &p = *r.p;
    if (p.P == 0) return MOE_OK;
    const bool em = p.layout == MOE_LAYOUT_EXPERT_MAJOR;
    const int bn = (p.H % 256 == 0) ? 256 : 128;
    CUtensorMap mA, mB;
    if (!make_map_u8(&mA, r.act, p.P, p.I, F_BM) || !make_map_u8(&mB, w2q, p.E * p.H, p.I, bn))
        return MOE_ERR_CUDA;
    F8Args g = base_args_f8(r);
    g.bn = bn; g.nb = (int)(p.H / bn); g.kb = (int)(p.I / F_BK);
    g.a_mode = 1; g.a_cap = 0; g.a_scale = r.act_scales; g.a_scale_ld = p.P;
    g.b_rows = p.H; g.b_scale = w2s;
    g.mode = 1; g.out_ld = p.H; g.out_bf16 = p.eo_bf16;
    if (em) { g.out = expert_out; g.out_mode = 0; g.out_cap = p.cap; }
    else { g.out = r.ypick; g.out_mode = 1; g.out_cap = 0; }
    return launch_gemm_fp8<1>(mA, mB, g, (p.P / F_BM + p.E) * g.nb, s);
}

}  // namespace moe
