// Internal declarations shared by the library's translation units: workspace plan,
// kernel launch wrappers and small device helpers.  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/moe.h"

namespace moe {

constexpr int kRouteThreads = 256;   // 8 warps per routing block
constexpr int kRouteWarps = kRouteThreads / 32;
constexpr int kTileM = 128;          // GEMM rows per tile (one tcgen05 M=128 MMA)
constexpr uint64_t kHandleMagic = 0x4d6f4545702d3130ull;

// Byte offsets of every region of the workspace, derived from the geometry alone.
struct Plan {
    int64_t T, W, Tr, cap, E, k, H, I, P;   // P = T*k picks
    int layout;
    int quant;      // moe_quant
    int eo_bf16;    // expert_out (and the RM/FLAT per-pick rows) in bf16
    int act_pair;   // bf16 geometry: SwiGLU activation as a bf16 (hi, lo) pair
    int64_t nrecv;  // rows of the receive buffer: E*cap (EM) or W*cap (RM/FLAT)
    int tb;         // tokens per routing block
    int nbpr;       // routing blocks per logical rank
    int nb;         // routing blocks in total (W * nbpr)
    size_t status, counts, offsets, mprefix, mprefix2, pick_pos, pick_src, slot, layout_range,
        blk_hist, blk_base, recv_row, recv_count, num_recv, recv_src, recv_topk_idx,
        recv_topk_w, blk_dhist, blk_dbase, recv_x, recv_scales, act, act_lo, act_scales, apick,
        apick_scales, ypick, direct_row, direct_w, total;
};

// Returns MOE_OK or a moe_error for an invalid geometry.
int make_plan(const moe_geom &g, Plan *p);

// Workspace pointers of one dispatch.
struct Routing {
    const Plan *p;
    int32_t *status, *counts, *offsets, *mprefix, *mprefix2, *pick_pos, *pick_src, *slot, *layout_range,
        *blk_hist, *blk_base, *recv_row, *recv_count, *num_recv, *recv_src, *recv_topk_idx,
        *blk_dhist, *blk_dbase;
    float *recv_topk_w;
    uint16_t *recv_x, *act, *act_lo, *apick;   // act (and act_lo for the pair): SwiGLU output
    void *ypick;    // RM/FLAT per-pick GEMM2 rows: float32, or bf16 with eo_bf16
    // RM/FLAT, per pick in pick-list order: the expert_out row (d*cap + r) when the pick is
    // the only local pick of its received row, else -1; and that pick's routing weight.
    // Written by the dispatch row scatter; the bf16 second GEMM then stores weight * y
    // straight into expert_out for such picks, and the local-pick reduction skips the row.
    int32_t *direct_row;
    float *direct_w;
    // the two GEMMs' tile counters for the dynamic tile order ([0..1] first GEMM, [2..3]
    // second), right after the status word; zeroed with it by the routing launch, and by
    // each GEMM for its next launch; NULL when the routing runs without a workspace
    int32_t *sched;
    // FP8 geometry: recv_x / act / apick hold e4m3 codes (one byte per element); their
    // scales are column-block major ([cols/128][rows]); act_lo is unused
    float *recv_scales, *act_scales, *apick_scales;
};

Routing carve(const Plan &p, void *ws);

// ---- launchers (return cudaGetLastError of the launch) -------------------------------
// Also clears the status word (before any routing kernel can set a bit).
cudaError_t launch_routing(const Routing &r, const void *ids, int ids64, const float *topk_w,
                           const int32_t *active, cudaStream_t s);
int routing_launches(const Plan &p);   // kernels launch_routing queues for this geometry
cudaError_t launch_dispatch_copy(const Routing &r, const uint16_t *x, cudaStream_t s);
// expert_out: float32, or bf16 when the plan's eo_bf16 is set.  skip_single: rows with one
// local pick were already written by the second GEMM (direct_row)
cudaError_t launch_reduce_ranks(const Routing &r, void *expert_out, bool skip_single, cudaStream_t s);
cudaError_t launch_combine(const Routing &r, const void *expert_out, const float *topk_w,
                           uint16_t *out, cudaStream_t s);
// RANK_MAJOR / FLAT: the combine fused with the rank reduction (multi-pick rows summed from
// the per-pick rows on the fly; bf16 geometries whose second GEMM wrote the one-pick rows)
cudaError_t launch_combine_fused(const Routing &r, const void *expert_out, uint16_t *out, cudaStream_t s);
cudaError_t launch_prepare_w1(const moe_geom &g, const uint16_t *w1, uint16_t *w1p,
                              cudaStream_t s);
// Grouped SwiGLU FFN: GEMM1 (+SiLU*mul) into act, GEMM2 into expert_out (EM) or the
// per-pick scratch (RM/FLAT).  Return MOE_OK or a moe_error.
int launch_gemm1(const Routing &r, const uint16_t *w1p, cudaStream_t s);
int launch_gemm2(const Routing &r, const uint16_t *w2, void *expert_out, cudaStream_t s);

// ---- FP8 (moe_quant MOE_QUANT_FP8_E4M3) -----------------------------------------------
cudaError_t launch_dispatch_quant(const Routing &r, const uint16_t *x, cudaStream_t s);
// 128x128-block quantisation of bf16 [E, rows, cols] weights; w1_inter = I interleaves the
// gate/up row blocks of W1 (0: keep the order)
cudaError_t launch_quantize_weights_fp8(const uint16_t *w, int64_t E, int64_t rows, int64_t cols,
                                        int64_t w1_inter, uint8_t *q, float *sc, cudaStream_t s);
cudaError_t launch_prepare_w1_fp8(const moe_geom &g, const uint8_t *w1q, const float *w1s,
                                  uint8_t *w1qp, float *w1sp, cudaStream_t s);
int launch_gemm1_fp8(const Routing &r, const uint8_t *w1qp, const float *w1sp, cudaStream_t s);
int launch_gemm2_fp8(const Routing &r, const uint8_t *w2q, const float *w2s, void *expert_out,
                     cudaStream_t s);

int num_sms();   // SM count of the current device (cached per device)
int check_device();   // MOE_OK on a compute capability 10.3 device, else a moe_error
int device_ordinal();   // the current device, or -1 (only ordinals below 64 are served)

// ---- programmatic dependent launch -----------------------------------------------------
// The layer's kernels are launched with programmatic stream serialization, so the launch of
// a kernel is processed while the previous one in the stream runs and its CTAs start as
// soon as that kernel has finished.  Each kernel waits (pdl_wait) until the previous one
// has completed and its memory is visible before it touches global memory; the GEMMs set
// up barriers and tensor memory first.  No kernel triggers its dependents early
// (griddepcontrol.launch_dependents): measured on GB300, an early trigger saved 3% on the
// 64-token batch but cost 3% on the 1024-token Mixtral-like batch under graph replay.
// The data order is the plain stream order.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_begin() { pdl_wait(); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace moe
