/*
 * moe.h - C ABI of a one-GPU Mixture-of-Experts expert-parallel layer for GB300 (sm_103a):
 *
 *     moe_dispatch  ->  moe_expert_ffn  ->  moe_combine
 *
 * The "world" of source ranks is a logical partition of one token batch that lives in one
 * device buffer: token t belongs to logical rank t / max_tok and expert e lives on logical
 * rank e / (num_experts / world).  There is no transport and no collective; the pages'
 * all-to-all exchange becomes a row permutation inside one HBM.
 *
 * Sources (page title, section):
 *   [MC-EP]  Mooncake EP user guide, "Mooncake EP API reference": Buffer.dispatch /
 *            Buffer.combine / Buffer.get_ep_buffer_size_hint, the packed
 *            local-expert-major receive layout and its handle, the input assertions.
 *   [FI-3]   FlashInfer "MoE-EP implementation & usage", section 3 "Algorithm / layout
 *            contracts": EXPERT_MAJOR / RANK_MAJOR / FLAT receive buffers, compute
 *            routing and combine rules.
 *   [FI-2]   same page, section 2 "Call stack": dispatch -> per-expert grouped GEMM
 *            (no routing) -> combine -> [num_tokens, hidden] bf16.
 *   [FI-4]   same page, section 4 step 1: w1 [E, 2*I, H], w2 [E, H, I].
 *
 * Conventions for every entry point:
 *   - Every pointer argument named *_dev, every pointer inside moe_handle and the
 *     workspace are DEVICE pointers of the current CUDA device.  Host pointers are named
 *     *_host.  The caller owns and allocates all memory; the library never allocates,
 *     frees or keeps global state beyond cached device attributes.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *     stream-ordered and asynchronous: they return once the kernels are queued and never
 *     synchronise the host (moe_get_status excepted).
 *   - Return value: MOE_OK (0) or a negative moe_error.  Host-detected errors return
 *     before anything is queued.  Errors found by the kernels (bad expert ids, an
 *     overflowing expert region, a device wait that gave up) set bits of the handle's
 *     device status word, read with moe_get_status; the offending pick is dropped,
 *     never written out of bounds.
 *   - bf16 arrays hold IEEE bfloat16 bit patterns (uint16).
 */
#ifndef COMBINE_TOPK_IDS_MOE_H
#define COMBINE_TOPK_IDS_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Receive layout [FI-3]. */
typedef enum {
    MOE_LAYOUT_EXPERT_MAJOR = 0, /* [num_experts, world*max_tok, hidden], rows pre-assigned to experts */
    MOE_LAYOUT_RANK_MAJOR = 1,   /* per destination rank: [world(source), max_tok, hidden]             */
    MOE_LAYOUT_FLAT = 2          /* per destination rank: [num_recv, hidden] token-major               */
} moe_layout;

/* EpAlgorithm [FI-3]: recorded in the geometry; both run the same kernels on one GPU. */
typedef enum { MOE_ALGO_LOW_LATENCY = 0, MOE_ALGO_HIGH_THROUGHPUT = 1 } moe_algorithm;

typedef enum { MOE_IDS_INT32 = 0, MOE_IDS_INT64 = 1 } moe_ids_dtype;

/*
 * Precision of the received rows and of the expert GEMMs [MC-EP Buffer.dispatch use_fp8:
 * with it the dispatch returns (packed FP8 data, packed scales) instead of bf16 rows].
 *   MOE_QUANT_NONE      bf16 rows, bf16 x bf16 -> fp32 GEMMs (moe_expert_ffn).
 *   MOE_QUANT_FP8_E4M3  the dispatch quantises every token row to OCP e4m3 ("fn": bias 7,
 *                       largest finite 448, no infinities) with one float32 scale per 128
 *                       columns; the FFN (moe_expert_ffn_fp8) runs e4m3 x e4m3 -> fp32
 *                       GEMMs on FP8 weights with one scale per 128 x 128 block and
 *                       quantises the SwiGLU activation the same way per 128 columns.
 *   Quantisation of a block with largest magnitude amax (all float32, IEEE rounding):
 *       a = max(amax, 2^-100); scale = a / 448; code = e4m3_rne_satfinite(v * (448 / a));
 *   the dequantised value is code * scale.  The page leaves the scale granularity and
 *   rule open; this is the library's reading.
 */
typedef enum { MOE_QUANT_NONE = 0, MOE_QUANT_FP8_E4M3 = 1 } moe_quant;

/*
 * Element type of expert_out (the expert stage's output and combine's input) and of the
 * per-pick rows the RANK_MAJOR / FLAT expert stage reduces [FI-3: the packed buffers that
 * return to combine are bf16].
 *   MOE_EXPERT_OUT_FLOAT32   float32 (default).
 *   MOE_EXPERT_OUT_BFLOAT16  bfloat16, rounded to nearest even from the fp32 GEMM result
 *                            (and, for RANK_MAJOR / FLAT, once more after the fp32 sum over
 *                            the row's local picks); combine accumulates in fp32 as before.
 *                            Half the bytes of the largest intermediate, at the price of
 *                            one or two extra bf16 roundings before the final one.
 */
typedef enum { MOE_EXPERT_OUT_FLOAT32 = 0, MOE_EXPERT_OUT_BFLOAT16 = 1 } moe_expert_out_dtype;

/*
 * The SwiGLU activation as the second GEMM's operand (bf16 geometries; FP8 geometries
 * quantise it to e4m3 instead).  The expert GEMMs take bf16 operands [FI-4 step 3]; the
 * layer's output is checked against the expert FFN evaluated in full precision from the
 * bf16 weights [FI-4 step 6], which only the pair reaches within the output tolerance.
 *   MOE_ACT_BF16_PAIR  (default, 0) act carried as act_hi = bf16(act) plus
 *                      act_lo = bf16(act - act_hi), about 16 significant bits: GEMM2 runs
 *                      both halves (two bf16 MMAs per k-step), so y tracks the unrounded
 *                      activation to about 2e-4.
 *   MOE_ACT_BF16       act = bf16_rne(silu(g) * u), one bf16 x bf16 GEMM: faster (about
 *                      20% of the layer on tensor-bound batches), but each bf16 code is a
 *                      rounding decision on a tensor-core sum; codes that land on the other
 *                      side of a midpoint move y by |W2| x one bf16 step, which on long
 *                      GEMMs puts some outputs outside 2e-2*|ref| + 1e-3 of the
 *                      full-precision FFN.
 */
typedef enum { MOE_ACT_BF16_PAIR = 0, MOE_ACT_BF16 = 1 } moe_act_precision;

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARGUMENT = -1,      /* null pointer, non-positive size, bad enum          */
    MOE_ERR_EXPERTS_NOT_DIVISIBLE = -2, /* num_experts % world != 0            [MC-EP] asserts */
    MOE_ERR_HIDDEN_ALIGNMENT = -3,      /* hidden % 128 != 0                    [MC-EP] asserts */
    MOE_ERR_INTERMEDIATE_ALIGNMENT = -4,/* intermediate % 128 != 0 (GEMM tiling)               */
    MOE_ERR_TOO_MANY_TOKENS = -5,       /* num_tokens > world*max_tok  [MC-EP] max_tok rule     */
    MOE_ERR_TOPK = -6,                  /* top_k < 1 or > MOE_MAX_TOPK                          */
    MOE_ERR_IDS_DTYPE = -7,             /* ids dtype not int32/int64                            */
    MOE_ERR_WORKSPACE_TOO_SMALL = -8,   /* workspace_bytes < moe_workspace_size()               */
    MOE_ERR_MISALIGNED = -9,            /* a device pointer breaks its alignment rule           */
    MOE_ERR_BAD_HANDLE = -10,           /* handle not filled by moe_dispatch                    */
    MOE_ERR_CUDA = -11,                 /* a CUDA runtime call or kernel launch failed          */
    MOE_ERR_NOT_BUILT_FOR_DEVICE = -12, /* device is not compute capability 10.3 (sm_103a)      */
    MOE_ERR_LIMIT = -13                 /* world, num_experts or hidden beyond the limits below */
} moe_error;

/* Device status bits (moe_get_status). */
#define MOE_STATUS_BAD_EXPERT_ID 0x1  /* an id outside [-1, num_experts): pick dropped          */
#define MOE_STATUS_EM_OVERFLOW 0x2    /* EXPERT_MAJOR region full (a token named one expert
                                         twice): the later picks were dropped                 */
#define MOE_STATUS_TIMEOUT 0x4        /* a bounded device wait gave up; outputs are invalid    */
#define MOE_STATUS_INACTIVE_RANK 0x8  /* picks were dropped by the active_ranks mask
                                         (informational)                                      */

/* Event slots of moe_handle.events (per-kernel timing). */
#define MOE_EV_DISPATCH_BEGIN 0
#define MOE_EV_ROUTING_END 1   /* after the three routing kernels                         */
#define MOE_EV_DISPATCH_END 2  /* after the row scatter                                   */
#define MOE_EV_FFN_BEGIN 3
#define MOE_EV_GATHER_END 4    /* recorded right after MOE_EV_FFN_BEGIN (the pick-ordered
                                  RANK_MAJOR / FLAT rows are written by moe_dispatch)      */
#define MOE_EV_GEMM1_END 5     /* after GEMM1 + SwiGLU                                    */
#define MOE_EV_GEMM2_END 6     /* after GEMM2                                             */
#define MOE_EV_FFN_END 7       /* after the RANK_MAJOR / FLAT local-pick reduction        */
#define MOE_EV_COMBINE_BEGIN 8
#define MOE_EV_COMBINE_END 9
#define MOE_EV_COUNT 10

#define MOE_MAX_TOPK 32
#define MOE_MAX_WORLD 64
#define MOE_MAX_EXPERTS 2048
#define MOE_MAX_HIDDEN 65536

/* EP geometry, the analogue of FleetParams [FI-3 table; section 1] plus the FFN size. */
typedef struct {
    int32_t world;        /* W: logical ranks                                              */
    int32_t max_tok;      /* Tr: num_max_dispatch_tokens_per_rank [MC-EP]                  */
    int32_t num_tokens;   /* T <= W*Tr; token t belongs to logical rank t / Tr             */
    int32_t hidden;       /* H, multiple of 128                                            */
    int32_t num_experts;  /* E, multiple of W; expert e lives on rank e / (E/W)            */
    int32_t top_k;        /* k                                                             */
    int32_t intermediate; /* I: SwiGLU FFN width, multiple of 128                          */
    int32_t layout;       /* moe_layout                                                    */
    int32_t algorithm;    /* moe_algorithm                                                 */
    int32_t quant;        /* moe_quant: precision of the received rows and expert GEMMs    */
    int32_t expert_out_dtype; /* moe_expert_out_dtype                                      */
    int32_t act_precision;    /* moe_act_precision                                         */
} moe_geom;

/*
 * Dispatch handle: the analogue of Mooncake's (packed_recv_src_info,
 * packed_recv_layout_range, max_tok, hidden, num_experts) tuple [MC-EP].  moe_dispatch
 * fills it with device pointers into the caller's workspace; it stays valid until the
 * workspace is reused by another moe_dispatch, and must only be passed to the
 * moe_expert_ffn / moe_combine of the same dispatch ([MC-EP]: a handle is never reused
 * across unrelated dispatch/combine pairs).  cap = W*Tr below; R = offsets[E].
 */
typedef struct {
    moe_geom geom;
    void *recv_x;              /* bf16 (FP8: e4m3 codes, one byte each).
                                  EM: [E, cap, H]; RM: [W(dst), W(src)*Tr, H];
                                  FLAT: [W(dst), cap, H].  Rows past the counts are
                                  unspecified and never read.                            */
    float *recv_scales;        /* FP8 only (else NULL): scales of recv_x, column-block
                                  major: scale of row r, columns [128b, 128b+128) at
                                  recv_scales[b * nrows + r], nrows = E*cap (EM) or
                                  W*cap (RM/FLAT)                                        */
    int32_t *counts;           /* [E] rows of expert e (packed_recv_count)               */
    int32_t *offsets;          /* [E+1] exclusive prefix of counts: the expert-grouped
                                  pick list of the FFN                                   */
    int32_t *pick_pos;         /* [T*k] position of pick (t,j) in the pick list, or -1   */
    int32_t *pick_src;         /* [T*k] first R entries: t*k+j of each pick-list entry
                                  (packed_recv_src_info, in compact form)               */
    int32_t *slot;             /* EM: [T*k] recv row e*cap + rank of pick in expert e,
                                  or -1.  Unused (untouched) for RM/FLAT.                */
    int32_t *layout_range;     /* EM: [E][W][2] (begin, count) of each source rank's rows
                                  inside expert e's region (packed_recv_layout_range)    */
    int32_t *recv_row;         /* RM/FLAT: [T][W] row of token t in destination d's
                                  region, or -1 if t has no pick on d                    */
    int32_t *recv_count;       /* RM/FLAT: [W(dst)][W(src)] tokens received per pair     */
    int32_t *num_recv;         /* RM/FLAT: [W] tokens received per destination           */
    int32_t *recv_src;         /* RM/FLAT: [W][cap] token of each received row           */
    int32_t *recv_topk_idx;    /* RM/FLAT: [W][cap][k] LOCAL expert id, -1 = non-local
                                  pick [FI-3], int32                                     */
    float *recv_topk_weights;  /* RM/FLAT: [W][cap][k] topk weight, 0 for non-local      */
    int32_t *status;           /* device status word (MOE_STATUS_* bits)                 */
    void *ffn_act;             /* written by the FFN: the SwiGLU activation, [R, I] in
                                  pick-list order (row offsets[e] + position), the second
                                  GEMM's operand.  bf16: the high half of the pair
                                  (MOE_ACT_BF16: the bf16 activation); FP8:
                                  e4m3 codes                                             */
    float *ffn_act_scales;     /* FP8 only (else NULL): scales of ffn_act, column-block
                                  major [I/128][T*k] (row p, block b at b*T*k + p)        */
    void *pick_rows;           /* RM/FLAT (else NULL): [R, H] the row of every kept pick in
                                  pick-list order, x[pick_src[p] / k] at row p, written by
                                  moe_dispatch beside the receive buffer as the first
                                  GEMM's operand (bf16, or FP8 e4m3 codes)               */
    float *pick_row_scales;    /* RM/FLAT FP8 only (else NULL): scales of pick_rows,
                                  column-block major [H/128][T*k]                        */
    void *workspace;           /* base of the workspace the handle lives in              */
    size_t workspace_bytes;
    /* Optional per-kernel timing, the analogue of FlashInfer's enable_timing stage events
       (section 2): when `events` is non-NULL, every call records the cudaEvent_t
       events[slot] (slots MOE_EV_*, slot < num_events, NULL entries skipped) on its stream
       between its kernels.  Caller-owned events; moe_dispatch keeps these two fields of the
       handle it is given and fills the rest. */
    void **events;
    int32_t num_events;
    uint64_t magic;            /* set by moe_dispatch                                    */
} moe_handle;

/*
 * moe_workspace_size - bytes of device workspace one dispatch/ffn/combine cycle needs
 * for geometry *g: receive buffer, routing metadata, FFN intermediates and scratch.
 * The analogue of Buffer.get_ep_buffer_size_hint [MC-EP]: size it for the peak
 * num_tokens (max_tok per rank), not the mean.  Writes the size to *bytes.
 * Errors: the geometry checks listed under moe_error.
 */
int moe_workspace_size(const moe_geom *g, size_t *bytes);

/*
 * moe_expert_out_size - bytes of the expert_out buffer moe_expert_ffn writes (float32, or
 * bf16 with MOE_EXPERT_OUT_BFLOAT16):
 * EM [E, cap, H]; RM/FLAT [W, cap, H] (the receive layout, float32).
 */
int moe_expert_out_size(const moe_geom *g, size_t *bytes);

/*
 * moe_dispatch - route and scatter one token batch [MC-EP Buffer.dispatch; FI-3].
 *   x_dev           bf16 [T, H], 16-byte aligned, row-major contiguous
 *   topk_ids_dev    [T, k] int32 or int64 (ids_dtype), global expert ids, -1 = masked
 *                   pick [MC-EP]; an id outside [-1, E) sets MOE_STATUS_BAD_EXPERT_ID
 *                   and that pick is dropped
 *   topk_weights_dev float32 [T, k]: copied into recv_topk_weights for RM/FLAT (the
 *                   received routing); unused for EM (may be NULL there)
 *   active_ranks_dev int32 [W] EP rank-health mask [MC-EP Buffer.dispatch active_ranks],
 *                   or NULL (all active).  A rank with 0 has failed: picks whose expert lives
 *                   on it and all picks of the tokens it owns are dropped (not dispatched,
 *                   computed or combined; such tokens combine to zero) and
 *                   MOE_STATUS_INACTIVE_RANK is set.  Read by the kernels at dispatch time.
 *   workspace_dev   >= moe_workspace_size bytes, 256-byte aligned; overwritten
 *   h               host struct filled on success
 * Computes (deterministically; atomics decide no position): per-expert counts and
 * offsets, the position of every pick in its expert's rows in ascending (token, pick)
 * order, the EM slots and layout ranges or the RM/FLAT per-destination rows, local
 * ids and weights, then copies each token row to every place it is received.  For RM/FLAT
 * it also writes every kept pick's row in pick-list order into the workspace, the operand
 * moe_expert_ffn reads (so the FFN sees the rows as dispatched: later writes to recv_x do
 * not reach an RM/FLAT FFN).  With
 * g->quant = MOE_QUANT_FP8_E4M3 each token row is quantised once (e4m3 codes plus one
 * scale per 128 columns, moe_quant rule) as it is copied: recv_x holds the codes and
 * recv_scales the scales.
 */
int moe_dispatch(const moe_geom *g, const void *x_dev, const void *topk_ids_dev,
                 int ids_dtype, const float *topk_weights_dev, const int32_t *active_ranks_dev,
                 void *workspace_dev, size_t workspace_bytes, moe_handle *h, void *stream);

/*
 * moe_prepare_weights - one-time re-layout of w1 [E, 2I, H] (gate rows [0, I), up rows
 * [I, 2I) per expert [FI-4]) into w1_prepared_dev of the same size: inside each expert,
 * blocks of 128 gate rows and the matching 128 up rows alternate, so one 256-column GEMM
 * tile holds both halves of the SwiGLU for 128 output columns.  Both bf16, 16-byte
 * aligned, distinct buffers.
 */
int moe_prepare_weights(const moe_geom *g, const void *w1_dev, void *w1_prepared_dev,
                        void *stream);

/*
 * moe_expert_ffn - per-expert grouped SwiGLU FFN on the received rows [FI-2; FI-3]:
 * for each expert e and each of its rows x: h = x W1[e]^T (fp32 accumulate),
 * act = silu(h[:I]) * h[I:] as a bf16 pair (MOE_ACT_BF16_PAIR) or one bf16 (MOE_ACT_BF16),
 * y = act W2[e]^T (fp32).
 *   EM:      expert_out[e*cap + r] = y of row r (top_k = 1 per dispatched row)
 *   RM/FLAT: expert_out[d*cap + r] = sum over the row's LOCAL picks j (ascending) of
 *            recv_topk_weights[d][r][j] * y_j; non-local picks are masked to weight 0
 *   w1_prepared_dev bf16 from moe_prepare_weights; w2_dev bf16 [E, H, I]
 *   expert_out_dev  float32 or bf16 (geom expert_out_dtype), moe_expert_out_size bytes,
 *                   16-byte aligned
 * Runs on tcgen05 tensor cores (bf16 x bf16 -> fp32 in tensor memory).
 */
int moe_expert_ffn(const moe_handle *h, const void *w1_prepared_dev, const void *w2_dev,
                   void *expert_out_dev, void *stream);

/*
 * moe_combine - return expert outputs to token order [MC-EP Buffer.combine; FI-3]:
 *   EM:      out[t] = bf16( sum over kept picks j ascending of
 *                           topk_weights[t, j] * expert_out[slot[t, j]] )
 *   RM/FLAT: out[t] = bf16( sum over destinations d ascending that received t of
 *                           expert_out[d*cap + recv_row[t, d]] )   (unweighted)
 *   expert_out_dev   float32 or bf16 (geom expert_out_dtype), as moe_expert_ffn wrote it
 *   topk_weights_dev float32 [T, k] (EM; ignored and may be NULL for RM/FLAT)
 *   out_dev          bf16 [T, H], 16-byte aligned
 * fp32 accumulation, one round-to-nearest-even to bf16.  Tokens without any kept
 * pick get zeros.
 */
int moe_combine(const moe_handle *h, const void *expert_out_dev,
                const float *topk_weights_dev, void *out_dev, void *stream);

/*
 * moe_quantize_weights_fp8 - one-time FP8 quantisation of bf16 expert weights for
 * moe_expert_ffn_fp8 (geometry with quant = MOE_QUANT_FP8_E4M3).  Every 128 x 128 block of
 * w1[e] [2I, H] and w2[e] [H, I] is quantised with the rule of moe_quant (amax over the
 * block).  W1 is written in the gate/up interleaved order of moe_prepare_weights (blocks of
 * 128 gate rows and the matching 128 up rows alternate), its block scales likewise:
 *   w1_dev            bf16 [E, 2I, H]          w2_dev            bf16 [E, H, I]
 *   w1q_prepared_dev  e4m3 [E, 2I, H]          w1_scales_prepared_dev float [E, 2I/128, H/128]
 *   w2q_dev           e4m3 [E, H, I]           w2_scales_dev     float [E, H/128, I/128]
 * All 16-byte aligned (scales 4-byte), distinct buffers.
 */
int moe_quantize_weights_fp8(const moe_geom *g, const void *w1_dev, const void *w2_dev,
                             void *w1q_prepared_dev, float *w1_scales_prepared_dev, void *w2q_dev,
                             float *w2_scales_dev, void *stream);

/*
 * moe_prepare_weights_fp8 - the gate/up interleave of moe_prepare_weights for W1 that is
 * already FP8 (e4m3 codes [E, 2I, H] with float block scales [E, 2I/128, H/128], rows
 * [0, I) gate and [I, 2I) up per expert): writes the interleaved codes and scales that
 * moe_expert_ffn_fp8 reads.  W2 needs no preparation.  Distinct, 16-byte aligned buffers.
 */
int moe_prepare_weights_fp8(const moe_geom *g, const void *w1q_dev, const float *w1_scales_dev,
                            void *w1q_prepared_dev, float *w1_scales_prepared_dev, void *stream);

/*
 * moe_expert_ffn_fp8 - moe_expert_ffn for a handle of an FP8 dispatch: per expert e,
 * h = x^ W1^[e]^T with e4m3 x e4m3 products accumulated in fp32 (tensor memory), every
 * 128-column k-block's partial sum scaled by its row scale times its weight-block scale
 * and added in fp32; act = silu(h[:I]) * h[I:] in fp32, quantised per 128 columns
 * (moe_quant rule) into ffn_act / ffn_act_scales; y = act^ W2^[e]^T the same way, fp32.
 * expert_out as in moe_expert_ffn.  Weights from moe_quantize_weights_fp8 or
 * moe_prepare_weights_fp8.  MOE_ERR_INVALID_ARGUMENT for a bf16 handle (and
 * moe_expert_ffn returns it for an FP8 handle).
 */
int moe_expert_ffn_fp8(const moe_handle *h, const void *w1q_prepared_dev,
                       const float *w1_scales_prepared_dev, const void *w2q_dev,
                       const float *w2_scales_dev, void *expert_out_dev, void *stream);

/*
 * moe_forward_host - the whole layer end to end from HOST buffers, on one stream:
 * moe_dispatch (all ranks active) -> moe_expert_ffn -> moe_combine of x_host /
 * topk_ids_host / topk_weights_host (same shapes as in moe_dispatch) into out_host (bf16
 * [T, H]).  When all four host buffers are page-locked (cudaHostAlloc / registered), the
 * kernels read the inputs from host memory and the combine writes out_host directly
 * (over NVLink-C2C on GB300); x_dev, topk_ids_dev, topk_weights_dev and out_dev are then
 * not used and may be NULL.  Otherwise the inputs are copied into those device buffers
 * first and out_dev is copied to out_host last (the copies of pageable memory
 * synchronise).  bf16 geometries only (MOE_ERR_INVALID_ARGUMENT for FP8).  Asynchronous
 * like the other calls: out_host is valid once the stream has been synchronised; the
 * host inputs must stay unchanged until then.  Returns the first error of the
 * sequence.
 * expert_out_dev is scratch here: for RANK_MAJOR / FLAT the rank reduction of received
 * rows with several local picks is folded into the combine, which sums their per-pick
 * rows on the fly in the same order, so out_host equals the three calls' output bit for
 * bit while those rows of expert_out_dev are left unwritten.
 */
int moe_forward_host(const moe_geom *g, const void *x_host, const void *topk_ids_host,
                     int ids_dtype, const float *topk_weights_host, void *out_host,
                     void *x_dev, void *topk_ids_dev, float *topk_weights_dev, void *out_dev,
                     const void *w1_prepared_dev, const void *w2_dev, void *expert_out_dev,
                     void *workspace_dev, size_t workspace_bytes, moe_handle *h, void *stream);

/*
 * moe_get_status - wait for `stream`, then read the handle's device status word
 * (MOE_STATUS_* bits, 0 = clean) into *status_host.  The only synchronising call.
 */
int moe_get_status(const moe_handle *h, int32_t *status_host, void *stream);

/*
 * moe_route_noalloc - EXPERT_MAJOR routing that allocates nothing and needs no workspace.
 * The pages have no counterpart of this call; it exists for callers that can only pass
 * input and output buffers (plugin hosts and engines that own all device memory and
 * plan it ahead of time) and so can neither give moe_dispatch a workspace nor let the
 * library call cudaMalloc.
 *   Computes exactly the routing outputs moe_dispatch produces for an EXPERT_MAJOR
 *   geometry, into caller buffers: counts_dev [E], offsets_dev [E+1], pick_pos_dev
 *   [T*k], pick_src_dev [T*k], slot_dev [T*k], layout_range_dev [E][W][2] (all int32,
 *   same meaning as the moe_handle fields) and status_dev (one int32, MOE_STATUS_* bits,
 *   cleared by the call).  No rows are copied.
 *   Scratch: a static device array of MOE_NOALLOC_SCRATCH_BYTES compiled into the library
 *   (held by every GPU that loads it until the process exits).  The routing needs
 *   (2 * E * nb + 2 * E + 2) * 4 bytes of it, nb being the routing chunk count of the geometry
 *   (about 256 for large batches); a larger geometry returns MOE_ERR_LIMIT.
 *   The first call on each device looks the array's address up (cudaGetSymbolAddress)
 *   with that device current; make that first call before any stream capture.  The
 *   address is kept for that device until the process exits: after cudaDeviceReset (or
 *   any other teardown of the device's primary context) this entry point must not be
 *   called again in the same process.
 *   Every call shares the one array, so calls that overlap on the GPU (issued on different
 *   streams of one device without ordering between them) race on it and corrupt each
 *   other's results: order them on one stream.
 *   Errors: MOE_ERR_INVALID_ARGUMENT for a non-EXPERT_MAJOR geometry or a NULL buffer,
 *   the geometry errors of moe_workspace_size, MOE_ERR_LIMIT beyond the scratch size,
 *   MOE_ERR_NOT_BUILT_FOR_DEVICE on a device other than compute capability 10.3.
 */
#define MOE_NOALLOC_SCRATCH_BYTES (1u << 20)
int moe_route_noalloc(const moe_geom *g, const void *topk_ids_dev, int ids_dtype,
                      int32_t *counts_dev, int32_t *offsets_dev, int32_t *pick_pos_dev,
                      int32_t *pick_src_dev, int32_t *slot_dev, int32_t *layout_range_dev,
                      int32_t *status_dev, void *stream);

/*
 * moe_launches_per_layer - number of kernels one moe_dispatch + moe_expert_ffn +
 * moe_combine of geometry *g queues (routing is one kernel for batches of at most 3072
 * picks over at most 64 experts and three otherwise; RANK_MAJOR / FLAT add the
 * local-pick reduction).  Written to *n.
 */
int moe_launches_per_layer(const moe_geom *g, int32_t *n);

/*
 * moe_selftest_wait_expiry - exercises the device-side failure path without faulting or
 * hanging the GPU: one CTA waits on an mbarrier that nothing will complete, through the
 * same bounded wait every tcgen05 GEMM kernel uses.  After the wait limit (2 s) the wait
 * gives up, ORs MOE_STATUS_TIMEOUT into *status_dev (device int32) and the kernel returns;
 * the context stays usable.  Stream-ordered and asynchronous.  The pages have no
 * counterpart; it exists so that tests can check the expiry path on a real GPU.
 * Errors: MOE_ERR_INVALID_ARGUMENT (NULL status), MOE_ERR_NOT_BUILT_FOR_DEVICE,
 * MOE_ERR_CUDA.
 */
int moe_selftest_wait_expiry(int32_t *status_dev, void *stream);

/* moe_strerror - static text for a moe_error code. */
const char *moe_strerror(int err);

#ifdef __cplusplus
}
#endif
#endif /* COMBINE_TOPK_IDS_MOE_H */
