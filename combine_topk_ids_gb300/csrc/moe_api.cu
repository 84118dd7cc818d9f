// C ABI of the layer (declared in include/moe.h): geometry checks, workspace plan,
// handle bookkeeping and the launch sequence of each call.  No allocation, no host
// synchronisation except in moe_get_status.
#include <cstring>
#include <mutex>

#include "moe_internal.cuh"

namespace moe {

namespace {
inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
inline bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct DeviceInfo {
    int checked = 0;   // 0 unknown, 1 compute capability 10.3, -1 other
    int sms = 0;
};
std::mutex g_dev_mutex;
DeviceInfo g_dev[64];

const DeviceInfo *device_info() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(g_dev_mutex);
    DeviceInfo &d = g_dev[dev];
    if (d.checked == 0) {
        int major = 0, minor = 0, sms = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        d.checked = (major == 10 && minor == 3) ? 1 : -1;
        d.sms = sms;
    }
    return &d;
}

}  // namespace

int check_device() {
    const DeviceInfo *d = device_info();
    if (!d) return MOE_ERR_CUDA;
    return d->checked == 1 ? MOE_OK : MOE_ERR_NOT_BUILT_FOR_DEVICE;
}

int device_ordinal() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
    return dev;
}

int num_sms() {
    const DeviceInfo *d = device_info();
    return (d && d->sms > 0) ? d->sms : 1;
}

int make_plan(const moe_geom &g, Plan *p) {
    if (g.world < 1 || g.max_tok < 1 || g.num_tokens < 0 || g.hidden < 1 || g.num_experts < 1 ||
        g.intermediate < 1)
        return MOE_ERR_INVALID_ARGUMENT;
    if (g.layout < 0 || g.layout > 2 || g.algorithm < 0 || g.algorithm > 1 || g.quant < 0 ||
        g.quant > 1 || g.expert_out_dtype < 0 || g.expert_out_dtype > 1 || g.act_precision < 0 ||
        g.act_precision > 1)
        return MOE_ERR_INVALID_ARGUMENT;
    if (g.top_k < 1 || g.top_k > MOE_MAX_TOPK) return MOE_ERR_TOPK;
    if (g.num_experts % g.world != 0) return MOE_ERR_EXPERTS_NOT_DIVISIBLE;
    if (g.hidden % 128 != 0) return MOE_ERR_HIDDEN_ALIGNMENT;
    if (g.intermediate % 128 != 0) return MOE_ERR_INTERMEDIATE_ALIGNMENT;
    if (g.world > MOE_MAX_WORLD || g.num_experts > MOE_MAX_EXPERTS || g.hidden > MOE_MAX_HIDDEN)
        return MOE_ERR_LIMIT;
    const int64_t cap = (int64_t)g.world * g.max_tok;
    if (g.num_tokens > cap) return MOE_ERR_TOO_MANY_TOKENS;
    const int64_t P = (int64_t)g.num_tokens * g.top_k;
    // slots, rows and pick positions are int32 on the device
    if ((int64_t)g.num_experts * cap >= ((int64_t)1 << 31) || P >= ((int64_t)1 << 31) ||
        (int64_t)g.world * cap >= ((int64_t)1 << 31))
        return MOE_ERR_LIMIT;

    Plan &q = *p;
    q.T = g.num_tokens; q.W = g.world; q.Tr = g.max_tok; q.cap = cap; q.E = g.num_experts;
    q.k = g.top_k; q.H = g.hidden; q.I = g.intermediate; q.P = P; q.layout = g.layout;
    q.quant = g.quant;
    q.eo_bf16 = g.expert_out_dtype == MOE_EXPERT_OUT_BFLOAT16;
    q.act_pair = g.quant == MOE_QUANT_NONE && g.act_precision == MOE_ACT_BF16_PAIR;
    // routing chunk: about 256 chunks over the whole capacity, 32..1024 tokens each
    int64_t want = (cap + 255) / 256;
    int tb = 32;
    while (tb < want && tb < 1024) tb <<= 1;
    q.tb = tb;
    q.nbpr = (int)((g.max_tok + tb - 1) / tb);
    q.nb = g.world * q.nbpr;

    const bool em = g.layout == MOE_LAYOUT_EXPERT_MAJOR;
    const bool f8 = g.quant == MOE_QUANT_FP8_E4M3;
    const int64_t E = q.E, W = q.W, k = q.k, H = q.H, I = q.I, nb = q.nb;
    const int64_t eb = f8 ? 1 : 2;   // bytes per element of rows and activations
    q.nrecv = (em ? E : W) * cap;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t o = off;
        off = align_up(off + bytes, 256);
        return o;
    };
    q.status = take(4 * 5);   // status word, then the GEMMs' four tile counters
    q.counts = take(4 * E);
    q.offsets = take(4 * (E + 1));
    q.mprefix = take(4 * (E + 1));
    q.mprefix2 = take(4 * (E + 1));
    q.pick_pos = take(4 * P);
    q.pick_src = take(4 * P);
    q.slot = take(4 * P);
    q.layout_range = take(8 * E * W);
    q.blk_hist = take(4 * E * nb);
    q.blk_base = take(4 * E * nb);
    q.recv_row = take(em ? 0 : 4 * q.T * W);
    q.recv_count = take(4 * W * W);
    q.num_recv = take(4 * W);
    q.recv_src = take(em ? 0 : 4 * W * cap);
    q.recv_topk_idx = take(em ? 0 : 4 * W * cap * k);
    q.recv_topk_w = take(em ? 0 : 4 * W * cap * k);
    q.blk_dhist = take(4 * W * nb);
    q.blk_dbase = take(4 * W * nb);
    q.recv_x = take(eb * q.nrecv * H);
    q.recv_scales = take(f8 ? 4 * q.nrecv * (H / 128) : 0);
    q.act = take(eb * P * I);
    q.act_lo = take(q.act_pair ? 2 * P * I : 0);
    q.act_scales = take(f8 ? 4 * P * (I / 128) : 0);
    q.apick = take(em ? 0 : eb * P * H);
    q.apick_scales = take(em || !f8 ? 0 : 4 * P * (H / 128));
    q.ypick = take(em ? 0 : (q.eo_bf16 ? 2 : 4) * P * H);
    q.direct_row = take(em ? 0 : 4 * P);
    q.direct_w = take(em ? 0 : 4 * P);
    q.total = off;
    return MOE_OK;
}

Routing carve(const Plan &p, void *ws) {
    char *b = static_cast<char *>(ws);
    Routing r;
    r.p = &p;
    auto i32 = [&](size_t o) { return reinterpret_cast<int32_t *>(b + o); };
    r.status = i32(p.status); r.sched = r.status + 1; r.counts = i32(p.counts); r.offsets = i32(p.offsets);
    r.mprefix = i32(p.mprefix); r.mprefix2 = i32(p.mprefix2); r.pick_pos = i32(p.pick_pos); r.pick_src = i32(p.pick_src);
    r.slot = i32(p.slot); r.layout_range = i32(p.layout_range); r.blk_hist = i32(p.blk_hist);
    r.blk_base = i32(p.blk_base); r.recv_row = i32(p.recv_row); r.recv_count = i32(p.recv_count);
    r.num_recv = i32(p.num_recv); r.recv_src = i32(p.recv_src);
    r.recv_topk_idx = i32(p.recv_topk_idx); r.blk_dhist = i32(p.blk_dhist);
    r.blk_dbase = i32(p.blk_dbase);
    r.recv_topk_w = reinterpret_cast<float *>(b + p.recv_topk_w);
    r.recv_x = reinterpret_cast<uint16_t *>(b + p.recv_x);
    r.act = reinterpret_cast<uint16_t *>(b + p.act);
    r.act_lo = p.act_pair ? reinterpret_cast<uint16_t *>(b + p.act_lo) : nullptr;
    r.apick = reinterpret_cast<uint16_t *>(b + p.apick);
    r.ypick = b + p.ypick;
    r.direct_row = p.layout != MOE_LAYOUT_EXPERT_MAJOR ? i32(p.direct_row) : nullptr;
    r.direct_w = p.layout != MOE_LAYOUT_EXPERT_MAJOR ? reinterpret_cast<float *>(b + p.direct_w) : nullptr;
    const bool f8 = p.quant == MOE_QUANT_FP8_E4M3;
    r.recv_scales = f8 ? reinterpret_cast<float *>(b + p.recv_scales) : nullptr;
    r.act_scales = f8 ? reinterpret_cast<float *>(b + p.act_scales) : nullptr;
    r.apick_scales = f8 && p.layout != MOE_LAYOUT_EXPERT_MAJOR ? reinterpret_cast<float *>(b + p.apick_scales)
                                                               : nullptr;
    return r;
}

namespace {
inline void record(const moe_handle *h, int slot, cudaStream_t s) {
    if (h && h->events && slot < h->num_events && h->events[slot])
        cudaEventRecord(static_cast<cudaEvent_t>(h->events[slot]), s);
}

// Device address of a page-locked host buffer, or NULL for any other pointer.
const void *mapped_host(const void *p) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();   // clear the error of an unknown pointer
        return nullptr;
    }
    return at.type == cudaMemoryTypeHost ? at.devicePointer : nullptr;
}

int handle_plan(const moe_handle *h, Plan *p) {
    if (!h || h->magic != kHandleMagic || !h->workspace) return MOE_ERR_BAD_HANDLE;
    int rc = make_plan(h->geom, p);
    if (rc != MOE_OK) return MOE_ERR_BAD_HANDLE;
    if (h->workspace_bytes < p->total) return MOE_ERR_BAD_HANDLE;
    return MOE_OK;
}
}  // namespace

}  // namespace moe

using namespace moe;

extern "C" {

int moe_workspace_size(const moe_geom *g, size_t *bytes) {
    if (!g || !bytes) return MOE_ERR_INVALID_ARGUMENT;
    Plan p;
    int rc = make_plan(*g, &p);
    if (rc != MOE_OK) return rc;
    *bytes = p.total;
    return MOE_OK;
}

int moe_expert_out_size(const moe_geom *g, size_t *bytes) {
    if (!g || !bytes) return MOE_ERR_INVALID_ARGUMENT;
    Plan p;
    int rc = make_plan(*g, &p);
    if (rc != MOE_OK) return rc;
    const int64_t rows = (p.layout == MOE_LAYOUT_EXPERT_MAJOR ? p.E : p.W) * p.cap;
    *bytes = (size_t)rows * (size_t)p.H * (p.eo_bf16 ? 2 : 4);
    return MOE_OK;
}

int moe_dispatch(const moe_geom *g, const void *x_dev, const void *topk_ids_dev, int ids_dtype,
                 const float *topk_weights_dev, const int32_t *active_ranks_dev, void *workspace_dev,
                 size_t workspace_bytes, moe_handle *h, void *stream) {
    if (!g || !h || !workspace_dev) return MOE_ERR_INVALID_ARGUMENT;
    if (ids_dtype != MOE_IDS_INT32 && ids_dtype != MOE_IDS_INT64) return MOE_ERR_IDS_DTYPE;
    Plan p;
    int rc = make_plan(*g, &p);
    if (rc != MOE_OK) return rc;
    const bool em = g->layout == MOE_LAYOUT_EXPERT_MAJOR;
    if (p.T > 0 && (!x_dev || !topk_ids_dev || (!em && !topk_weights_dev)))
        return MOE_ERR_INVALID_ARGUMENT;
    if (!aligned(workspace_dev, 256) || (x_dev && !aligned(x_dev, 16)) ||
        (topk_ids_dev && !aligned(topk_ids_dev, ids_dtype == MOE_IDS_INT64 ? 8 : 4)) ||
        (topk_weights_dev && !aligned(topk_weights_dev, 4)) ||
        (active_ranks_dev && !aligned(active_ranks_dev, 4)))
        return MOE_ERR_MISALIGNED;
    if (workspace_bytes < p.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
    if ((rc = check_device()) != MOE_OK) return rc;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    Routing r = carve(p, workspace_dev);
    void **events = h->events;
    const int32_t num_events = h->num_events;
    std::memset(h, 0, sizeof(*h));
    h->events = events;
    h->num_events = num_events;
    h->geom = *g;
    h->recv_x = r.recv_x;
    h->recv_scales = r.recv_scales;
    h->ffn_act = r.act;
    h->ffn_act_scales = r.act_scales;
    h->pick_rows = g->layout != MOE_LAYOUT_EXPERT_MAJOR ? (void *)r.apick : nullptr;
    h->pick_row_scales = r.apick_scales;
    h->counts = r.counts;
    h->offsets = r.offsets;
    h->pick_pos = r.pick_pos;
    h->pick_src = r.pick_src;
    h->slot = r.slot;
    h->layout_range = r.layout_range;
    if (!em) {
        h->recv_row = r.recv_row;
        h->recv_count = r.recv_count;
        h->num_recv = r.num_recv;
        h->recv_src = r.recv_src;
        h->recv_topk_idx = r.recv_topk_idx;
        h->recv_topk_weights = r.recv_topk_w;
    }
    h->status = r.status;
    h->workspace = workspace_dev;
    h->workspace_bytes = workspace_bytes;

    record(h, MOE_EV_DISPATCH_BEGIN, s);
    // launch_routing clears the status word before any kernel can set a bit
    if (launch_routing(r, topk_ids_dev, ids_dtype == MOE_IDS_INT64, topk_weights_dev,
                       active_ranks_dev, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    record(h, MOE_EV_ROUTING_END, s);
    const cudaError_t ce = p.quant == MOE_QUANT_FP8_E4M3
                               ? launch_dispatch_quant(r, static_cast<const uint16_t *>(x_dev), s)
                               : launch_dispatch_copy(r, static_cast<const uint16_t *>(x_dev), s);
    if (ce != cudaSuccess) return MOE_ERR_CUDA;
    record(h, MOE_EV_DISPATCH_END, s);
    h->magic = kHandleMagic;
    return MOE_OK;
}

int moe_prepare_weights(const moe_geom *g, const void *w1_dev, void *w1_prepared_dev, void *stream) {
    if (!g || !w1_dev || !w1_prepared_dev || w1_dev == w1_prepared_dev) return MOE_ERR_INVALID_ARGUMENT;
    Plan p;
    int rc = make_plan(*g, &p);
    if (rc != MOE_OK) return rc;
    if (!aligned(w1_dev, 16) || !aligned(w1_prepared_dev, 16)) return MOE_ERR_MISALIGNED;
    if ((rc = check_device()) != MOE_OK) return rc;
    return launch_prepare_w1(*g, static_cast<const uint16_t *>(w1_dev),
                             static_cast<uint16_t *>(w1_prepared_dev),
                             static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? MOE_OK
               : MOE_ERR_CUDA;
}

namespace moe {
namespace {
// The bf16 expert stage.  reduce = false (RANK_MAJOR / FLAT inside moe_forward_host): the
// rank reduction is left to the fused combine, so expert_out's multi-pick rows stay unwritten.
int expert_ffn(const moe_handle *h, const void *w1_prepared_dev, const void *w2_dev, void *expert_out_dev,
               void *stream, bool reduce) {
    Plan p;
    int rc = handle_plan(h, &p);
    if (rc != MOE_OK) return rc;
    if (!w1_prepared_dev || !w2_dev || !expert_out_dev) return MOE_ERR_INVALID_ARGUMENT;
    if (p.quant != MOE_QUANT_NONE) return MOE_ERR_INVALID_ARGUMENT;   // moe_expert_ffn_fp8
    if (!aligned(w1_prepared_dev, 16) || !aligned(w2_dev, 16) || !aligned(expert_out_dev, 16))
        return MOE_ERR_MISALIGNED;
    if ((rc = check_device()) != MOE_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    Routing r = carve(p, h->workspace);
    const bool em = p.layout == MOE_LAYOUT_EXPERT_MAJOR;
    record(h, MOE_EV_FFN_BEGIN, s);
    record(h, MOE_EV_GATHER_END, s);   // RM/FLAT pick rows were written by moe_dispatch
    if ((rc = launch_gemm1(r, static_cast<const uint16_t *>(w1_prepared_dev), s)) != MOE_OK) return rc;
    record(h, MOE_EV_GEMM1_END, s);
    if ((rc = launch_gemm2(r, static_cast<const uint16_t *>(w2_dev), expert_out_dev, s)) != MOE_OK)
        return rc;
    record(h, MOE_EV_GEMM2_END, s);
    if (!em && reduce && launch_reduce_ranks(r, expert_out_dev, true, s) != cudaSuccess) return MOE_ERR_CUDA;
    record(h, MOE_EV_FFN_END, s);
    return MOE_OK;
}

// moe_combine's launch; fused: RANK_MAJOR / FLAT combine that also forms the multi-pick
// rows' sums (after expert_ffn with reduce = false)
int combine(const moe_handle *h, const void *expert_out_dev, const float *topk_weights_dev, void *out_dev,
            void *stream, bool fused) {
    Plan p;
    int rc = handle_plan(h, &p);
    if (rc != MOE_OK) return rc;
    const bool em = p.layout == MOE_LAYOUT_EXPERT_MAJOR;
    if (p.T > 0 && (!expert_out_dev || !out_dev || (em && !topk_weights_dev)))
        return MOE_ERR_INVALID_ARGUMENT;
    if ((expert_out_dev && !aligned(expert_out_dev, 16)) || (out_dev && !aligned(out_dev, 16)) ||
        (topk_weights_dev && !aligned(topk_weights_dev, 4)))
        return MOE_ERR_MISALIGNED;
    if ((rc = check_device()) != MOE_OK) return rc;
    Routing r = carve(p, h->workspace);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    record(h, MOE_EV_COMBINE_BEGIN, s);
    const cudaError_t ce = fused && !em
                               ? launch_combine_fused(r, expert_out_dev, static_cast<uint16_t *>(out_dev), s)
                               : launch_combine(r, expert_out_dev, topk_weights_dev, static_cast<uint16_t *>(out_dev), s);
    if (ce != cudaSuccess) return MOE_ERR_CUDA;
    record(h, MOE_EV_COMBINE_END, s);
    return MOE_OK;
}
}  // namespace
}  // namespace moe

int moe_expert_ffn(const moe_handle *h, const void *w1_prepared_dev, const void *w2_dev,
                   void *expert_out_dev, void *stream) {
    return moe::expert_ffn(h, w1_prepared_dev, w2_dev, expert_out_dev, stream, true);
}

int moe_expert_ffn_fp8(const moe_handle *h, const void *w1q_prepared_dev,
                       const float *w1_scales_prepared_dev, const void *w2q_dev,
                       const float *w2_scales_dev, void *expert_out_dev, void *stream) {
    Plan p;
    int rc = handle_plan(h, &p);
    if (rc != MOE_OK) return rc;
    if (p.quant != MOE_QUANT_FP8_E4M3) return MOE_ERR_INVALID_ARGUMENT;
    if (!w1q_prepared_dev || !w1_scales_prepared_dev || !w2q_dev || !w2_scales_dev || !expert_out_dev)
        return MOE_ERR_INVALID_ARGUMENT;
    if (!aligned(w1q_prepared_dev, 16) || !aligned(w2q_dev, 16) || !aligned(expert_out_dev, 16) ||
        !aligned(w1_scales_prepared_dev, 4) || !aligned(w2_scales_dev, 4))
        return MOE_ERR_MISALIGNED;
    if ((rc = check_device()) != MOE_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    Routing r = carve(p, h->workspace);
    const bool em = p.layout == MOE_LAYOUT_EXPERT_MAJOR;
    record(h, MOE_EV_FFN_BEGIN, s);
    record(h, MOE_EV_GATHER_END, s);   // RM/FLAT pick rows were written by moe_dispatch
    if ((rc = launch_gemm1_fp8(r, static_cast<const uint8_t *>(w1q_prepared_dev), w1_scales_prepared_dev,
                               s)) != MOE_OK)
        return rc;
    record(h, MOE_EV_GEMM1_END, s);
    if ((rc = launch_gemm2_fp8(r, static_cast<const uint8_t *>(w2q_dev), w2_scales_dev, expert_out_dev,
                               s)) != MOE_OK)
        return rc;
    record(h, MOE_EV_GEMM2_END, s);
    if (!em && launch_reduce_ranks(r, expert_out_dev, false, s) != cudaSuccess) return MOE_ERR_CUDA;
    record(h, MOE_EV_FFN_END, s);
    return MOE_OK;
}

int moe_quantize_weights_fp8(const moe_geom *g, const void *w1_dev, const void *w2_dev,
                             void *w1q_prepared_dev, float *w1_scales_prepared_dev, void *w2q_dev,
                             float *w2_scales_dev, void *stream) {
    if (!g || !w1_dev || !w2_dev || !w1q_prepared_dev || !w1_scales_prepared_dev || !w2q_dev ||
        !w2_scales_dev)
        return MOE_ERR_INVALID_ARGUMENT;
    Plan p;
    int rc = make_plan(*g, &p);
    if (rc != MOE_OK) return rc;
    if (!aligned(w1_dev, 16) || !aligned(w2_dev, 16) || !aligned(w1q_prepared_dev, 16) ||
        !aligned(w2q_dev, 16) || !aligned(w1_scales_prepared_dev, 4) || !aligned(w2_scales_dev, 4))
        return MOE_ERR_MISALIGNED;
    if ((rc = check_device()) != MOE_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (launch_quantize_weights_fp8(static_cast<const uint16_t *>(w1_dev), p.E, 2 * p.I, p.H, p.I,
                                    static_cast<uint8_t *>(w1q_prepared_dev), w1_scales_prepared_dev,
                                    s) != cudaSuccess ||
        launch_quantize_weights_fp8(static_cast<const uint16_t *>(w2_dev), p.E, p.H, p.I, 0,
                                    static_cast<uint8_t *>(w2q_dev), w2_scales_dev, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

int moe_prepare_weights_fp8(const moe_geom *g, const void *w1q_dev, const float *w1_scales_dev,
                            void *w1q_prepared_dev, float *w1_scales_prepared_dev, void *stream) {
    if (!g || !w1q_dev || !w1_scales_dev || !w1q_prepared_dev || !w1_scales_prepared_dev ||
        w1q_dev == w1q_prepared_dev || (const void *)w1_scales_dev == (const void *)w1_scales_prepared_dev)
        return MOE_ERR_INVALID_ARGUMENT;
    Plan p;
    int rc = make_plan(*g, &p);
    if (rc != MOE_OK) return rc;
    if (!aligned(w1q_dev, 16) || !aligned(w1q_prepared_dev, 16) || !aligned(w1_scales_dev, 4) ||
        !aligned(w1_scales_prepared_dev, 4))
        return MOE_ERR_MISALIGNED;
    if ((rc = check_device()) != MOE_OK) return rc;
    return launch_prepare_w1_fp8(*g, static_cast<const uint8_t *>(w1q_dev), w1_scales_dev,
                                 static_cast<uint8_t *>(w1q_prepared_dev), w1_scales_prepared_dev,
                                 static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? MOE_OK
               : MOE_ERR_CUDA;
}

int moe_combine(const moe_handle *h, const void *expert_out_dev, const float *topk_weights_dev,
                void *out_dev, void *stream) {
    return moe::combine(h, expert_out_dev, topk_weights_dev, out_dev, stream, false);
}

int moe_forward_host(const moe_geom *g, const void *x_host, const void *topk_ids_host,
                     int ids_dtype, const float *topk_weights_host, void *out_host,
                     void *x_dev, void *topk_ids_dev, float *topk_weights_dev, void *out_dev,
                     const void *w1_prepared_dev, const void *w2_dev, void *expert_out_dev,
                     void *workspace_dev, size_t workspace_bytes, moe_handle *h, void *stream) {
    if (!g || !h) return MOE_ERR_INVALID_ARGUMENT;
    if (ids_dtype != MOE_IDS_INT32 && ids_dtype != MOE_IDS_INT64) return MOE_ERR_IDS_DTYPE;
    Plan p;
    int rc = make_plan(*g, &p);
    if (rc != MOE_OK) return rc;
    if (p.quant != MOE_QUANT_NONE) return MOE_ERR_INVALID_ARGUMENT;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (p.T > 0 && (!x_host || !topk_ids_host || !topk_weights_host || !out_host))
        return MOE_ERR_INVALID_ARGUMENT;
    // Page-locked host buffers are addressable by the kernels (one address space, and on
    // GB300 a coherent NVLink-C2C link to the Grace memory): the row scatter and the
    // routing then read the batch straight from host memory and the combine writes the
    // result straight into it, instead of staging copies through the device buffers.
    if (p.T > 0) {
        const void *xm = mapped_host(x_host), *im = mapped_host(topk_ids_host),
                   *wm = mapped_host(topk_weights_host);
        void *om = const_cast<void *>(mapped_host(out_host));
        if (xm && im && wm && om && aligned(xm, 16) && aligned(om, 16) &&
            aligned(im, ids_dtype == MOE_IDS_INT64 ? 8 : 4) && aligned(wm, 4)) {
            int rc2 = moe_dispatch(g, xm, im, ids_dtype, static_cast<const float *>(wm), nullptr, workspace_dev,
                                   workspace_bytes, h, stream);
            if (rc2 == MOE_OK) rc2 = moe::expert_ffn(h, w1_prepared_dev, w2_dev, expert_out_dev, stream, false);
            if (rc2 == MOE_OK)
                rc2 = moe::combine(h, expert_out_dev, static_cast<const float *>(wm), om, stream, true);
            return rc2;
        }
    }
    if (p.T > 0) {
        if (!x_dev || !topk_ids_dev || !topk_weights_dev) return MOE_ERR_INVALID_ARGUMENT;
        const size_t xb = (size_t)p.T * p.H * 2, pb = (size_t)p.P;
        if (cudaMemcpyAsync(x_dev, x_host, xb, cudaMemcpyHostToDevice, s) != cudaSuccess ||
            cudaMemcpyAsync(topk_ids_dev, topk_ids_host, pb * (ids_dtype == MOE_IDS_INT64 ? 8 : 4),
                            cudaMemcpyHostToDevice, s) != cudaSuccess ||
            cudaMemcpyAsync(topk_weights_dev, topk_weights_host, pb * 4, cudaMemcpyHostToDevice, s) !=
                cudaSuccess)
            return MOE_ERR_CUDA;
    }
    if ((rc = moe_dispatch(g, x_dev, topk_ids_dev, ids_dtype, topk_weights_dev, nullptr,
                           workspace_dev, workspace_bytes, h, stream)) != MOE_OK)
        return rc;
    if ((rc = moe::expert_ffn(h, w1_prepared_dev, w2_dev, expert_out_dev, stream, false)) != MOE_OK) return rc;
    if ((rc = moe::combine(h, expert_out_dev, topk_weights_dev, out_dev, stream, true)) != MOE_OK) return rc;
    if (p.T > 0 &&
        cudaMemcpyAsync(out_host, out_dev, (size_t)p.T * p.H * 2, cudaMemcpyDeviceToHost, s) !=
            cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

int moe_get_status(const moe_handle *h, int32_t *status_host, void *stream) {
    if (!h || !status_host) return MOE_ERR_INVALID_ARGUMENT;
    if (h->magic != kHandleMagic || !h->status) return MOE_ERR_BAD_HANDLE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t v = 0;
    if (cudaMemcpyAsync(&v, h->status, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return MOE_ERR_CUDA;
    *status_host = v;
    return MOE_OK;
}

int moe_launches_per_layer(const moe_geom *g, int32_t *n) {
    if (!g || !n) return MOE_ERR_INVALID_ARGUMENT;
    Plan p;
    int rc = make_plan(*g, &p);
    if (rc != MOE_OK) return rc;
    if (p.T == 0) {
        *n = routing_launches(p);
        return MOE_OK;
    }
    const bool em = p.layout == MOE_LAYOUT_EXPERT_MAJOR;
    // routing, row scatter, GEMM1, GEMM2, (RM/FLAT local-pick reduction), combine
    *n = routing_launches(p) + 1 + 2 + (em ? 0 : 1) + 1;
    return MOE_OK;
}

const char *moe_strerror(int err) {
    switch (err) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARGUMENT: return "invalid argument (null pointer, bad size or enum)";
    case MOE_ERR_EXPERTS_NOT_DIVISIBLE: return "num_experts must be divisible by world";
    case MOE_ERR_HIDDEN_ALIGNMENT: return "hidden must be a multiple of 128";
    case MOE_ERR_INTERMEDIATE_ALIGNMENT: return "intermediate must be a multiple of 128";
    case MOE_ERR_TOO_MANY_TOKENS: return "num_tokens exceeds world * max_tok";
    case MOE_ERR_TOPK: return "top_k must be in [1, 32]";
    case MOE_ERR_IDS_DTYPE: return "topk_ids dtype must be int32 or int64";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace smaller than moe_workspace_size()";
    case MOE_ERR_MISALIGNED: return "device pointer misaligned";
    case MOE_ERR_BAD_HANDLE: return "handle not filled by moe_dispatch";
    case MOE_ERR_CUDA: return "CUDA call or kernel launch failed";
    case MOE_ERR_NOT_BUILT_FOR_DEVICE: return "library built for sm_103a only (compute capability 10.3)";
    case MOE_ERR_LIMIT: return "geometry beyond library limits";
    default: return "unknown error";
    }
}

}  // extern "C"
