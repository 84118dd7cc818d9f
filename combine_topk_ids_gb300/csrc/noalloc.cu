// moe_route_noalloc: EXPERT_MAJOR routing whose scratch lives in a static device array.
//
// Who needs it: hosts that hand a library only its input and output buffers and own every
// byte of device memory themselves (plugin interfaces of inference runtimes, engines with a
// fixed memory budget planned ahead of time).  Such callers cannot provide the routing
// workspace that moe_dispatch carves its per-chunk histograms from, and the library must
// not call cudaMalloc on their behalf (it would bypass their allocator and their memory
// accounting).  This entry point computes the same routing outputs as moe_dispatch without
// any allocation: its scratch is a fixed array compiled into the library.
#include <mutex>

#include "moe_internal.cuh"

namespace moe {
namespace {

// Per-chunk expert histograms and their exclusive bases ([E][nb] int32 each) plus the two
// GEMM row-block prefixes ([E+1] each): 2*E*nb + 2*(E+1) ints must fit.  Every GPU that
// loads the library holds this array until the process exits.
constexpr size_t kScratchBytes = MOE_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) int32_t g_route_scratch[kScratchBytes / sizeof(int32_t)];

std::mutex g_mutex;
int32_t *g_scratch_ptr[64];   // device address of g_route_scratch, per device

// Device address of the scratch array on the current device, looked up once per device.
int32_t *scratch_on_current_device(int *err) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        *err = MOE_ERR_CUDA;
        return nullptr;
    }
    std::lock_guard<std::mutex> lk(g_mutex);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || !p) {
            *err = MOE_ERR_CUDA;
            return nullptr;
        }
        g_scratch_ptr[dev] = static_cast<int32_t *>(p);
    }
    return g_scratch_ptr[dev];
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" int moe_route_noalloc(const moe_geom *g, const void *topk_ids_dev, int ids_dtype,
                                 int32_t *counts_dev, int32_t *offsets_dev, int32_t *pick_pos_dev,
                                 int32_t *pick_src_dev, int32_t *slot_dev,
                                 int32_t *layout_range_dev, int32_t *status_dev, void *stream) {
    if (!g || !counts_dev || !offsets_dev || !layout_range_dev || !status_dev)
        return MOE_ERR_INVALID_ARGUMENT;
    if (g->layout != MOE_LAYOUT_EXPERT_MAJOR) return MOE_ERR_INVALID_ARGUMENT;
    if (ids_dtype != MOE_IDS_INT32 && ids_dtype != MOE_IDS_INT64) return MOE_ERR_IDS_DTYPE;
    Plan p;
    int rc = make_plan(*g, &p);
    if (rc != MOE_OK) return rc;
    if (p.T > 0 && (!topk_ids_dev || !pick_pos_dev || !pick_src_dev || !slot_dev))
        return MOE_ERR_INVALID_ARGUMENT;
    // scratch: blk_hist [E*nb], blk_base [E*nb], mprefix [E+1], mprefix2 [E+1]
    const size_t hist_ints = (size_t)p.E * p.nb;
    const size_t need = 2 * hist_ints + 2 * ((size_t)p.E + 1);
    if (need * sizeof(int32_t) > kScratchBytes) return MOE_ERR_LIMIT;
    if ((rc = check_device()) != MOE_OK) return rc;

    int err = MOE_OK;
    int32_t *scratch = scratch_on_current_device(&err);
    if (!scratch) return err;

    Routing r{};
    r.p = &p;
    r.status = status_dev;
    r.counts = counts_dev;
    r.offsets = offsets_dev;
    r.pick_pos = pick_pos_dev;
    r.pick_src = pick_src_dev;
    r.slot = slot_dev;
    r.layout_range = layout_range_dev;
    r.blk_hist = scratch;
    r.blk_base = scratch + hist_ints;
    r.mprefix = scratch + 2 * hist_ints;
    r.mprefix2 = r.mprefix + p.E + 1;
    // every scratch entry the kernels read is written earlier in the same call, so the
    // previous call's contents never need clearing; the status output starts at 0, which
    // launch_routing sees to before any routing kernel can set a bit
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return launch_routing(r, topk_ids_dev, ids_dtype == MOE_IDS_INT64, nullptr, nullptr, s) ==
                   cudaSuccess
               ? MOE_OK
               : MOE_ERR_CUDA;
}
