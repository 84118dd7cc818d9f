// Self-test of the device-side failure path: a bounded mbarrier wait that nothing will ever
// satisfy.  The wait is the same helper every tcgen05 GEMM uses (tc_common.cuh): after its
// limit it raises the CTA's abort flag, sets MOE_STATUS_TIMEOUT in the status word and
// returns, and the kernel exits normally.  Nothing faults, traps or hangs.
#include "tc_common.cuh"

namespace moe {
namespace {

__global__ void wait_expiry_kernel(int32_t *status) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);   // one arrival expected, none will come
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, &abort_flag, status);
    __syncthreads();
}

}  // namespace
}  // namespace moe

extern "C" int moe_selftest_wait_expiry(int32_t *status_dev, void *stream) {
    if (!status_dev) return MOE_ERR_INVALID_ARGUMENT;
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (major != 10 || minor != 3) return MOE_ERR_NOT_BUILT_FOR_DEVICE;
    moe::wait_expiry_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status_dev);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
