// tim_selftest.cu -- failure-detection self-test of the pipelines' bounded waits.
//
// Every mbarrier wait in the library's kernels gives up after a time budget,
// raises the CTA's abort flag, lets in-flight copies land and records
// TIM_ERR_TIMEOUT in the status word, instead of hanging the GPU.  This kernel
// runs that path on purpose without any fault: one warp waits on an mbarrier
// that nothing ever arrives on, with the caller's budget, and records the
// status.  The context stays usable; tim_check() reports TIM_ERR_TIMEOUT.
#include "../../include/tim.h"
#include "tim_internal.h"
#include "tim_ptx.cuh"

namespace {

__global__ void selftest_wait_kernel(int *status, uint64_t budget_ns, int *observed)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        tim::mbar_init(tim::smem_u32(&bar), 1);
        tim::fence_mbar_init();
        abort_flag = 0;
    }
    __syncwarp();
    // phase 0 never completes: nothing arrives on the barrier
    const bool ok = tim::mbar_wait(tim::smem_u32(&bar), 0u, &abort_flag, budget_ns);
    __syncwarp();
    if (threadIdx.x == 0) {
        *observed = ok ? 1 : 0;
        if (!ok)
            atomicCAS(status, 0, static_cast<int>(TIM_ERR_TIMEOUT));
    }
}

__device__ int g_selftest_observed;

} // namespace

extern "C" int tim_selftest_wait_timeout(uint32_t budget_us, tim_stream_t stream)
{
    if (budget_us == 0 || budget_us > 1000000u)
        return tim::record_error(TIM_ERR_INVALID_ARG, "budget_us must be in [1, 1000000]");
    int dev = 0, major = 0, minor = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e != cudaSuccess)
        return tim::record_error(TIM_ERR_CUDA, cudaGetErrorString(e));
    if (major != 10 || minor != 3)
        return tim::record_error(TIM_ERR_UNSUPPORTED_DEVICE, "this library needs sm_103a (GB300)");
    int *status = nullptr;
    int *observed = nullptr;
    if ((e = tim::status_word_address(&status)) != cudaSuccess ||
        (e = cudaGetSymbolAddress(reinterpret_cast<void **>(&observed), g_selftest_observed)) != cudaSuccess)
        return tim::record_error(TIM_ERR_CUDA, cudaGetErrorString(e));
    selftest_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        status, static_cast<uint64_t>(budget_us) * 1000ull, observed);
    if ((e = cudaGetLastError()) != cudaSuccess)
        return tim::record_error(TIM_ERR_CUDA, cudaGetErrorString(e));
    return tim::record_error(TIM_OK, "");
}
