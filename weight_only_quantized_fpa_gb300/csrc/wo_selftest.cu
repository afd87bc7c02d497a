// wo_selftest.cu -- wo_selftest_wait_timeout: exercises the bounded-wait
// failure path of the kernels (an mbarrier wait that runs out records an
// error code in the workspace header and the CTA winds down) without any GPU
// fault: the waited-on barrier simply never completes.
#include <cuda_runtime.h>

#include "wo_internal.h"
#include "wo_sm100.cuh"

namespace wo {
namespace {

constexpr unsigned kSelftestCode = 99;  // error word written by the self-test

__global__ void wait_timeout_kernel(unsigned* err, unsigned long long limit_ns)
{
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        sm100::mbar_init(&bar, 1);  // one arrival expected; none ever comes
        abort_flag = 0;
        sm100::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0)
        sm100::mbar_wait_bounded(&bar, 0, &abort_flag, err, kSelftestCode, limit_ns);
}

}  // namespace

cudaError_t launch_wait_timeout(unsigned* err, unsigned limit_us, cudaStream_t s)
{
    wait_timeout_kernel<<<1, 32, 0, s>>>(err, (unsigned long long)limit_us * 1000ull);
    return cudaGetLastError();
}

}  // namespace wo

extern "C" wo_status wo_selftest_wait_timeout(void* workspace, size_t workspace_bytes,
                                              unsigned limit_us, void* stream)
{
    if (!workspace || workspace_bytes < wo::kWsHeader ||
        (reinterpret_cast<uintptr_t>(workspace) % 256) != 0 || limit_us < 1 || limit_us > 1000000)
        return WO_ERR_INVALID_ARG;
    return wo::launch_wait_timeout(static_cast<unsigned*>(workspace), limit_us,
                                   static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? WO_OK
               : WO_ERR_CUDA;
}
