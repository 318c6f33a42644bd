// wait_probe.cu -- mha_check_wait_timeout: runs the pipelines' bounded mbarrier wait against a
// barrier nothing ever arrives at, so the failure path (timeout -> abort flag -> status word ->
// orderly exit) can be exercised without faulting or hanging the GPU.
#include <stdint.h>

#include "../../include/mha.h"
#include "internal.h"
#include "ptx.cuh"

namespace mha {
namespace {

// Two waiters on one never-completed barrier: the first gives up after limit_ns, records
// MHA_ERR_TIMEOUT and raises the CTA abort flag; the second sees the flag and returns too.
__global__ void wait_probe_kernel(int* status, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if ((threadIdx.x & 31) == 0) mbar_wait(smem_u32(&bar), 0, &abort_flag, status, limit_ns);
    __syncwarp();  // whole warps reach the CTA barrier
    __syncthreads();
}

}  // namespace
}  // namespace mha

extern "C" mha_status mha_check_wait_timeout(mha_t handle, int64_t limit_ns, void* stream) {
    if (handle == nullptr || limit_ns <= 0 || limit_ns > 10000000000ll) return MHA_ERR_INVALID_ARG;
    if (handle->ws == nullptr) return MHA_ERR_WORKSPACE;
    mha::wait_probe_kernel<<<1, 64, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<int*>(handle->ws), (uint64_t)limit_ns);
    return cudaGetLastError() == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
}
