// Test entry points (include/mita_testing.h): the device-side error reports
// of the operator's kernels, driven from the host without a fault.
#include "common.cuh"
#include "mita_testing.h"
#include "tc_util.cuh"

namespace mita {
cudaError_t testing_bucket(mita_plan_s* p, const int32_t* route, cudaStream_t st);   // staged.cu
}

namespace {

// One warp: an mbarrier expecting one arrival that never comes; the bounded
// wait gives up after `budget` cycles and the kernel reports the timeout.
__global__ void wait_timeout_kernel(long long budget, int32_t* status) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t ub = (uint32_t)__cvta_generic_to_shared(&bar);
    if (threadIdx.x == 0) {
        mita::tc::mbar_init(ub, 1);
        mita::tc::mbar_fence_init();
    }
    __syncwarp();
    if (threadIdx.x == 0 && !mita::tc::mbar_wait_bounded(ub, 0, budget))
        atomicExch(status, (int)MITA_ERR_TIMEOUT);
}

}  // namespace

extern "C" int mita_testing_bucket(mita_plan_t p, const int32_t* route, struct CUstream_st* stream) {
    if (!p || !route || ((uintptr_t)route & 15u)) return MITA_ERR_INVALID_ARG;
    if (mita::testing_bucket(p, route, (cudaStream_t)stream) != cudaSuccess) return MITA_ERR_CUDA;
    p->done_valid = 0;   // mita_get_status() waits for the device
    return MITA_OK;
}

extern "C" int mita_testing_wait(mita_plan_t p, long long budget_cycles, struct CUstream_st* stream) {
    if (!p || budget_cycles < 1 || budget_cycles > (1LL << 31)) return MITA_ERR_INVALID_ARG;
    wait_timeout_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(budget_cycles, p->status);
    if (cudaGetLastError() != cudaSuccess) return MITA_ERR_CUDA;
    p->done_valid = 0;
    return MITA_OK;
}
