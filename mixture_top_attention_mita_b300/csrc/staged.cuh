// Stage-by-stage MiTA kernels: launcher declarations.
#pragma once
#include "common.cuh"

namespace mita {
size_t staged_attend_smem(const Shape& s);
cudaError_t run_staged(mita_plan_s* p, const void* Q, const void* K, const void* V, void* out,
                       int32_t* idx, int32_t* route, cudaStream_t st);
}  // namespace mita
