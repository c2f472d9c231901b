// One-kernel MiTA forward for short sequences: launcher declarations.
#pragma once
#include "common.cuh"

namespace mita {
bool fused_supported(const Shape& s, mita_dtype_t dtype);

cudaError_t run_fused(mita_plan_s* p, const void* Q, const void* K, const void* V, void* out,
                      int32_t* idx, int32_t* route, int keep_landmarks, cudaStream_t st);
}  // namespace mita
