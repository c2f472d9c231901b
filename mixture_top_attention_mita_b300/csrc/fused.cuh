// One-kernel MiTA forward for short sequences: launcher declarations.
#pragma once
#include "common.cuh"

namespace mita {
bool fused_supported(const Shape& s, mita_dtype_t dtype);
// Pooling matrix of the one-kernel path (bf16 0/1, landmark x token), built on
// the host and kept in the plan workspace.
size_t fused_pool_bytes(const Shape& s);
void fused_pool_matrix(const Shape& s, uint16_t* dst);
cudaError_t run_fused(mita_plan_s* p, const void* Q, const void* K, const void* V, void* out,
                      int32_t* idx, int32_t* route, int keep_landmarks, cudaStream_t st);
}  // namespace mita
