// Stage-by-stage MiTA kernels: launcher declarations.
#pragma once
#include "common.cuh"

namespace mita {
size_t staged_attend_smem(const Shape& s, int ns);   // dynamic shared bytes, ns experts per query
// Step 3 of the staged path (exact top-k over raw scores S [BH, m, N] fp32),
// reused by the tiled path for rows longer than its bitmap select takes;
// `chained`: the launch may overlap the previous kernel (see launch.cuh).
cudaError_t staged_topk(const Shape& s, const float* S, int32_t* idx, cudaStream_t st, bool chained = false);
// Backward of the operator (routes s = 1) into fp32 dQ, dK, dV [BH, N, d].
cudaError_t run_backward(mita_plan_s* p, const void* Q, const void* K, const void* V, const void* dOut, float* dQ,
                         float* dK, float* dV, cudaStream_t st);
cudaError_t run_staged(mita_plan_s* p, const void* Q, const void* K, const void* V, void* out,
                       int32_t* idx, int32_t* route, cudaStream_t st);
}  // namespace mita
