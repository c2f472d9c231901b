// Tensor-core tiled MiTA forward for long sequences: launcher declarations.
#pragma once
#include "common.cuh"

namespace mita {
bool tiled_supported(const Shape& s, mita_dtype_t dtype);
size_t tiled_part_bytes(const Shape& s);   // landmark-value partials in the plan workspace
int tiled_max_tiles(const Shape& s);       // attention tiles per head, upper bound
// Q_l (bf16, d = 64 or 128) by the tiled path's pool kernel, which also resets
// each landmark's row max and min (rowmax, then rowmin = rowmax + BH m) and
// query count.
cudaError_t tiled_pool(const Shape& s, const void* Q, void* Ql, uint32_t* rowmax, int32_t* counts, cudaStream_t st);
// The tiled path's top-k of rows up to 4096 keys (raw scores S [BH, m, N]
// with each row's max and min from the score kernel; idx [BH, m, k]).
bool tiled_topk_supported(const Shape& s);
cudaError_t tiled_topk(const Shape& s, const float* S, const uint32_t* rowmax, int32_t* idx, cudaStream_t st);
// Landmark values by the tiled path's tensor-core kernel (bf16 V_l, and V_l in
// fp32 with each row's {max raw score, sum of the numerators} as the backward
// needs them); part is the tiled workspace's split partials.
cudaError_t tiled_values_stats(const Shape& s, const float* S, const uint32_t* rowmax, const void* V, float* part,
                               void* Vl, float* Vl32, float* stats, int32_t* status, cudaStream_t st);
cudaError_t run_tiled(mita_plan_s* p, const void* Q, const void* K, const void* V, void* out,
                      int32_t* idx, int32_t* route, cudaStream_t st);
}  // namespace mita
