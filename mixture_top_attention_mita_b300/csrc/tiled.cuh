// Tensor-core tiled MiTA forward for long sequences: launcher declarations.
#pragma once
#include "common.cuh"

namespace mita {
bool tiled_supported(const Shape& s, mita_dtype_t dtype);
size_t tiled_part_bytes(const Shape& s);   // landmark-value partials in the plan workspace
int tiled_max_tiles(const Shape& s);       // attention tiles per head, upper bound
cudaError_t run_tiled(mita_plan_s* p, const void* Q, const void* K, const void* V, void* out,
                      int32_t* idx, int32_t* route, cudaStream_t st);
}  // namespace mita
