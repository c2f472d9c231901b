// tcgen05 kernels of the tiled path: launcher declarations.  `chain`: the
// launch may overlap the previous kernel on the stream (see launch.cuh).
#pragma once
#include "common.cuh"

namespace mita {
// Raw landmark scores S [BH, m, N] fp32 and each row's max / min as order keys.
cudaError_t tc_scores(const Shape& s, const void* Ql, const void* K, float* S, uint32_t* rowmax,
                      uint32_t* rowmin, int32_t* status, cudaStream_t st, bool chain);
// Split-K partials [BH, splits, m, d + 1] of the landmark values (numerators
// exp2(S * cs - max * cs) applied to V; last column: their sum).
cudaError_t tc_values(const Shape& s, const float* S, const uint32_t* rowmax, const void* V, float* part,
                      float cs, int32_t* status, cudaStream_t st, bool chain);
int tc_value_splits(const Shape& s);
// Scores and routes in one launch (m <= 256): raw scores with each row's max
// and min, and every query's route with the per-landmark counts (added).
bool tc_scores_route_supported(const Shape& s);
cudaError_t tc_scores_route(const Shape& s, const void* Ql, const void* K, const void* Q, float* S, uint32_t* rowmax,
                            uint32_t* rowmin, int32_t* route, int32_t* counts, int32_t* status, cudaStream_t st,
                            bool chain);
int tc_value_keys(const Shape& s);   // keys per split
// Route of every query (first argmax of q . Q_l) and per-landmark query counts (added).
cudaError_t tc_route(const Shape& s, const void* Q, const void* Ql, int32_t* route, int32_t* counts,
                     int32_t* status, cudaStream_t st, bool chain);
}  // namespace mita
