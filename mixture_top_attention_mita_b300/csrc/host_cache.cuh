// Host-side state of the launch path, kept across forwards so that a forward
// costs only its launches: 2-D bf16 TMA maps (encoded once per base address,
// row length, row count and box), the dynamic shared-memory limit of each
// kernel (raised once to the largest size asked for) and per-SM occupancy.
// All three are guarded by one mutex; every entry is a pure function of its
// key, so a cached entry is never stale.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>

namespace mita {

// Map over `rows` rows of `d` bf16 values (row pitch 2*d bytes), boxes of
// box_cols x box_rows, 128-byte swizzle, rows past the end read as zero.
// Returns false when the driver entry point is missing or rejects the map.
bool tma_map_bf16(CUtensorMap* map, const void* base, int d, size_t rows, int box_cols, int box_rows);

// cudaFuncAttributeMaxDynamicSharedMemorySize of `func` raised to at least `bytes`.
cudaError_t ensure_smem_attr(const void* func, int bytes);

// Resident blocks per SM of `func` at `threads` threads and `smem` dynamic
// shared bytes (after ensure_smem_attr); 0 when the query fails.
int blocks_per_sm(const void* func, int threads, int smem);

}  // namespace mita
