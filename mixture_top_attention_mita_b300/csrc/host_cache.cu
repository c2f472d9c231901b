// Host-side caches of the launch path (see host_cache.cuh).
#include "host_cache.cuh"

#include <mutex>

namespace mita {
namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

std::mutex g_mu;

EncodeTiledFn encode_fn() {   // under g_mu
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (EncodeTiledFn)p;
    }
    return fn;
}

struct MapEntry {
    const void* base;
    int d, box_cols, box_rows;
    size_t rows;
    int device;
    CUtensorMap map;
};
constexpr int kMaps = 64;
MapEntry g_maps[kMaps];
int g_nmaps = 0, g_next = 0;

struct FuncEntry {
    const void* func;
    int device, smem_set;
};
constexpr int kFuncs = 64;
FuncEntry g_funcs[kFuncs];
int g_nfuncs = 0;

struct OccEntry {
    const void* func;
    int device, threads, smem, blocks;
};
constexpr int kOcc = 64;
OccEntry g_occ[kOcc];
int g_nocc = 0, g_occ_next = 0;

int current_device() {
    int dev = 0;
    cudaGetDevice(&dev);
    return dev;
}

}  // namespace

bool tma_map_bf16(CUtensorMap* map, const void* base, int d, size_t rows, int box_cols, int box_rows) {
    const int dev = current_device();
    std::lock_guard<std::mutex> lock(g_mu);
    for (int i = 0; i < g_nmaps; ++i) {
        const MapEntry& e = g_maps[i];
        if (e.base == base && e.d == d && e.rows == rows && e.box_cols == box_cols && e.box_rows == box_rows &&
            e.device == dev) {
            *map = e.map;
            return true;
        }
    }
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)d * 2};
    const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    if (fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    const int slot = g_nmaps < kMaps ? g_nmaps++ : (g_next++ % kMaps);
    g_maps[slot] = MapEntry{base, d, box_cols, box_rows, rows, dev, *map};
    return true;
}

cudaError_t ensure_smem_attr(const void* func, int bytes) {
    const int dev = current_device();
    std::lock_guard<std::mutex> lock(g_mu);
    FuncEntry* f = nullptr;
    for (int i = 0; i < g_nfuncs; ++i)
        if (g_funcs[i].func == func && g_funcs[i].device == dev) f = &g_funcs[i];
    if (f && f->smem_set >= bytes) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    if (!f && g_nfuncs < kFuncs) f = &g_funcs[g_nfuncs++];
    if (f) *f = FuncEntry{func, dev, bytes};
    return cudaSuccess;
}

int blocks_per_sm(const void* func, int threads, int smem) {
    const int dev = current_device();
    std::lock_guard<std::mutex> lock(g_mu);
    for (int i = 0; i < g_nocc; ++i) {
        const OccEntry& o = g_occ[i];
        if (o.func == func && o.device == dev && o.threads == threads && o.smem == smem) return o.blocks;
    }
    int blocks = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, func, threads, smem) != cudaSuccess) return 0;
    const int slot = g_nocc < kOcc ? g_nocc++ : (g_occ_next++ % kOcc);
    g_occ[slot] = OccEntry{func, dev, threads, smem, blocks};
    return blocks;
}

}  // namespace mita
