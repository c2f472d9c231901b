// Allocation-free variant of the stage-by-stage forward.
//
// Some callers cannot call cudaMalloc: code embedded in a host framework
// that owns all device memory through its own pool and forbids raw device
// allocations, and latency-critical loops in which an allocation would
// implicitly synchronise the device.  They cannot create a plan either,
// since mita_plan() allocates the workspace.  mita_forward_noalloc() runs
// the same stage kernels as the staged path with their scratch (landmark
// queries and values, landmark scores, query buckets, status word) carved
// out of one fixed device array that the library declares at file scope.
#include <mutex>

#include "common.cuh"
#include "staged.cuh"

namespace {

// The shared scratch.  Every GPU that loads the library holds it until the
// process exits.
constexpr size_t kScratchBytes = (size_t)MITA_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

// Device address of g_scratch per device.  In host code the symbol name is
// only a host-side stand-in, so the address is looked up once per device
// with that device current.
constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int scratch_address(int device, void** out) {
    if (device < 0 || device >= kMaxDevices) return MITA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_addr[device]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess) {
            cudaGetLastError();
            return MITA_ERR_CUDA;
        }
        g_addr[device] = p;
    }
    *out = g_addr[device];
    return MITA_OK;
}

}  // namespace

extern "C" uint64_t mita_noalloc_scratch_bytes(void) { return (uint64_t)kScratchBytes; }

extern "C" int mita_forward_noalloc(int B, int H, int N, int d, mita_grid_t grid, int m, int k,
                                    mita_dtype_t dtype, const void* Q, const void* K, const void* V,
                                    void* out, int32_t* expert_idx, int32_t* route,
                                    struct CUstream_st* stream) {
    if (B < 1 || H < 1 || N < 1 || d < 1 || m < 1 || k < 1 || k > N) return MITA_ERR_INVALID_ARG;
    if (grid.gh < 1 || grid.gw < 1 || grid.ph < 1 || grid.pw < 1) return MITA_ERR_INVALID_ARG;
    if ((long long)grid.gh * grid.gw != N || (long long)grid.ph * grid.pw != m) return MITA_ERR_INVALID_ARG;
    if (grid.ph > grid.gh || grid.pw > grid.gw) return MITA_ERR_INVALID_ARG;
    if (dtype != MITA_F32 && dtype != MITA_BF16) return MITA_ERR_INVALID_ARG;
    if (!Q || !K || !V || !out) return MITA_ERR_INVALID_ARG;
    auto mis = [](const void* p) { return ((uintptr_t)p & 15u) != 0; };
    if (mis(Q) || mis(K) || mis(V) || mis(out) || (expert_idx && mis(expert_idx)) || (route && mis(route)))
        return MITA_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return MITA_ERR_UNSUPPORTED;
    if (m > 1024 || k > 4096 || m + k > 4096 || (long long)B * H > 65535) return MITA_ERR_UNSUPPORTED;

    // Carve the stage buffers out of the scratch; refuse shapes that do not fit.
    const size_t BH = (size_t)B * H, e = dtype == MITA_BF16 ? 2 : 4;
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t o = off; off = align_up(off + bytes, 256); return o; };
    const size_t oQl = take(BH * m * d * e), oVl = take(BH * m * d * e);
    const size_t oS = take(BH * m * (size_t)N * 4);
    const size_t oIdx = take(expert_idx ? 0 : BH * m * (size_t)k * 4);
    const size_t oRoute = take(route ? 0 : BH * (size_t)N * 4);
    const size_t oCnt = take(BH * m * 4), oOff = take(BH * (m + 1) * 4), oPerm = take(BH * (size_t)N * 4);
    const size_t oStatus = take(256);
    if (off > kScratchBytes) return MITA_ERR_UNSUPPORTED;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MITA_ERR_CUDA;
    void* base = nullptr;
    int rc = scratch_address(dev, &base);
    if (rc != MITA_OK) return rc;

    mita_plan_s p = {};
    p.s = mita::Shape{B, H, N, d, m, k, grid.gh, grid.gw, grid.ph, grid.pw};
    p.dtype = dtype;
    p.device = dev;
    p.path_opt = MITA_PATH_STAGED;
    char* b = (char*)base;
    p.ws = base;
    p.ws_bytes = off;
    p.Ql = b + oQl;
    p.Vl = b + oVl;
    p.S = (float*)(b + oS);
    p.idx = (int32_t*)(b + oIdx);
    p.route = (int32_t*)(b + oRoute);
    p.counts = (int32_t*)(b + oCnt);
    p.offsets = (int32_t*)(b + oOff);
    p.perm = (int32_t*)(b + oPerm);
    p.status = (int32_t*)(b + oStatus);

    cudaStream_t st = (cudaStream_t)stream;
    // The status word is the only scratch that must start at zero (the
    // bucket kernel clears its own counters; every other buffer is written
    // before it is read).
    if (cudaMemsetAsync(p.status, 0, 4, st) != cudaSuccess) return MITA_ERR_CUDA;
    cudaError_t err = mita::run_staged(&p, Q, K, V, out, expert_idx ? expert_idx : p.idx,
                                       route ? route : p.route, st);
    return err == cudaSuccess ? MITA_OK : MITA_ERR_CUDA;
}
