// C ABI of the MiTA forward operator: plan validation, workspace, path
// choice and dispatch.  The operator and every argument are described in
// include/mita.h.
#include <stdlib.h>
#include <string.h>

#include "common.cuh"
#include "fused.cuh"
#include "staged.cuh"
#include "tiled.cuh"

using mita::Shape;

namespace {

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

int resolve_path(const mita_plan_s* p) {
    if (p->path_opt != MITA_PATH_AUTO) return p->path_opt;
    if (p->routes_s > 1) return MITA_PATH_STAGED;   // s > 1: the staged kernels only
    if (mita::fused_supported(p->s, p->dtype)) return MITA_PATH_FUSED;
    if (mita::tiled_supported(p->s, p->dtype)) return MITA_PATH_TILED;
    return MITA_PATH_STAGED;
}

}  // namespace

extern "C" {

const char* mita_strerror(int code) {
    switch (code) {
        case MITA_OK: return "ok";
        case MITA_ERR_INVALID_ARG: return "invalid argument";
        case MITA_ERR_UNSUPPORTED: return "unsupported shape or option";
        case MITA_ERR_CUDA: return "CUDA runtime error";
        case MITA_ERR_TIMEOUT: return "device wait timed out";
        case MITA_ERR_OOM: return "out of device memory";
        case MITA_ERR_DEVICE: return "kernel reported invalid data";
        default: return "unknown status";
    }
}

int mita_plan(mita_plan_t* plan, int B, int H, int N, int d, mita_grid_t grid, int m, int k,
              mita_dtype_t dtype) {
    if (!plan) return MITA_ERR_INVALID_ARG;
    *plan = nullptr;
    if (B < 1 || H < 1 || N < 1 || d < 1 || m < 1 || k < 1 || k > N) return MITA_ERR_INVALID_ARG;
    if (grid.gh < 1 || grid.gw < 1 || grid.ph < 1 || grid.pw < 1) return MITA_ERR_INVALID_ARG;
    if ((long long)grid.gh * grid.gw != N || (long long)grid.ph * grid.pw != m) return MITA_ERR_INVALID_ARG;
    if (grid.ph > grid.gh || grid.pw > grid.gw) return MITA_ERR_INVALID_ARG;
    if (dtype != MITA_F32 && dtype != MITA_BF16) return MITA_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return MITA_ERR_UNSUPPORTED;
    if (m > 1024 || k > 4096 || m + k > 4096) return MITA_ERR_UNSUPPORTED;
    if ((long long)B * H > 65535) return MITA_ERR_UNSUPPORTED;
    if ((double)B * H * N * d >= 1099511627776.0) return MITA_ERR_UNSUPPORTED;

    mita_plan_s* p = (mita_plan_s*)calloc(1, sizeof(mita_plan_s));
    if (!p) return MITA_ERR_OOM;
    p->s = Shape{B, H, N, d, m, k, grid.gh, grid.gw, grid.ph, grid.pw};
    p->dtype = dtype;
    p->path_opt = MITA_PATH_AUTO;
    if (cudaGetDevice(&p->device) != cudaSuccess) { free(p); return MITA_ERR_CUDA; }

    const size_t BH = (size_t)B * H, e = dtype == MITA_BF16 ? 2 : 4;
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t o = off; off = align_up(off + bytes, 256); return o; };
    const size_t oQl = take(BH * m * d * e), oVl = take(BH * m * d * e);
    const size_t oS = take(BH * m * (size_t)N * 4);
    const size_t oIdx = take(BH * m * (size_t)k * 4), oRoute = take(BH * (size_t)N * 4);
    const size_t oCnt = take(BH * m * 4), oOff = take(BH * (m + 1) * 4), oPerm = take(BH * (size_t)N * 4);
    const size_t oStatus = take(256);
    // backward (fp32): dQ_l, dV_l, V_l, then per landmark row {max S, sum of weights}
    const size_t oGradL = take((3 * BH * m * d + 2 * BH * m) * 4);
    const bool tiled = mita::tiled_supported(p->s, dtype);
    const size_t oRowmax = take(tiled ? 2 * BH * m * 4 : 0);   // row max, then row min
    const size_t oVpart = take(tiled ? mita::tiled_part_bytes(p->s) : 0);
    const size_t oCursor = take(tiled ? BH * m * 4 : 0);
    const size_t oTiles = take(tiled ? BH * (size_t)mita::tiled_max_tiles(p->s) * 4 : 0);
    const size_t oNtiles = take(tiled ? BH * 4 : 0);

    p->ws_bytes = off;
    if (cudaMalloc(&p->ws, p->ws_bytes) != cudaSuccess) {
        cudaGetLastError();
        free(p);
        return MITA_ERR_OOM;
    }
    char* b = (char*)p->ws;
    p->Ql = b + oQl;
    p->Vl = b + oVl;
    p->S = (float*)(b + oS);
    p->idx = (int32_t*)(b + oIdx);
    p->route = (int32_t*)(b + oRoute);
    p->counts = (int32_t*)(b + oCnt);
    p->offsets = (int32_t*)(b + oOff);
    p->perm = (int32_t*)(b + oPerm);
    p->status = (int32_t*)(b + oStatus);
    p->dQl = (float*)(b + oGradL);
    p->dVl = p->dQl + BH * m * d;
    if (tiled) {
        p->rowmax = (uint32_t*)(b + oRowmax);
        p->vpart = (float*)(b + oVpart);
        p->cursor = (int32_t*)(b + oCursor);
        p->tiles = (int32_t*)(b + oTiles);
        p->ntiles = (int32_t*)(b + oNtiles);
    }
    if (cudaMemset(p->status, 0, 256) != cudaSuccess) {
        cudaFree(p->ws);
        free(p);
        return MITA_ERR_CUDA;
    }
    *plan = p;
    return MITA_OK;
}

int mita_set_option(mita_plan_t p, int option, int value) {
    if (!p) return MITA_ERR_INVALID_ARG;
    if (option == MITA_OPT_PATH) {
        if (value != MITA_PATH_AUTO && value != MITA_PATH_STAGED && value != MITA_PATH_FUSED &&
            value != MITA_PATH_TILED)
            return MITA_ERR_INVALID_ARG;
        p->path_opt = value;
        return MITA_OK;
    }
    if (option == MITA_OPT_KEEP_LANDMARKS) {
        if (value != 0 && value != 1) return MITA_ERR_INVALID_ARG;
        p->keep_landmarks = value;
        return MITA_OK;
    }
    if (option == MITA_OPT_ROUTING_ONLY) {
        if (value != 0 && value != 1) return MITA_ERR_INVALID_ARG;
        p->routing_only = value;
        return MITA_OK;
    }
    if (option == MITA_OPT_ROUTES) {
        if (value < 1 || value > mita::kMaxRoutes || value > p->s.m) return MITA_ERR_INVALID_ARG;
        p->routes_s = value;
        return MITA_OK;
    }
    return MITA_ERR_INVALID_ARG;
}

int mita_get_path(mita_plan_t p) {
    if (!p) return -MITA_ERR_INVALID_ARG;
    const int path = resolve_path(p);
    if (path != MITA_PATH_STAGED && p->routes_s > 1) return -MITA_ERR_UNSUPPORTED;
    if (path == MITA_PATH_FUSED && !mita::fused_supported(p->s, p->dtype)) return -MITA_ERR_UNSUPPORTED;
    if (path == MITA_PATH_TILED && !p->rowmax) return -MITA_ERR_UNSUPPORTED;
    return path;
}

int mita_forward(mita_plan_t p, const void* Q, const void* K, const void* V, void* out, int32_t* expert_idx,
                 int32_t* route, struct CUstream_st* stream) {
    if (!p || !Q || !K || !V || !out) return MITA_ERR_INVALID_ARG;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(out)) return MITA_ERR_INVALID_ARG;
    if ((expert_idx && !aligned16(expert_idx)) || (route && !aligned16(route))) return MITA_ERR_INVALID_ARG;
    int32_t* idx = expert_idx ? expert_idx : p->idx;
    int32_t* rt = route ? route : p->route;
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t err;
    const int path = resolve_path(p);
    if (path != MITA_PATH_STAGED && p->routes_s > 1) return MITA_ERR_UNSUPPORTED;
    if (path == MITA_PATH_FUSED) {
        if (!mita::fused_supported(p->s, p->dtype)) return MITA_ERR_UNSUPPORTED;
        err = mita::run_fused(p, Q, K, V, out, idx, rt, p->keep_landmarks, st);
    } else if (path == MITA_PATH_TILED) {
        if (!p->rowmax) return MITA_ERR_UNSUPPORTED;
        err = mita::run_tiled(p, Q, K, V, out, idx, rt, st);
    } else {
        err = mita::run_staged(p, Q, K, V, out, idx, rt, st);
    }
    if (err != cudaSuccess) return MITA_ERR_CUDA;
    p->landmarks_valid = p->keep_landmarks || path != MITA_PATH_FUSED;
    return MITA_OK;
}

int mita_backward(mita_plan_t p, const void* Q, const void* K, const void* V, const void* dOut, float* dQ,
                  float* dK, float* dV, struct CUstream_st* stream) {
    if (!p || !Q || !K || !V || !dOut || !dQ || !dK || !dV) return MITA_ERR_INVALID_ARG;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(dOut) || !aligned16(dQ) || !aligned16(dK) ||
        !aligned16(dV))
        return MITA_ERR_INVALID_ARG;
    if (p->routes_s > 1) return MITA_ERR_UNSUPPORTED;
    if (mita::run_backward(p, Q, K, V, dOut, dQ, dK, dV, (cudaStream_t)stream) != cudaSuccess) return MITA_ERR_CUDA;
    return MITA_OK;
}

int mita_get_status(mita_plan_t p) {
    if (!p) return MITA_ERR_INVALID_ARG;
    int prev = 0;
    cudaGetDevice(&prev);
    cudaSetDevice(p->device);
    int32_t st = 0;
    int rc = MITA_OK;
    if (cudaDeviceSynchronize() != cudaSuccess) rc = MITA_ERR_CUDA;
    else if (cudaMemcpy(&st, p->status, 4, cudaMemcpyDeviceToHost) != cudaSuccess) rc = MITA_ERR_CUDA;
    else {
        rc = st;
        cudaMemset(p->status, 0, 4);
    }
    cudaSetDevice(prev);
    return rc;
}

int mita_get_landmarks(mita_plan_t p, void* Ql, void* Vl, struct CUstream_st* stream) {
    if (!p || !Ql || !Vl || !p->landmarks_valid) return MITA_ERR_INVALID_ARG;
    const size_t bytes = (size_t)p->s.BH() * p->s.m * p->s.d * (p->dtype == MITA_BF16 ? 2 : 4);
    cudaStream_t st = (cudaStream_t)stream;
    if (cudaMemcpyAsync(Ql, p->Ql, bytes, cudaMemcpyDeviceToDevice, st) != cudaSuccess) return MITA_ERR_CUDA;
    if (cudaMemcpyAsync(Vl, p->Vl, bytes, cudaMemcpyDeviceToDevice, st) != cudaSuccess) return MITA_ERR_CUDA;
    return MITA_OK;
}

int mita_launch_count(mita_plan_t p, uint64_t* launches) {
    if (!p || !launches) return MITA_ERR_INVALID_ARG;
    *launches = p->launches;
    return MITA_OK;
}

int mita_workspace_bytes(mita_plan_t p, uint64_t* bytes) {
    if (!p || !bytes) return MITA_ERR_INVALID_ARG;
    *bytes = p->ws_bytes;
    return MITA_OK;
}

void mita_destroy(mita_plan_t p) {
    if (!p) return;
    int prev = 0;
    cudaGetDevice(&prev);
    cudaSetDevice(p->device);
    cudaDeviceSynchronize();
    cudaFree(p->ws);
    cudaSetDevice(prev);
    free(p);
}

}  // extern "C"
