// C ABI of the MiTA forward operator: plan validation, workspace, path
// choice and dispatch.  The operator and every argument are described in
// include/mita.h.
#include <stdlib.h>
#include <algorithm>
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

// One device allocation of `bytes` on the plan's device (MITA_ERR_OOM on failure).
int alloc_region(mita_plan_s* p, void** out, size_t bytes) {
    int prev = 0;
    cudaGetDevice(&prev);
    cudaSetDevice(p->device);
    const cudaError_t e = cudaMalloc(out, bytes);
    cudaSetDevice(prev);
    if (e != cudaSuccess) {
        cudaGetLastError();
        *out = nullptr;
        return MITA_ERR_OOM;
    }
    p->ws_bytes += bytes;
    return MITA_OK;
}

// The regions a path needs beyond the core: raw scores for the staged and
// tiled paths (and the backward), the tiled path's own buffers, and the
// backward's fp32 region.  Each is allocated once, the first time it is
// needed: at plan time for the path the plan starts on, else when an option
// or the first backward call selects a path that needs it.
int ensure_scores(mita_plan_s* p) {
    if (p->ws_S) return MITA_OK;
    const mita::Shape& s = p->s;
    int rc = alloc_region(p, &p->ws_S, (size_t)s.BH() * s.m * s.N * 4);
    if (rc == MITA_OK) p->S = (float*)p->ws_S;
    return rc;
}

int ensure_tiled(mita_plan_s* p) {
    if (p->ws_tiled || !mita::tiled_supported(p->s, p->dtype)) return MITA_OK;
    int rc = ensure_scores(p);
    if (rc != MITA_OK) return rc;
    const mita::Shape& s = p->s;
    const size_t BH = (size_t)s.BH();
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t o = off; off = align_up(off + bytes, 256); return o; };
    const size_t oRowmax = take(2 * BH * s.m * 4);   // row max, then row min
    const size_t oVpart = take(mita::tiled_part_bytes(s));
    const size_t oCursor = take(BH * s.m * 4);
    const size_t oTiles = take(BH * (size_t)mita::tiled_max_tiles(s) * 8);   // int2 per tile
    const size_t oNtiles = take(BH * 4);
    if ((rc = alloc_region(p, &p->ws_tiled, off)) != MITA_OK) return rc;
    char* b = (char*)p->ws_tiled;
    p->rowmax = (uint32_t*)(b + oRowmax);
    p->vpart = (float*)(b + oVpart);
    p->cursor = (int32_t*)(b + oCursor);
    p->tiles = (int32_t*)(b + oTiles);
    p->ntiles = (int32_t*)(b + oNtiles);
    return MITA_OK;
}

int ensure_grad(mita_plan_s* p) {
    if (p->ws_grad) return MITA_OK;
    int rc = ensure_scores(p);
    if (rc != MITA_OK) return rc;
    const mita::Shape& s = p->s;
    const size_t BH = (size_t)s.BH();
    // dQ_l, dV_l, V_l in fp32 [BH, m, d] each, then per landmark row {max S, sum of weights}
    if ((rc = alloc_region(p, &p->ws_grad, (3 * BH * s.m * s.d + 2 * BH * s.m) * 4)) != MITA_OK) return rc;
    p->dQl = (float*)p->ws_grad;
    p->dVl = p->dQl + BH * s.m * s.d;
    return MITA_OK;
}

// Regions for the path the plan currently resolves to.
int ensure_path(mita_plan_s* p) {
    const int path = resolve_path(p);
    if (path == MITA_PATH_STAGED) return ensure_scores(p);
    if (path == MITA_PATH_TILED) return ensure_tiled(p);
    return MITA_OK;
}

// ---------------------------------------------------------------- host forward
// mita_forward_host streams the heads through the device in kHostChunks
// chunks, two staging slots deep.
constexpr int kHostChunks = 8;

size_t io_size(const mita_plan_s* p) { return p->dtype == MITA_BF16 ? 2 : 4; }

// Byte offsets of one staging slot: Q, K, V and out of `hc` heads, then
// their experts and routes, then (tiled-capable shapes) value partials sized
// for the larger of the two chunk shapes a call uses.
struct HostSlot {
    size_t q, k, v, o, idx, route, part, bytes;
};

mita::Shape chunk_shape(const mita::Shape& s, int heads) {
    mita::Shape c = s;
    c.B = 1;
    c.H = heads;
    return c;
}

HostSlot host_slot(const mita_plan_s* p, int hc) {
    const mita::Shape& s = p->s;
    HostSlot L{};
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t o = off; off = align_up(off + bytes, 256); return o; };
    const size_t act = (size_t)hc * s.N * s.d * io_size(p);
    L.q = take(act);
    L.k = take(act);
    L.v = take(act);
    L.o = take(act);
    L.idx = take((size_t)hc * s.m * s.k * 4);
    L.route = take((size_t)hc * s.N * 4);
    size_t part = 0;
    if (mita::tiled_supported(s, p->dtype)) {
        const int BH = s.BH(), last = BH - (BH - 1) / hc * hc;
        part = std::max(mita::tiled_part_bytes(chunk_shape(s, hc)), mita::tiled_part_bytes(chunk_shape(s, last)));
    }
    L.part = take(part);
    L.bytes = off;
    return L;
}

// The copy streams and events on the plan's device, then the two staging
// slots (one allocation), on the first mita_forward_host() call.
int ensure_host(mita_plan_s* p) {
    if (p->ws_host) return MITA_OK;
    if (!p->ev_out[1]) {
        int prev = 0;
        cudaGetDevice(&prev);
        cudaSetDevice(p->device);
        bool ok = (p->h2d || cudaStreamCreateWithFlags(&p->h2d, cudaStreamNonBlocking) == cudaSuccess) &&
                  (p->d2h || cudaStreamCreateWithFlags(&p->d2h, cudaStreamNonBlocking) == cudaSuccess);
        cudaEvent_t* evs[7] = {&p->ev_start, &p->ev_in[0], &p->ev_in[1], &p->ev_comp[0],
                               &p->ev_comp[1], &p->ev_out[0], &p->ev_out[1]};
        for (int i = 0; ok && i < 7; ++i)
            ok = *evs[i] || cudaEventCreateWithFlags(evs[i], cudaEventDisableTiming) == cudaSuccess;
        cudaSetDevice(prev);
        if (!ok) {
            cudaGetLastError();
            return MITA_ERR_CUDA;
        }
    }
    const int BH = p->s.BH();
    p->host_heads = (BH + kHostChunks - 1) / kHostChunks;
    p->host_slot_bytes = host_slot(p, p->host_heads).bytes;
    return alloc_region(p, &p->ws_host, 2 * p->host_slot_bytes);
}

void free_plan(mita_plan_s* p) {
    int prev = 0;
    cudaGetDevice(&prev);
    cudaSetDevice(p->device);
    cudaDeviceSynchronize();
    if (p->ws) cudaFree(p->ws);
    if (p->ws_S) cudaFree(p->ws_S);
    if (p->ws_tiled) cudaFree(p->ws_tiled);
    if (p->ws_grad) cudaFree(p->ws_grad);
    if (p->ws_host) cudaFree(p->ws_host);
    if (p->done) cudaEventDestroy(p->done);
    if (p->aux) cudaStreamDestroy(p->aux);
    if (p->h2d) cudaStreamDestroy(p->h2d);
    if (p->d2h) cudaStreamDestroy(p->d2h);
    cudaEvent_t evs[7] = {p->ev_start, p->ev_in[0], p->ev_in[1], p->ev_comp[0], p->ev_comp[1], p->ev_out[0],
                          p->ev_out[1]};
    for (cudaEvent_t e : evs)
        if (e) cudaEventDestroy(e);
    cudaSetDevice(prev);
    free(p);
}

// Remember the stream's last launch for mita_get_status(); a launch captured
// into a graph completes only when the graph runs, so then the status waits
// for the whole device instead.
void note_launch(mita_plan_s* p, cudaStream_t st) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cap) != cudaSuccess) {
        cudaGetLastError();
        p->done_valid = 0;
        return;
    }
    if (cap != cudaStreamCaptureStatusNone) {
        p->done_valid = 0;
        return;
    }
    p->done_valid = cudaEventRecord(p->done, st) == cudaSuccess;
    if (!p->done_valid) cudaGetLastError();
}

// The path a forward takes, or -status when the plan cannot run it.
int forward_path(const mita_plan_s* p) {
    const int path = resolve_path(p);
    if (path != MITA_PATH_STAGED && p->routes_s > 1) return -MITA_ERR_UNSUPPORTED;
    if (path == MITA_PATH_FUSED && !mita::fused_supported(p->s, p->dtype)) return -MITA_ERR_UNSUPPORTED;
    if (path == MITA_PATH_TILED && !p->rowmax) return -MITA_ERR_UNSUPPORTED;
    if (path == MITA_PATH_STAGED && !p->S) return -MITA_ERR_UNSUPPORTED;
    return path;
}

// Enqueue the forward of plan p's heads on `path` (device pointers).
cudaError_t run_path(mita_plan_s* p, int path, const void* Q, const void* K, const void* V, void* out, int32_t* idx,
                     int32_t* rt, cudaStream_t st) {
    if (path == MITA_PATH_FUSED) return mita::run_fused(p, Q, K, V, out, idx, rt, p->keep_landmarks, st);
    if (path == MITA_PATH_TILED) return mita::run_tiled(p, Q, K, V, out, idx, rt, st);
    return mita::run_staged(p, Q, K, V, out, idx, rt, st);
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
    const size_t oIdx = take(BH * m * (size_t)k * 4), oRoute = take(BH * (size_t)N * 4);
    const size_t oCnt = take(BH * m * 4), oOff = take(BH * (m + 1) * 4), oPerm = take(BH * (size_t)N * 4);
    const size_t oStatus = take(256);

    if (alloc_region(p, &p->ws, off) != MITA_OK) {
        free(p);
        return MITA_ERR_OOM;
    }
    char* b = (char*)p->ws;
    p->Ql = b + oQl;
    p->Vl = b + oVl;
    p->idx = (int32_t*)(b + oIdx);
    p->route = (int32_t*)(b + oRoute);
    p->counts = (int32_t*)(b + oCnt);
    p->offsets = (int32_t*)(b + oOff);
    p->perm = (int32_t*)(b + oPerm);
    p->status = (int32_t*)(b + oStatus);
    if (cudaEventCreateWithFlags(&p->done, cudaEventDisableTiming) != cudaSuccess ||
        cudaStreamCreateWithFlags(&p->aux, cudaStreamNonBlocking) != cudaSuccess ||
        cudaMemset(p->status, 0, 256) != cudaSuccess) {
        cudaGetLastError();
        free_plan(p);
        return MITA_ERR_CUDA;
    }
    const int rc = ensure_path(p);
    if (rc != MITA_OK) {
        free_plan(p);
        return rc;
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
        return ensure_path(p);
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
        return ensure_path(p);
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
    const int path = forward_path(p);
    if (path < 0) return -path;
    if (run_path(p, path, Q, K, V, out, idx, rt, st) != cudaSuccess) return MITA_ERR_CUDA;
    note_launch(p, st);
    p->landmarks_valid = p->keep_landmarks || path != MITA_PATH_FUSED;
    return MITA_OK;
}

int mita_forward_host(mita_plan_t p, const void* Q, const void* K, const void* V, void* out, int32_t* expert_idx,
                      int32_t* route, struct CUstream_st* stream) {
    if (!p || !Q || !K || !V || !out) return MITA_ERR_INVALID_ARG;
    const int path = forward_path(p);
    if (path < 0) return -path;
    int rc = ensure_host(p);
    if (rc != MITA_OK) return rc;
    const mita::Shape& s = p->s;
    const size_t e = io_size(p);
    const int BH = s.BH(), hc = p->host_heads, nc = (BH + hc - 1) / hc;
    const HostSlot L = host_slot(p, hc);
    cudaStream_t st = (cudaStream_t)stream;
    // the copies in wait for the caller's stream position at this call (and
    // so for the previous call's last copy out); chunk c reuses the slot of
    // chunk c - 2 once that chunk's results have left it
#define MITA_CK(x)                              \
    do {                                        \
        if ((x) != cudaSuccess) {               \
            cudaGetLastError();                 \
            return MITA_ERR_CUDA;               \
        }                                       \
    } while (0)
    MITA_CK(cudaEventRecord(p->ev_start, st));
    MITA_CK(cudaStreamWaitEvent(p->h2d, p->ev_start, 0));
    MITA_CK(cudaStreamWaitEvent(p->d2h, p->ev_start, 0));
    mita_plan_s sub = *p;
    for (int c = 0; c < nc; ++c) {
        const int slot = c & 1, h0 = c * hc, nh = std::min(hc, BH - h0);
        char* base = (char*)p->ws_host + slot * p->host_slot_bytes;
        const size_t act = (size_t)nh * s.N * s.d * e, aoff = (size_t)h0 * s.N * s.d * e;
        const size_t ib = (size_t)nh * s.m * s.k * 4, ioff = (size_t)h0 * s.m * s.k * 4;
        const size_t rb = (size_t)nh * s.N * 4, roff = (size_t)h0 * s.N * 4;
        if (c >= 2) MITA_CK(cudaStreamWaitEvent(p->h2d, p->ev_out[slot], 0));
        MITA_CK(cudaMemcpyAsync(base + L.q, (const char*)Q + aoff, act, cudaMemcpyHostToDevice, p->h2d));
        MITA_CK(cudaMemcpyAsync(base + L.k, (const char*)K + aoff, act, cudaMemcpyHostToDevice, p->h2d));
        MITA_CK(cudaMemcpyAsync(base + L.v, (const char*)V + aoff, act, cudaMemcpyHostToDevice, p->h2d));
        MITA_CK(cudaEventRecord(p->ev_in[slot], p->h2d));
        MITA_CK(cudaStreamWaitEvent(st, p->ev_in[slot], 0));
        // the chunk as a plan of its own over the same workspace: landmarks
        // at the chunk's place, value partials in the slot
        sub.s = chunk_shape(s, nh);
        sub.Ql = (char*)p->Ql + (size_t)h0 * s.m * s.d * e;
        sub.Vl = (char*)p->Vl + (size_t)h0 * s.m * s.d * e;
        if (L.part) sub.vpart = (float*)(base + L.part);
        sub.launches = 0;
        const cudaError_t err = run_path(&sub, path, base + L.q, base + L.k, base + L.v, base + L.o,
                                         (int32_t*)(base + L.idx), (int32_t*)(base + L.route), st);
        p->launches += sub.launches;
        MITA_CK(err);
        MITA_CK(cudaEventRecord(p->ev_comp[slot], st));
        MITA_CK(cudaStreamWaitEvent(p->d2h, p->ev_comp[slot], 0));
        MITA_CK(cudaMemcpyAsync((char*)out + aoff, base + L.o, act, cudaMemcpyDeviceToHost, p->d2h));
        if (expert_idx)
            MITA_CK(cudaMemcpyAsync((char*)expert_idx + ioff, base + L.idx, ib, cudaMemcpyDeviceToHost, p->d2h));
        if (route) MITA_CK(cudaMemcpyAsync((char*)route + roff, base + L.route, rb, cudaMemcpyDeviceToHost, p->d2h));
        MITA_CK(cudaEventRecord(p->ev_out[slot], p->d2h));
    }
    // the copies out run in order: the last one's event covers them all
    MITA_CK(cudaStreamWaitEvent(st, p->ev_out[(nc - 1) & 1], 0));
#undef MITA_CK
    note_launch(p, st);
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
    int rc = ensure_grad(p);
    // the tiled path's row keys let the backward recompute the forward's
    // scores and routes with its kernels
    if (rc == MITA_OK) rc = ensure_tiled(p);
    if (rc != MITA_OK) return rc;
    if (mita::run_backward(p, Q, K, V, dOut, dQ, dK, dV, (cudaStream_t)stream) != cudaSuccess) return MITA_ERR_CUDA;
    note_launch(p, (cudaStream_t)stream);
    return MITA_OK;
}

int mita_get_status(mita_plan_t p) {
    if (!p) return MITA_ERR_INVALID_ARG;
    int prev = 0;
    cudaGetDevice(&prev);
    cudaSetDevice(p->device);
    int32_t st = 0;
    int rc = MITA_OK;
    // wait for the plan's last launch only (the whole device after a
    // captured one), then read and clear the status word on the plan's own
    // non-blocking stream, which waits for no other stream
    const cudaError_t w = p->done_valid ? cudaEventSynchronize(p->done) : cudaDeviceSynchronize();
    if (w != cudaSuccess) rc = MITA_ERR_CUDA;
    else if (cudaMemcpyAsync(&st, p->status, 4, cudaMemcpyDeviceToHost, p->aux) != cudaSuccess ||
             cudaMemsetAsync(p->status, 0, 4, p->aux) != cudaSuccess || cudaStreamSynchronize(p->aux) != cudaSuccess)
        rc = MITA_ERR_CUDA;
    else
        rc = st;
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
    free_plan(p);
}

}  // extern "C"
