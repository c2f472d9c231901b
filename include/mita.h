/*
 * mita.h -- C ABI of the B300 (sm_103a) Mixture-of-Top-k Attention forward
 * operator.
 *
 * The operator (36Kr / 新智元 "注意力也是FFN？从快权重出发，重新理解高效注意力",
 * section "用少量地标查询，同时构造全局概括与细节专家"; English version "Is
 * Attention Also FFN? ...", section "Construct global generalization and
 * detail experts at the same time with a small number of landmark queries"),
 * per (batch, head), with Q, K, V of N tokens x d features:
 *   1. m landmark queries Q_l by local average pooling of Q over the token
 *      grid (adaptive bins [floor(i*G/P), ceil((i+1)*G/P)) per axis);
 *   2. landmark scores Q_l . K^T / sqrt(d)   (m x N);
 *   3. routed expert i = the k keys with the highest scores of landmark i
 *      (ties to the lower key index);
 *   4. landmark values V_l = softmax(scores) . V; (Q_l, V_l) is the shared
 *      expert of m key-value pairs;
 *   5. each query is routed (s = 1) to the landmark with the highest
 *      q . Q_l / sqrt(d) (ties to the lower landmark index);
 *   6. each query takes one softmax over the m shared pairs and the k raw
 *      key-value pairs of its routed expert.
 * The attention is non-causal and the scale is fixed at 1/sqrt(d).
 *
 * Precision contract: inputs and out are MITA_F32 or MITA_BF16.  All sums are
 * fp32.  Q_l is the correctly rounded mean in the I/O type; V_l is rounded
 * to the I/O type; out is rounded to nearest even.  Top-k and routing compare
 * the unscaled fp32 dot products; -0.0 compares equal to +0.0.
 *
 * Every function returns a mita_status_t (0 = MITA_OK) unless noted.  No
 * function synchronises the host with the device except mita_get_status()
 * and mita_destroy().
 */
#ifndef MITA_H
#define MITA_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;                       /* = cudaStream_t */
typedef struct mita_plan_s* mita_plan_t;

typedef enum { MITA_F32 = 0, MITA_BF16 = 1 } mita_dtype_t;

typedef enum {
    MITA_OK = 0,
    MITA_ERR_INVALID_ARG = 1,   /* bad size, null or misaligned pointer     */
    MITA_ERR_UNSUPPORTED = 2,   /* valid but outside the built kernels      */
    MITA_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed     */
    MITA_ERR_TIMEOUT = 4,       /* a bounded device wait ran out            */
    MITA_ERR_OOM = 5,           /* workspace allocation failed              */
    MITA_ERR_DEVICE = 6         /* a kernel flagged bad data (status word)  */
} mita_status_t;

/* Token grid and landmark grid.  2-D: gh x gw tokens in row-major order
 * pooled to ph x pw landmarks (landmark i = row * pw + col).  1-D sequence:
 * gh = ph = 1, gw = N, pw = m. */
typedef struct {
    int gh, gw;
    int ph, pw;
} mita_grid_t;

/* Create a plan for B x H heads of N tokens, head dim d, m landmarks and
 * top-k width k, with inputs of type dtype.
 * Requirements (else MITA_ERR_INVALID_ARG): B, H, N >= 1; gh*gw == N;
 * ph*pw == m; 1 <= ph <= gh; 1 <= pw <= gw; 1 <= k <= N; plan != NULL.
 * Supported (else MITA_ERR_UNSUPPORTED): d in {64, 128}; m <= 1024;
 * k <= 4096; m + k <= 4096; B*H*N*d < 2^40.
 * The plan owns a device workspace on the current device, freed by
 * mita_destroy().  mita_plan() allocates the part every path needs and the
 * part of the path the plan starts on (MITA_ERR_OOM if that fails); a path
 * chosen later by mita_set_option(), and the first mita_backward(), may add
 * one allocation each, so make those calls before any stream capture.
 * mita_forward() never allocates.  *plan is set to NULL on failure. */
int mita_plan(mita_plan_t* plan, int B, int H, int N, int d, mita_grid_t grid,
              int m, int k, mita_dtype_t dtype);

/* Run the forward operator asynchronously on `stream` (NULL = legacy default
 * stream).  Device pointers, all contiguous and 16-byte aligned:
 *   Q, K, V     [B, H, N, d] of the plan's dtype (read only);
 *   out         [B, H, N, d] of the plan's dtype (written);
 *   expert_idx  [B, H, m, k] int32, each expert's key indices in ascending
 *               order (written; may be NULL);
 *   route       [B, H, N] int32, the landmark each query is routed to
 *               (written; may be NULL).
 * The caller owns every buffer; out must not alias Q, K or V.  Calls on one
 * plan share its workspace: they must be ordered on one stream.  Returns
 * MITA_ERR_INVALID_ARG for a null/misaligned pointer and MITA_ERR_CUDA if a
 * launch fails; data errors found by kernels are reported by
 * mita_get_status(). */
int mita_forward(mita_plan_t plan, const void* Q, const void* K, const void* V, void* out,
                 int32_t* expert_idx, int32_t* route, struct CUstream_st* stream);

/* The forward of mita_forward() on tensors in HOST memory: Q, K, V, out,
 * expert_idx and route have the layouts and types of mita_forward() but
 * point to host memory (page-locked -- cudaMallocHost or cudaHostRegister --
 * for the copies to overlap; pageable memory gives the same results with the
 * copies serialised).  No alignment is required; expert_idx and route may be
 * NULL.  The heads go through the device in at most 8 chunks (B*H / 8
 * heads each, rounded up), each a run of consecutive heads: while chunk c is
 * copied to the device, chunk c - 1's
 * forward runs on `stream` and chunk c - 2's results are copied back, on two
 * copy streams the plan owns, so a call takes about as long as its larger
 * copy direction.  The kernels, and so the results, are those of
 * mita_forward() on the same path for a plan of the chunk's heads.
 * Ordering: the copies to the device start once `stream` reaches this call,
 * and `stream` passes the call's end only after the last result is in host
 * memory, so synchronising `stream` (or an event recorded on it after the
 * call) makes out, expert_idx and route readable; the host buffers must stay
 * valid and unwritten until then.  The first call on a plan allocates two
 * staging slots of device memory (each one chunk's Q, K, V, out, experts and
 * routes, plus the tiled path's value partials for a chunk: about a quarter
 * of Q, K, V and out together at 8 chunks; MITA_ERR_OOM if that fails) and
 * creates the copy streams and their events (MITA_ERR_CUDA): make it before
 * any stream capture.  Calls on one plan
 * share the slots: order them on one stream.  Returns MITA_ERR_INVALID_ARG
 * for a null Q, K, V or out, MITA_ERR_UNSUPPORTED where mita_forward()
 * would, MITA_ERR_CUDA if a copy or launch fails to enqueue; data errors are
 * reported by mita_get_status(), as for mita_forward(). */
int mita_forward_host(mita_plan_t plan, const void* Q, const void* K, const void* V, void* out,
                      int32_t* expert_idx, int32_t* route, struct CUstream_st* stream);

/* Wait for the plan's last mita_forward() / mita_backward() launch and
 * return the device status word of the plan's kernels since the last call
 * (MITA_OK or MITA_ERR_DEVICE / MITA_ERR_TIMEOUT), then clear it.  It waits
 * on that launch's stream position only (an event), not on the whole
 * device; after a launch captured into a CUDA graph it waits for the whole
 * device, and after a graph replay the caller synchronises first. */
int mita_get_status(mita_plan_t plan);

/* Free the workspace and the plan (NULL is a no-op).  Synchronises the
 * plan's device first. */
void mita_destroy(mita_plan_t plan);

/* Backward pass (routes s = 1; the routing-only option is honoured): given
 * the output gradient dOut ([B, H, N, d], plan dtype, device), writes the
 * input gradients dQ, dK, dV ([B, H, N, d], fp32, device, overwritten) on
 * `stream`.  The forward's discrete choices (experts and routes) are
 * recomputed from Q and K exactly as mita_forward makes them and held
 * constant; gradients flow through the output softmax, the landmark values
 * V_l = softmax(Q_l K^T / sqrt d) V and the bin means into Q; the roundings of
 * Q_l, V_l and out to the I/O type pass gradients unchanged (the reading of
 * 36Kr / 新智元 "注意力也是FFN？", which trains the operator end to end without
 * stating its gradients).  Runs the stage-by-stage kernels with fp32
 * atomics (sums in a nondeterministic order).  MITA_ERR_UNSUPPORTED when the
 * plan routes to s > 1 experts; MITA_ERR_INVALID_ARG for a null or
 * misaligned pointer.  The first call on a plan allocates the backward's
 * fp32 workspace (MITA_ERR_OOM if that fails): make it before capturing a
 * backward in a graph. */
int mita_backward(mita_plan_t plan, const void* Q, const void* K, const void* V, const void* dOut, float* dQ,
                  float* dK, float* dV, struct CUstream_st* stream);

/* Static string for a status code (never NULL). */
const char* mita_strerror(int code);

/* Plan options (set before mita_forward; return MITA_ERR_INVALID_ARG for an
 * unknown option or value):
 *   MITA_OPT_PATH            MITA_PATH_AUTO (default) picks the fastest
 *                            built path for the shape; MITA_PATH_STAGED
 *                            forces the stage-by-stage kernels;
 *                            MITA_PATH_FUSED forces the one-kernel path for
 *                            short sequences and MITA_PATH_TILED the
 *                            tensor-core kernel chain for long ones
 *                            (MITA_ERR_UNSUPPORTED at forward time if the
 *                            shape does not fit the forced path).
 *   MITA_OPT_KEEP_LANDMARKS  1: mita_forward also stores Q_l and V_l in the
 *                            workspace for mita_get_landmarks().
 *   MITA_OPT_ROUTING_ONLY    1: the routing-only variant (the ablation of
 *                            36Kr / 新智元 "注意力也是FFN？", section
 *                            "长序列建模：训练时间从10.6小时降至2.4小时"): the
 *                            shared expert is dropped and each query takes
 *                            one softmax over its routed expert's k keys
 *                            alone; landmarks, experts and routes are
 *                            unchanged.  0 (default): the m shared pairs
 *                            join every query's softmax.
 *   MITA_OPT_ROUTES          s, the experts per query (1 <= s <= min(m, 8);
 *                            default 1): each query is routed to its s best
 *                            landmarks (ties to the lower index) and takes
 *                            one softmax over the shared pairs and the union
 *                            of those experts' keys, each key once; route[]
 *                            holds the best landmark.  s > 1 runs on the
 *                            staged path (AUTO picks it; a forced fused or
 *                            tiled path gives MITA_ERR_UNSUPPORTED). */
typedef enum {
    MITA_OPT_PATH = 0,
    MITA_OPT_KEEP_LANDMARKS = 1,
    MITA_OPT_ROUTING_ONLY = 2,
    MITA_OPT_ROUTES = 3
} mita_option_t;
typedef enum { MITA_PATH_AUTO = 0, MITA_PATH_STAGED = 1, MITA_PATH_FUSED = 2, MITA_PATH_TILED = 3 } mita_path_t;
int mita_set_option(mita_plan_t plan, int option, int value);

/* Path the next mita_forward() will take (a mita_path_t value other than
 * AUTO), or a negative status on error: -MITA_ERR_UNSUPPORTED when a forced
 * path does not fit the plan's shape. */
int mita_get_path(mita_plan_t plan);

/* Copy the landmark queries Q_l and landmark values V_l of the last forward
 * ([B, H, m, d] each, plan dtype, device pointers) on `stream`.  Requires
 * MITA_OPT_KEEP_LANDMARKS = 1 before that forward (else
 * MITA_ERR_INVALID_ARG). */
int mita_get_landmarks(mita_plan_t plan, void* Ql, void* Vl, struct CUstream_st* stream);

/* Bytes of device workspace the plan holds. */
int mita_workspace_bytes(mita_plan_t plan, uint64_t* bytes);

/* Number of kernels this plan has launched since it was created (every
 * mita_forward adds the launches of the path it took). */
int mita_launch_count(mita_plan_t plan, uint64_t* launches);

/* ---------------------------------------------------------------------
 * Allocation-free forward.  The method description has no counterpart of
 * this entry point: it exists for callers that cannot call cudaMalloc --
 * code embedded in a host framework that owns all device memory through its
 * own pool and forbids raw device allocations, and latency-critical loops
 * in which an allocation would implicitly synchronise the device.  Such
 * callers cannot create a plan either, because mita_plan() allocates.
 *
 * mita_forward_noalloc() computes the same result as mita_forward() on the
 * stage-by-stage path, with the same arguments as mita_plan() followed by
 * those of mita_forward().  It allocates nothing: its scratch (landmark
 * queries and values, landmark scores, query buckets, a status word) lives
 * in one fixed device array of MITA_NOALLOC_SCRATCH_BYTES that the library
 * declares statically; every GPU that loads the library holds that array
 * until the process exits.  It calls no cudaMalloc, cudaFree or allocating
 * library routine.
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and caches it; make that first call before any
 *     stream capture.
 *   - A shape whose scratch does not fit (mita_noalloc_scratch_bytes())
 *     returns MITA_ERR_UNSUPPORTED; argument errors are those of mita_plan()
 *     and mita_forward().
 *   - Every call shares the one array, and a call leaves its contents
 *     behind.  Calls that overlap on the GPU (different streams, or
 *     different host threads, on one device) race on it: order them on one
 *     stream.
 *   - Kernel data checks have no plan to report to: a call returns only
 *     launch errors.
 */
#define MITA_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

int mita_forward_noalloc(int B, int H, int N, int d, mita_grid_t grid, int m, int k,
                         mita_dtype_t dtype, const void* Q, const void* K, const void* V, void* out,
                         int32_t* expert_idx, int32_t* route, struct CUstream_st* stream);

/* Size in bytes of the fixed scratch array used by mita_forward_noalloc(). */
uint64_t mita_noalloc_scratch_bytes(void);

#ifdef __cplusplus
}
#endif

#endif /* MITA_H */
