/*
 * moe.h -- C ABI of the routed Mixture-of-Experts layer for one GB300 (sm_103a).
 *
 * The layer (four stages):
 *   1. softmax top-k router: fp32 softmax over E expert logits, top-k with the
 *      lowest index winning a tie, weights renormalised over the k picks
 *      [vllm.cpp PR #481 "gate(#378): the first DEVICE run of the warp MoE
 *      router", warp-router commit; daScript PR #3988 "dasLLAMA vulkan: a MoE
 *      that fits the card ...", routed-block commit: TopKRows];
 *   2. token-to-expert dispatch: per-expert histogram, exclusive scan, stable
 *      permutation [daScript PR #3988, routed-block commit: MoeSched];
 *   3. grouped SwiGLU expert MLP over int4 offset-binary weights (value =
 *      nibble - 8) with one fp16 scale per 32 K-columns: gate+up, silu(gate)*up,
 *      down [colibri PR #418 "Vulkan backend: expert tier + dense + MLA
 *      attention on any Vulkan 1.2 GPU", Summary, Correctness and "Grouped
 *      scales in the Vulkan kernels"]; or over MXFP4 weights (e2m1 codes, one
 *      ue8m0 scale per 32 K-columns, the same PR's fmt=7), per expert set;
 *   4. weighted combine onto the residual plus an optional shared expert scaled
 *      by sigmoid(x . g) [daScript PR #3988, decode span commit: DecCombineSh;
 *      the combine-folded residual commit: shared row, then the slots in
 *      order, then the residual].
 *
 * Conventions for every entry point
 *   - Pointers to tensors are DEVICE pointers, owned by the caller; the library
 *     never frees or retains them.  Struct pointers (moe_experts, moe_shared)
 *     and `status` out-parameters are HOST pointers, read/written during the
 *     call only.
 *   - bf16 and fp16 tensors are passed as uint16_t bit patterns.  Tensors are
 *     dense row-major with the shapes stated per argument.
 *   - `stream` is a cudaStream_t passed as an opaque pointer (NULL = the legacy
 *     default stream).  Every call only enqueues work on `stream`, returns
 *     without synchronising, and allocates no device memory: scratch comes from
 *     the caller's workspace `ws` of at least the size the matching
 *     *_workspace_size() function returns (256-byte aligned).
 *   - Arguments are validated on the host before any launch; a failed check
 *     returns MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED and enqueues nothing.
 *     A launch failure returns MOE_ERR_CUDA.  No C++ exception crosses the ABI.
 *   - Faults found on the device (a routed id outside [0, E), a bounded wait
 *     that ran out) are recorded in a status word inside the workspace and the
 *     kernel skips the affected work; moe_device_status() reads and clears it.
 *   - There is no CPU fallback: without a usable sm_103a device every call that
 *     would launch returns MOE_ERR_CUDA.
 *
 * Weight layout ("CPU byte layout", uploaded with a plain copy, colibri #418):
 *   moe_q4.q  uint8  [n_mat][rows][K/2]: column c of a row is nibble (c & 1) of
 *             byte c/2 (low nibble = even column); value = nibble - 8
 *   moe_q4.s  fp16   [n_mat][rows][K/32]: scale of columns 32g .. 32g+31
 *   routed experts (n_mat = E): gate, up: rows = I, K = H; down: rows = H, K = I
 *   shared expert  (n_mat = 1): gate, up: rows = I_sh, K = H; down: rows = H, K = I_sh
 * MXFP4 weights (fmt = MOE_WFMT_MXFP4; colibri #418, the fmt=7 note of its Kimi K3 tier: e2m1
 * codes through a table, one ue8m0 scale per 32 inputs, the exponents expanded at upload):
 *   moe_q4.q  the same layout; each nibble is an e2m1 code (OCP Microscaling formats: sign bit
 *             3, exponent bits 2..1 with bias 1, mantissa bit 0), uploaded as stored
 *   moe_q4.s  fp16 [n_mat][rows][K/32] = 2^(e - 128) for the group's ue8m0 exponent e, as
 *             written by moe_mxfp4_scales(): half the MX scale, because the kernels read an
 *             e2m1 code as the integer 2v (v the code's value), exactly
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

typedef void* moe_stream_t; /* a cudaStream_t */

enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = -1,     /* null pointer, size out of range, workspace too small */
    MOE_ERR_UNSUPPORTED = -2,     /* valid request the library does not serve */
    MOE_ERR_CUDA = -3,            /* a CUDA call or launch failed (no device, bad stream, ...) */
    MOE_ERR_DEVICE_TIMEOUT = -4,  /* a bounded device-side wait ran out (recorded on device) */
    MOE_ERR_DEVICE_INDEX = -5,    /* a routed expert id outside [0, E) (recorded on device) */
    MOE_ERR_DEVICE_RANGE = -6     /* an MXFP4 scale exponent outside [104, 140] (recorded on device) */
};

enum {
    MOE_WFMT_INT4 = 0,   /* offset-binary int4 (nibble - 8), fp16 scale per 32 columns */
    MOE_WFMT_MXFP4 = 1   /* e2m1 codes, expanded ue8m0 scale per 32 columns (moe_mxfp4_scales) */
};

enum {
    MOE_ARM_AUTO = 0,  /* GEMV while T * k <= MOE_AUTO_GEMV_ROWS_PER_EXPERT * E and, with a shared
                          expert, T <= MOE_AUTO_GEMV_MAX_T_SHARED; grouped GEMM otherwise */
    MOE_ARM_GEMV = 1,  /* bandwidth arm: fused int4 GEMV, weights streamed once per call */
    MOE_ARM_GEMM = 2   /* tensor arm: grouped GEMM on tcgen05 / TMEM */
};

/* Size limits checked on the host. */
#define MOE_MAX_E 256
#define MOE_MAX_K 32
/* Arm choice of MOE_ARM_AUTO, from a sweep of both arms over T on one GB300 (the GEMV arm
 * streams each routed expert's weights once per pass of up to 4 of its tokens, and the shared
 * expert's once per 4 tokens of the batch; the GEMM arm costs a latency floor of ~200 us). */
#define MOE_AUTO_GEMV_ROWS_PER_EXPERT 4
#define MOE_AUTO_GEMV_MAX_T_SHARED 16
#define MOE_MAX_H 24576

typedef struct {
    const uint8_t* q;   /* device, uint8 [n_mat][rows][K/2] */
    const uint16_t* s;  /* device, fp16  [n_mat][rows][K/32] */
} moe_q4;

typedef struct {
    int E, H, I;        /* 1 <= E <= 256; H, I positive multiples of 32; H <= 24576 */
    moe_q4 gate, up, down;
    int fmt;            /* MOE_WFMT_INT4 (0) or MOE_WFMT_MXFP4 (1), all three matrices alike */
} moe_experts;

typedef struct {
    int I_sh;           /* positive multiple of 32 */
    moe_q4 gate, up, down;
    const uint16_t* g;  /* device, bf16 [H] gate vector; NULL = ungated (weight 1) */
    int fmt;            /* MOE_WFMT_*, independent of the routed experts' format */
} moe_shared;

/* Upload step of MXFP4 weights: expands n ue8m0 exponents e8 (device, uint8) into the fp16
 * scales the kernels read, s[i] = 2^(e8[i] - 128) (device, fp16 [n], 2-byte aligned; written
 * for every i).  Exponents in [104, 140] give exact products with every e2m1 code in fp16;
 * an exponent outside that range (255, the MX NaN, included) writes 0 and records
 * MOE_ERR_DEVICE_RANGE in the status word of the workspace ws (at least 4096 bytes, from
 * moe_workspace_init or zeroed), which moe_device_status() reads.  Asynchronous on stream.
 * Returns MOE_ERR_INVALID_ARG for null pointers or a short workspace. */
MOE_API int moe_mxfp4_scales(const uint8_t* e8, size_t n, uint16_t* s, void* ws, size_t ws_bytes,
                             moe_stream_t stream);

/* Text of a status code (static storage). */
MOE_API const char* moe_status_string(int status);

/* Library version string, e.g. "moe-gb300 0.1 sm_103a". */
MOE_API const char* moe_version(void);

/* Router logits (stage 1, its GEMV/GEMM: one dot product per expert row and,
 * when g != NULL, the shared-expert gate as one extra row whose logit is stored
 * after the E router logits, daScript PR #3988 decode span commit).
 *   x       bf16 [T][H]        W_r bf16 [E][H]        g bf16 [H] or NULL
 *   logits  fp32 [T][E + (g != NULL)], fp32 accumulation of bf16 products.
 * T <= 32 runs a GEMV; larger T runs a tcgen05 GEMM when H % 64 == 0,
 * E <= 256 and x, W_r, g are 16-byte aligned (else a tiled fp32 GEMM).  The
 * tensor-core kernel's bounded waits cannot report a timeout through this call
 * (it has no workspace status word).
 * T = 0 is a no-op. */
MOE_API int moe_router_logits(const uint16_t* x, const uint16_t* W_r, const uint16_t* g,
                      int T, int H, int E, float* logits, moe_stream_t stream);

/* Softmax top-k router (stage 1; one warp per token, the logit row held in
 * registers, one read of the row: vllm.cpp PR #481).
 *   logits     fp32 (logits_is_bf16 = 0) or bf16 (= 1) [T][ld], ld >= E; only
 *              the first E entries of a row are read
 *   topk_ids   int32 [T][k]: the k experts with the largest logits, ties broken
 *              towards the lower index, written in ascending expert id
 *   topk_w     fp32  [T][k]: softmax(row)[id] / sum of softmax over the k picks
 * A NaN logit is treated as -inf for selection.  1 <= k <= min(E, 32),
 * E <= 256. */
MOE_API int moe_router_topk(const void* logits, int logits_is_bf16, int ld, int T, int E,
                    int k, int32_t* topk_ids, float* topk_w, moe_stream_t stream);

/* Router variants (daScript PR #3988, routed block commit: among the router shapes the pages
 * name are a router or selection bias and renormalised, scaled weights).  The picks are the k
 * largest of logits[t][e] + sel_bias[e] (lowest index on a tie, NaN never picked), written in
 * ascending expert id; the weights come from the unbiased logits:
 *   p = softmax(logits[t]) over all E;  topk_w = (renormalize ? p[id] / sum of p over the picks
 *   : p[id]) * scale.
 *   sel_bias  device fp32 [E], 4-byte aligned, or NULL (no bias)
 *   scale     finite (else MOE_ERR_INVALID_ARG)
 * Other arguments and limits as moe_router_topk; sel_bias = NULL, renormalize = 1, scale = 1
 * is moe_router_topk. */
MOE_API int moe_router_topk_v(const void* logits, int logits_is_bf16, int ld, int T, int E, int k,
                              const float* sel_bias, int renormalize, float scale, int32_t* topk_ids,
                              float* topk_w, moe_stream_t stream);

/* Dispatch (stage 2): atomic-free per-expert histogram, exclusive scan and a
 * stable permutation of the T*k slots a = t*k + j.
 *   counts   int32 [E] or NULL     offsets int32 [E+1] (offsets[E] = T*k)
 *   perm     int32 [T*k]: bucket by bucket (ascending expert), the slots in
 *            ascending order;  inv int32 [T*k]: inv[perm[r]] = r
 * An id outside [0, E) sets MOE_ERR_DEVICE_INDEX in the workspace status word
 * and is left out of every bucket. */
MOE_API size_t moe_dispatch_workspace_size(int T, int k, int E);
MOE_API int moe_dispatch(const int32_t* topk_ids, int T, int k, int E, int32_t* counts,
                 int32_t* offsets, int32_t* perm, int32_t* inv, void* ws,
                 size_t ws_bytes, moe_stream_t stream);

/* moe_dispatch without a workspace (the pages have no counterpart: this entry point
 * exists for callers, not for the method).  Some callers cannot allocate device memory
 * when they dispatch: a host framework whose device memory pool is fixed at start-up, a
 * serving runtime's plugin callback that is not allowed to allocate, or a latency-bound
 * loop that cannot afford the device synchronisation an allocation implies.  This variant
 * runs the same kernels as moe_dispatch with their scratch in one array compiled into the
 * library (about 66 KiB, held on every GPU that loads the library until the process
 * exits), and allocates nothing.
 *   Arguments and outputs are those of moe_dispatch; T*k must not exceed
 *   MOE_DISPATCH_STATIC_MAX_SLOTS (else MOE_ERR_INVALID_ARG, nothing enqueued).
 *   A call looks up the array's device address on the current device (again on every call
 *   whose stream is not being captured, so a device reset does not leave a stale address);
 *   make the first call on a device before any stream capture.
 *   Every call on a device shares the one array and each call clears its status word first:
 *   calls that overlap on the GPU (other streams, other host threads) race and must be
 *   serialised by the caller.  An id outside [0, E) is left out of every bucket (its inv
 *   entry is -1); there is no status word to read back. */
#define MOE_DISPATCH_STATIC_MAX_SLOTS (1 << 20)
MOE_API int moe_dispatch_static(const int32_t* topk_ids, int T, int k, int E, int32_t* counts,
                                int32_t* offsets, int32_t* perm, int32_t* inv, moe_stream_t stream);

/* Expert MLP (stage 3) for every dispatched row, unweighted:
 *   rows fp32 [T*k][H]: rows[r] = W_d[e] (silu(W_g[e] x_t) * (W_u[e] x_t)) with
 *   a = perm[r], t = a / k, e the bucket holding r (offsets[e] <= r < offsets[e+1]).
 *   x bf16 [T][H], rows: 16-byte aligned (else MOE_ERR_INVALID_ARG);
 *   offsets/perm as produced by moe_dispatch.
 *   arm: MOE_ARM_* (which kernels compute it). */
MOE_API size_t moe_expert_mlp_workspace_size(int T, int k, int E, int H, int I);
MOE_API int moe_expert_mlp(const uint16_t* x, int T, int k, const moe_experts* W,
                   const int32_t* offsets, const int32_t* perm, float* rows,
                   int arm, void* ws, size_t ws_bytes, moe_stream_t stream);

/* Combine (stage 4): y[t] = shared[t] + sum_j topk_w[t][j] * rows[inv[t*k+j]]
 * + residual[t], summed in that order (shared row, slots by j, residual).
 *   rows fp32 [T*k][H] (dispatch order)   inv int32 [T*k]   topk_w fp32 [T][k]
 *   shared fp32 [T][H] or NULL (already gated)   residual bf16 [T][H] or NULL
 *   y fp32 [T][H] */
MOE_API int moe_combine(const float* rows, const int32_t* inv, const float* topk_w,
                const float* shared, const uint16_t* residual, int T, int k, int H,
                float* y, moe_stream_t stream);

/* The whole layer: logits (with the shared gate row), top-k, dispatch, expert
 * MLP with the combine fused into the down projection, shared expert.
 *   x bf16 [T][H]; residual bf16 [T][H] or NULL; W_r bf16 [E][H];
 *   sh: shared expert or NULL; y fp32 [T][H];
 *   topk_ids_out int32 [T][k] / topk_w_out fp32 [T][k]: optional copies.
 * T = 0 is a no-op. */
MOE_API size_t moe_workspace_size(int T, int E, int k, int H, int I, int I_sh);
MOE_API int moe_layer_forward(const uint16_t* x, const uint16_t* residual, const uint16_t* W_r,
                      const moe_experts* W, const moe_shared* sh, int T, int k,
                      float* y, int32_t* topk_ids_out, float* topk_w_out, int arm,
                      void* ws, size_t ws_bytes, moe_stream_t stream);

/* RMSNorm of the layer output for the next layer (daScript PR #3988, combine-folded residual
 * commit: after the routed block the residual row is normed for the next layer; the combine
 * above already adds the residual, so this is the norm step):
 *   y_norm[t][h] = bf16(y[t][h] / sqrt(mean_h y[t][h]^2 + eps) * gamma[h])
 *   y fp32 [T][H] (16-byte aligned), gamma bf16 [H], y_norm bf16 [T][H] (both 8-byte aligned);
 *   H a multiple of 32, eps >= 0 and finite (else MOE_ERR_INVALID_ARG).  The sum of squares is
 *   fp32 in a fixed order; the output is rounded to nearest even. */
MOE_API int moe_rmsnorm(const float* y, const uint16_t* gamma, int T, int H, float eps, uint16_t* y_norm,
                        moe_stream_t stream);

/* moe_layer_forward with the RMSNorm of its y: y receives the layer output, y_norm its RMSNorm
 * with norm_gamma bf16 [H] and eps, bit-identical to moe_rmsnorm on that y.  The tensor arm's
 * combine norms each row as it writes it (no extra launch, no second pass over y in HBM); the GEMV arm,
 * whose combine is folded into the down projection, runs the norm as one more launch on the
 * same stream. */
MOE_API int moe_layer_forward_norm(const uint16_t* x, const uint16_t* residual, const uint16_t* W_r,
                                   const moe_experts* W, const moe_shared* sh, int T, int k, float* y,
                                   const uint16_t* norm_gamma, float eps, uint16_t* y_norm,
                                   int32_t* topk_ids_out, float* topk_w_out, int arm, void* ws,
                                   size_t ws_bytes, moe_stream_t stream);

/* Clears the head of a workspace (its first 4096 bytes: the device status word, the GEMV
 * arm's task claim counters, the decode routing's completion count, the down projection's
 * column counters and the test hook below) on `stream`.  A workspace must start with a zero
 * head: call this once on a new workspace, or allocate it zero-filled.  The calls above leave
 * the head zero again (except a recorded status); after a call that recorded
 * MOE_ERR_DEVICE_TIMEOUT the counters may not be zero, so call this again before reusing the
 * workspace. */
MOE_API int moe_workspace_init(void* ws, size_t ws_bytes, moe_stream_t stream);

/* Test support for the bounded device waits (a device-side wait gives up, records a status
 * and lets its kernel return instead of hanging the GPU).  Sets the workspace's
 * test hook on `stream`: the next calls that run the tensor arm's gate/up kernel with this
 * workspace use wait_limit_cycles (> 0; 0 keeps the default of about two seconds) as the
 * limit of its waits, and its first CTA withholds the token-tile copy of its second K-step,
 * so that its MMA thread's wait runs out: that CTA records MOE_ERR_DEVICE_TIMEOUT in the
 * status word, every role of it stops, it waits (bounded) for its own copies and MMAs, frees
 * its tensor memory and returns; the rest of the call runs to completion with that CTA's
 * share of the output unspecified.  moe_workspace_init clears the hook.  Returns
 * MOE_ERR_INVALID_ARG for a null, short or misaligned workspace or a negative limit. */
MOE_API int moe_workspace_test_timeout(void* ws, size_t ws_bytes, long long wait_limit_cycles,
                                       moe_stream_t stream);

/* Synchronises `stream`, copies the device status word of a workspace used by
 * the calls above into *status (MOE_OK or a MOE_ERR_DEVICE_* code) and clears
 * it.  Returns MOE_OK, or MOE_ERR_CUDA / MOE_ERR_INVALID_ARG. */
MOE_API int moe_device_status(void* ws, size_t ws_bytes, int* status, moe_stream_t stream);

/* Measurement support (not part of the layer).
 * moe_launch_count: number of kernels this library has launched in the process.
 * moe_profile_enable(1): from now on every kernel launch is bracketed by a CUDA event pair on
 *   its stream (moe_profile_enable(0) stops; both reset the totals).
 * moe_profile_read: waits for the recorded events and returns, per kernel name, the summed
 *   device time in ms and the number of launches.  names receives up to max_n
 *   NUL-terminated names of name_len bytes each; *n receives the number of kernel names. */
MOE_API long long moe_launch_count(void);
MOE_API int moe_profile_enable(int on);
MOE_API int moe_profile_read(int max_n, char* names, int name_len, double* ms, long* launches, int* n);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
