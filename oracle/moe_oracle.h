/*
 * moe_oracle.h -- plain fp64 CPU oracle of the routed Mixture-of-Experts layer.
 *
 * TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.  Only the tests, the smoke
 * check and the benchmark's CPU-baseline leg load this library.  It shares no
 * code, header, table or helper with the CUDA library, and nothing in the CUDA
 * library calls it.
 *
 * Sources (web pages; the method is stated there in prose, no code is given):
 *   [colibri #418]   "Vulkan backend: expert tier + dense + MLA attention on any
 *                    Vulkan 1.2 GPU" (colibri PR #418): int4 offset-binary
 *                    weights, grouped scales, the fused gate+up+silu->down group.
 *   [dasLLAMA #3988] "dasLLAMA vulkan: a MoE that fits the card serves on the
 *                    whole-model resident driver" (daScript PR #3988): router
 *                    GEMM/GEMV, per-row top-k, bucket schedule, sigmoid-gated
 *                    shared expert, combine order.
 *   [vllm.cpp #481]  "gate(#378): the first DEVICE run of the warp MoE router"
 *                    (vllm.cpp PR #481): softmax top-k router guards.
 *
 * Every function returns 0 on success or a negative code (-1 bad argument,
 * -2 non-finite input).  All outputs are caller-allocated host arrays.
 * Weight layout (expert-major, row-major, "CPU byte layout" of colibri #418):
 *   q[e][row][K/2]  uint8, column c in nibble (c & 1) of byte c/2 (low first)
 *   s[e][row][K/32] fp16 bits, one scale per 32 consecutive K-columns
 * gate/up: rows = I, K = H;  down: rows = H, K = I.
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

double mo_bf16_to_f64(uint16_t bits);
double mo_f16_to_f64(uint16_t bits);

/* Worker threads for independent rows (router logits per token, dispatched
 * expert rows, shared-expert tokens); default 1.  Every row is computed by the
 * same sequential loop whatever the count, so results are bit-identical. */
void mo_set_threads(int n);
int mo_get_threads(void);

/* Dequantise rows x K of one int4 matrix into w[rows][K] (fp64). */
int mo_dequant(const uint8_t* q, const uint16_t* s, int rows, int K, double* w);

/* MXFP4 weights (colibri PR #418, the fmt=7 note of its Kimi K3 Vulkan tier: e2m1 nibbles
 * decoded through a table, one ue8m0 scale per 32 inputs).  The element and scale encodings are
 * those of the OCP Microscaling (MX) formats: e2m1 has the sign in bit 3, a 2-bit exponent
 * (bits 2..1, bias 1) and a 1-bit mantissa (bit 0), exponent field 0 meaning the subnormal
 * value mantissa * 2^-1; ue8m0 is the power of two 2^(e - 127), e = 255 NaN.  Layout as for
 * int4 (nibble (c & 1) of byte c/2, low first; the pages do not state the nibble order, the
 * int4 layout's order is taken), exponents e8[row][K/32] one byte each. */
double mo_e2m1_to_f64(int nibble);
double mo_ue8m0_to_f64(uint8_t e);
int mo_dequant_mxfp4(const uint8_t* q, const uint8_t* e8, int rows, int K, double* w);

/* Weight formats of the _fmt functions below: the scale pointers are fp16 bits (uint16_t) for
 * MO_FMT_INT4 and ue8m0 exponents (uint8_t) for MO_FMT_MXFP4. */
#define MO_FMT_INT4 0
#define MO_FMT_MXFP4 1

/* logits[t][e] = sum_h x[t][h] * W_r[e][h] for e < E; when g != NULL also
 * logits[t][E] = sum_h x[t][h] * g[h] (the shared-expert gate row).  Row
 * stride of logits is E + (g != NULL). */
int mo_router_logits(const uint16_t* x, const uint16_t* W_r, const uint16_t* g,
                     int T, int H, int E, double* logits);

/* Softmax top-k with lowest-index tie-break and renormalised weights.
 * logits: T rows of stride ld (>= E); ids[t][j] ascending expert id;
 * w[t][j] = softmax(logits[t])[ids[t][j]] / sum over the k selected. */
int mo_router_topk(const double* logits, int ld, int T, int E, int k,
                   int32_t* ids, double* w);

/* Router variants (daScript PR #3988 "dasLLAMA vulkan: a MoE that fits the card ...", routed
 * block commit, which names a router or selection bias and renormalised, scaled weights among
 * the router shapes): selection over s_e = l_e + bias_e (bias NULL: 0), k rounds of argmax with
 * the lowest index keeping a tie, picks in ascending expert id; weights from the unbiased
 * logits: p = softmax(l) over all E, w_j = p[id_j] / sum over the picks of p when renormalize,
 * else p[id_j]; then times scale.  bias = NULL, renormalize = 1, scale = 1 is mo_router_topk. */
int mo_router_topk_v(const double* logits, int ld, int T, int E, int k, const double* bias,
                     int renormalize, double scale, int32_t* ids, double* w);

/* RMSNorm of the layer output (daScript PR #3988, combine-folded residual commit: the add + RMS
 * step after the routed block sums the FFN row onto the residual, then norms the row for the
 * next layer):
 * out[t][h] = y[t][h] / sqrt(mean_h y[t][h]^2 + eps) * gamma[h], gamma bf16 [H]. */
int mo_rmsnorm(const double* y, const uint16_t* gamma, int T, int H, double eps, double* out);

/* Per-expert histogram, exclusive scan and stable permutation of the T*k slots. */
int mo_dispatch(const int32_t* ids, int T, int k, int E, int32_t* counts,
                int32_t* offsets, int32_t* perm, int32_t* inv);

/* One SwiGLU expert on one bf16 hidden row: o = W_d (silu(W_g x) * (W_u x)).
 * gq/gs, uq/us: rows = I, K = H; dq/ds: rows = H, K = I.  o has H entries. */
int mo_expert_row(const uint16_t* x_row, int H, int I,
                  const uint8_t* gq, const uint16_t* gs,
                  const uint8_t* uq, const uint16_t* us,
                  const uint8_t* dq, const uint16_t* ds, double* o);
int mo_expert_row_fmt(const uint16_t* x_row, int H, int I, int fmt,
                      const uint8_t* gq, const void* gs,
                      const uint8_t* uq, const void* us,
                      const uint8_t* dq, const void* ds, double* o);

/* Expert outputs for every dispatched row r (dispatch order): a = perm[r],
 * t = a / k, e = ids[a]; rows[r][:] = expert e applied to x[t].  When
 * token_mask != NULL only rows whose token has token_mask[t] != 0 are computed
 * (the others are left untouched). */
int mo_expert_mlp(const uint16_t* x, int T, int H, int I, int E, int k,
                  const uint8_t* gate_q, const uint16_t* gate_s,
                  const uint8_t* up_q, const uint16_t* up_s,
                  const uint8_t* down_q, const uint16_t* down_s,
                  const int32_t* ids, const int32_t* perm,
                  const uint8_t* token_mask, double* rows);
int mo_expert_mlp_fmt(const uint16_t* x, int T, int H, int I, int E, int k, int fmt,
                      const uint8_t* gate_q, const void* gate_s,
                      const uint8_t* up_q, const void* up_s,
                      const uint8_t* down_q, const void* down_s,
                      const int32_t* ids, const int32_t* perm,
                      const uint8_t* token_mask, double* rows);

/* Shared expert: y_sh[t] = gate_t * W_d(silu(W_g x_t) * (W_u x_t)), where
 * gate_t = 1 / (1 + exp(-x_t . g)) when g != NULL and 1 otherwise. */
int mo_shared_expert(const uint16_t* x, int T, int H, int I_sh,
                     const uint8_t* gate_q, const uint16_t* gate_s,
                     const uint8_t* up_q, const uint16_t* up_s,
                     const uint8_t* down_q, const uint16_t* down_s,
                     const uint16_t* g, const uint8_t* token_mask, double* y_sh);
int mo_shared_expert_fmt(const uint16_t* x, int T, int H, int I_sh, int fmt,
                         const uint8_t* gate_q, const void* gate_s,
                         const uint8_t* up_q, const void* up_s,
                         const uint8_t* down_q, const void* down_s,
                         const uint16_t* g, const uint8_t* token_mask, double* y_sh);

/* y[t][n] = residual[t][n] + shared[t][n] + sum_j w[t][j] * rows[inv[t*k+j]][n]
 * (residual bf16 and shared may be NULL). */
int mo_combine(const double* rows, const int32_t* inv, const double* w,
               const double* shared, const uint16_t* residual,
               int T, int k, int H, const uint8_t* token_mask, double* y);

/* Whole layer.  Router logits are computed in fp64 and rounded to fp32 before
 * selection (the router consumes fp32 logits); the shared gate logit is used
 * unrounded.  Optional outputs: logits_f32 [T][E] (the rounded values), ids,
 * w.  y [T][H].  token_mask as above (routing runs for every token). */
int mo_layer_forward(const uint16_t* x, const uint16_t* residual,
                     const uint16_t* W_r, int T, int H, int I, int E, int k,
                     const uint8_t* gate_q, const uint16_t* gate_s,
                     const uint8_t* up_q, const uint16_t* up_s,
                     const uint8_t* down_q, const uint16_t* down_s,
                     int I_sh,
                     const uint8_t* sh_gate_q, const uint16_t* sh_gate_s,
                     const uint8_t* sh_up_q, const uint16_t* sh_up_s,
                     const uint8_t* sh_down_q, const uint16_t* sh_down_s,
                     const uint16_t* sh_g, const uint8_t* token_mask,
                     double* logits_f32, int32_t* ids, double* w, double* y);
/* The same layer with the routed experts in format fmt_r and the shared expert in fmt_s. */
int mo_layer_forward_fmt(const uint16_t* x, const uint16_t* residual,
                         const uint16_t* W_r, int T, int H, int I, int E, int k, int fmt_r,
                         const uint8_t* gate_q, const void* gate_s,
                         const uint8_t* up_q, const void* up_s,
                         const uint8_t* down_q, const void* down_s,
                         int I_sh, int fmt_s,
                         const uint8_t* sh_gate_q, const void* sh_gate_s,
                         const uint8_t* sh_up_q, const void* sh_up_s,
                         const uint8_t* sh_down_q, const void* sh_down_s,
                         const uint16_t* sh_g, const uint8_t* token_mask,
                         double* logits_f32, int32_t* ids, double* w, double* y);

#ifdef __cplusplus
}
#endif
#endif
