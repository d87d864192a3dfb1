// internal.h -- launchers shared between the C-ABI layer (api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace moe {

// Counts a kernel launch and, when timing is on, brackets it with CUDA events (profile.cu).
class KernelScope {
   public:
    KernelScope(const char* name, cudaStream_t st);
    ~KernelScope();
    KernelScope(const KernelScope&) = delete;
    KernelScope& operator=(const KernelScope&) = delete;

   private:
    cudaStream_t st_;
    int idx_;
};

// tmap.cu: 2D tensor map (inner dimension first), cached per parameter set.
bool tmap_2d(CUtensorMap* out, CUtensorMapDataType dtype, const void* base, uint64_t inner, uint64_t rows,
             uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swizzle);

// router.cu
// Decode routing in the logits launch (T <= 32): top-k ids/w of every token and the dispatch
// (counts, offsets, perm, inv, active list), run by the row CTA that finishes last; `done` is a
// completion count that is zero between calls (workspace head).
struct DecodeRoute {
    int k = 0;
    int32_t* ids = nullptr;       // null: logits only
    float* w = nullptr;
    int32_t* counts = nullptr;
    int32_t* offsets = nullptr;
    int32_t* perm = nullptr;
    int32_t* inv = nullptr;
    int32_t* active = nullptr;
    int32_t* n_active = nullptr;
    int* status = nullptr;
    int* done = nullptr;
};
// xq/xmeta (optional): also quantise x for the GEMV arm in the same launch (decode batches).
cudaError_t launch_router_logits(const uint16_t* x, const uint16_t* W_r, const uint16_t* g, int T, int H,
                                 int E, float* logits, cudaStream_t st, int16_t* xq = nullptr,
                                 int2* xmeta = nullptr, int x_gld = 0, int* status = nullptr,
                                 const DecodeRoute* route = nullptr);
// router_tc.cu: tcgen05 logits GEMM for T > 32 (status: device timeout record, may be null)
// (H % 64 == 0, 1 <= E <= 256, x / W_r / g 16-byte aligned)
bool router_tc_supported(const void* x, const void* W_r, const void* g, int H, int E);
// ksplit > 1: partial logits of ksplit equal K ranges in planes T * (E + (g != 0)) floats apart
// (router_tc_ksplit(H) picks up to 4 ranges of at least 4 K-steps); the planes sum to the logits.
int router_tc_ksplit(int H);
cudaError_t launch_router_logits_tc(const uint16_t* x, const uint16_t* W_r, const uint16_t* g, int T, int H, int E,
                                    float* logits, int* status, cudaStream_t st, int ksplit = 1);
// group row stride of the quantised activations: K/32 rounded up to a multiple of 4
inline int act_gld(int K) { return ((K / 32) + 3) & ~3; }
// bias (fp32 [E], selection only), renorm, scale: the router variants (defaults: plain softmax top-k)
cudaError_t launch_router_topk(const void* logits, bool is_bf16, int ld, int T, int E, int k, int32_t* ids,
                               float* w, cudaStream_t st, const float* bias = nullptr, bool renorm = true,
                               float scale = 1.f);
// The same top-k (fp32 logits, no variants) with each CTA of kCountedWarps * tpw tokens counting
// its picks per expert into row blockIdx.x of cta_cnt [ceil(T / (kCountedWarps tpw))][E]: the
// count table of a dispatch whose CTAs take kCountedWarps tpw k slots each
// (launch_dispatch_counted).
constexpr int kCountedWarps = 16;
// parts > 1: the logits arrive as `parts` partial planes (T * ld floats apart, plane 0 at `logits`);
// each warp sums them in plane order into plane 0 (the final logits) before its top-k.
cudaError_t launch_router_topk_counted(float* logits, int ld, int T, int E, int k, int tpw, int32_t* ids, float* w,
                                       int* cta_cnt, cudaStream_t st, int parts = 1);

// dispatch.cu
size_t dispatch_scratch_bytes(int n_slots, int E);
// The scatter alone, for a count table written by the router (CTA c counted slots [c spc, (c + 1)
// spc)): offsets, counts, active list, perm and inv, and (tiles != nullptr) the tensor arm's tile
// list.  Needs dispatch_counted_supported(nblk, E).
bool dispatch_counted_supported(int nblk, int E);
cudaError_t launch_dispatch_counted(const int32_t* ids, int n_slots, int E, int spc, int nblk, const int* cta_cnt,
                                    int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv, int32_t* active,
                                    int32_t* n_active, int* status, int* tiles, int* n_tiles, cudaStream_t st);
cudaError_t launch_dispatch(const int32_t* ids, int n_slots, int E, int32_t* counts, int32_t* offsets,
                            int32_t* perm, int32_t* inv, int32_t* active, int32_t* n_active, void* scratch,
                            int* status, cudaStream_t st);

// gemv.cu -- bandwidth arm
struct QuantArgs {
    const void* src0 = nullptr;
    int src0_bf16 = 0, rows0 = 0, K0 = 32;
    int16_t* q0 = nullptr;
    int2* meta0 = nullptr;        // {scale bits, integer sum} per group
    int gld0 = 0;                 // row stride of meta0 in groups (0: K/32)
    int kc0 = 512;                // slice width of the stored order of q0
    const void* src1 = nullptr;
    int src1_bf16 = 0, rows1 = 0, K1 = 32;
    int16_t* q1 = nullptr;
    int2* meta1 = nullptr;
    int gld1 = 0;
    int kc1 = 512;
};
cudaError_t launch_quantize(const QuantArgs& a, cudaStream_t st);

struct GemvArgs {
    // TMA maps of the weights (uint8, box 256 B x 32 rows) and scales (fp16, box 16 x 32 rows)
    CUtensorMap tm_gate, tm_up, tm_down, tm_gate_s, tm_up_s, tm_down_s;
    CUtensorMap tm_sh_gate, tm_sh_up, tm_sh_down, tm_sh_gate_s, tm_sh_up_s, tm_sh_down_s;
    int ws_gu, ws_d, ws_sh_gu, ws_sh_d;  // scale maps valid (else scales are read directly)
    int T, k, H, I;
    int max_active;               // host-side upper bound of n_active (grid sizing)
    // routed experts
    const uint8_t* gate_q;
    const uint16_t* gate_s;
    const uint8_t* up_q;
    const uint16_t* up_s;
    const uint8_t* down_q;
    const uint16_t* down_s;
    int fp4_r, fp4_s;             // MXFP4 codes (else int4) in the routed / shared matrices
    // shared expert (sh_I == 0: none)
    int sh_I;
    const uint8_t* sh_gate_q;
    const uint16_t* sh_gate_s;
    const uint8_t* sh_up_q;
    const uint16_t* sh_up_s;
    const uint8_t* sh_down_q;
    const uint16_t* sh_down_s;
    const float* sh_gate_logit;   // &logits[0][E] (stride logit_ld) or nullptr = ungated
    int logit_ld;
    // routing
    const int32_t* offsets;
    const int32_t* perm;
    const int32_t* active;
    const int32_t* n_active;
    const float* topk_w;
    // quantised activations: int16 values, {scale, sum} per group (row stride *_gld groups)
    const int16_t* xq;            // [T][H]
    const int2* xmeta;
    int16_t* hq;                  // [T*k][I] dispatch order
    int2* hmeta;
    int16_t* sh_hq;               // [T][I_sh]
    int2* sh_hmeta;
    int x_gld, h_gld, sh_gld;
    // outputs
    float* rows_out;              // ROWS mode: [T*k][H] unweighted, dispatch order
    float* sh_rows_out;           // ROWS mode: [T][H] gated shared rows
    float* slot_term;             // COMBINE mode: [T*k][H] weighted, slot order
    float* sh_term;               // COMBINE mode: [T][H] gated shared rows
    int* col_counter;             // COMBINE mode: [H/32] zero between calls
    int* task_counter;            // [4] task claim counters (gate/up, down), zero between calls
    int* status;                  // device status word (bounded-wait timeouts)
    const uint16_t* residual;     // COMBINE mode
    float* y;                     // COMBINE mode: [T][H]
};
// Builds the tensor maps of GemvArgs from its weight pointers; false if encoding fails.
bool gemv_tensor_maps(GemvArgs& p, int E);
cudaError_t launch_gateup_gemv(const GemvArgs& p, cudaStream_t st);
cudaError_t launch_down_gemv(const GemvArgs& p, bool combine, cudaStream_t st);

// gemm_sm100.cu -- tensor arm (tcgen05 / TMEM grouped GEMM)
struct GemmPlan {
    int T, k, E, H, I, sh_I;
    int ntile_max;                // host upper bound of routed tiles
    int sh_tiles;                 // shared-expert tiles (ceil(T / tile))
    // routing
    const int32_t* offsets;
    const int32_t* perm;
    const float* topk_w;
    const float* sh_gate_logit;
    int logit_ld;
    // weights
    const uint8_t* gate_q;
    const uint16_t* gate_s;
    const uint8_t* up_q;
    const uint16_t* up_s;
    const uint8_t* down_q;
    const uint16_t* down_s;
    const uint8_t* sh_gate_q;
    const uint16_t* sh_gate_s;
    const uint8_t* sh_up_q;
    const uint16_t* sh_up_s;
    const uint8_t* sh_down_q;
    const uint16_t* sh_down_s;
    int fp4_r, fp4_s;             // MXFP4 codes (else int4) in the routed / shared matrices
    // activations / scratch
    const uint16_t* x;            // bf16 [T][H]
    uint16_t* x16;                // fp16 [T*k + T][H]: dispatch-order rows, then token-order rows
    uint16_t* h16;                // fp16 [T*k][I]
    uint16_t* sh_h16;             // fp16 [T][I_sh]
    int* tiles;                   // [3 * ntile_max] (expert, row start, rows)
    int* n_tiles;
    int tiles_ready;              // the dispatch already wrote the tile list
    int* status;
    // outputs
    float* rows_out;              // ROWS mode [T*k][H], unweighted, dispatch order
    float* slot_out;              // SLOT mode [T*k][H], weighted, slot order
    float* sh_out;                // [T][H] gated shared rows
};
constexpr int kGemmTileN = 256;   // tokens per tile
int gemm_ntile_max(int n_slots, int E);
bool gemm_supported(int H, int I, int I_sh);
cudaError_t launch_gemm_arm(const GemmPlan& p, bool rows_mode, cudaStream_t st);

// MXFP4 upload: fp16 2^(e - 128) per ue8m0 exponent; out-of-range exponents record
// MOE_ERR_DEVICE_RANGE in *status.
cudaError_t launch_mxfp4_scales(const uint8_t* e8, size_t n, uint16_t* s, int* status, cudaStream_t st);

// norm.cu: RMSNorm of the layer output into bf16 rows (H % 4 == 0, y 16-byte and gamma/out
// 8-byte aligned)
cudaError_t launch_rmsnorm(const float* y, const uint16_t* gamma, int T, int H, float eps, uint16_t* out,
                           cudaStream_t st);

// combine.cu
cudaError_t launch_combine(const float* rows, const int32_t* inv, const float* topk_w, bool weighted_slots,
                           const float* shared, const uint16_t* residual, int T, int k, int H, float* y,
                           cudaStream_t st);

}  // namespace moe
