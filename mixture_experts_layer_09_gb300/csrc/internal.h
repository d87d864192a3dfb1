// internal.h -- launchers shared between the C-ABI layer (api.cu) and the kernel files.
#pragma once

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

// router.cu
cudaError_t launch_router_logits(const uint16_t* x, const uint16_t* W_r, const uint16_t* g, int T, int H,
                                 int E, float* logits, cudaStream_t st);
cudaError_t launch_router_topk(const void* logits, bool is_bf16, int ld, int T, int E, int k, int32_t* ids,
                               float* w, cudaStream_t st);

// dispatch.cu
size_t dispatch_scratch_bytes(int n_slots, int E);
cudaError_t launch_dispatch(const int32_t* ids, int n_slots, int E, int32_t* counts, int32_t* offsets,
                            int32_t* perm, int32_t* inv, int32_t* active, int32_t* n_active, void* scratch,
                            int* status, cudaStream_t st);

// gemv.cu -- bandwidth arm
struct QuantArgs {
    const void* src0 = nullptr;
    int src0_bf16 = 0, rows0 = 0, K0 = 32;
    int16_t* q0 = nullptr;
    float* sc0 = nullptr;
    int* sum0 = nullptr;
    const void* src1 = nullptr;
    int src1_bf16 = 0, rows1 = 0, K1 = 32;
    int16_t* q1 = nullptr;
    float* sc1 = nullptr;
    int* sum1 = nullptr;
};
cudaError_t launch_quantize(const QuantArgs& a, cudaStream_t st);

struct GemvArgs {
    int T, k, H, I;
    int max_active;               // host-side upper bound of n_active (grid sizing)
    // routed experts
    const uint8_t* gate_q;
    const uint16_t* gate_s;
    const uint8_t* up_q;
    const uint16_t* up_s;
    const uint8_t* down_q;
    const uint16_t* down_s;
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
    // quantised activations
    const int16_t* xq;
    const float* xsc;
    const int* xsum;
    float* h;                     // [T*k][I] dispatch order
    float* sh_h;                  // [T][I_sh]
    const int16_t* hq;
    const float* hsc;
    const int* hsum;
    const int16_t* sh_hq;
    const float* sh_hsc;
    const int* sh_hsum;
    // outputs
    float* rows_out;              // ROWS mode: [T*k][H] unweighted, dispatch order
    float* sh_rows_out;           // ROWS mode: [T][H] gated shared rows
    const uint16_t* residual;     // COMBINE mode
    float* y;                     // COMBINE mode: [T][H]
};
bool gemv_supported(int H, int I, int I_sh);
cudaError_t launch_gateup_gemv(const GemvArgs& p, int num_sms, cudaStream_t st);
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
    // activations / scratch
    const uint16_t* x;            // bf16 [T][H]
    uint16_t* x16;                // fp16 [T*k + T][H]: dispatch-order rows, then token-order rows
    uint16_t* h16;                // fp16 [T*k][I]
    uint16_t* sh_h16;             // fp16 [T][I_sh]
    int* tiles;                   // [ntile_max] packed (expert, row start, rows)
    int* n_tiles;
    int* status;
    // outputs
    float* rows_out;              // ROWS mode [T*k][H], unweighted, dispatch order
    float* slot_out;              // SLOT mode [T*k][H], weighted, slot order
    float* sh_out;                // [T][H] gated shared rows
};
constexpr int kGemmTileN = 128;   // tokens per tile
int gemm_ntile_max(int n_slots, int E);
bool gemm_supported(int H, int I, int I_sh);
cudaError_t launch_gemm_arm(const GemmPlan& p, bool rows_mode, cudaStream_t st);

// combine.cu
cudaError_t launch_combine(const float* rows, const int32_t* inv, const float* topk_w, bool weighted_slots,
                           const float* shared, const uint16_t* residual, int T, int k, int H, float* y,
                           cudaStream_t st);

}  // namespace moe
