// norm.h -- the layer output's RMSNorm done inside the tensor arm's combine (combine.cu): one CTA
// per token row combines the row, then norms it; the bits equal launch_rmsnorm's on the same y.
#pragma once
#include <cuda_runtime.h>
#include <cstdint>

namespace moe {

struct NormOut {
    const uint16_t* gamma;  // [H] bf16, 8-byte aligned
    float eps;
    uint16_t* y_norm;       // [T][H] bf16, 8-byte aligned
};

// launch_combine's inputs and y, plus y_norm = RMSNorm(y) with gamma and eps.
cudaError_t launch_combine_norm(const float* rows, const int32_t* inv, const float* topk_w, bool weighted_slots,
                                const float* shared, const uint16_t* residual, int T, int k, int H, float* y,
                                const NormOut& norm, cudaStream_t st);

}  // namespace moe
