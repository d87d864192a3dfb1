// norm.cu -- RMSNorm of the layer output for the next layer, as its own launch (the arms whose
// combine does not norm its rows, and the moe_rmsnorm stage call).  The arithmetic and its
// order live in norm.cuh.  One CTA of 256 threads per token row: float4 loads, the sum of
// squares in fp32, one reciprocal square root, bf16 stores.
#include "common.cuh"
#include "internal.h"
#include "norm.cuh"

namespace moe {

__global__ void __launch_bounds__(kNormThreads) rmsnorm_kernel(const float* __restrict__ y,
                                                               const uint16_t* __restrict__ gamma, int H, float eps,
                                                               uint16_t* __restrict__ out) {
    pdl_wait();
    pdl_trigger();
    __shared__ float part[kNormThreads / 32];
    const int t = blockIdx.x;
    const float4* row = reinterpret_cast<const float4*>(y + static_cast<size_t>(t) * H);
    const int n4 = H / 4;
    float ss = 0.f;
    for (int c = threadIdx.x; c < n4; c += kNormThreads) ss = sq_acc4(row[c], ss);
    const float inv = row_inv_rms(ss, part, H, eps);
    uint2* orow = reinterpret_cast<uint2*>(out + static_cast<size_t>(t) * H);
    for (int c = threadIdx.x; c < n4; c += kNormThreads) orow[c] = norm4(row[c], inv, gamma, c);
}

cudaError_t launch_rmsnorm(const float* y, const uint16_t* gamma, int T, int H, float eps, uint16_t* out,
                           cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    KernelScope ks_("rmsnorm", st);
    return launch_pdl(rmsnorm_kernel, dim3(T), dim3(kNormThreads), 0, st, y, gamma, H, eps, out);
}

}  // namespace moe
