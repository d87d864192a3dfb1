// combine.cu -- stage 4 of the routed MoE layer when it is not fused into the down projection.
//
// y[t] = shared[t] + sum_j w[t][j] * o[t][j] + residual[t], summed in that order: the gated
// shared row first, then the routed slots in order, then the residual (daScript PR #3988
// "dasLLAMA vulkan: a MoE that fits the card ...", combine-folded residual commit, which
// fixed this order because the natural one moved a router near-tie downstream).
// Rows come either unweighted in dispatch order (read through inv, weighted here) or already
// weighted in slot order (written that way by the tensor arm's down epilogue).
#include "common.cuh"
#include "internal.h"

namespace moe {

template <bool WEIGHTED_SLOTS>
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ rows,
                                                      const int32_t* __restrict__ inv,
                                                      const float* __restrict__ topk_w,
                                                      const float* __restrict__ shared,
                                                      const uint16_t* __restrict__ residual, int T, int k,
                                                      int H, float* __restrict__ y) {
    pdl_wait();
    pdl_trigger();
    // T * H / 4 < 2^31 for every supported shape (checked by the launcher): 32-bit index math
    const int H4 = H / 4;
    const int total = T * H4;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
        const int t = i / H4;
        const int n4 = i - t * H4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (shared) acc = __ldg(reinterpret_cast<const float4*>(shared + static_cast<size_t>(t) * H) + n4);
        for (int j = 0; j < k; ++j) {
            const int a = t * k + j;
            float4 v;
            if (WEIGHTED_SLOTS) {
                v = __ldg(reinterpret_cast<const float4*>(rows + static_cast<size_t>(a) * H) + n4);
            } else {
                const int r = __ldg(inv + a);
                const float w = __ldg(topk_w + a);
                v = __ldg(reinterpret_cast<const float4*>(rows + static_cast<size_t>(r) * H) + n4);
                v.x *= w; v.y *= w; v.z *= w; v.w *= w;
            }
            acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
        }
        if (residual) {
            const uint2 rb = __ldg(reinterpret_cast<const uint2*>(residual + static_cast<size_t>(t) * H) + n4);
            acc.x += __uint_as_float(rb.x << 16);
            acc.y += __uint_as_float(rb.x & 0xffff0000u);
            acc.z += __uint_as_float(rb.y << 16);
            acc.w += __uint_as_float(rb.y & 0xffff0000u);
        }
        reinterpret_cast<float4*>(y + static_cast<size_t>(t) * H)[n4] = acc;
    }
}

cudaError_t launch_combine(const float* rows, const int32_t* inv, const float* topk_w, bool weighted_slots,
                           const float* shared, const uint16_t* residual, int T, int k, int H, float* y,
                           cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    const long total = static_cast<long>(T) * (H / 4);
    if (total >= (1L << 31)) return cudaErrorInvalidValue;
    long blocks = (total + 255) / 256;
    if (blocks > 152L * 16) blocks = 152L * 16;
    KernelScope ks_("combine", st);
    const dim3 grid(static_cast<unsigned>(blocks)), block(256);
    if (weighted_slots)
        return launch_pdl(combine_kernel<true>, grid, block, 0, st, rows, inv, topk_w, shared, residual, T, k, H, y);
    return launch_pdl(combine_kernel<false>, grid, block, 0, st, rows, inv, topk_w, shared, residual, T, k, H, y);
}

}  // namespace moe
