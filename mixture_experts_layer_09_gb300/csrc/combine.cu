// combine.cu -- stage 4 of the routed MoE layer when it is not fused into the down projection.
//
// y[t] = shared[t] + sum_j w[t][j] * o[t][j] + residual[t], summed in that order: the gated
// shared row first, then the routed slots in order, then the residual (daScript PR #3988
// "dasLLAMA vulkan: a MoE that fits the card ...", combine-folded residual commit, which
// fixed this order because the natural one moved a router near-tie downstream).
// Rows come either unweighted in dispatch order (read through inv, weighted here) or already
// weighted in slot order (written that way by the tensor arm's down epilogue).
// With a norm output the combine also norms each row it finishes (the same commit's add + RMS
// step): one CTA per token row, the row's sum of squares taken as it is written, then the row
// read back by the threads that wrote it.  That removes the norm's own launch and its second
// pass over y from HBM; the bits match the separate norm kernel (norm.cuh).
#include "common.cuh"
#include "internal.h"
#include "norm.cuh"
#include "norm.h"

namespace moe {

struct CombineIn {
    const float* rows;
    const int32_t* inv;
    const float* topk_w;
    const float* shared;
    const uint16_t* residual;
    int k, H;
};

// Column group n4 (four floats) of token t's output.
template <bool WEIGHTED_SLOTS>
__device__ __forceinline__ float4 combine4(const CombineIn& a, int t, int n4) {
    const int H = a.H;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (a.shared) acc = __ldg(reinterpret_cast<const float4*>(a.shared + static_cast<size_t>(t) * H) + n4);
    for (int j = 0; j < a.k; ++j) {
        const int s = t * a.k + j;
        float4 v;
        if (WEIGHTED_SLOTS) {
            v = __ldg(reinterpret_cast<const float4*>(a.rows + static_cast<size_t>(s) * H) + n4);
        } else {
            const int r = __ldg(a.inv + s);
            const float w = __ldg(a.topk_w + s);
            v = __ldg(reinterpret_cast<const float4*>(a.rows + static_cast<size_t>(r) * H) + n4);
            v.x *= w; v.y *= w; v.z *= w; v.w *= w;
        }
        acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    if (a.residual) {
        const uint2 rb = __ldg(reinterpret_cast<const uint2*>(a.residual + static_cast<size_t>(t) * H) + n4);
        acc.x += __uint_as_float(rb.x << 16);
        acc.y += __uint_as_float(rb.x & 0xffff0000u);
        acc.z += __uint_as_float(rb.y << 16);
        acc.w += __uint_as_float(rb.y & 0xffff0000u);
    }
    return acc;
}

template <bool WEIGHTED_SLOTS>
__global__ void __launch_bounds__(256) combine_kernel(const __grid_constant__ CombineIn a, int T,
                                                      float* __restrict__ y) {
    pdl_wait();
    pdl_trigger();
    // T * H / 4 < 2^31 for every supported shape (checked by the launcher): 32-bit index math
    const int H4 = a.H / 4;
    const int total = T * H4;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
        const int t = i / H4;
        const int n4 = i - t * H4;
        reinterpret_cast<float4*>(y + static_cast<size_t>(t) * a.H)[n4] = combine4<WEIGHTED_SLOTS>(a, t, n4);
    }
}

// One CTA per token row: combine, then norm the row (norm.cuh's ownership and order).
template <bool WEIGHTED_SLOTS>
__global__ void __launch_bounds__(kNormThreads) combine_norm_kernel(const __grid_constant__ CombineIn a,
                                                                    float* __restrict__ y,
                                                                    const uint16_t* __restrict__ gamma, float eps,
                                                                    uint16_t* __restrict__ y_norm) {
    pdl_wait();
    pdl_trigger();
    __shared__ float part[kNormThreads / 32];
    const int t = blockIdx.x, H4 = a.H / 4;
    float4* row = reinterpret_cast<float4*>(y + static_cast<size_t>(t) * a.H);
    float ss = 0.f;
    for (int c = threadIdx.x; c < H4; c += kNormThreads) {
        const float4 v = combine4<WEIGHTED_SLOTS>(a, t, c);
        row[c] = v;
        ss = sq_acc4(v, ss);
    }
    const float inv = row_inv_rms(ss, part, a.H, eps);
    uint2* orow = reinterpret_cast<uint2*>(y_norm + static_cast<size_t>(t) * a.H);
    for (int c = threadIdx.x; c < H4; c += kNormThreads) orow[c] = norm4(row[c], inv, gamma, c);
}

cudaError_t launch_combine(const float* rows, const int32_t* inv, const float* topk_w, bool weighted_slots,
                           const float* shared, const uint16_t* residual, int T, int k, int H, float* y,
                           cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    const long total = static_cast<long>(T) * (H / 4);
    if (total >= (1L << 31)) return cudaErrorInvalidValue;
    const CombineIn a{rows, inv, topk_w, shared, residual, k, H};
    long blocks = (total + 255) / 256;
    if (blocks > 152L * 16) blocks = 152L * 16;
    KernelScope ks_("combine", st);
    const dim3 grid(static_cast<unsigned>(blocks)), block(256);
    if (weighted_slots) return launch_pdl(combine_kernel<true>, grid, block, 0, st, a, T, y);
    return launch_pdl(combine_kernel<false>, grid, block, 0, st, a, T, y);
}

cudaError_t launch_combine_norm(const float* rows, const int32_t* inv, const float* topk_w, bool weighted_slots,
                                const float* shared, const uint16_t* residual, int T, int k, int H, float* y,
                                const NormOut& norm, cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    const CombineIn a{rows, inv, topk_w, shared, residual, k, H};
    KernelScope ks_("combine_norm", st);
    const dim3 grid(static_cast<unsigned>(T)), block(kNormThreads);
    if (weighted_slots)
        return launch_pdl(combine_norm_kernel<true>, grid, block, 0, st, a, y, norm.gamma, norm.eps, norm.y_norm);
    return launch_pdl(combine_norm_kernel<false>, grid, block, 0, st, a, y, norm.gamma, norm.eps, norm.y_norm);
}

}  // namespace moe
