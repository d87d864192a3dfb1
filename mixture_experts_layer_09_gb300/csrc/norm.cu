// norm.cu -- RMSNorm of the layer output for the next layer (daScript PR #3988 "dasLLAMA
// vulkan: a MoE that fits the card ...", combine-folded residual commit: the add + RMS step
// after the routed block sums the FFN row onto the residual, then norms the row for the next
// layer).  The combine already lands on the residual, so this pass reads y once more:
//   y_norm[t][h] = bf16(y[t][h] * rsqrt(mean_h y[t][h]^2 + eps) * gamma[h]).
// One CTA of 256 threads per token row: float4 loads, the sum of squares in fp32 reduced in a
// fixed order (per warp, then over the 8 warps), one reciprocal square root, bf16 stores.
#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"

namespace moe {

__global__ void __launch_bounds__(256) rmsnorm_kernel(const float* __restrict__ y, const uint16_t* __restrict__ gamma,
                                                      int H, float eps, uint16_t* __restrict__ out) {
    pdl_wait();
    pdl_trigger();
    __shared__ float part[8];
    const int t = blockIdx.x, lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const float4* row = reinterpret_cast<const float4*>(y + static_cast<size_t>(t) * H);
    const int n4 = H / 4;
    float ss = 0.f;
    for (int c = threadIdx.x; c < n4; c += 256) {
        const float4 v = row[c];
        ss = fmaf(v.x, v.x, ss);
        ss = fmaf(v.y, v.y, ss);
        ss = fmaf(v.z, v.z, ss);
        ss = fmaf(v.w, v.w, ss);
    }
    ss = warp_sum(ss);
    if (lane == 0) part[wid] = ss;
    __syncthreads();
    const float tot = ((part[0] + part[1]) + (part[2] + part[3])) + ((part[4] + part[5]) + (part[6] + part[7]));
    const float inv = rsqrtf(tot / static_cast<float>(H) + eps);
    uint2* orow = reinterpret_cast<uint2*>(out + static_cast<size_t>(t) * H);
    const uint2* grow = reinterpret_cast<const uint2*>(gamma);
    for (int c = threadIdx.x; c < n4; c += 256) {
        const float4 v = row[c];
        const uint2 g = __ldg(grow + c);
        const float o0 = v.x * inv * bf16_to_f32(static_cast<uint16_t>(g.x & 0xffffu));
        const float o1 = v.y * inv * bf16_to_f32(static_cast<uint16_t>(g.x >> 16));
        const float o2 = v.z * inv * bf16_to_f32(static_cast<uint16_t>(g.y & 0xffffu));
        const float o3 = v.w * inv * bf16_to_f32(static_cast<uint16_t>(g.y >> 16));
        const uint32_t lo = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(o0))) |
                            (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(o1))) << 16);
        const uint32_t hi = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(o2))) |
                            (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(o3))) << 16);
        orow[c] = make_uint2(lo, hi);
    }
}

cudaError_t launch_rmsnorm(const float* y, const uint16_t* gamma, int T, int H, float eps, uint16_t* out,
                           cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    KernelScope ks_("rmsnorm", st);
    return launch_pdl(rmsnorm_kernel, dim3(T), dim3(256), 0, st, y, gamma, H, eps, out);
}

}  // namespace moe
