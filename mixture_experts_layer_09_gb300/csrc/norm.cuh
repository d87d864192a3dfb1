// norm.cuh -- the RMSNorm arithmetic shared by the standalone norm kernel and the combine that
// norms its own rows (daScript PR #3988 "dasLLAMA vulkan: a MoE that fits the card ...",
// combine-folded residual commit: after the routed block lands on the residual, the row is
// normed for the next layer):
//   y_norm[t][h] = bf16(y[t][h] * rsqrt(mean_h y[t][h]^2 + eps) * gamma[h]).
// A row is handled by one CTA of 256 threads, thread i owning the float4 columns i, i + 256, ...
// Both users keep that ownership and the reduction order below, so a row normed inside the
// combine is bit-identical to the same row normed by the separate launch.
#pragma once
#include <cuda_bf16.h>

#include "common.cuh"

namespace moe {

constexpr int kNormThreads = 256;

__device__ __forceinline__ float sq_acc4(float4 v, float ss) {
    ss = fmaf(v.x, v.x, ss);
    ss = fmaf(v.y, v.y, ss);
    ss = fmaf(v.z, v.z, ss);
    return fmaf(v.w, v.w, ss);
}

// 1 / rms of a row from its 8 per-warp sums of squares, added in a fixed tree.
__device__ __forceinline__ float inv_rms_of_parts(const float* part, int H, float eps) {
    const float tot = ((part[0] + part[1]) + (part[2] + part[3])) + ((part[4] + part[5]) + (part[6] + part[7]));
    return rsqrtf(tot / static_cast<float>(H) + eps);
}

// 1 / rms of the row from each thread's partial sum of squares: per warp, then over the 8 warps.
// `part` is 8 floats of shared memory; every thread of the CTA calls this.
__device__ __forceinline__ float row_inv_rms(float ss, float* part, int H, float eps) {
    ss = warp_sum(ss);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
    __syncthreads();
    return inv_rms_of_parts(part, H, eps);
}

// Four normed bf16 values of column group c (gamma read through the read-only path).
__device__ __forceinline__ uint2 norm4(float4 v, float inv, const uint16_t* __restrict__ gamma, int c) {
    const uint2 g = __ldg(reinterpret_cast<const uint2*>(gamma) + c);
    const float o0 = v.x * inv * bf16_to_f32(static_cast<uint16_t>(g.x & 0xffffu));
    const float o1 = v.y * inv * bf16_to_f32(static_cast<uint16_t>(g.x >> 16));
    const float o2 = v.z * inv * bf16_to_f32(static_cast<uint16_t>(g.y & 0xffffu));
    const float o3 = v.w * inv * bf16_to_f32(static_cast<uint16_t>(g.y >> 16));
    const uint32_t lo = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(o0))) |
                        (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(o1))) << 16);
    const uint32_t hi = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(o2))) |
                        (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(o3))) << 16);
    return make_uint2(lo, hi);
}

}  // namespace moe
