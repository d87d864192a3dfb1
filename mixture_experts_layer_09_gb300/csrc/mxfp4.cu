// mxfp4.cu -- upload step of MXFP4 expert weights (colibri PR #418, the fmt=7 note of its Kimi K3
// Vulkan tier: the e2m1 codes are uploaded exactly as stored and the host expands the ue8m0
// exponents at upload).
//
// Each ue8m0 exponent e becomes the fp16 scale 2^(e - 128).  The expert kernels read an e2m1
// code as the integer 2v (v the code's value, |2v| <= 12), so half the MX scale 2^(e - 127)
// gives back v * 2^(e - 127).  Every product 2v * 2^(e - 128) is exact in fp16 when
// e - 128 lies in [-24, 12] (the top code 12 * 2^12 stays below 65504; 2^-24 is fp16's
// smallest step); an exponent outside that range, the MX NaN code 255 among them, writes 0
// and records MOE_ERR_DEVICE_RANGE with its index and value.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace moe {

__global__ void __launch_bounds__(256) mxfp4_scales_kernel(const uint8_t* __restrict__ e8, size_t n,
                                                           uint16_t* __restrict__ s, int* status) {
    pdl_wait();
    pdl_trigger();
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
        const int e = e8[i];
        const int p = e - 128;
        uint16_t b = 0;
        if (p >= -14 && p <= 12)
            b = static_cast<uint16_t>((p + 15) << 10);  // normal: biased exponent p + 15, mantissa 0
        else if (p >= -24 && p < -14)
            b = static_cast<uint16_t>(1u << (p + 24));  // subnormal: 2^(p + 24) steps of 2^-24
        else
            record_status(status, MOE_ERR_DEVICE_RANGE, static_cast<int>(i & 0x7fffffff), e);
        s[i] = b;
    }
}

cudaError_t launch_mxfp4_scales(const uint8_t* e8, size_t n, uint16_t* s, int* status, cudaStream_t st) {
    if (n == 0) return cudaSuccess;
    const size_t blocks = std::min<size_t>((n + 255) / 256, 152 * 8);  // grid-stride beyond 8 per SM
    KernelScope ks_("mxfp4_scales", st);
    return launch_pdl(mxfp4_scales_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st, e8, n, s, status);
}

}  // namespace moe
