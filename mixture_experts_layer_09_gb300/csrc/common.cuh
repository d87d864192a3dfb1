// common.cuh -- device helpers shared by the layer's kernels (sm_103a only).
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <utility>

#include "../../include/moe.h"

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ < 1000)
#error "this library is written for sm_103a (Blackwell) only"
#endif

namespace moe {

constexpr int kWarp = 32;
constexpr size_t kWsAlign = 256;
// Head of every workspace: the device status word at offset 0, the GEMV task claim counters
// at kWsTaskOffset and, from kWsCounterOffset, the per-column-block counters of the GEMV down
// projection.  The kernels leave every counter at zero when they finish.
constexpr size_t kWsHead = 4096;
constexpr size_t kWsCounterOffset = 1024;
constexpr size_t kWsTaskOffset = 512;  // GEMV task claim counters (4 ints)
constexpr size_t kWsRouteOffset = 528;  // decode routing: row-CTA completion count (1 int)
// Test hook (16 bytes, zero in normal use): a wait limit in clock cycles (int64, 0 = the
// default) and an int that makes the tensor arm's gate/up kernel withhold one token-tile copy
// in its first CTA, so that a bounded wait runs out (moe_workspace_test_timeout).
constexpr size_t kWsTestHookOffset = 544;
struct TestHook {
    long long wait_limit;
    int withhold_copy;
    int pad;
};
constexpr int kMaxColBlocks = static_cast<int>((kWsHead - kWsCounterOffset) / sizeof(int));  // H <= 24576

// Device status word layout (first 256 bytes of every workspace).
struct DevStatus {
    int code;        // first MOE_ERR_DEVICE_* recorded, 0 when clean
    int detail[3];   // where it happened (kernel-specific)
};

__device__ __forceinline__ void record_status(int* st, int code, int d0 = 0, int d1 = 0) {
    if (st && atomicCAS(st, 0, code) == 0) {
        st[1] = d0;
        st[2] = d1;
    }
}

__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// 128-bit streaming load of data read once per call (weights): no L1 allocation.
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ uint4 ldg_nc(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

__host__ __device__ constexpr inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Programmatic dependent launch.  Every kernel of the library is launched with programmatic
// stream serialisation, so it may start while the previous kernel of the stream drains; it
// must call pdl_wait() before it reads or writes any memory that earlier work touches.  Once
// pdl_wait() returns, every earlier kernel of the stream has completed and its writes are
// visible.  pdl_trigger() lets the next kernel start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace moe
