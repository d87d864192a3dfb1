// router_tc.cu -- router logits for prefill batches on the 5th-generation tensor cores.
//
// logits[t][e] = x[t] . W_r[e] for e < E, and logits[t][E] = x[t] . g for the shared-expert
// gate (daScript PR #3988 "dasLLAMA vulkan: a MoE that fits the card ...", decode span commit:
// the gate logit is one more router row past the router's logits).  A CTA takes 128 tokens
// (MMA M = 128) and all E (+1) router rows (MMA N, rounded up to 16, split at 256): bf16 A and
// B in 128-byte-swizzled K-major tiles, fp32 accumulators in tensor memory.  Warp 0 brings the
// token tile (two boxes) and the router rows by TMA, one copy per lane, and writes the gate row
// into the B tile itself; warp 1 issues the MMAs; warps 2-5 read the accumulators and store the
// logits.  Waits are bounded.  With ksplit > 1 (prefill layer) the grid's y index takes one of
// ksplit equal K ranges and the epilogue writes that range's partial logits to plane y of the
// output (planes T * ld apart); the consumer sums the planes in order.
#include <cuda.h>

#include <algorithm>

#include "async.cuh"
#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace moe {

namespace {
constexpr int RM = 128;       // tokens per CTA
constexpr int RK = 64;        // K per stage (128 bytes of bf16)
constexpr int kMaxStages = 8;
constexpr int kTileA = RM * RK * 2;
constexpr int kSmemBudget = 227 * 1024;
static_assert(kTileA % 1024 == 0, "swizzled tiles stay 1024-aligned");

struct RouterTcArgs {
    CUtensorMap tm_x;   // bf16 [T][H], box 64 x 64
    CUtensorMap tm_w;   // bf16 [E][H], box 64 x E
    const uint16_t* g;  // bf16 [H] or nullptr
    int T, H, E, ld;
    int tile_b;         // bytes of one B tile: round16(E + (g != 0)) rows of 128 bytes
    int stages;         // pipeline depth, 2 .. kMaxStages
    int ksplit;         // K ranges (grid y); plane y of logits holds range y's partial sums
    float* logits;
    int* status;
};

// smem: [stages][A tile | B tile] | g copy (H bf16, when g != 0) | barriers
__host__ __device__ inline int g_bytes(int H, bool has_g) { return has_g ? ((H * 2 + 1023) & ~1023) : 0; }
}  // namespace

__global__ void __launch_bounds__(192, 1) router_logits_tc_kernel(const __grid_constant__ RouterTcArgs p) {
    const int t0 = blockIdx.x * RM;
    const int ncols = p.E + (p.g ? 1 : 0);
    const int nk = p.H / RK / p.ksplit;          // K-steps of this CTA's range
    const int kb0 = static_cast<int>(blockIdx.y) * nk;
    const int RS = p.stages;
    const int stage_bytes = kTileA + p.tile_b;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* gbuf = smem + RS * stage_bytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(gbuf + g_bytes(p.H, p.g != nullptr));
    uint64_t* empty = full + kMaxStages;
    uint64_t* accum = empty + kMaxStages;
    uint64_t* drain = accum + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < RS; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        mbar_init(accum, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (p.g) {
        // the gate row once per CTA, so that no stage waits on a global load
        for (int i = threadIdx.x; i < p.H / 8; i += blockDim.x)
            reinterpret_cast<uint4*>(gbuf)[i] = ldg_nc(p.g + static_cast<size_t>(i) * 8);
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&p.tm_x);
        prefetch_tmap(&p.tm_w);
    }
    if (warp == 1) tmem_alloc(tmem_slot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // everything above reads only the router weights: it overlaps the previous launch's tail
    pdl_wait();
    pdl_trigger();

    if (warp == 0) {
        // ---------------- producer: token tile + router rows by TMA, gate row by hand
        int issued = 0;
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % RS;
            bool ok = true;
            if (kb >= RS && lane == 0) ok = mbar_wait(empty + s, ((kb / RS) & 1) ^ 1, abort_flag, p.status, 21);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            uint8_t* sa = smem + s * stage_bytes;
            uint8_t* sb = sa + kTileA;
            if (p.g && lane < 8) {
                // row E of the B tile: 8 chunks of 16 bytes, in the tile's 128-byte swizzle
                const uint4 v = reinterpret_cast<const uint4*>(gbuf + (kb0 + kb) * RK * 2)[lane];
                *reinterpret_cast<uint4*>(sb + p.E * 128 + ((lane ^ (p.E & 7)) << 4)) = v;
                fence_proxy_async_smem();
            }
            __syncwarp();  // the gate row's writes, before lane 0's arrive releases the stage
            if (lane == 0) mbar_arrive_expect_tx(full + s, kTileA + p.E * RK * 2);
            __syncwarp();
            // the token tile as two 64-row boxes and the router rows, each from its own lane:
            // copies issued by one thread are served one after another
            if (lane < 2)
                tma_load_2d(sa + lane * (RM / 2) * 128, &p.tm_x, (kb0 + kb) * RK, t0 + lane * (RM / 2), full + s);
            if (lane == 2) tma_load_2d(sb, &p.tm_w, (kb0 + kb) * RK, 0, full + s);
            issued = kb + 1;
        }
        if (*abort_flag && lane == 0) {
            for (int kb = max(0, issued - RS); kb < issued; ++kb) {
                const long long c0 = clock64();
                while (!mbar_try_wait(full + kb % RS, (kb / RS) & 1) && clock64() - c0 < kWaitLimitCycles) {
                }
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer
        if (lane == 0) {
            const int n0 = min(256, (ncols + 15) & ~15);          // first column chunk
            const int n1 = ((ncols + 15) & ~15) - n0;             // rest (only when E + 1 > 256)
            const uint32_t id0 = idesc_f16_m128(n0, true);
            const uint32_t id1 = n1 > 0 ? idesc_f16_m128(n1, true) : 0;
            bool any = false;
            for (int kb = 0; kb < nk; ++kb) {
                const int s = kb % RS;
                if (!mbar_wait(full + s, (kb / RS) & 1, abort_flag, p.status, 22)) break;
                tc_fence_after();
                const uint32_t a0 = smem_u32(smem + s * stage_bytes), b0 = a0 + kTileA;
#pragma unroll
                for (int kk = 0; kk < RK / 16; ++kk) {
                    const uint32_t acc = (kb > 0 || kk > 0) ? 1u : 0u;
                    const uint64_t ad = sw128_kmajor_desc(a0 + kk * 32);
                    mma_f16(tmem, ad, sw128_kmajor_desc(b0 + kk * 32), id0, acc);
                    if (n1 > 0) mma_f16(tmem + 256, ad, sw128_kmajor_desc(b0 + 256 * 128 + kk * 32), id1, acc);
                }
                mma_commit(empty + s);
                any = true;
            }
            if (!*abort_flag) {
                mma_commit(accum);
            } else if (any) {
                mma_commit(drain);
                const long long c0 = clock64();
                while (!mbar_try_wait(drain, 0) && clock64() - c0 < kWaitLimitCycles) {
                }
            }
        }
    } else {
        // ---------------- epilogue: lane quadrant q holds tokens t0 + 32q .. t0 + 32q + 31.
        // Each 16-column chunk goes through shared memory (stage 0, idle once the accumulator is
        // final), so that the stores run along the rows of the logits rather than down a column.
        bool go = __all_sync(0xffffffffu, mbar_wait(accum, 0, abort_flag, p.status, 23));
        go = named_barrier_or(1, 128, !go) ? false : go;  // the four epilogue warps agree
        if (go) {
            tc_fence_after();
            const int q = warp & 3;
            const int et = threadIdx.x - 64;  // 0 .. 127
            const uint32_t tbase = tmem + (static_cast<uint32_t>(q * 32) << 16);
            float* stg = reinterpret_cast<float*>(smem);  // [128][17]
            float* out = p.logits + (static_cast<size_t>(blockIdx.y) * p.T + t0) * p.ld;
            const int nrow = min(RM, p.T - t0);
            for (int c0 = 0; c0 < ncols; c0 += 16) {
                float v[16];
                tmem_ld16(tbase + c0, v);
#pragma unroll
                for (int j = 0; j < 16; ++j) stg[(q * 32 + lane) * 17 + j] = v[j];
                named_barrier(1, 128);
#pragma unroll
                for (int m = 0; m < 16; ++m) {
                    const int i = et + 128 * m, row = i >> 4, col = i & 15;
                    if (row < nrow && c0 + col < ncols) out[static_cast<size_t>(row) * p.ld + c0 + col] = stg[row * 17 + col];
                }
                named_barrier(1, 128);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

bool router_tc_supported(const void* x, const void* W_r, const void* g, int H, int E) {
    const auto aligned = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15) == 0; };
    return H % RK == 0 && E >= 1 && E <= 256 && aligned(x) && aligned(W_r) && aligned(g);
}

int router_tc_ksplit(int H) {
    const int steps = H / RK;
    for (int s = 4; s > 1; s >>= 1)
        if (steps % s == 0 && steps / s >= 4) return s;
    return 1;
}

cudaError_t launch_router_logits_tc(const uint16_t* x, const uint16_t* W_r, const uint16_t* g, int T, int H, int E,
                                    float* logits, int* status, cudaStream_t st, int ksplit) {
    RouterTcArgs a{};
    if (ksplit < 1 || (H / RK) % ksplit) return cudaErrorInvalidValue;
    a.ksplit = ksplit;
    if (!tmap_2d(&a.tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, static_cast<uint64_t>(H), static_cast<uint64_t>(T),
                 static_cast<uint64_t>(H) * 2, RK, RM / 2, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    if (!tmap_2d(&a.tm_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, W_r, static_cast<uint64_t>(H), static_cast<uint64_t>(E),
                 static_cast<uint64_t>(H) * 2, RK, static_cast<uint32_t>(E), CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    const int ncols = E + (g ? 1 : 0);
    a.g = g;
    a.T = T;
    a.H = H;
    a.E = E;
    a.ld = ncols;
    a.tile_b = ((ncols + 15) & ~15) * RK * 2;
    const int fixed = 1024 + g_bytes(H, g != nullptr) + 256;
    a.stages = std::min(kMaxStages, (kSmemBudget - fixed) / (kTileA + a.tile_b));
    if (a.stages < 2) return cudaErrorInvalidValue;
    a.logits = logits;
    a.status = status;
    const size_t smem = static_cast<size_t>(fixed) + static_cast<size_t>(a.stages) * (kTileA + a.tile_b);
    static cudaError_t attr =
        cudaFuncSetAttribute(router_logits_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBudget);
    if (attr != cudaSuccess) return attr;
    KernelScope ks_("router_logits_tc", st);
    return launch_pdl(router_logits_tc_kernel, dim3((T + RM - 1) / RM, ksplit), dim3(192), smem, st, a);
}

}  // namespace moe
