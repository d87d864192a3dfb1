// gemm_sm100.cu -- tensor arm of the expert MLP (prefill batches): grouped GEMMs on the
// 5th-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// Each expert's bucket of dispatched rows is cut into tiles of up to 128 rows (daScript
// PR #3988 "dasLLAMA vulkan: a MoE that fits the card ...", routed-block commit: the bucket
// schedule places the buckets and their tiles; a tile with no rows returns at once).  A CTA
// computes one (weight row block of 128, token tile) pair:
//   A = 128 weight rows, int4 offset-binary with fp16 scales per 32 columns (colibri PR #418
//       "Vulkan backend: expert tier + dense + MLA attention on any Vulkan 1.2 GPU",
//       Correctness and "Grouped scales in the Vulkan kernels"), expanded by four producer
//       warps into fp16 (nibble - 8) * scale directly in the 128-byte-swizzled K-major
//       layout the tensor core reads;
//   B = the tile's activation rows (fp16), brought in by TMA with the same swizzle;
//   D = A * B^T in tensor memory (fp32), 128 lanes x N columns, N = tile rows rounded to 16.
// Gate and up run as two accumulators of one CTA, so the epilogue forms silu(g) * u (the
// fused gate+up+silu of colibri PR #418, Summary) and writes h in fp16.  The down GEMM's
// epilogue writes either the unweighted rows (dispatch order), the rows weighted by their
// top-k weight in slot order (the tensor arm's combine feed), or the shared expert's rows
// scaled by sigmoid of its gate logit.
//
// Roles in a CTA of 576 threads: warp 0 issues the TMA loads of B, warp 1 owns the tensor
// memory and issues the MMAs (one thread), warps 2-17 dequantise A (four threads per weight
// row: with one CTA per SM the dequantisation is latency-bound, so more warps carry it) and
// then run the epilogue (each warp one TMEM lane quadrant and a quarter of the columns).
// Every mbarrier wait is bounded; a wait that runs out records MOE_ERR_DEVICE_TIMEOUT in the
// status word, stops the CTA's loops, drains its own copies and MMAs, frees its tensor
// memory and returns.
#include <cuda.h>

#include "async.cuh"
#include "tcgen05.cuh"
#include "common.cuh"
#include "internal.h"

namespace moe {

constexpr int BM = 128;           // weight rows per tile (MMA M)
constexpr int BN = kGemmTileN;    // tokens per tile (MMA N upper bound)
constexpr int BK = 64;            // K per pipeline stage: 128 bytes of fp16 per row
constexpr int kTileBytesA = BM * BK * 2;
constexpr int kTileBytesB = BN * BK * 2;
constexpr int kStagesGU = 3;
constexpr int kStagesDN = 4;
#ifndef MOE_GEMM_TPR
#define MOE_GEMM_TPR 4
#endif
constexpr int kTpr = MOE_GEMM_TPR;              // dequantising threads per weight row
constexpr int kCpt = 8 / kTpr;                  // 16-byte chunks (8 K-columns) per thread per K-step
constexpr int kDqThreads = BM * kTpr;           // dequantising / epilogue threads (warps 2..)
constexpr int kPrefetch = 4;                    // K-steps of raw weights in flight per thread
constexpr int kGemmThreads = 64 + kDqThreads;   // + TMA warp + MMA warp

struct GemmK {
    CUtensorMap tm_r;     // B operand of routed tiles
    CUtensorMap tm_s;     // B operand of shared-expert tiles
    int T, k, E;
    int K_r, K_s;         // reduction length (H for gate/up, I or I_sh for down)
    int M_r, M_s;         // weight rows (I or I_sh for gate/up, H for down)
    int mblk_r, mblk_s;   // weight row blocks
    int ctas_r;           // routed CTAs in the grid (ntile_max * mblk_r)
    int out_mode;         // down: 0 rows (unweighted, dispatch order), 1 weighted slots
    int sh_row0;          // B row of the first shared token in tm_s
    const int* tiles;     // [2 * ntile] (expert, first dispatch row)
    const int* n_tiles;
    const int32_t* offsets;
    const int32_t* perm;
    const float* topk_w;
    const float* sh_gate_logit;
    int logit_ld;
    const uint8_t* qa_r;  // gate (gate/up) or down (down) of the routed experts
    const uint16_t* sa_r;
    const uint8_t* qb_r;  // up (gate/up only)
    const uint16_t* sb_r;
    const uint8_t* qa_s;
    const uint16_t* sa_s;
    const uint8_t* qb_s;
    const uint16_t* sb_s;
    uint16_t* h_r;        // gate/up out: fp16 [T*k][M_r]
    uint16_t* h_s;        // gate/up out: fp16 [T][M_s]
    float* out_r;         // down out: [T*k][H]
    float* out_s;         // down out: [T][H]
    int* status;
};


// 8 nibbles (columns 0..7 at bits 4c) times one fp16 scale -> 8 fp16 values, stored in the
// K order [c0 c4 c1 c5 c2 c6 c3 c7] (the activations are stored in the same order, so the
// product over K is unchanged and no byte permute is needed).
__device__ __forceinline__ uint4 dequant8(uint32_t w, __half2 s2) {
    const uint32_t t0 = (w & 0x000F000Fu) | 0x64006400u;          // c0, c4 as 1024 + n
    const uint32_t t1 = ((w >> 4) & 0x000F000Fu) | 0x64006400u;   // c1, c5
    const uint32_t t2 = ((w >> 8) & 0x000F000Fu) | 0x64006400u;   // c2, c6
    const uint32_t t3 = ((w >> 12) & 0x000F000Fu) | 0x64006400u;  // c3, c7
    const __half2 k1032 = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));
    uint4 out;
    __half2 v;
    v = __hmul2(__hsub2(*reinterpret_cast<const __half2*>(&t0), k1032), s2);
    out.x = *reinterpret_cast<uint32_t*>(&v);
    v = __hmul2(__hsub2(*reinterpret_cast<const __half2*>(&t1), k1032), s2);
    out.y = *reinterpret_cast<uint32_t*>(&v);
    v = __hmul2(__hsub2(*reinterpret_cast<const __half2*>(&t2), k1032), s2);
    out.z = *reinterpret_cast<uint32_t*>(&v);
    v = __hmul2(__hsub2(*reinterpret_cast<const __half2*>(&t3), k1032), s2);
    out.w = *reinterpret_cast<uint32_t*>(&v);
    return out;
}

// Position of column c (0..7) of an 8-column group in that K order.
__host__ __device__ constexpr inline int kperm8(int c) { return (c & 3) * 2 + (c >> 2); }

// One K-step (64 columns) of a thread's part of a weight row: kCpt words of nibbles (8 columns
// each) and the scale of their group (a part never straddles two 32-column groups).
struct RawK {
    uint32_t q[kCpt];
    uint16_t s;
};

__device__ __forceinline__ RawK load_raw(const uint8_t* qrow, const uint16_t* srow, int kb, int part, bool valid) {
    RawK r;
    if (valid) {
        const uint8_t* src = qrow + kb * 32 + part * kCpt * 4;
        if constexpr (kCpt == 4) {
            const uint4 v = ldg_nc(src);
            r.q[0] = v.x; r.q[1] = v.y; r.q[2] = v.z; r.q[3] = v.w;
        } else {
            const uint2 v = __ldg(reinterpret_cast<const uint2*>(src));
            r.q[0] = v.x; r.q[1] = v.y;
        }
        r.s = __ldg(srow + kb * 2 + (part * kCpt) / 4);
    } else {
#pragma unroll
        for (int j = 0; j < kCpt; ++j) r.q[j] = 0x88888888u;  // all zero weights
        r.s = 0;
    }
    return r;
}

// Writes chunks part*kCpt .. part*kCpt+kCpt-1 of `row` into a 128-byte-swizzled K-major tile.
__device__ __forceinline__ void store_dequant(uint8_t* tile, int row, int part, const RawK& r) {
    const __half2 s2 = __half2half2(__ushort_as_half(r.s));
    uint8_t* rowp = tile + row * 128;
#pragma unroll
    for (int j = 0; j < kCpt; ++j) {
        const int c = part * kCpt + j;
        *reinterpret_cast<uint4*>(rowp + ((c ^ (row & 7)) << 4)) = dequant8(r.q[j], s2);
    }
}

template <int MODE>  // 0 = gate+up (two accumulators, SwiGLU epilogue), 1 = down
__global__ void __launch_bounds__(kGemmThreads, 1) moe_gemm_kernel(const __grid_constant__ GemmK p) {
    pdl_wait();
    pdl_trigger();
    constexpr int S = MODE == 0 ? kStagesGU : kStagesDN;
    constexpr int NMAT = MODE == 0 ? 2 : 1;
    constexpr int kStageBytes = NMAT * kTileBytesA + kTileBytesB;
    constexpr uint32_t kTmemCols = MODE == 0 ? 2 * BN : BN;

    // ---- which tile this CTA computes
    const bool shared = static_cast<int>(blockIdx.x) >= p.ctas_r;
    int e, row0, nrows, mblk, K, M;
    if (!shared) {
        const int tix = blockIdx.x / p.mblk_r;
        mblk = blockIdx.x % p.mblk_r;
        if (tix >= *p.n_tiles) return;  // tile beyond the schedule: nothing to do
        e = p.tiles[2 * tix];
        row0 = p.tiles[2 * tix + 1];
        nrows = min(BN, p.offsets[e + 1] - row0);
        K = p.K_r;
        M = p.M_r;
    } else {
        const int sid = blockIdx.x - p.ctas_r;
        const int tix = sid / p.mblk_s;
        mblk = sid % p.mblk_s;
        e = -1;
        row0 = tix * BN;
        nrows = min(BN, p.T - row0);
        K = p.K_s;
        M = p.M_s;
    }
    if (nrows <= 0) return;
    const int nk = K / BK;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full_a = reinterpret_cast<uint64_t*>(smem + S * kStageBytes);
    uint64_t* full_b = full_a + S;
    uint64_t* empty = full_b + S;
    uint64_t* accum = empty + S;
    uint64_t* drain = accum + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* row_slot = const_cast<int*>(abort_flag) + 1;           // [BN] down: slot of each tile row
    float* row_w = reinterpret_cast<float*>(row_slot + BN);     // [BN] down: its weight / shared gate

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_a + s, kDqThreads / 32);  // one arrival per dequantising warp
            mbar_init(full_b + s, 1);
            mbar_init(empty + s, 1);
        }
        mbar_init(accum, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    auto stage_a = [&](int s, int mat) { return smem + s * kStageBytes + mat * kTileBytesA; };
    auto stage_b = [&](int s) { return smem + s * kStageBytes + NMAT * kTileBytesA; };

    if (warp == 0) {
        // ---------------- TMA producer of B
        if (lane == 0) {
            const CUtensorMap* tm = shared ? &p.tm_s : &p.tm_r;
            const int brow = shared ? p.sh_row0 + row0 : row0;
            int issued = 0;
            for (int kb = 0; kb < nk; ++kb) {
                const int s = kb % S;
                if (kb >= S && !mbar_wait(empty + s, ((kb / S) & 1) ^ 1, abort_flag, p.status, 1)) break;
                mbar_arrive_expect_tx(full_b + s, kTileBytesB);
                tma_load_2d(stage_b(s), tm, kb * BK, brow, full_b + s);
                issued = kb + 1;
            }
            if (*abort_flag) {
                // let the copies this thread started land before the CTA leaves
                for (int kb = max(0, issued - S); kb < issued; ++kb) {
                    const long long t0 = clock64();
                    while (!mbar_try_wait(full_b + kb % S, (kb / S) & 1) && clock64() - t0 < kWaitLimitCycles) {
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer
        if (lane == 0) {
            const int nmma = (nrows + 15) & ~15;
            const uint32_t idesc = idesc_f16_m128(nmma);
            bool any = false;
            for (int kb = 0; kb < nk; ++kb) {
                const int s = kb % S;
                const uint32_t par = (kb / S) & 1;
                if (!mbar_wait(full_b + s, par, abort_flag, p.status, 2)) break;
                if (!mbar_wait(full_a + s, par, abort_flag, p.status, 3)) break;
                tc_fence_after();
                const uint32_t b0 = smem_u32(stage_b(s));
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk) {
                    const uint64_t bd = sw128_kmajor_desc(b0 + kk * 32);
                    const uint32_t acc = (kb > 0 || kk > 0) ? 1u : 0u;
#pragma unroll
                    for (int mat = 0; mat < NMAT; ++mat) {
                        const uint64_t ad = sw128_kmajor_desc(smem_u32(stage_a(s, mat)) + kk * 32);
                        mma_f16(tmem + mat * BN, ad, bd, idesc, acc);
                    }
                }
                mma_commit(empty + s);
                any = true;
            }
            if (!*abort_flag) {
                mma_commit(accum);
            } else if (any) {
                mma_commit(drain);  // wait for this thread's MMAs before tensor memory is freed
                const long long t0 = clock64();
                while (!mbar_try_wait(drain, 0) && clock64() - t0 < kWaitLimitCycles) {
                }
            }
        }
    } else {
        // ---------------- A producers (8 warps: two threads per weight row), then the epilogue
        const int dt = threadIdx.x - 64;
        const int pr = dt / kTpr, half = dt % kTpr;  // weight row within the block, part of its K-step
        const int wrow = mblk * BM + pr;        // weight row within the matrix
        const bool valid = wrow < M;
        const size_t grow = shared ? static_cast<size_t>(wrow) : static_cast<size_t>(e) * M + wrow;
        const uint8_t* qa = (shared ? p.qa_s : p.qa_r) + grow * (K / 2);
        const uint16_t* sa = (shared ? p.sa_s : p.sa_r) + grow * (K / 32);
        const uint8_t* qb = nullptr;
        const uint16_t* sb = nullptr;
        if (MODE == 0) {
            qb = (shared ? p.qb_s : p.qb_r) + grow * (K / 2);
            sb = (shared ? p.sb_s : p.sb_r) + grow * (K / 32);
        }
        if (MODE == 1) {
            // the epilogue's per-row data, loaded now so it is not on the epilogue's path
            if (dt < nrows) {
                const int r = row0 + dt;
                if (shared) {
                    float gate = 1.f;
                    if (p.sh_gate_logit) gate = 1.f / (1.f + expf(-__ldg(p.sh_gate_logit + static_cast<size_t>(r) * p.logit_ld)));
                    row_slot[dt] = r;
                    row_w[dt] = gate;
                } else if (p.out_mode == 1) {  // weighted slot rows; rows mode needs no table
                    const int a = __ldg(p.perm + r);
                    row_slot[dt] = a;
                    row_w[dt] = __ldg(p.topk_w + a);
                }
            }
        }
        // raw weights kPrefetch K-steps ahead in registers; one lane per warp waits for a free
        // stage and one arrives for the warp (after __syncwarp orders the warp's writes), so
        // that 256 threads do not poll and arrive on one barrier word every K-step
        RawK ra[kPrefetch], rb[kPrefetch];
#pragma unroll
        for (int d = 0; d < kPrefetch; ++d) {
            ra[d] = load_raw(qa, sa, d, half, valid && d < nk);
            if (MODE == 0) rb[d] = load_raw(qb, sb, d, half, valid && d < nk);
        }
        bool ok = true;
        for (int kb0 = 0; kb0 < nk && ok; kb0 += kPrefetch) {
#pragma unroll
            for (int d = 0; d < kPrefetch; ++d) {
                const int kb = kb0 + d;
                if (kb >= nk) break;
                const int s = kb % S;
                if (kb >= S) {
                    bool free_ok = true;
                    if (lane == 0) free_ok = mbar_wait(empty + s, ((kb / S) & 1) ^ 1, abort_flag, p.status, 4);
                    if (!__shfl_sync(0xffffffffu, free_ok, 0)) {
                        ok = false;
                        break;
                    }
                }
                store_dequant(stage_a(s, 0), pr, half, ra[d]);
                if (MODE == 0) store_dequant(stage_a(s, 1), pr, half, rb[d]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(full_a + s);
                if (kb + kPrefetch < nk) {
                    ra[d] = load_raw(qa, sa, kb + kPrefetch, half, valid);
                    if (MODE == 0) rb[d] = load_raw(qb, sb, kb + kPrefetch, half, valid);
                }
            }
        }
        named_barrier(2, kDqThreads);  // row_slot / row_w visible to every epilogue thread
        // ---------------- epilogue (tcgen05.ld is warp-collective: decide per warp)
        // The tile is staged in the pipeline's shared memory (free once the accumulators are
        // final): row c = token row of the tile, 128 output columns; then each thread writes
        // one token row with a bulk copy.  Gate/up stage fp16 h in the down GEMM's K order,
        // down stages fp32 (weighted) outputs bound for the row's slot or token.
        bool go = __all_sync(0xffffffffu, ok);
        if (go) go = __all_sync(0xffffffffu, mbar_wait(accum, 0, abort_flag, p.status, 5));
        go = named_barrier_or(2, kDqThreads, !go) ? false : go;  // all epilogue warps agree
        if (go) {
            tc_fence_after();
            const int q = warp & 3;                 // tensor-memory lane quadrant of this warp
            const int m = q * 32 + lane;            // accumulator row = weight row in the block
            const int ch = (warp - 2) >> 2;         // column share handled by this warp
            const uint32_t tbase = tmem + (static_cast<uint32_t>(q * 32) << 16);
            constexpr int kCols = BN / (kDqThreads / 128);
            const int cbeg = ch * kCols, cend = min(nrows, cbeg + kCols);
            if (MODE == 0) {
                uint16_t* stile = reinterpret_cast<uint16_t*>(smem);           // [BN][BM] fp16
                const int pos = (m & ~7) + kperm8(m & 7);                     // K order of the down GEMM
                for (int c0 = cbeg; c0 < cend; c0 += 32) {
                    float g[32], u[32];
                    tmem_ld32x2(tbase + c0, tbase + BN + c0, g, u);
#pragma unroll
                    for (int cc = 0; cc < 32; ++cc) {
                        if (c0 + cc < cend) {
                            const float h = __fdividef(g[cc] * u[cc], 1.f + __expf(-g[cc]));
                            stile[(c0 + cc) * BM + pos] = __half_as_ushort(__float2half_rn(h));
                        }
                    }
                }
            } else {
                float* stile = reinterpret_cast<float*>(smem);                 // [BN][BM] fp32
                const bool weighted = shared || p.out_mode == 1;
                for (int c0 = cbeg; c0 < cend; c0 += 32) {
                    float d[32];
                    tmem_ld32(tbase + c0, d);
#pragma unroll
                    for (int cc = 0; cc < 32; ++cc) {
                        if (c0 + cc < cend) stile[(c0 + cc) * BM + m] = weighted ? row_w[c0 + cc] * d[cc] : d[cc];
                    }
                }
            }
            fence_proxy_async_smem();  // the tile's generic writes, before the bulk copies read it
            named_barrier(2, kDqThreads);
            if (dt < nrows) {
                const int cols = min(BM, M - mblk * BM);
                if (MODE == 0) {
                    uint16_t* hout = shared ? p.h_s : p.h_r;
                    bulk_store(hout + static_cast<size_t>(row0 + dt) * M + mblk * BM,
                               reinterpret_cast<const uint16_t*>(smem) + dt * BM, cols * 2);
                } else {
                    const size_t orow = shared ? static_cast<size_t>(row0 + dt)
                                               : (p.out_mode == 1 ? static_cast<size_t>(row_slot[dt])
                                                                  : static_cast<size_t>(row0 + dt));
                    float* out = shared ? p.out_s : p.out_r;
                    bulk_store(out + orow * M + mblk * BM, reinterpret_cast<const float*>(smem) + dt * BM, cols * 4);
                }
                bulk_store_wait();
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------------------------------------------ small helpers
// Tile list from the bucket offsets: tiles of up to BN rows per expert, expert-major.
__global__ void __launch_bounds__(256) build_tiles_kernel(const int32_t* __restrict__ offsets, int E,
                                                          int* __restrict__ tiles, int* __restrict__ n_tiles) {
    pdl_wait();
    pdl_trigger();
    __shared__ int warp_tot[8];
    const int e = threadIdx.x, lane = e & 31, w = e >> 5;
    const int cnt = (e < E) ? offsets[e + 1] - offsets[e] : 0;
    const int nt = (cnt + BN - 1) / BN;
    int incl = nt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) warp_tot[w] = incl;
    __syncthreads();
    int base = incl - nt;
    for (int i = 0; i < w; ++i) base += warp_tot[i];
    if (e == 255) *n_tiles = base + nt;
    for (int j = 0; j < nt; ++j) {
        tiles[2 * (base + j)] = e;
        tiles[2 * (base + j) + 1] = offsets[e] + j * BN;
    }
}

// x16[r] = fp16(x[perm[r] / k]) for the T*k dispatched rows, then x16[T*k + t] = fp16(x[t]);
// each group of 8 columns is stored in the K order of the dequantised weight tiles.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint16_t* __restrict__ x,
                                                          const int32_t* __restrict__ perm, int T, int k, int H,
                                                          int with_tokens, uint16_t* __restrict__ x16) {
    pdl_wait();
    pdl_trigger();
    const int n_rows = T * k + (with_tokens ? T : 0);
    const int H8 = H / 8;
    const long total = static_cast<long>(n_rows) * H8;
    for (long i = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<long>(gridDim.x) * blockDim.x) {
        const int r = static_cast<int>(i / H8), c = static_cast<int>(i % H8);
        const int t = (r < T * k) ? __ldg(perm + r) / k : r - T * k;
        const uint4 v = ldg_nc(x + static_cast<size_t>(t) * H + c * 8);
        const uint32_t in[4] = {v.x, v.y, v.z, v.w};
        uint16_t h[8];  // columns 0..7 as fp16
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            h[2 * j] = __half_as_ushort(__float2half_rn(__uint_as_float(in[j] << 16)));
            h[2 * j + 1] = __half_as_ushort(__float2half_rn(__uint_as_float(in[j] & 0xffff0000u)));
        }
        // stored in the GEMM's K order [c0 c4 c1 c5 c2 c6 c3 c7]
        uint32_t out[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) out[j] = static_cast<uint32_t>(h[j]) | (static_cast<uint32_t>(h[j + 4]) << 16);
        reinterpret_cast<uint4*>(x16 + static_cast<size_t>(r) * H)[c] = make_uint4(out[0], out[1], out[2], out[3]);
    }
}

// ------------------------------------------------------------------ host side
// 2D fp16 tensor [rows][K], box = 64 x BN, 128-byte swizzle, zero fill outside.
static bool make_tmap(CUtensorMap* m, const void* base, int K, int rows) {
    return tmap_2d(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, base, static_cast<uint64_t>(K), static_cast<uint64_t>(rows),
                   static_cast<uint64_t>(K) * 2, BK, BN, CU_TENSOR_MAP_SWIZZLE_128B);
}

int gemm_ntile_max(int n_slots, int E) { return (n_slots + BN - 1) / BN + E; }

bool gemm_supported(int H, int I, int I_sh) {
    return H % BK == 0 && I % BK == 0 && (I_sh <= 0 || I_sh % BK == 0);
}

template <int MODE>
static size_t gemm_smem_bytes() {
    constexpr int S = MODE == 0 ? kStagesGU : kStagesDN;
    constexpr int NMAT = MODE == 0 ? 2 : 1;
    return static_cast<size_t>(S) * (NMAT * kTileBytesA + kTileBytesB) + 1024 + 256 + 8 * BN;
}

template <int MODE>
static cudaError_t set_smem_attr() {
    static cudaError_t once = cudaFuncSetAttribute(moe_gemm_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(gemm_smem_bytes<MODE>()));
    return once;
}

cudaError_t launch_gemm_arm(const GemmPlan& p, bool rows_mode, cudaStream_t st) {
    cudaError_t err;
    const int n_slots = p.T * p.k;
    const bool has_sh = p.sh_I > 0;
    if ((err = set_smem_attr<0>()) != cudaSuccess) return err;
    if ((err = set_smem_attr<1>()) != cudaSuccess) return err;
    // 1. activations in dispatch order (and token order for the shared expert), fp16
    {
        const long total = static_cast<long>(n_slots + (has_sh ? p.T : 0)) * (p.H / 8);
        long blocks = (total + 255) / 256;
        if (blocks > 152L * 8) blocks = 152L * 8;
        if (blocks < 1) blocks = 1;
        {
            KernelScope ks_("gather_rows", st);
            err = launch_pdl(gather_rows_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st, p.x, p.perm,
                             p.T, p.k, p.H, has_sh ? 1 : 0, p.x16);
        }
    }
    // 2. tile schedule
    {
        KernelScope ks_("build_tiles", st);
        if (err == cudaSuccess)
            err = launch_pdl(build_tiles_kernel, dim3(1), dim3(256), 0, st, static_cast<const int32_t*>(p.offsets), p.E,
                             p.tiles, p.n_tiles);
    }
    if (err != cudaSuccess) return err;

    // 3. gate + up
    GemmK g{};
    g.T = p.T;
    g.k = p.k;
    g.E = p.E;
    g.tiles = p.tiles;
    g.n_tiles = p.n_tiles;
    g.offsets = p.offsets;
    g.perm = p.perm;
    g.topk_w = p.topk_w;
    g.sh_gate_logit = p.sh_gate_logit;
    g.logit_ld = p.logit_ld;
    g.status = p.status;
    g.K_r = p.H;
    g.K_s = p.H;
    g.M_r = p.I;
    g.M_s = has_sh ? p.sh_I : BM;
    g.mblk_r = (p.I + BM - 1) / BM;
    g.mblk_s = has_sh ? (p.sh_I + BM - 1) / BM : 1;
    g.ctas_r = p.ntile_max * g.mblk_r;
    g.sh_row0 = n_slots;
    if (!make_tmap(&g.tm_r, p.x16, p.H, n_slots + (has_sh ? p.T : 0))) return cudaErrorInvalidValue;
    g.tm_s = g.tm_r;
    g.qa_r = p.gate_q;
    g.sa_r = p.gate_s;
    g.qb_r = p.up_q;
    g.sb_r = p.up_s;
    g.qa_s = p.sh_gate_q;
    g.sa_s = p.sh_gate_s;
    g.qb_s = p.sh_up_q;
    g.sb_s = p.sh_up_s;
    g.h_r = p.h16;
    g.h_s = p.sh_h16;
    {
        const int ctas = g.ctas_r + (has_sh ? p.sh_tiles * g.mblk_s : 0);
        {
            KernelScope ks_("gemm_gateup", st);
            err = launch_pdl(moe_gemm_kernel<0>, dim3(ctas), dim3(kGemmThreads), gemm_smem_bytes<0>(), st, g);
        }
        if (err != cudaSuccess) return err;
    }
    // 4. down (+ weighting / shared gate in the epilogue)
    GemmK d = g;
    d.K_r = p.I;
    d.K_s = has_sh ? p.sh_I : BK;
    d.M_r = p.H;
    d.M_s = p.H;
    d.mblk_r = (p.H + BM - 1) / BM;
    d.mblk_s = d.mblk_r;
    d.ctas_r = p.ntile_max * d.mblk_r;
    d.sh_row0 = 0;
    d.out_mode = rows_mode ? 0 : 1;
    if (!make_tmap(&d.tm_r, p.h16, p.I, n_slots)) return cudaErrorInvalidValue;
    if (has_sh) {
        if (!make_tmap(&d.tm_s, p.sh_h16, p.sh_I, p.T)) return cudaErrorInvalidValue;
    } else {
        d.tm_s = d.tm_r;
    }
    d.qa_r = p.down_q;
    d.sa_r = p.down_s;
    d.qb_r = nullptr;
    d.sb_r = nullptr;
    d.qa_s = p.sh_down_q;
    d.sa_s = p.sh_down_s;
    d.qb_s = nullptr;
    d.sb_s = nullptr;
    d.out_r = rows_mode ? p.rows_out : p.slot_out;
    d.out_s = p.sh_out;
    {
        const int ctas = d.ctas_r + (has_sh ? p.sh_tiles * d.mblk_s : 0);
        {
            KernelScope ks_("gemm_down", st);
            err = launch_pdl(moe_gemm_kernel<1>, dim3(ctas), dim3(kGemmThreads), gemm_smem_bytes<1>(), st, d);
        }
        if (err != cudaSuccess) return err;
    }
    return cudaSuccess;
}

}  // namespace moe
