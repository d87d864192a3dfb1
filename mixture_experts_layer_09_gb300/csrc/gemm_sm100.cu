// gemm_sm100.cu -- tensor arm of the expert MLP (prefill batches): grouped GEMMs on the
// 5th-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// Each expert's bucket of dispatched rows is cut into token tiles of up to 256 rows, balanced
// within the bucket (daScript PR #3988 "dasLLAMA vulkan: a MoE that fits the card ...",
// routed-block commit: the bucket schedule places the buckets and their tiles).  The A operand
// is int4 offset-binary weight rows with fp16 scales per 32 columns (colibri PR #418 "Vulkan
// backend: expert tier + dense + MLA attention on any Vulkan 1.2 GPU", Correctness and
// "Grouped scales in the Vulkan kernels"), expanded by producer warps into fp16
// (nibble - 8) * scale directly in the 128-byte-swizzled K-major layout the tensor core
// reads (MXFP4 rows, the fmt=7 format of the same PR: fp16 2v * 2^(e - 128) per e2m1 code,
// exact, chosen per work item); B is the tile's activation rows (fp16), brought in by TMA with
// the same swizzle; D = A * B^T accumulates in tensor memory (fp32), 128 lanes x N columns,
// N = tile rows rounded to 16.
//
// Gate/up (moe_gateup_kernel): one CTA per (128 features, token tile); gate and up are two
// accumulators of 256 columns, so the epilogue forms silu(g) * u (the fused gate+up+silu of
// colibri PR #418, Summary) and writes h in fp16, staged in shared memory and stored one token
// row per bulk copy.  Down (moe_down_kernel): persistent, one CTA per SM walking its work
// items; two 256-column accumulators let one item's epilogue run during the next item's main
// loop; the epilogue writes the unweighted rows (dispatch order), the rows weighted by their
// top-k weight in slot order (the tensor arm's combine feed), or the shared expert's rows
// scaled by sigmoid of its gate logit.  (The gate/up pair needs all 512 columns for one tile,
// so it cannot double-buffer at this tile size; pairing 64 gate with 64 up rows would fit in
// 256 columns but halves the work per pipeline stage, and measured slower.)
//
// Every mbarrier wait is bounded; a wait that runs out records MOE_ERR_DEVICE_TIMEOUT in the
// status word and every role of the CTA stops; the CTA drains its own copies and MMAs, frees
// its tensor memory and returns.
#include <cuda.h>

#include <algorithm>

#include "async.cuh"
#include "tcgen05.cuh"
#include "common.cuh"
#include "fp4.cuh"
#include "internal.h"

namespace moe {

constexpr int BM = 128;           // A rows per tile (MMA M)
constexpr int BN = kGemmTileN;    // tokens per tile (MMA N upper bound)
constexpr int BNB = 128;          // token rows per B TMA box
constexpr int BK = 64;            // K per pipeline stage: 128 bytes of fp16 per row
constexpr int kTileBytesA = BM * BK * 2;
constexpr int kTileBytesB = BN * BK * 2;
static_assert(BN <= 256 && BN % BNB == 0, "one MMA per K-slice, whole TMA boxes");

// gate/up kernel: 3 stages of (gate A, up A, B); 4 dequantising threads per A row
constexpr int kGuStages = 3;
constexpr int kGuStageBytes = 2 * kTileBytesA + kTileBytesB;
constexpr int kGuTpr = 4;
constexpr int kGuDqThreads = BM * kGuTpr;
constexpr int kGuThreads = 64 + kGuDqThreads;
constexpr int kGuPrefetch = 4;
// down kernel: 4 stages of (A, B); 2 dequantising threads per A row; 4 epilogue warps
constexpr int kDnStages = 4;
constexpr int kDnStageBytes = kTileBytesA + kTileBytesB;
constexpr int kDnTpr = 2;
constexpr int kDnDqThreads = BM * kDnTpr;
constexpr int kDnDqWarps = kDnDqThreads / 32;
constexpr int kDnEpiWarp0 = 2 + kDnDqWarps;
constexpr int kDnEpiThreads = 128;
constexpr int kDnThreads = 64 + kDnDqThreads + kDnEpiThreads;
constexpr int kDnPrefetch = 2;
constexpr int kAccCols = 256;     // tensor-memory columns of one down accumulator
constexpr int kEpiChunk = 32;     // down epilogue: token columns per tensor-memory load
constexpr int kBarEpi = 3;        // named barrier of the down epilogue warps

struct GemmK {
    CUtensorMap tm_r;     // B operand of routed tiles
    CUtensorMap tm_s;     // B operand of shared-expert tiles
    int T, k, E;
    int K_r, K_s;         // reduction length (H for gate/up, I or I_sh for down)
    int M_r, M_s;         // output features (I or I_sh for gate/up, H for down)
    int mblk_r, mblk_s;   // 128-row blocks of the output features
    int items_r;          // routed work items (ntile_max * mblk_r); shared items follow
    int items;            // all work items (the gate/up grid)
    int out_mode;         // down: 0 rows (unweighted, dispatch order), 1 weighted slots
    int fp4_r, fp4_s;     // MXFP4 codes (else int4) in the routed / shared matrices
    int sh_row0;          // B row of the first shared token in tm_s
    const int* tiles;     // [3 * ntile] (expert, first dispatch row, rows)
    const int* n_tiles;
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

struct Item {
    bool shared;
    int e, row0, nrows, mblk, K, M;
};

// Work item t: the shared expert's items first (the longest: full token tiles and, for down, the
// longest K), then the routed ones (tile-major, row blocks inner), so that the last wave holds
// short items.  False when the item is past the tile schedule or has no rows (every role skips
// it alike).
__device__ __forceinline__ bool item_at(const GemmK& p, int t, int n_tiles, Item& it) {
    const int n_sh = p.items - p.items_r;
    if (t >= n_sh) {
        const int rt = t - n_sh;
        const int tix = rt / p.mblk_r;
        if (tix >= n_tiles) return false;
        it.shared = false;
        it.mblk = rt % p.mblk_r;
        it.e = __ldg(p.tiles + 3 * tix);
        it.row0 = __ldg(p.tiles + 3 * tix + 1);
        it.nrows = __ldg(p.tiles + 3 * tix + 2);
        it.K = p.K_r;
        it.M = p.M_r;
    } else {
        const int tix = t / p.mblk_s;
        it.shared = true;
        it.mblk = t % p.mblk_s;
        it.e = -1;
        it.row0 = tix * BN;
        it.nrows = min(BN, p.T - it.row0);
        it.K = p.K_s;
        it.M = p.M_s;
    }
    return it.nrows > 0;
}

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

// One K-step (64 columns) of a thread's part of a weight row: CPT words of nibbles (8 columns
// each, CPT = 8 / threads per row) and the scale of their 32-column group.
template <int CPT>
struct RawK {
    uint32_t q[CPT];
    uint16_t s;
};

template <int CPT>
__device__ __forceinline__ RawK<CPT> load_raw(const uint8_t* qrow, const uint16_t* srow, int kb, int part, bool valid) {
    static_assert(CPT == 2 || CPT == 4, "a part stays inside one 32-column scale group");
    RawK<CPT> r;
    if (valid) {
        const uint8_t* src = qrow + kb * 32 + part * CPT * 4;
        if constexpr (CPT == 4) {
            const uint4 v = ldg_nc(src);
            r.q[0] = v.x; r.q[1] = v.y; r.q[2] = v.z; r.q[3] = v.w;
        } else {
            const uint2 v = __ldg(reinterpret_cast<const uint2*>(src));
            r.q[0] = v.x; r.q[1] = v.y;
        }
        r.s = __ldg(srow + kb * 2 + (part * CPT) / 4);
    } else {
#pragma unroll
        for (int j = 0; j < CPT; ++j) r.q[j] = 0x88888888u;  // all zero weights
        r.s = 0;
    }
    return r;
}

// Writes chunks part*CPT .. part*CPT+CPT-1 of `row` into a 128-byte-swizzled K-major tile;
// FP4: the words hold e2m1 codes (the same K order, fp4.cuh).
template <int CPT, bool FP4>
__device__ __forceinline__ void store_dequant(uint8_t* tile, int row, int part, const RawK<CPT>& r) {
    const __half2 s2 = __half2half2(__ushort_as_half(r.s));
    uint8_t* rowp = tile + row * 128;
#pragma unroll
    for (int j = 0; j < CPT; ++j) {
        const int c = part * CPT + j;
        *reinterpret_cast<uint4*>(rowp + ((c ^ (row & 7)) << 4)) = FP4 ? e2m1x8_to_f16(r.q[j], s2) : dequant8(r.q[j], s2);
    }
}

template <int CPT>
__device__ __forceinline__ void store_dequant(uint8_t* tile, int row, int part, const RawK<CPT>& r, bool fp4) {
    if (fp4)
        store_dequant<CPT, true>(tile, row, part, r);
    else
        store_dequant<CPT, false>(tile, row, part, r);
}

// TMA of a tile's B rows for one K-step: one 128-row box per lane (copies issued by one thread
// are served one after another), only the boxes that hold tile rows.  Called by a whole warp.
__device__ __forceinline__ void load_b_stage(uint8_t* dst, const CUtensorMap* tm, int kb, int brow, int nrows,
                                             uint64_t* bar, int lane) {
    const int nbox = (nrows + BNB - 1) / BNB;
    if (lane == 0) mbar_arrive_expect_tx(bar, nbox * BNB * BK * 2);
    __syncwarp();
    if (lane < nbox) tma_load_2d(dst + lane * BNB * 128, tm, kb * BK, brow + lane * BNB, bar);
}

// ------------------------------------------------------------------ gate + up (+ SwiGLU)
// One CTA per work item (128 features, token tile).  Warp 0 issues the TMA loads of B, warp 1
// owns the tensor memory and issues the MMAs (one thread), warps 2-17 dequantise the gate and
// up rows (four threads per row) and then run the epilogue (each warp one tensor-memory lane
// quadrant and a quarter of the token columns).
__global__ void __launch_bounds__(kGuThreads, 1) moe_gateup_kernel(const __grid_constant__ GemmK p) {
    pdl_wait();
    pdl_trigger();
    constexpr int S = kGuStages;
    constexpr int CPT = 8 / kGuTpr;
    // the workspace's test hook (zero in normal use): a shorter wait limit, and a token-tile copy
    // that the first CTA withholds so that its MMA thread's wait runs out
    const TestHook hook = *reinterpret_cast<const TestHook*>(reinterpret_cast<const char*>(p.status) + kWsTestHookOffset);
    const long long wl = hook.wait_limit > 0 ? hook.wait_limit : kWaitLimitCycles;
    const bool withhold = hook.withhold_copy != 0 && blockIdx.x == 0;
    Item w;
    if (!item_at(p, blockIdx.x, __ldg(p.n_tiles), w)) return;  // no rows: nothing to do
    const int nk = w.K / BK;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full_a = reinterpret_cast<uint64_t*>(smem + S * kGuStageBytes);
    uint64_t* full_b = full_a + S;
    uint64_t* empty = full_b + S;
    uint64_t* accum = empty + S;
    uint64_t* drain = accum + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_a + s, kGuDqThreads / 32);  // one arrival per dequantising warp
            mbar_init(full_b + s, 1);
            mbar_init(empty + s, 1);
        }
        mbar_init(accum, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) tmem_alloc(tmem_slot, 2 * BN);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    auto stage_a = [&](int s, int mat) { return smem + s * kGuStageBytes + mat * kTileBytesA; };
    auto stage_b = [&](int s) { return smem + s * kGuStageBytes + 2 * kTileBytesA; };

    if (warp == 0) {
        // ---------------- TMA producer of B
        const CUtensorMap* tm = w.shared ? &p.tm_s : &p.tm_r;
        const int brow = w.shared ? p.sh_row0 + w.row0 : w.row0;
        int issued = 0;
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % S;
            bool ok = true;
            if (kb >= S && lane == 0) ok = mbar_wait(empty + s, ((kb / S) & 1) ^ 1, abort_flag, p.status, 1, wl);
            if (!__shfl_sync(0xffffffffu, ok, 0)) break;
            if (!(withhold && kb == 1)) load_b_stage(stage_b(s), tm, kb, brow, w.nrows, full_b + s, lane);
            issued = kb + 1;
        }
        if (*abort_flag && lane == 0) {
            // let the copies this warp started land before the CTA leaves
            for (int kb = max(0, issued - S); kb < issued; ++kb) {
                const long long t0 = clock64();
                while (!mbar_try_wait(full_b + kb % S, (kb / S) & 1) && clock64() - t0 < wl) {
                }
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer: gate into columns 0.., up into columns BN..
        if (lane == 0) {
            const uint32_t idesc = idesc_f16_m128((w.nrows + 15) & ~15);
            bool any = false;
            for (int kb = 0; kb < nk; ++kb) {
                const int s = kb % S;
                const uint32_t par = (kb / S) & 1;
                if (!mbar_wait(full_b + s, par, abort_flag, p.status, 2, wl)) break;
                if (!mbar_wait(full_a + s, par, abort_flag, p.status, 3, wl)) break;
                tc_fence_after();
                const uint32_t b0 = smem_u32(stage_b(s));
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk) {
                    const uint64_t bd = sw128_kmajor_desc(b0 + kk * 32);
                    const uint32_t acc = (kb > 0 || kk > 0) ? 1u : 0u;
#pragma unroll
                    for (int mat = 0; mat < 2; ++mat)
                        mma_f16(tmem + mat * BN, sw128_kmajor_desc(smem_u32(stage_a(s, mat)) + kk * 32), bd, idesc, acc);
                }
                mma_commit(empty + s);
                any = true;
            }
            if (!*abort_flag) {
                mma_commit(accum);
            } else if (any) {
                mma_commit(drain);  // wait for this thread's MMAs before tensor memory is freed
                const long long t0 = clock64();
                while (!mbar_try_wait(drain, 0) && clock64() - t0 < wl) {
                }
            }
        }
    } else {
        // ---------------- gate and up producers (kGuTpr threads per feature), then the epilogue
        const int dt = threadIdx.x - 64;
        const int pr = dt / kGuTpr, part = dt % kGuTpr;  // feature within the block, part of its K-step
        const int f = w.mblk * BM + pr;
        const bool valid = f < w.M;
        const size_t grow = w.shared ? static_cast<size_t>(f) : static_cast<size_t>(w.e) * w.M + f;
        const uint8_t* qa = (w.shared ? p.qa_s : p.qa_r) + grow * (w.K / 2);
        const uint16_t* sa = (w.shared ? p.sa_s : p.sa_r) + grow * (w.K / 32);
        const uint8_t* qb = (w.shared ? p.qb_s : p.qb_r) + grow * (w.K / 2);
        const uint16_t* sb = (w.shared ? p.sb_s : p.sb_r) + grow * (w.K / 32);
        const bool fp4 = w.shared ? p.fp4_s : p.fp4_r;
        // raw weights kGuPrefetch K-steps ahead in registers; one lane per warp waits for a free
        // stage and one arrives for the warp (after __syncwarp orders the warp's writes)
        RawK<CPT> ra[kGuPrefetch], rb[kGuPrefetch];
#pragma unroll
        for (int d = 0; d < kGuPrefetch; ++d) {
            ra[d] = load_raw<CPT>(qa, sa, d, part, valid && d < nk);
            rb[d] = load_raw<CPT>(qb, sb, d, part, valid && d < nk);
        }
        bool ok = true;
        for (int kb0 = 0; kb0 < nk && ok; kb0 += kGuPrefetch) {
#pragma unroll
            for (int d = 0; d < kGuPrefetch; ++d) {
                const int kb = kb0 + d;
                if (kb >= nk) break;
                const int s = kb % S;
                if (kb >= S) {
                    bool free_ok = true;
                    if (lane == 0) free_ok = mbar_wait(empty + s, ((kb / S) & 1) ^ 1, abort_flag, p.status, 4, wl);
                    if (!__shfl_sync(0xffffffffu, free_ok, 0)) {
                        ok = false;
                        break;
                    }
                }
                store_dequant<CPT>(stage_a(s, 0), pr, part, ra[d], fp4);
                store_dequant<CPT>(stage_a(s, 1), pr, part, rb[d], fp4);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(full_a + s);
                if (kb + kGuPrefetch < nk) {
                    ra[d] = load_raw<CPT>(qa, sa, kb + kGuPrefetch, part, valid);
                    rb[d] = load_raw<CPT>(qb, sb, kb + kGuPrefetch, part, valid);
                }
            }
        }
        // ---------------- epilogue (tcgen05.ld is warp-collective: decide per warp).  The tile
        // is staged in the pipeline's shared memory (free once the accumulators are final) as
        // fp16 h in the down GEMM's K order, then each thread writes one token row by bulk copy.
        bool go = __all_sync(0xffffffffu, ok);
        if (go) go = __all_sync(0xffffffffu, mbar_wait(accum, 0, abort_flag, p.status, 5, wl));
        go = named_barrier_or(2, kGuDqThreads, !go) ? false : go;  // all epilogue warps agree
        if (go) {
            tc_fence_after();
            const int q = warp & 3;                 // tensor-memory lane quadrant of this warp
            const int m = q * 32 + lane;            // accumulator row = feature in the block
            const int ch = (warp - 2) >> 2;         // column share handled by this warp
            const uint32_t tbase = tmem + (static_cast<uint32_t>(q * 32) << 16);
            constexpr int kCols = BN / (kGuDqThreads / 128);
            const int cbeg = ch * kCols, cend = min(w.nrows, cbeg + kCols);
            uint16_t* stile = reinterpret_cast<uint16_t*>(smem);  // [BN][BM] fp16
            const int pos = (m & ~7) + kperm8(m & 7);
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
            fence_proxy_async_smem();  // the tile's generic writes, before the bulk copies read it
            named_barrier(2, kGuDqThreads);
            if (dt < w.nrows) {
                const int cols = min(BM, w.M - w.mblk * BM);
                uint16_t* hout = w.shared ? p.h_s : p.h_r;
                bulk_store(hout + static_cast<size_t>(w.row0 + dt) * w.M + w.mblk * BM, stile + dt * BM, cols * 2);
                bulk_store_wait();
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 2 * BN);
    }
}

// ------------------------------------------------------------------ down (persistent)
// One CTA per SM walks work items blockIdx.x, + gridDim.x, ...; item n accumulates into
// tensor-memory buffer n & 1.  Warp 0 issues the TMA loads of B; warp 1 owns the tensor memory
// and issues the MMAs (one thread); warps 2-9 dequantise A (two threads per row); warps 10-13
// run the epilogue, one tensor-memory lane quadrant each, storing straight from registers (a
// warp's 32 lanes are 32 consecutive output columns of one token row).
__global__ void __launch_bounds__(kDnThreads, 1) moe_down_kernel(const __grid_constant__ GemmK p) {
    pdl_wait();
    pdl_trigger();
    constexpr int S = kDnStages;
    constexpr int CPT = 8 / kDnTpr;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full_a = reinterpret_cast<uint64_t*>(smem + S * kDnStageBytes);
    uint64_t* full_b = full_a + S;
    uint64_t* empty = full_b + S;
    uint64_t* tfull = empty + S;   // [2] accumulator ready for the epilogue
    uint64_t* tempty = tfull + 2;  // [2] accumulator drained by the epilogue
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* row_out = const_cast<int*>(abort_flag) + 1;            // [2][BN] output row of each tile row
    float* row_w = reinterpret_cast<float*>(row_out + 2 * BN);  // [2][BN] its weight / shared gate

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_a + s, kDnDqWarps);  // one arrival per dequantising warp
            mbar_init(full_b + s, 1);
            mbar_init(empty + s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull + b, 1);
            mbar_init(tempty + b, kDnEpiThreads / 32);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) tmem_alloc(tmem_slot, 2 * kAccCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int n_tiles = __ldg(p.n_tiles);

    auto stage_a = [&](int s) { return smem + s * kDnStageBytes; };
    auto stage_b = [&](int s) { return smem + s * kDnStageBytes + kTileBytesA; };

    if (warp == 0) {
        // ---------------- TMA producer of B
        uint32_t it = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < p.items && ok; t += gridDim.x) {
            Item w;
            if (!item_at(p, t, n_tiles, w)) continue;
            const CUtensorMap* tm = w.shared ? &p.tm_s : &p.tm_r;
            const int brow = w.shared ? p.sh_row0 + w.row0 : w.row0;
            const int nk = w.K / BK;
            for (int kb = 0; kb < nk; ++kb) {
                const int s = it % S;
                if (it >= S && lane == 0) ok = mbar_wait(empty + s, ((it / S) & 1) ^ 1, abort_flag, p.status, 1);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                load_b_stage(stage_b(s), tm, kb, brow, w.nrows, full_b + s, lane);
                ++it;
            }
        }
        if (*abort_flag && lane == 0) {
            // let the copies this warp started land before the CTA leaves
            for (uint32_t j = it > static_cast<uint32_t>(S) ? it - S : 0; j < it; ++j) {
                const long long t0 = clock64();
                while (!mbar_try_wait(full_b + j % S, (j / S) & 1) && clock64() - t0 < kWaitLimitCycles) {
                }
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer
        if (lane == 0) {
            uint32_t it = 0, n = 0;
            bool ok = true, any = false;
            for (int t = blockIdx.x; t < p.items && ok; t += gridDim.x) {
                Item w;
                if (!item_at(p, t, n_tiles, w)) continue;
                const int b = n & 1;
                if (n >= 2 && !mbar_wait(tempty + b, ((n >> 1) & 1) ^ 1, abort_flag, p.status, 6)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t idesc = idesc_f16_m128((w.nrows + 15) & ~15);
                const uint32_t dacc = tmem + b * kAccCols;
                const int nk = w.K / BK;
                for (int kb = 0; kb < nk; ++kb) {
                    const int s = it % S;
                    const uint32_t par = (it / S) & 1;
                    if (!mbar_wait(full_b + s, par, abort_flag, p.status, 2) ||
                        !mbar_wait(full_a + s, par, abort_flag, p.status, 3)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(stage_a(s)), b0 = smem_u32(stage_b(s));
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        mma_f16(dacc, sw128_kmajor_desc(a0 + kk * 32), sw128_kmajor_desc(b0 + kk * 32), idesc,
                                (kb > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(empty + s);
                    any = true;
                    ++it;
                }
                if (!ok) break;
                mma_commit(tfull + b);
                ++n;
            }
            if (*abort_flag && any) {
                mma_commit(drain);  // wait for this thread's MMAs before tensor memory is freed
                const long long t0 = clock64();
                while (!mbar_try_wait(drain, 0) && clock64() - t0 < kWaitLimitCycles) {
                }
            }
        }
    } else if (warp < kDnEpiWarp0) {
        // ---------------- A producers (kDnTpr threads per row of W_d)
        const int dt = threadIdx.x - 64;
        const int pr = dt / kDnTpr, part = dt % kDnTpr;  // A row of the item, part of its K-step
        uint32_t it = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < p.items && ok; t += gridDim.x) {
            Item w;
            if (!item_at(p, t, n_tiles, w)) continue;
            const int wrow = w.mblk * BM + pr;
            const bool valid = wrow < w.M;
            const size_t grow = w.shared ? static_cast<size_t>(wrow) : static_cast<size_t>(w.e) * w.M + wrow;
            const uint8_t* qa = (w.shared ? p.qa_s : p.qa_r) + grow * (w.K / 2);
            const uint16_t* sa = (w.shared ? p.sa_s : p.sa_r) + grow * (w.K / 32);
            const bool fp4 = w.shared ? p.fp4_s : p.fp4_r;
            const int nk = w.K / BK;
            // raw weights kDnPrefetch K-steps ahead in registers; one lane per warp waits for a
            // free stage and one arrives for the warp (after __syncwarp orders its writes)
            RawK<CPT> ra[kDnPrefetch];
#pragma unroll
            for (int d = 0; d < kDnPrefetch; ++d) ra[d] = load_raw<CPT>(qa, sa, d, part, valid && d < nk);
            for (int kb0 = 0; kb0 < nk && ok; kb0 += kDnPrefetch) {
#pragma unroll
                for (int d = 0; d < kDnPrefetch; ++d) {
                    const int kb = kb0 + d;
                    if (kb >= nk) break;
                    const int s = it % S;
                    if (it >= S) {
                        bool free_ok = true;
                        if (lane == 0) free_ok = mbar_wait(empty + s, ((it / S) & 1) ^ 1, abort_flag, p.status, 4);
                        if (!__shfl_sync(0xffffffffu, free_ok, 0)) {
                            ok = false;
                            break;
                        }
                    }
                    store_dequant<CPT>(stage_a(s), pr, part, ra[d], fp4);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(full_a + s);
                    if (kb + kDnPrefetch < nk) ra[d] = load_raw<CPT>(qa, sa, kb + kDnPrefetch, part, valid);
                    ++it;
                }
            }
        }
    } else {
        // ---------------- epilogue: warp q = warp & 3 reads tensor-memory lanes 32q .. 32q+31
        const int et = threadIdx.x - 64 - kDnDqThreads;
        const int q = warp & 3, m = q * 32 + lane;
        uint32_t n = 0;
        for (int t = blockIdx.x; t < p.items; t += gridDim.x) {
            Item w;
            if (!item_at(p, t, n_tiles, w)) continue;
            const int b = n & 1;
            int* ro = row_out + b * BN;
            float* rw = row_w + b * BN;
            // the tile's output rows and weights, while the main loop runs (two copies: the
            // previous item's may still be in use by a slower epilogue warp)
            for (int i = et; i < w.nrows; i += kDnEpiThreads) {
                const int r = w.row0 + i;
                if (w.shared) {
                    float gate = 1.f;
                    if (p.sh_gate_logit)
                        gate = 1.f / (1.f + expf(-__ldg(p.sh_gate_logit + static_cast<size_t>(r) * p.logit_ld)));
                    ro[i] = r;
                    rw[i] = gate;
                } else if (p.out_mode == 1) {
                    const int a = __ldg(p.perm + r);
                    ro[i] = a;
                    rw[i] = __ldg(p.topk_w + a);
                } else {
                    ro[i] = r;
                    rw[i] = 1.f;
                }
            }
            bool ok = true;
            if (lane == 0) ok = mbar_wait(tfull + b, (n >> 1) & 1, abort_flag, p.status, 5);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (named_barrier_or(kBarEpi, kDnEpiThreads, !ok)) break;  // every epilogue warp stops alike
            tc_fence_after();
            const uint32_t tb = tmem + (static_cast<uint32_t>(q * 32) << 16) + b * kAccCols;
            const int col = w.mblk * BM + m;
            float* out = w.shared ? p.out_s : p.out_r;
            for (int c0 = 0; c0 < w.nrows; c0 += kEpiChunk) {
                const int nc = min(kEpiChunk, w.nrows - c0);
                float d[32];
                tmem_ld32(tb + c0, d);
                if (col < w.M) {
#pragma unroll
                    for (int cc = 0; cc < 32; ++cc)
                        if (cc < nc) out[static_cast<size_t>(ro[c0 + cc]) * w.M + col] = rw[c0 + cc] * d[cc];
                }
            }
            tc_fence_before();  // this warp's tensor-memory reads, before the buffer is handed back
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty + b);
            ++n;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 2 * kAccCols);
    }
}

// ------------------------------------------------------------------ small helpers
// Tile list from the bucket offsets, expert-major: a bucket of c rows takes ceil(c / BN) tiles
// of ceil(c / tiles) rows each (the last one may be shorter), so that no tile is a short tail
// that pays a whole pass over the expert's weights for a few rows.
__global__ void __launch_bounds__(256) build_tiles_kernel(const int32_t* __restrict__ offsets, int E,
                                                          int* __restrict__ tiles, int* __restrict__ n_tiles) {
    pdl_wait();
    pdl_trigger();
    __shared__ int warp_tot[8];
    const int e = threadIdx.x, lane = e & 31, w = e >> 5;
    const int cnt = (e < E) ? offsets[e + 1] - offsets[e] : 0;
    const int nt = (cnt + BN - 1) / BN;
    const int per = nt > 0 ? (cnt + nt - 1) / nt : 0;
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
        tiles[3 * (base + j)] = e;
        tiles[3 * (base + j) + 1] = offsets[e] + j * per;
        tiles[3 * (base + j) + 2] = max(0, min(per, cnt - j * per));
    }
}

// x16[r] = fp16(x[perm[r] / k]) for the T*k dispatched rows, then x16[T*k + t] = fp16(x[t]);
// each group of 8 columns is stored in the K order of the dequantised weight tiles.  One warp
// per row: lane l takes the 16-byte pieces l, l + 32, ..., four loads in flight before the
// stores.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint16_t* __restrict__ x,
                                                          const int32_t* __restrict__ perm, int T, int k, int H,
                                                          int with_tokens, uint16_t* __restrict__ x16) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int n_rows = T * k + (with_tokens ? T : 0);
    const int H8 = H / 8;
    const int nw = gridDim.x * (blockDim.x >> 5);
    for (int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < n_rows; r += nw) {
        int t = r - T * k;
        if (r < T * k) {
            int a = 0;
            if (lane == 0) a = __ldg(perm + r);
            t = __shfl_sync(0xffffffffu, a, 0) / k;
        }
        const uint16_t* src = x + static_cast<size_t>(t) * H;
        uint4* dst = reinterpret_cast<uint4*>(x16 + static_cast<size_t>(r) * H);
        for (int c0 = 0; c0 < H8; c0 += 4 * 32) {
            uint4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int c = c0 + u * 32 + lane;
                if (c < H8) v[u] = ldg_nc(src + static_cast<size_t>(c) * 8);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int c = c0 + u * 32 + lane;
                if (c >= H8) break;
                const uint32_t in[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
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
                dst[c] = make_uint4(out[0], out[1], out[2], out[3]);
            }
        }
    }
}

// ------------------------------------------------------------------ host side
// 2D fp16 tensor [rows][K], box = 64 x BN, 128-byte swizzle, zero fill outside.
static bool make_tmap(CUtensorMap* m, const void* base, int K, int rows) {
    return tmap_2d(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, base, static_cast<uint64_t>(K), static_cast<uint64_t>(rows),
                   static_cast<uint64_t>(K) * 2, BK, BNB, CU_TENSOR_MAP_SWIZZLE_128B);
}

int gemm_ntile_max(int n_slots, int E) { return (n_slots + BN - 1) / BN + E; }

bool gemm_supported(int H, int I, int I_sh) {
    return H % BK == 0 && I % BK == 0 && (I_sh <= 0 || I_sh % BK == 0);
}

static size_t gateup_smem_bytes() { return 1024 + static_cast<size_t>(kGuStages) * kGuStageBytes + 256; }

static size_t down_smem_bytes() {
    // stages | barriers, tensor-memory slot, abort flag | two row tables
    return 1024 + static_cast<size_t>(kDnStages) * kDnStageBytes + 256 + 2 * BN * 8;
}

static int sm_count() {
    static int n = [] {
        int dev = 0, v = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        return v > 0 ? v : 148;
    }();
    return n;
}

static cudaError_t set_smem_attrs() {
    static cudaError_t once = [] {
        cudaError_t e = cudaFuncSetAttribute(moe_gateup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(gateup_smem_bytes()));
        if (e != cudaSuccess) return e;
        return cudaFuncSetAttribute(moe_down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(down_smem_bytes()));
    }();
    return once;
}

cudaError_t launch_gemm_arm(const GemmPlan& p, bool rows_mode, cudaStream_t st) {
    cudaError_t err;
    const int n_slots = p.T * p.k;
    const bool has_sh = p.sh_I > 0;
    if ((err = set_smem_attrs()) != cudaSuccess) return err;
    // 1. activations in dispatch order (and token order for the shared expert), fp16
    {
        const long rows = n_slots + (has_sh ? p.T : 0);  // one warp per row, 8 per block
        long blocks = (rows + 7) / 8;
        if (blocks > static_cast<long>(sm_count()) * 8) blocks = static_cast<long>(sm_count()) * 8;
        if (blocks < 1) blocks = 1;
        {
            KernelScope ks_("gather_rows", st);
            err = launch_pdl(gather_rows_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st, p.x, p.perm,
                             p.T, p.k, p.H, has_sh ? 1 : 0, p.x16);
        }
    }
    // 2. tile schedule (unless the dispatch wrote it)
    if (!p.tiles_ready) {
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
    g.fp4_r = p.fp4_r;
    g.fp4_s = p.fp4_s;
    g.E = p.E;
    g.tiles = p.tiles;
    g.n_tiles = p.n_tiles;
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
    g.items_r = p.ntile_max * g.mblk_r;
    g.items = g.items_r + (has_sh ? p.sh_tiles * g.mblk_s : 0);
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
        KernelScope ks_("gemm_gateup", st);
        err = launch_pdl(moe_gateup_kernel, dim3(g.items), dim3(kGuThreads), gateup_smem_bytes(), st, g);
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
    d.items_r = p.ntile_max * d.mblk_r;
    d.items = d.items_r + (has_sh ? p.sh_tiles * d.mblk_s : 0);
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
        KernelScope ks_("gemm_down", st);
        err = launch_pdl(moe_down_kernel, dim3(std::min(d.items, sm_count())), dim3(kDnThreads), down_smem_bytes(),
                         st, d);
        if (err != cudaSuccess) return err;
    }
    return cudaSuccess;
}

}  // namespace moe
