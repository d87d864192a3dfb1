// gemv.cu -- bandwidth arm of the expert MLP (decode batches): fused int4 GEMVs.
//
// The expert weights are int4 offset-binary (value = nibble - 8) with one fp16 scale per 32
// K-columns, uploaded in the CPU byte layout (colibri PR #418 "Vulkan backend: expert tier +
// dense + MLA attention on any Vulkan 1.2 GPU", Correctness and "Grouped scales in the Vulkan
// kernels": the scale is applied to the packed-word partial).  A 16-byte chunk of a weight
// row is 32 nibbles = exactly one scale group, so the partial of a chunk is
//     sum_c (n_c - 8) * a_c  =  sum_c n_c * a_c  -  8 * sum_c a_c
// and the group scale multiplies that partial.  Activations a (hidden rows x; the SwiGLU
// product h for the down projection) are held as int16 with one power-of-two scale per 32
// values, so sum_c n_c * a_c is an exact integer dot product (dp2a: two int16 by two 8-bit
// nibbles per instruction).  The only rounding is the activation's: bf16 hidden values within
// 2^7 of their group's largest magnitude convert exactly, smaller ones round at 2^-15 of it;
// h rounds at 2^-15 of its group's largest magnitude.
// MXFP4 matrices (e2m1 codes, the fmt=7 format of colibri PR #418's Kimi K3 tier) take the same
// path: a chunk's codes expand to the signed bytes 2v (fp4.cuh), the dot product stays exact,
// there is no offset term, and the upload-expanded scale 2^(e - 128) multiplies the partial.
// The format is per matrix set (routed or shared), chosen per stage.
//
// Work layout (both kernels): a CTA owns 32 consecutive weight rows of one expert; each of its
// 8 warps owns 4 of them, with 8 lanes per row splitting the row's chunks, so every 128-bit
// load instruction of a warp reads 4 rows x 128 contiguous bytes.
//   gateup_gemv   g = W_g x, u = W_u x for the expert's bucket, h = silu(g) * u; the 32 rows
//                 of a CTA are one quantisation group of h, so h is written directly as int16
//                 with its scale and integer sum.
//   down_gemv     o = W_d h for the bucket.  Mode ROWS writes o per dispatched row; mode
//                 COMBINE writes w * o per (token, slot) and the gated shared row, and the
//                 last CTA to finish a block of 32 output columns sums, per token, the shared
//                 row, then the slots in order j, then the residual (daScript PR #3988
//                 "dasLLAMA vulkan: a MoE that fits the card ...", combine-folded residual
//                 commit) -- the combine runs inside the down projection's launch.
// The shared expert, when present, is one more expert whose bucket is every token.
#include <algorithm>

#include "async.cuh"
#include "common.cuh"
#include "fp4.cuh"
#include "internal.h"
#include "quant.cuh"

namespace moe {


// ------------------------------------------------------------------ activation quantisation
struct QuantSeg {
    const void* src;  // bf16 (is_bf16) or fp32 rows [rows][K]
    int is_bf16;
    int rows, K;
    int16_t* q;       // [rows][K], dp2a order within each 8-column word
    int2* meta;       // [rows][gld] {scale bits, integer sum}
    int gld;          // group row stride (>= K/32)
    int kc;           // slice width of the stored order
};

__global__ void __launch_bounds__(256) quantize_rows_kernel(QuantSeg s0, QuantSeg s1) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    long gw = (static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const long n0 = static_cast<long>(s0.rows) * (s0.K / 32);
    const long n1 = static_cast<long>(s1.rows) * (s1.K / 32);
    QuantSeg s = s0;
    if (gw >= n0) {
        gw -= n0;
        if (gw >= n1) return;  // whole warp leaves together
        s = s1;
    }
    const int ng = s.K / 32;
    const long row = gw / ng;
    const int grp = static_cast<int>(gw % ng);
    const size_t idx = static_cast<size_t>(row) * s.K + grp * 32 + lane;
    const float v = s.is_bf16 ? bf16_to_f32(static_cast<const uint16_t*>(s.src)[idx])
                              : static_cast<const float*>(s.src)[idx];
    quantize_group(v, lane, s.q + static_cast<size_t>(row) * act_row(s.K), grp, s.kc, s.meta + row * s.gld + grp);
}

cudaError_t launch_quantize(const QuantArgs& a, cudaStream_t st) {
    QuantSeg s0{a.src0, a.src0_bf16, a.rows0, a.K0, a.q0, a.meta0, a.gld0 ? a.gld0 : a.K0 / 32, a.kc0};
    QuantSeg s1{a.src1, a.src1_bf16, a.rows1, a.K1, a.q1, a.meta1, a.gld1 ? a.gld1 : a.K1 / 32, a.kc1};
    if (!a.src1) { s1.rows = 0; s1.K = 32; }
    const long warps = static_cast<long>(s0.rows) * (s0.K / 32) + static_cast<long>(s1.rows) * (s1.K / 32);
    if (warps == 0) return cudaSuccess;
    const long blocks = (warps + 7) / 8;
    KernelScope ks_("quantize_rows", st);
    return launch_pdl(quantize_rows_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st, s0, s1);
}

// ------------------------------------------------------------------ int4 x int16 chunk dot
struct Nib {  // one 16-byte weight chunk split into its even and odd nibble bytes
    uint32_t lo[4], hi[4];
};

__device__ __forceinline__ Nib split_nibbles(const uint4 w) {
    Nib n;
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        n.lo[m] = ww[m] & 0x0F0F0F0Fu;          // columns 8m + 0, 2, 4, 6
        n.hi[m] = (ww[m] >> 4) & 0x0F0F0F0Fu;   // columns 8m + 1, 3, 5, 7
    }
    return n;
}

// The same split of an MXFP4 chunk: signed bytes 2v of the e2m1 codes (no offset to remove).
__device__ __forceinline__ Nib split_e2m1(const uint4 w) {
    Nib n;
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int m = 0; m < 4; ++m) e2m1x8_to_i8(ww[m], n.lo[m], n.hi[m]);
    return n;
}

template <bool FP4>
__device__ __forceinline__ Nib split_chunk(const uint4 w) {
    if constexpr (FP4)
        return split_e2m1(w);
    else
        return split_nibbles(w);
}

// sum over the 32 columns of a chunk of nibble * activation; a = 32 int16 in dp2a order.
// Four independent accumulators (one per 8-column word) keep the dp2a chains short.
__device__ __forceinline__ int dot_nib(const Nib& n, const uint4 (&a)[4]) {
    int acc[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        acc[m] = __dp2a_lo(static_cast<int>(a[m].x), static_cast<int>(n.lo[m]), 0);
        acc[m] = __dp2a_hi(static_cast<int>(a[m].y), static_cast<int>(n.lo[m]), acc[m]);
        acc[m] = __dp2a_lo(static_cast<int>(a[m].z), static_cast<int>(n.hi[m]), acc[m]);
        acc[m] = __dp2a_hi(static_cast<int>(a[m].w), static_cast<int>(n.hi[m]), acc[m]);
    }
    return (acc[0] + acc[1]) + (acc[2] + acc[3]);
}

__device__ __forceinline__ void load_act(const int16_t* p, uint4 (&a)[4]) {
    const uint4* q = reinterpret_cast<const uint4*>(p);
#pragma unroll
    for (int m = 0; m < 4; ++m) a[m] = __ldg(q + m);
}

__device__ __forceinline__ float silu(float z) { return z / (1.f + expf(-z)); }

__device__ __forceinline__ float f16_to_f32(uint16_t b) { return __half2float(__ushort_as_half(b)); }

// Sum over the 8 lanes that share a row (lanes 8q .. 8q+7).
__device__ __forceinline__ float row_sum8(float v) {
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    v += __shfl_xor_sync(0xffffffffu, v, 4);
    return v;
}


// ------------------------------------------------------------------ pipelined GEMV kernels
// Persistent CTAs, two per SM.  Work is a list of tasks -- (expert, block of 32 weight rows)
// -- split into contiguous ranges, one per CTA.  A producer warp walks its range and streams
// each task in K-slices into a ring of shared-memory stages: TMA boxes of the 32 weight rows
// (256 bytes x 32 rows per box) and of their fp16 scales, one bulk copy per bucket token of
// its int16 activation slice and one of its {scale, sum} pairs, and a small header (task,
// pass, token rows, slots, weights) written before the stage's mbarrier arrive.  Eight
// consumer warps then work from shared memory only: warp w owns rows 4w .. 4w+3 of the task,
// 8 lanes per row, lane % 8 taking chunks lane % 8, +8, +16, ... of the slice, so one weight
// read covers 4 rows x 128 contiguous bytes and a row's sum meets by three shuffles.
//
// MODE 0 (gate/up): g = W_g x, u = W_u x, h = silu(g) * u; the 32 rows of a task are one
//   quantisation group of h, so h is written as int16 with its scale and integer sum.
// MODE 1 (down, combine): o = W_d h; w * o goes to the slot-ordered term buffer (the gated
//   shared row to its own buffer).  Tasks run in column-block-major order; when a CTA leaves a
//   block of 32 output columns it publishes how many of the block's tasks it did, and the CTA
//   completing the block sums per token the shared row, the slots in order j and the residual
//   (daScript PR #3988 "dasLLAMA vulkan: a MoE that fits the card ...", combine-folded
//   residual commit).
// MODE 2 (down, rows): o per dispatched row, unweighted.
// The shared expert is one more expert whose bucket is every token.

constexpr int kBoxB = 256;  // bytes of one weight TMA box row (512 K-columns)
constexpr int kCW = 8;      // consumer warps
// producer lanes issuing a stage's copies: weight boxes from lane 0, scale boxes, activation
// slices and their {scale, sum} pairs from these lanes on (one copy per lane)
constexpr int kLaneScale = 8, kLaneAct = 16, kLaneMeta = 24;

template <int MODE>
struct Pipe {
    static constexpr int NMAT = (MODE == 0) ? 2 : 1;
    static constexpr int KC = (MODE == 0) ? kSliceX : kSliceH;  // K columns per slice
    static constexpr int NBOX = KC / 2 / kBoxB;         // weight boxes per matrix per slice
    static constexpr int CPL = KC / 32 / 8;             // chunks per lane per slice
    static constexpr int TB = 4;                         // tokens per pass
    static constexpr int GRP = KC / 32;                  // scale groups per slice
    static constexpr int WMAT = 32 * KC / 2;             // bytes of one matrix's slice
    static constexpr int OFF_WS = NMAT * WMAT;
    static constexpr int OFF_A = OFF_WS + NMAT * 32 * GRP * 2;
    static constexpr int OFF_AM = OFF_A + TB * KC * 2;
    static constexpr int OFF_HDR = OFF_AM + TB * GRP * 8;
    // the boxes are unswizzled, so stage bases need 128-byte alignment only; four stages of
    // either mode leave room for two CTAs per SM
    static constexpr int STAGE = (OFF_HDR + 256 + 127) / 128 * 128;
    static constexpr int STAGES = 4;
    static_assert(OFF_WS % 128 == 0 && OFF_A % 128 == 0 && OFF_AM % 16 == 0, "copy destinations aligned");
    static_assert(NMAT * NBOX <= kLaneScale && TB == 4, "one copy per producer lane; four tokens per pass");
};

struct StageHdr {
    int end;            // 1: no more work for this CTA
    int shared, e, rb;  // task
    int K, t0, nb;      // reduction length, first bucket row of the pass, tokens in the pass
    int first, last;    // first / last slice of the pass
    int task_end;       // this pass is the task's last
    int sl;             // slice index
    int arow[4];        // activation rows (tokens for gate/up, dispatch rows or tokens for down)
    int slot[4];        // MODE 1 routed: slot a = perm[row]
    float wgt[4];       // MODE 1: top-k weight of the slot, or the shared gate
};

struct TaskDesc {
    bool shared;
    int e, rb, K, b0, b1, wrow;
    int arow0[4], slot0[4];  // the first pass's tokens: activation rows and (down) slots
    float wgt0[4];           // and (down) their weights or the shared gate
};

// Activation row, slot and weight of bucket row r of a task (r < b1).
template <int MODE>
__device__ __forceinline__ void pass_row(const GemvArgs& p, bool shared, int r, int& arow, int& slot, float& wgt) {
    slot = 0;
    wgt = 0.f;
    if (MODE == 0) {
        arow = shared ? r : __ldg(p.perm + r) / p.k;
    } else {
        arow = r;
        if (shared) {
            wgt = 1.f;
            if (p.sh_gate_logit) wgt = 1.f / (1.f + expf(-__ldg(p.sh_gate_logit + static_cast<size_t>(r) * p.logit_ld)));
        } else if (MODE == 1) {
            slot = __ldg(p.perm + r);
            wgt = __ldg(p.topk_w + slot);
        }
    }
}

template <int MODE>
__device__ __forceinline__ void task_desc(const GemvArgs& p, int t, int n_act, int nrb, TaskDesc& tk) {
    const int routed = n_act * nrb;
    const int rows_per_expert = (MODE == 0) ? p.I : p.H;
    if (t < routed) {
        tk.shared = false;
        tk.rb = t % nrb;
        tk.e = __ldg(p.active + t / nrb);
        tk.b0 = __ldg(p.offsets + tk.e);
        tk.b1 = __ldg(p.offsets + tk.e + 1);
        tk.K = (MODE == 0) ? p.H : p.I;
        tk.wrow = tk.e * rows_per_expert + tk.rb * 32;
    } else {
        tk.shared = true;
        tk.e = -1;
        tk.rb = t - routed;
        tk.b0 = 0;
        tk.b1 = p.T;
        tk.K = (MODE == 0) ? p.H : p.sh_I;
        tk.wrow = tk.rb * 32;
    }
    // the first pass's per-token loads now, with the descriptor, not on the producer's path
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        tk.arow0[i] = 0;
        tk.slot0[i] = 0;
        tk.wgt0[i] = 0.f;
        if (tk.b0 + i < tk.b1) pass_row<MODE>(p, tk.shared, tk.b0 + i, tk.arow0[i], tk.slot0[i], tk.wgt0[i]);
    }
}

// MODE 1: publish `cnt` finished tasks of column block cb; the CTA that completes the block
// sums, per token, the shared row, the slots in order and the residual, then resets the counter.
__device__ __forceinline__ void combine_flush(const GemvArgs& p, int cb, int cnt, int n_act, int* last_flag) {
    // the consumers' term stores happen before thread 0's fence (barrier), and the fence orders
    // them before the count (release); the completing CTA fences after reading the count (acquire)
    named_barrier(1, kCW * 32);
    if (threadIdx.x == 0) {
        const int expected = n_act + (p.sh_I > 0 ? 1 : 0);
        __threadfence();
        *last_flag = (atomicAdd(p.col_counter + cb, cnt) + cnt == expected);
        __threadfence();
    }
    named_barrier(1, kCW * 32);
    if (*last_flag) {
        __threadfence();
        const int H = p.H;
        // every term's load is issued before the sum (eight slots at a time), and the adds keep
        // the order shared, slots 0..k-1, residual
        for (int idx = threadIdx.x; idx < p.T * 32; idx += kCW * 32) {
            const int tt = idx >> 5, nn = cb * 32 + (idx & 31);
            const size_t at = static_cast<size_t>(tt) * H + nn;
            float y = (p.sh_I > 0) ? __ldcg(p.sh_term + at) : 0.f;
            const float res = p.residual ? bf16_to_f32(p.residual[at]) : 0.f;
            const float* slots = p.slot_term + static_cast<size_t>(tt) * p.k * H + nn;
            for (int j0 = 0; j0 < p.k; j0 += 8) {
                float v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) v[u] = (j0 + u < p.k) ? __ldcg(slots + static_cast<size_t>(j0 + u) * H) : 0.f;
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (j0 + u < p.k) y += v[u];
            }
            if (p.residual) y += res;
            p.y[at] = y;
        }
        if (threadIdx.x == 0) p.col_counter[cb] = 0;  // ready for the next call
    }
    named_barrier(1, kCW * 32);
}

// One slice with staged scales for NB tokens: chunks ks, ks + 8, ... below nch (a slice
// shorter than KC, as the last or only slice of a short K, ends early; when nch is a multiple
// of 8 every lane stops at the same chunk).
template <int MODE, int NB, bool FP4>
__device__ __forceinline__ void stage_dot(const uint8_t* st, int ks, int lrow, int nch,
                                          float (&acc)[Pipe<MODE>::TB][Pipe<MODE>::NMAT]) {
    using P = Pipe<MODE>;
    constexpr int NMAT = P::NMAT;
#pragma unroll
    for (int j = 0; j < P::CPL; ++j) {
        const int c = ks + 8 * j;
        if (c >= nch) break;
        Nib nw[NMAT];
        float fs[NMAT];
#pragma unroll
        for (int m = 0; m < NMAT; ++m) {
            nw[m] = split_chunk<FP4>(
                *reinterpret_cast<const uint4*>(st + m * P::WMAT + (c >> 4) * 32 * kBoxB + lrow * kBoxB + (c & 15) * 16));
            fs[m] = f16_to_f32(*reinterpret_cast<const uint16_t*>(st + P::OFF_WS + (m * 32 + lrow) * P::GRP * 2 + c * 2));
        }
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            uint4 av[4];
            const uint4* ap = reinterpret_cast<const uint4*>(st + P::OFF_A + b * P::KC * 2);
#pragma unroll
            for (int q = 0; q < 4; ++q) av[q] = ap[((c >> 3) * 4 + q) * 8 + (c & 7)];
            const int2 amv = reinterpret_cast<const int2*>(st + P::OFF_AM)[b * P::GRP + c];
            const float asc = __int_as_float(amv.x);
            const int off = FP4 ? 0 : 8 * amv.y;  // int4: sum of (n - 8) a = sum n a - 8 sum a
#pragma unroll
            for (int m = 0; m < NMAT; ++m)
                acc[b][m] = fmaf(static_cast<float>(dot_nib(nw[m], av) - off), fs[m] * asc, acc[b][m]);
        }
    }
}

// Down projection with the folded combine: this CTA's contiguous range [first, last) of the
// column-block-major task list (block cb: one task of each active expert, then the shared
// one), cut at equal shares of the estimated work.  A task costs about (4 + tokens) per pass
// of up to four tokens and per K-slice, so every block costs the same and a cut point maps to
// (block, expert) by one count over the experts' cost prefix.  Runs on the producer warp;
// n_act <= 256 (eight experts per lane).
__device__ __forceinline__ void balanced_range(const GemvArgs& p, int n_act, int nrb, int nsh, int lane, int& first,
                                               int& last) {
    constexpr int KC = Pipe<1>::KC;
    const long long nsl_r = (p.I + KC - 1) / KC;
    long long pre[8];  // exclusive cost prefix within the lane
    long long mine = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int a = lane * 8 + i;
        pre[i] = mine;
        if (a < n_act) {
            const int e = __ldg(p.active + a);
            const int cnt = __ldg(p.offsets + e + 1) - __ldg(p.offsets + e);
            mine += nsl_r * (4 * ((cnt + 3) / 4) + cnt);
        }
    }
    long long incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    const long long base = incl - mine;
    const long long routed = __shfl_sync(0xffffffffu, incl, 31);
    long long W = routed;
    if (nsh > 0) W += static_cast<long long>((p.sh_I + KC - 1) / KC) * (4 * ((p.T + 3) / 4) + p.T);
    if (W <= 0) W = 1;
    const long long C = W * nrb;
    const int per_cb = n_act + (nsh > 0 ? 1 : 0);
    auto cut = [&](long long pos) -> int {  // first task whose start cost is >= pos
        if (pos >= C) return nrb * per_cb;
        const long long cb = pos / W, rem = pos - cb * W;
        int n = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) n += (lane * 8 + i < n_act && base + pre[i] < rem) ? 1 : 0;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) n += __shfl_xor_sync(0xffffffffu, n, o);
        if (nsh > 0 && routed < rem) ++n;  // the shared expert's task
        return static_cast<int>(cb) * per_cb + n;
    };
    first = cut(C * blockIdx.x / gridDim.x);
    last = cut(C * (blockIdx.x + 1) / gridDim.x);
}

template <int MODE>
__global__ void __launch_bounds__((kCW + 1) * 32, 2) gemv_pipe_kernel(const __grid_constant__ GemvArgs p) {
    using P = Pipe<MODE>;
    constexpr int NMAT = P::NMAT, S = P::STAGES, TB = P::TB;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * P::STAGE);
    uint64_t* empty = full + S;
    float* red = reinterpret_cast<float*>(empty + S);  // MODE 0: [TB][2][32]
    volatile int* abort_flag = reinterpret_cast<volatile int*>(red + TB * 2 * 32);
    int* last_flag = const_cast<int*>(abort_flag) + 1;

    // set-up that reads nothing an earlier kernel writes runs before the dependency wait, during
    // the previous kernel's tail: the stage barriers and the TMA descriptors this mode uses
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, kCW);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kCW && lane == 0) {
        if (MODE == 0) {
            prefetch_tmap(&p.tm_gate);
            prefetch_tmap(&p.tm_up);
            prefetch_tmap(&p.tm_gate_s);
            prefetch_tmap(&p.tm_up_s);
            prefetch_tmap(&p.tm_sh_gate);
            prefetch_tmap(&p.tm_sh_up);
            prefetch_tmap(&p.tm_sh_gate_s);
            prefetch_tmap(&p.tm_sh_up_s);
        } else {
            prefetch_tmap(&p.tm_down);
            prefetch_tmap(&p.tm_down_s);
            prefetch_tmap(&p.tm_sh_down);
            prefetch_tmap(&p.tm_sh_down_s);
        }
    }
    __syncthreads();
    pdl_wait();
    pdl_trigger();

    if (warp == kCW) {
        // ---------------- producer
        const int n_act = *p.n_active;
        const int nrb = (MODE == 0) ? p.I / 32 : p.H / 32;
        const int nsh = (p.sh_I > 0) ? ((MODE == 0) ? p.sh_I / 32 : p.H / 32) : 0;
        const int ntask = n_act * nrb + nsh;
        const int per_cb = n_act + (nsh > 0 ? 1 : 0);
        // Gate/up (and the rows-mode down) claim chunks of tasks from a counter in the workspace
        // head, the next chunk claimed while the current one streams, the first chunk implied by
        // the CTA index: tasks differ in token count, and a fixed split left the slowest CTA far
        // behind the mean.  The down projection with the folded combine instead walks one
        // contiguous column-block-major range per CTA (it leaves each block at most once), cut by
        // estimated cost above four tokens and by task count below.
        int* next_ctr = p.task_counter + (MODE == 0 ? 0 : 2);
        int* done_ctr = next_ctr + 1;
        int CH, q0, r_last = ntask;
        if (MODE == 1) {
            if (p.T > 4) {
                balanced_range(p, n_act, nrb, nsh, lane, q0, r_last);
            } else {
                const int len = (ntask + gridDim.x - 1) / gridDim.x;
                q0 = min(ntask, static_cast<int>(blockIdx.x) * len);
                r_last = min(ntask, q0 + len);
            }
            CH = 32;
        } else {
            CH = max(1, min(32, ntask / (static_cast<int>(gridDim.x) * 8)));
            q0 = static_cast<int>(blockIdx.x) * CH;
        }
        uint32_t it = 0;
        while (q0 < r_last && !*abort_flag) {
          int qn = q0 + CH;
          if (MODE != 1) {
              if (lane == 0) qn = atomicAdd(next_ctr, CH) + static_cast<int>(gridDim.x) * CH;
          }
          const int last = min(r_last, q0 + CH);
          // the warp's lanes look up the chunk's task descriptors at once
          TaskDesc mine{};
          if (q0 + lane < last) {
              // MODE 1 walks column-block-major (block cb: experts in order, then the shared one)
              int t = q0 + lane;
              if (MODE == 1) {
                  const int cb = t / per_cb, a = t % per_cb;
                  t = a < n_act ? a * nrb + cb : n_act * nrb + cb;
              }
              task_desc<MODE>(p, t, n_act, nrb, mine);
          }
          const int wn = last - q0;
          for (int j = 0; j < wn && !*abort_flag; ++j) {
            TaskDesc tk;
            tk.shared = __shfl_sync(0xffffffffu, static_cast<int>(mine.shared), j);
            tk.e = __shfl_sync(0xffffffffu, mine.e, j);
            tk.rb = __shfl_sync(0xffffffffu, mine.rb, j);
            tk.K = __shfl_sync(0xffffffffu, mine.K, j);
            tk.b0 = __shfl_sync(0xffffffffu, mine.b0, j);
            tk.b1 = __shfl_sync(0xffffffffu, mine.b1, j);
            tk.wrow = __shfl_sync(0xffffffffu, mine.wrow, j);
            const CUtensorMap* tw[2];
            const CUtensorMap* ts[2];
            const int16_t* aq;
            const int2* am;
            int ag_ld, ws;
            if (MODE == 0) {
                tw[0] = tk.shared ? &p.tm_sh_gate : &p.tm_gate;
                tw[1] = tk.shared ? &p.tm_sh_up : &p.tm_up;
                ts[0] = tk.shared ? &p.tm_sh_gate_s : &p.tm_gate_s;
                ts[1] = tk.shared ? &p.tm_sh_up_s : &p.tm_up_s;
                ws = tk.shared ? p.ws_sh_gu : p.ws_gu;
                aq = p.xq; am = p.xmeta; ag_ld = p.x_gld;
            } else {
                tw[0] = tw[1] = tk.shared ? &p.tm_sh_down : &p.tm_down;
                ts[0] = ts[1] = tk.shared ? &p.tm_sh_down_s : &p.tm_down_s;
                ws = tk.shared ? p.ws_sh_d : p.ws_d;
                aq = tk.shared ? p.sh_hq : p.hq;
                am = tk.shared ? p.sh_hmeta : p.hmeta;
                ag_ld = tk.shared ? p.sh_gld : p.h_gld;
            }
            const int nsl = (tk.K + P::KC - 1) / P::KC;
            // the first pass's token data from the descriptor lane: lane b takes token b
            int farow = 0, fslot = 0;
            float fwgt = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int va = __shfl_sync(0xffffffffu, mine.arow0[i], j);
                const int vs = __shfl_sync(0xffffffffu, mine.slot0[i], j);
                const float vw = __shfl_sync(0xffffffffu, mine.wgt0[i], j);
                if (lane == i) {
                    farow = va;
                    fslot = vs;
                    fwgt = vw;
                }
            }
            for (int t0 = tk.b0; t0 < tk.b1 && !*abort_flag; t0 += TB) {
                const int nb = min(TB, tk.b1 - t0);
                int arow = farow, slot = fslot;
                float wgt = fwgt;
                if (t0 != tk.b0 && lane < nb) pass_row<MODE>(p, tk.shared, t0 + lane, arow, slot, wgt);
                for (int sl = 0; sl < nsl; ++sl, ++it) {
                    const int s = it % S;
                    if (it >= static_cast<uint32_t>(S)) {
                        // one lane waits; the warp takes its answer (uniform control flow)
                        bool ok = true;
                        if (lane == 0) ok = mbar_wait(empty + s, ((it / S) & 1) ^ 1, abort_flag, p.status, 11);
                        ok = __shfl_sync(0xffffffffu, ok, 0);
                        __syncwarp();
                        if (!ok) break;
                    }
                    uint8_t* st = smem + s * P::STAGE;
                    StageHdr* hd = reinterpret_cast<StageHdr*>(st + P::OFF_HDR);
                    if (lane == 0) {
                        hd->end = 0; hd->shared = tk.shared; hd->e = tk.e; hd->rb = tk.rb; hd->K = tk.K;
                        hd->t0 = t0; hd->nb = nb; hd->first = (sl == 0); hd->last = (sl == nsl - 1); hd->sl = sl;
                        hd->task_end = (t0 + TB >= tk.b1);
                    }
                    if (lane < nb) {
                        hd->arow[lane] = arow;
                        hd->slot[lane] = slot;
                        hd->wgt[lane] = wgt;
                    }
                    __syncwarp();
                    const int cols = min(P::KC, tk.K - sl * P::KC);
                    const uint32_t ab = act_row(cols) * 2;          // whole groups of 8 chunks
                    const uint32_t mb = ((cols / 32 + 3) & ~3) * 8;  // {scale, sum} pairs, padded
                    if (lane == 0) {
                        const uint32_t bytes = NMAT * (P::WMAT + (ws ? 32 * P::GRP * 2 : 0)) + nb * (ab + mb);
                        mbar_arrive_expect_tx(full + s, bytes);  // release: the header is visible
                    }
                    __syncwarp();
                    // every copy of the stage from its own lane: one thread's copies are served one
                    // after another, copies from different threads overlap
                    const int brow = __shfl_sync(0xffffffffu, arow, lane & 3);
                    if (lane < NMAT * P::NBOX) {
                        const int m = lane / P::NBOX, bx = lane % P::NBOX;
                        tma_load_2d(st + m * P::WMAT + bx * 32 * kBoxB, tw[m], sl * (P::KC / 2) + bx * kBoxB, tk.wrow,
                                    full + s);
                    } else if (lane >= kLaneScale && lane < kLaneScale + NMAT) {
                        const int m = lane - kLaneScale;
                        if (ws) tma_load_2d(st + P::OFF_WS + m * 32 * P::GRP * 2, ts[m], sl * P::GRP, tk.wrow, full + s);
                    } else if (lane >= kLaneAct && lane < kLaneAct + nb) {
                        const int b = lane - kLaneAct;
                        bulk_load(st + P::OFF_A + b * P::KC * 2,
                                  aq + static_cast<size_t>(brow) * act_row(tk.K) + sl * P::KC, ab, full + s);
                    } else if (lane >= kLaneMeta && lane < kLaneMeta + nb) {
                        const int b = lane - kLaneMeta;
                        bulk_load(st + P::OFF_AM + b * P::GRP * 8, am + static_cast<size_t>(brow) * ag_ld + sl * P::GRP,
                                  mb, full + s);
                    }
                }
            }
          }
          q0 = (MODE == 1) ? qn : __shfl_sync(0xffffffffu, qn, 0);
        }
        if (MODE != 1 && lane == 0) {
            // the last CTA to stop claiming puts the counter back to zero for the next call
            __threadfence();
            if (atomicAdd(done_ctr, 1) == static_cast<int>(gridDim.x) - 1) {
                atomicExch(next_ctr, 0);
                atomicExch(done_ctr, 0);
            }
        }
        // closing stage: a header with end = 1 and no copies
        if (!*abort_flag) {
            const int s = it % S;
            if (lane == 0 &&
                (it < static_cast<uint32_t>(S) || mbar_wait(empty + s, ((it / S) & 1) ^ 1, abort_flag, p.status, 13))) {
                reinterpret_cast<StageHdr*>(smem + s * P::STAGE + P::OFF_HDR)->end = 1;
                mbar_arrive_expect_tx(full + s, 0);
            }
            ++it;
        }
        if (*abort_flag && lane == 0) {
            // let the copies this warp started land before the CTA leaves (bounded)
            const uint32_t f0 = it > static_cast<uint32_t>(S) ? it - S : 0;
            for (uint32_t j = f0; j < it; ++j) {
                const long long c0 = clock64();
                while (!mbar_try_wait(full + j % S, (j / S) & 1) && clock64() - c0 < kWaitLimitCycles) {
                }
            }
        }
        return;
    }

    // ---------------- consumers
    const int ks = lane & 7;
    const int lrow = 4 * warp + (lane >> 3);  // row of the task owned by this lane group
    // scale rows for the direct path (when the scale rows cannot be staged by TMA)
    const int n_act_c = (MODE == 1) ? *p.n_active : 0;
    int run_cb = -1, run_cnt = 0;
    float acc[TB][NMAT];
    uint32_t it = 0;
    for (;; ++it) {
        const int s = it % S;
        bool ok = true;
        if (lane == 0) {
            ok = mbar_wait(full + s, (it / S) & 1, abort_flag, p.status, 12);
            if (!ok) {
                // grace wait: if the stage does complete, every consumer warp goes on together,
                // so no warp can be left alone at a named barrier; otherwise they all stop here
                const long long c0 = clock64();
                while (!(ok = mbar_try_wait(full + s, (it / S) & 1)) && clock64() - c0 < kWaitLimitCycles / 32) {
                }
            }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        __syncwarp();  // lane 0's acquire of the stage is ordered before the warp's reads
        const uint8_t* st = smem + s * P::STAGE;
        const StageHdr* hd = reinterpret_cast<const StageHdr*>(st + P::OFF_HDR);
        if (!ok || hd->end) break;
        const int nb = hd->nb, K = hd->K, sl = hd->sl;
        if (MODE == 1 && hd->rb != run_cb) {
            if (run_cb >= 0) combine_flush(p, run_cb, run_cnt, n_act_c, last_flag);
            run_cb = hd->rb;
            run_cnt = 0;
        }
        if (hd->first) {
#pragma unroll
            for (int b = 0; b < TB; ++b)
#pragma unroll
                for (int m = 0; m < NMAT; ++m) acc[b][m] = 0.f;
        }
        const bool ws = hd->shared ? ((MODE == 0) ? p.ws_sh_gu : p.ws_sh_d) : ((MODE == 0) ? p.ws_gu : p.ws_d);
        const bool fp4 = hd->shared ? p.fp4_s : p.fp4_r;
        const int nch = min(P::KC, K - sl * P::KC) / 32;
        if (ws && !fp4) {
            // staged scales: specialised on the token count
            switch (nb) {
                case 1: stage_dot<MODE, 1, false>(st, ks, lrow, nch, acc); break;
                case 2: stage_dot<MODE, 2, false>(st, ks, lrow, nch, acc); break;
                case 3: stage_dot<MODE, 3, false>(st, ks, lrow, nch, acc); break;
                default: stage_dot<MODE, 4, false>(st, ks, lrow, nch, acc); break;
            }
        } else if (ws) {
            switch (nb) {
                case 1: stage_dot<MODE, 1, true>(st, ks, lrow, nch, acc); break;
                case 2: stage_dot<MODE, 2, true>(st, ks, lrow, nch, acc); break;
                case 3: stage_dot<MODE, 3, true>(st, ks, lrow, nch, acc); break;
                default: stage_dot<MODE, 4, true>(st, ks, lrow, nch, acc); break;
            }
        } else {
#pragma unroll
            for (int j = 0; j < P::CPL; ++j) {
                const int c = ks + 8 * j;  // chunk within the slice
                if (c < nch) {
                    Nib nw[NMAT];
                    float fs[NMAT];
#pragma unroll
                    for (int m = 0; m < NMAT; ++m) {
                        const uint4 wv = *reinterpret_cast<const uint4*>(st + m * P::WMAT + (c >> 4) * 32 * kBoxB +
                                                                         lrow * kBoxB + (c & 15) * 16);
                        nw[m] = fp4 ? split_e2m1(wv) : split_nibbles(wv);
                        uint16_t sb;
                        if (ws) {
                            sb = *reinterpret_cast<const uint16_t*>(st + P::OFF_WS + (m * 32 + lrow) * P::GRP * 2 + c * 2);
                        } else {
                            const uint16_t* srow;
                            const int rows_pe = (MODE == 0) ? p.I : p.H;
                            if (MODE == 0)
                                srow = hd->shared ? (m ? p.sh_up_s : p.sh_gate_s) : (m ? p.up_s : p.gate_s);
                            else
                                srow = hd->shared ? p.sh_down_s : p.down_s;
                            const size_t wrow = hd->shared ? static_cast<size_t>(hd->rb) * 32 + lrow
                                                           : static_cast<size_t>(hd->e) * rows_pe + hd->rb * 32 + lrow;
                            sb = __ldg(srow + wrow * (K / 32) + sl * P::GRP + c);
                        }
                        fs[m] = f16_to_f32(sb);
                    }
#pragma unroll
                    for (int b = 0; b < TB; ++b) {
                        if (b < nb) {
                            uint4 av[4];
                            const uint4* ap = reinterpret_cast<const uint4*>(st + P::OFF_A + b * P::KC * 2);
#pragma unroll
                            for (int q = 0; q < 4; ++q) av[q] = ap[((c >> 3) * 4 + q) * 8 + (c & 7)];
                            const int2 amv = reinterpret_cast<const int2*>(st + P::OFF_AM)[b * P::GRP + c];
                            const float asc = __int_as_float(amv.x);
                            const int off = fp4 ? 0 : 8 * amv.y;
#pragma unroll
                            for (int m = 0; m < NMAT; ++m)
                                acc[b][m] = fmaf(static_cast<float>(dot_nib(nw[m], av) - off), fs[m] * asc, acc[b][m]);
                        }
                    }
                }
            }
        }
        // copy what the epilogue needs out of the header before the stage is released
        const bool last = hd->last, shared = hd->shared, task_end = hd->task_end;
        const int rb = hd->rb, t0 = hd->t0;
        int slot[TB];
        float wgt[TB];
#pragma unroll
        for (int b = 0; b < TB; ++b) {
            slot[b] = hd->slot[b];
            wgt[b] = hd->wgt[b];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty + s);
        if (!last) continue;
        // ---- end of a pass
        if (MODE == 0) {
#pragma unroll
            for (int b = 0; b < TB; ++b) {
                if (b >= nb) break;  // the pass's token count (warp-uniform)
#pragma unroll
                for (int m = 0; m < NMAT; ++m) {
                    const float v = row_sum8(acc[b][m]);
                    if (ks == 0) red[(b * 2 + m) * 32 + lrow] = v;
                }
            }
            named_barrier(1, kCW * 32);
            if (warp < nb) {
                const int b = warp;
                const float h = silu(red[(b * 2 + 0) * 32 + lane]) * red[(b * 2 + 1) * 32 + lane];
                const int M = shared ? p.sh_I : p.I;
                const int gld = shared ? p.sh_gld : p.h_gld;
                int16_t* hq = shared ? p.sh_hq : p.hq;
                int2* hm = shared ? p.sh_hmeta : p.hmeta;
                const size_t rr = static_cast<size_t>(t0 + b);
                quantize_group(h, lane, hq + rr * act_row(M), rb, kSliceH, hm + rr * gld + rb);
            }
            named_barrier(1, kCW * 32);
        } else {
            const int n = rb * 32 + lrow;  // output column of this lane group
#pragma unroll
            for (int b = 0; b < TB; ++b) {
                if (b >= nb) break;  // the pass's token count (warp-uniform)
                const float o = row_sum8(acc[b][0]);
                if (ks == 0) {
                    const int r = t0 + b;
                    if (shared) {
                        float* dst = (MODE == 1) ? p.sh_term : p.sh_rows_out;
                        dst[static_cast<size_t>(r) * p.H + n] = wgt[b] * o;
                    } else if (MODE == 1) {
                        p.slot_term[static_cast<size_t>(slot[b]) * p.H + n] = wgt[b] * o;
                    } else {
                        p.rows_out[static_cast<size_t>(r) * p.H + n] = o;
                    }
                }
            }
            if (MODE == 1 && task_end) ++run_cnt;
        }
    }
    if (MODE == 1 && run_cb >= 0 && !*abort_flag) combine_flush(p, run_cb, run_cnt, n_act_c, last_flag);
}

// Weight maps: uint8 [rows][K/2], box 256 bytes x 32 rows.  Scale maps: fp16 [rows][K/32],
// box 32 x 32 rows, only when a scale row is a multiple of 16 bytes (K % 256 == 0) and the
// pointer is 16-byte aligned; otherwise the consumers read scales directly.
static bool weight_maps(CUtensorMap* wm, CUtensorMap* sm, int* ws, const uint8_t* q, const uint16_t* s, int rows,
                        int K, int sbox) {
    if (!tmap_2d(wm, CU_TENSOR_MAP_DATA_TYPE_UINT8, q, static_cast<uint64_t>(K / 2), static_cast<uint64_t>(rows),
                 static_cast<uint64_t>(K / 2), kBoxB, 32, CU_TENSOR_MAP_SWIZZLE_NONE))
        return false;
    *ws = (K % 256 == 0) && (reinterpret_cast<uintptr_t>(s) & 15u) == 0;
    if (*ws && !tmap_2d(sm, CU_TENSOR_MAP_DATA_TYPE_UINT16, s, static_cast<uint64_t>(K / 32),
                        static_cast<uint64_t>(rows), static_cast<uint64_t>(K / 32) * 2, sbox, 32,
                        CU_TENSOR_MAP_SWIZZLE_NONE))
        return false;
    if (!*ws) *sm = *wm;
    return true;
}

bool gemv_tensor_maps(GemvArgs& p, int E) {
    int ws_up = 0;
    const int gb = Pipe<0>::GRP, db = Pipe<1>::GRP;
    if (!weight_maps(&p.tm_gate, &p.tm_gate_s, &p.ws_gu, p.gate_q, p.gate_s, E * p.I, p.H, gb)) return false;
    if (!weight_maps(&p.tm_up, &p.tm_up_s, &ws_up, p.up_q, p.up_s, E * p.I, p.H, gb)) return false;
    p.ws_gu = p.ws_gu && ws_up;
    if (!weight_maps(&p.tm_down, &p.tm_down_s, &p.ws_d, p.down_q, p.down_s, E * p.H, p.I, db)) return false;
    if (p.sh_I > 0) {
        if (!weight_maps(&p.tm_sh_gate, &p.tm_sh_gate_s, &p.ws_sh_gu, p.sh_gate_q, p.sh_gate_s, p.sh_I, p.H, gb))
            return false;
        if (!weight_maps(&p.tm_sh_up, &p.tm_sh_up_s, &ws_up, p.sh_up_q, p.sh_up_s, p.sh_I, p.H, gb)) return false;
        p.ws_sh_gu = p.ws_sh_gu && ws_up;
        if (!weight_maps(&p.tm_sh_down, &p.tm_sh_down_s, &p.ws_sh_d, p.sh_down_q, p.sh_down_s, p.H, p.sh_I, db))
            return false;
    } else {
        p.tm_sh_gate = p.tm_gate; p.tm_sh_up = p.tm_up; p.tm_sh_down = p.tm_down;
        p.tm_sh_gate_s = p.tm_gate_s; p.tm_sh_up_s = p.tm_up_s; p.tm_sh_down_s = p.tm_down_s;
        p.ws_sh_gu = p.ws_sh_d = 0;
    }
    return true;
}

template <int MODE>
static size_t pipe_smem_bytes() {
    using P = Pipe<MODE>;
    return 128 + static_cast<size_t>(P::STAGES) * P::STAGE + 2 * P::STAGES * sizeof(uint64_t) +
           P::TB * 2 * 32 * sizeof(float) + 16;
}

template <int MODE>
static cudaError_t pipe_attr() {
    static cudaError_t once = cudaFuncSetAttribute(gemv_pipe_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(pipe_smem_bytes<MODE>()));
    return once;
}

static int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 148;
    return n;
}

cudaError_t launch_gateup_gemv(const GemvArgs& p, cudaStream_t st) {
    cudaError_t e = pipe_attr<0>();
    if (e != cudaSuccess) return e;
    const int tasks = p.max_active * (p.I / 32) + (p.sh_I > 0 ? p.sh_I / 32 : 0);
    const int grid = std::max(1, std::min(tasks, 2 * sm_count()));
    KernelScope ks_("gateup_gemv", st);
    return launch_pdl(gemv_pipe_kernel<0>, dim3(grid), dim3((kCW + 1) * 32), pipe_smem_bytes<0>(), st, p);
}

cudaError_t launch_down_gemv(const GemvArgs& p, bool combine, cudaStream_t st) {
    cudaError_t e = combine ? pipe_attr<1>() : pipe_attr<2>();
    if (e != cudaSuccess) return e;
    const int tasks = (p.max_active + (p.sh_I > 0 ? 1 : 0)) * (p.H / 32);
    const int grid = std::max(1, std::min(tasks, 2 * sm_count()));
    KernelScope ks_(combine ? "down_gemv_combine" : "down_gemv_rows", st);
    if (combine) return launch_pdl(gemv_pipe_kernel<1>, dim3(grid), dim3((kCW + 1) * 32), pipe_smem_bytes<1>(), st, p);
    return launch_pdl(gemv_pipe_kernel<2>, dim3(grid), dim3((kCW + 1) * 32), pipe_smem_bytes<2>(), st, p);
}

}  // namespace moe
