// router.cu -- stage 1 of the routed MoE layer: router logits and the softmax top-k.
//
// Logits: one dot product per (token, router row) in fp32 over bf16 products, with the
// shared-expert gate vector as one more row past the router's E rows (daScript PR #3988
// "dasLLAMA vulkan: a MoE that fits the card ...", decode span commit: the gate logit is one
// more router GEMV row).  Decode batches (T <= 32) run a GEMV that reads every router row
// once; larger batches run a tcgen05 GEMM (router_tc.cu), or a tiled fp32 GEMM where H is not a
// multiple of 64 or E is above 256.
//
// Top-k: one warp per token with the whole logit row in registers, no shared memory, no
// block barrier and one read of the row (vllm.cpp PR #481 "gate(#378): the first DEVICE run
// of the warp MoE router", warp-router commit).  Selection is k rounds of a warp argmax with
// the lowest index winning a tie; weights are the fp32 softmax over all E logits renormalised
// over the k picks; the picks are written in ascending expert id.
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "quant.cuh"
#include "route_core.cuh"

namespace moe {

// ------------------------------------------------------------------ logits, decode GEMV
// Decode batches: one CTA per router row (and one for the gate row) reads the row once and
// dots it with every token in one pass (TB >= T); 256 threads, one 16-byte chunk of the row
// per thread per 2048 columns; the eight warp sums meet in a fixed order.  CTAs past the rows
// quantise x for the GEMV arm (one 32-value group per warp) when xq != nullptr, so that step
// costs no launch of its own.  With routing (r.ids != nullptr) the row CTA that finishes last
// (a completion count after a release fence) also runs the softmax top-k of every token and
// the dispatch of the fresh ids, so a decode batch routes in this one launch.
template <int TB, int VPT>
__global__ void __launch_bounds__(256) router_logits_gemv_kernel(
    const uint16_t* __restrict__ x, const uint16_t* __restrict__ W_r, const uint16_t* __restrict__ g,
    int T, int H, int E, int ld, float* __restrict__ logits, int nrows, int16_t* __restrict__ xq,
    int2* __restrict__ xmeta, int x_gld, DecodeRoute r) {
    pdl_wait();
    pdl_trigger();
    const int wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (static_cast<int>(blockIdx.x) >= nrows) {
        const int ng = H / 32;
        const int gw = (blockIdx.x - nrows) * 8 + wid;
        if (gw >= T * ng) return;
        const int t = gw / ng, grp = gw % ng;
        const float v = bf16_to_f32(x[static_cast<size_t>(t) * H + grp * 32 + lane]);
        quantize_group(v, lane, xq + static_cast<size_t>(t) * act_row(H), grp, kSliceX,
                       xmeta + static_cast<size_t>(t) * x_gld + grp);
        return;
    }
    const int row = blockIdx.x;  // 0..E-1 router rows, E = gate row
    const uint16_t* w = (row < E) ? W_r + static_cast<size_t>(row) * H : g;
    const int nch = H / 8;
    __shared__ float red[8][TB];
    float acc[TB];
#pragma unroll
    for (int i = 0; i < TB; ++i) acc[i] = 0.f;
    for (int c = threadIdx.x; c < nch; c += 256) {
        const uint4 wv = ldg_nc(w + static_cast<size_t>(c) * 8);
        float wf[8];
        const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            wf[2 * q] = __uint_as_float(ww[q] << 16);
            wf[2 * q + 1] = __uint_as_float(ww[q] & 0xffff0000u);
        }
#pragma unroll
        for (int i = 0; i < TB; ++i) {
            if (i < T) {
                const uint4 xv = ldg_nc(x + static_cast<size_t>(i) * H + static_cast<size_t>(c) * 8);
                const uint32_t xx[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    acc[i] = fmaf(__uint_as_float(xx[q] << 16), wf[2 * q], acc[i]);
                    acc[i] = fmaf(__uint_as_float(xx[q] & 0xffff0000u), wf[2 * q + 1], acc[i]);
                }
            }
        }
    }
#pragma unroll
    for (int i = 0; i < TB; ++i) {
        const float v = warp_sum(acc[i]);
        if (lane == 0) red[wid][i] = v;
    }
    __syncthreads();
    if (static_cast<int>(threadIdx.x) < T) {
        const int i = threadIdx.x;
        logits[static_cast<size_t>(i) * ld + row] =
            ((red[0][i] + red[1][i]) + (red[2][i] + red[3][i])) + ((red[4][i] + red[5][i]) + (red[6][i] + red[7][i]));
    }
    if (!r.ids) return;
    // ---- the last row CTA routes the batch
    __shared__ int is_last;
    __threadfence();  // this CTA's logits, before its count
    __syncthreads();
    if (threadIdx.x == 0) is_last = atomicAdd(r.done, 1) == nrows - 1;
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    extern __shared__ int dyn[];  // [T*k] ids | [rows][E] walk counts, rows = ceil(T*k / 32)
    const int k = r.k, n = T * k, rows = (n + 31) / 32;
    int* ids_s = dyn;
    int* hist = dyn + ((n + 3) & ~3);
    __shared__ int scratch[9];
    for (int i = threadIdx.x; i < rows * E; i += blockDim.x) hist[i] = 0;
    for (int t = wid; t < T; t += 8)
        topk_warp_row<CoherentF32, VPT>(reinterpret_cast<const CoherentF32*>(logits + static_cast<size_t>(t) * ld), E, k,
                                        ids_s + t * k, r.w + static_cast<size_t>(t) * k);
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += blockDim.x) r.ids[i] = ids_s[i];
    for (int q = wid; q < rows; q += 8)
        warp_walk(ids_s, q * 32, min(n, q * 32 + 32), E, hist + q * E, 0, r.perm, r.inv, r.status, true);
    __syncthreads();
    finalize_plan(hist, rows, E, n, r.counts, r.offsets, r.active, r.n_active, scratch);
    __syncthreads();
    for (int q = wid; q < rows; q += 8)
        warp_walk(ids_s, q * 32, min(n, q * 32 + 32), E, hist + q * E, 1, r.perm, r.inv, r.status, true);
    if (threadIdx.x == 0) *r.done = 0;  // ready for the next call
}

// ------------------------------------------------------------------ logits, prefill GEMM
// Tile: 64 tokens x 32 router rows, K step 32; 256 threads, each 4 tokens x 2 rows.
constexpr int RG_BT = 64, RG_BR = 32, RG_BK = 32;

__global__ void __launch_bounds__(256) router_logits_gemm_kernel(
    const uint16_t* __restrict__ x, const uint16_t* __restrict__ W_r, const uint16_t* __restrict__ g,
    int T, int H, int E, int nrows, int ld, float* __restrict__ logits) {
    pdl_wait();
    pdl_trigger();
    __shared__ float xs[RG_BK][RG_BT + 4];
    __shared__ float ws[RG_BK][RG_BR + 4];
    const int t0 = blockIdx.x * RG_BT, r0 = blockIdx.y * RG_BR;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;  // tx: rows (2 each), ty: tokens (4 each)
    float acc[4][2] = {};
    for (int k0 = 0; k0 < H; k0 += RG_BK) {
        // x tile: 64 tokens x 32 k = 2048 values, 8 per thread (one 16-byte load)
        {
            const int tt = threadIdx.x >> 2, kk = (threadIdx.x & 3) * 8;
            const int t = t0 + tt;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (t < T) v = ldg_nc(x + static_cast<size_t>(t) * H + k0 + kk);
            const uint32_t vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                xs[kk + 2 * q][tt] = __uint_as_float(vv[q] << 16);
                xs[kk + 2 * q + 1][tt] = __uint_as_float(vv[q] & 0xffff0000u);
            }
        }
        // router tile: 32 rows x 32 k = 1024 values, 4 per thread
        {
            const int rr = threadIdx.x >> 3, kk = (threadIdx.x & 7) * 4;
            const int r = r0 + rr;
            uint2 v = make_uint2(0, 0);
            if (r < nrows) {
                const uint16_t* src = (r < E) ? W_r + static_cast<size_t>(r) * H : g;
                v = *reinterpret_cast<const uint2*>(src + k0 + kk);
            }
            ws[kk + 0][rr] = __uint_as_float(v.x << 16);
            ws[kk + 1][rr] = __uint_as_float(v.x & 0xffff0000u);
            ws[kk + 2][rr] = __uint_as_float(v.y << 16);
            ws[kk + 3][rr] = __uint_as_float(v.y & 0xffff0000u);
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < RG_BK; ++kk) {
            float xv[4], wv[2];
#pragma unroll
            for (int i = 0; i < 4; ++i) xv[i] = xs[kk][ty * 4 + i];
#pragma unroll
            for (int j = 0; j < 2; ++j) wv[j] = ws[kk][tx * 2 + j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 2; ++j) acc[i][j] = fmaf(xv[i], wv[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int t = t0 + ty * 4 + i;
        if (t >= T) continue;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int r = r0 + tx * 2 + j;
            if (r < nrows) logits[static_cast<size_t>(t) * ld + r] = acc[i][j];
        }
    }
}

cudaError_t launch_router_logits(const uint16_t* x, const uint16_t* W_r, const uint16_t* g, int T, int H,
                                 int E, float* logits, cudaStream_t st, int16_t* xq, int2* xmeta, int x_gld,
                                 int* status, const DecodeRoute* route) {
    if (x_gld == 0) x_gld = H / 32;
    if (T == 0) return cudaSuccess;
    const int nrows = E + (g ? 1 : 0);
    const int ld = nrows;
    if (T <= 32) {
        const int qctas = xq ? (T * (H / 32) + 7) / 8 : 0;
        const DecodeRoute r = route ? *route : DecodeRoute{};
        const size_t smem = r.ids ? sizeof(int) * (((T * r.k + 3) & ~3) + static_cast<size_t>((T * r.k + 31) / 32) * E)
                                  : 0;
        KernelScope ks_(r.ids ? "router_gemv+topk+dispatch" : (xq ? "router_logits_gemv+quant_x" : "router_logits_gemv"),
                        st);
        const dim3 grid(nrows + qctas), block(256);
        const int vpt = E <= 64 ? 2 : (E <= 128 ? 4 : 8);
#define MOE_RG_CASE(TBV, V)                                                                                     \
    if (T <= TBV && vpt == V)                                                                                   \
        return launch_pdl(router_logits_gemv_kernel<TBV, V>, grid, block, smem, st, x, W_r, g, T, H, E, ld, logits, \
                          nrows, xq, xmeta, x_gld, r);
        MOE_RG_CASE(4, 2) MOE_RG_CASE(4, 4) MOE_RG_CASE(4, 8)
        MOE_RG_CASE(8, 2) MOE_RG_CASE(8, 4) MOE_RG_CASE(8, 8)
        MOE_RG_CASE(16, 2) MOE_RG_CASE(16, 4) MOE_RG_CASE(16, 8)
        MOE_RG_CASE(32, 2) MOE_RG_CASE(32, 4) MOE_RG_CASE(32, 8)
#undef MOE_RG_CASE
        return cudaErrorInvalidValue;
    }
    cudaError_t e;
    if (router_tc_supported(x, W_r, g, H, E)) {
        e = launch_router_logits_tc(x, W_r, g, T, H, E, logits, status, st);
    } else {
        KernelScope ks_("router_logits_gemm", st);
        const dim3 grid((T + RG_BT - 1) / RG_BT, (nrows + RG_BR - 1) / RG_BR);
        e = launch_pdl(router_logits_gemm_kernel, grid, dim3(256), 0, st, x, W_r, g, T, H, E, nrows, ld, logits);
    }
    if (e != cudaSuccess || !xq) return e;
    QuantArgs q;
    q.src0 = x; q.src0_bf16 = 1; q.rows0 = T; q.K0 = H; q.q0 = xq; q.meta0 = xmeta; q.gld0 = x_gld;
    return launch_quantize(q, st);
}

// ------------------------------------------------------------------ softmax top-k
// VPT = values per lane = ceil(E / 32); expert index of (lane, j) is lane + 32 * j.
template <typename Tin, int VPT>
__global__ void __launch_bounds__(256) router_topk_warp_kernel(const Tin* __restrict__ logits, int ld, int T, int E,
                                                               int k, int32_t* __restrict__ topk_ids,
                                                               float* __restrict__ topk_w,
                                                               const float* __restrict__ bias, int renorm,
                                                               float scale) {
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    topk_warp_row<Tin, VPT>(logits + static_cast<size_t>(t) * ld, E, k, topk_ids + static_cast<size_t>(t) * k,
                            topk_w + static_cast<size_t>(t) * k, bias, renorm != 0, scale);
}

// Counted variant (prefill layer): a CTA takes kCountedWarps * tpw consecutive tokens, in
// rounds of kCountedWarps (warp w takes token w of a round); its picks per expert go to row
// blockIdx.x of the dispatch count table.  The logit rows of rpr rounds at a time are staged in
// shared memory by the whole CTA (coalesced, every load in flight): with K-split router logits
// the partial planes are summed there, in plane order, and the sums also written back to plane 0
// (the shared gate's logit is read from it later); each warp then selects from its staged row.
constexpr int kCountedUnroll = 8;  // staged values per thread per batch (times the planes)

template <int VPT>
__global__ void __launch_bounds__(kCountedWarps * 32) router_topk_counted_kernel(float* logits, int ld, int T, int E,
                                                                                 int k, int tpw, int rpr,
                                                                                 int32_t* __restrict__ topk_ids,
                                                                                 float* __restrict__ topk_w,
                                                                                 int* __restrict__ cta_cnt, int parts) {
    extern __shared__ float rows_s[];  // [kCountedWarps * rpr][ld]
    __shared__ int hist[32 * VPT];
    for (int i = threadIdx.x; i < E; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    pdl_wait();
    pdl_trigger();
    const int w = threadIdx.x >> 5;
    const int c0 = blockIdx.x * kCountedWarps * tpw;  // the CTA's first token
    const int cend = min(T, c0 + kCountedWarps * tpw);
    const size_t plane = static_cast<size_t>(T) * ld;
    for (int j0 = 0; j0 < tpw; j0 += rpr) {
        // rounds j0 .. j0 + rpr - 1: tokens [r0, r1), contiguous rows of the logits
        const int r0 = min(cend, c0 + j0 * kCountedWarps);
        const int r1 = min(cend, r0 + rpr * kCountedWarps);
        const int nval = (r1 - r0) * ld;
        float* base = logits + static_cast<size_t>(r0) * ld;
        for (int i0 = 0; i0 < nval; i0 += kCountedUnroll * kCountedWarps * 32) {
            float v[kCountedUnroll][4];
#pragma unroll
            for (int u = 0; u < kCountedUnroll; ++u) {
                const int i = i0 + u * kCountedWarps * 32 + threadIdx.x;
#pragma unroll
                for (int q = 0; q < 4; ++q) v[u][q] = (i < nval && q < parts) ? __ldg(base + q * plane + i) : 0.f;
            }
#pragma unroll
            for (int u = 0; u < kCountedUnroll; ++u) {
                const int i = i0 + u * kCountedWarps * 32 + threadIdx.x;
                if (i < nval) {
                    float sum = v[u][0];
#pragma unroll
                    for (int q = 1; q < 4; ++q)
                        if (q < parts) sum += v[u][q];
                    rows_s[i] = sum;
                    if (parts > 1) base[i] = sum;
                }
            }
        }
        __syncthreads();
        for (int r = 0; r < rpr; ++r) {
            const int t = r0 + r * kCountedWarps + w;
            if (t < r1)
                topk_warp_row<SharedF32, VPT>(reinterpret_cast<const SharedF32*>(rows_s + (t - r0) * ld), E, k,
                                              topk_ids + static_cast<size_t>(t) * k,
                                              topk_w + static_cast<size_t>(t) * k, nullptr, true, 1.f, hist);
        }
        __syncthreads();  // the staged rows are replaced by the next rounds'
    }
    for (int e = threadIdx.x; e < E; e += blockDim.x) cta_cnt[static_cast<size_t>(blockIdx.x) * E + e] = hist[e];
}

// Rounds staged at once: as many as fit kCountedStageBytes of shared memory (at least one; with
// the kernel's static histogram this stays under the 48 KB a launch gets without opting in).
constexpr int kCountedStageBytes = 40 * 1024;
static int counted_rounds_per_stage(int tpw, int ld) {
    const int fit = kCountedStageBytes / (kCountedWarps * ld * static_cast<int>(sizeof(float)));
    return std::max(1, std::min(tpw, fit));
}

cudaError_t launch_router_topk_counted(float* logits, int ld, int T, int E, int k, int tpw, int32_t* ids, float* w,
                                       int* cta_cnt, cudaStream_t st, int parts) {
    if (T == 0) return cudaSuccess;
    if (parts < 1 || parts > 4) return cudaErrorInvalidValue;
    const int vpt = (E + 31) / 32;
    const int rpr = counted_rounds_per_stage(tpw, ld);
    const size_t smem = static_cast<size_t>(kCountedWarps) * rpr * ld * sizeof(float);
    if (smem > static_cast<size_t>(kCountedStageBytes)) return cudaErrorInvalidValue;
    const dim3 grid((T + kCountedWarps * tpw - 1) / (kCountedWarps * tpw)), block(kCountedWarps * 32);
    KernelScope ks_("router_topk+count", st);
    switch (vpt) {
#define MOE_TOPKC_CASE(V) \
    case V:                                                                                                   \
        return launch_pdl(router_topk_counted_kernel<V>, grid, block, smem, st, logits, ld, T, E, k, tpw, rpr, ids, \
                          w, cta_cnt, parts);
        MOE_TOPKC_CASE(1)
        MOE_TOPKC_CASE(2)
        MOE_TOPKC_CASE(3)
        MOE_TOPKC_CASE(4)
        MOE_TOPKC_CASE(5)
        MOE_TOPKC_CASE(6)
        MOE_TOPKC_CASE(7)
        MOE_TOPKC_CASE(8)
#undef MOE_TOPKC_CASE
        default: return cudaErrorInvalidValue;
    }
}

template <typename Tin>
static cudaError_t launch_topk_t(const Tin* logits, int ld, int T, int E, int k, int32_t* ids, float* w,
                                 const float* bias, bool renorm, float scale, cudaStream_t st) {
    const int vpt = (E + 31) / 32;
    const dim3 grid((T + 7) / 8), block(256);
    KernelScope ks_("router_topk", st);
    switch (vpt) {
#define MOE_TOPK_CASE(V) \
    case V:                                                                                                \
        return launch_pdl(router_topk_warp_kernel<Tin, V>, grid, block, 0, st, logits, ld, T, E, k, ids, w, bias, \
                          renorm ? 1 : 0, scale);
        MOE_TOPK_CASE(1)
        MOE_TOPK_CASE(2)
        MOE_TOPK_CASE(3)
        MOE_TOPK_CASE(4)
        MOE_TOPK_CASE(5)
        MOE_TOPK_CASE(6)
        MOE_TOPK_CASE(7)
        MOE_TOPK_CASE(8)
#undef MOE_TOPK_CASE
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_router_topk(const void* logits, bool is_bf16, int ld, int T, int E, int k, int32_t* ids,
                               float* w, cudaStream_t st, const float* bias, bool renorm, float scale) {
    if (T == 0) return cudaSuccess;
    if (is_bf16)
        return launch_topk_t(static_cast<const uint16_t*>(logits), ld, T, E, k, ids, w, bias, renorm, scale, st);
    return launch_topk_t(static_cast<const float*>(logits), ld, T, E, k, ids, w, bias, renorm, scale, st);
}

}  // namespace moe
