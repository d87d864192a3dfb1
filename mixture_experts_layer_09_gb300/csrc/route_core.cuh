// route_core.cuh -- device pieces of stage 1 (top-k of one logit row, one warp) and stage 2
// (per-warp histogram walk, CTA scans, bucket placement), shared by the stand-alone router and
// dispatch kernels and by the fused decode routing kernel.
#pragma once

#include "common.cuh"

namespace moe {

// ------------------------------------------------------------------ softmax top-k
// One warp per token with the whole logit row in registers, no shared memory, one read of the
// row (vllm.cpp PR #481 "gate(#378): the first DEVICE run of the warp MoE router", warp-router
// commit).  Selection is k rounds of a warp argmax with the lowest index winning a tie (per
// round one warp max over order-preserving integer keys of the scores and one warp min over
// the indices holding it); weights are the fp32 softmax over all E logits renormalised over
// the k picks -- computed as the softmax over the picked logits, which it equals -- or, for the
// unnormalised variant, the full softmax; the picks are written in ascending expert id.
template <typename Tin>
__device__ __forceinline__ float load_logit(const Tin* p);
template <>
__device__ __forceinline__ float load_logit<float>(const float* p) { return __ldg(p); }
template <>
__device__ __forceinline__ float load_logit<uint16_t>(const uint16_t* p) { return bf16_to_f32(__ldg(p)); }
// fp32 logits written earlier by other CTAs of the same kernel: coherent loads through L2
struct CoherentF32 {
    float v;
};
static_assert(sizeof(CoherentF32) == sizeof(float), "one logit per element");
template <>
__device__ __forceinline__ float load_logit<CoherentF32>(const CoherentF32* p) {
    return __ldcg(reinterpret_cast<const float*>(p));
}
// fp32 logits staged in shared memory by the calling CTA
struct SharedF32 {
    float v;
};
static_assert(sizeof(SharedF32) == sizeof(float), "one logit per element");
template <>
__device__ __forceinline__ float load_logit<SharedF32>(const SharedF32* p) {
    return p->v;
}

// VPT = values per lane = ceil(E / 32); expert index of (lane, j) is lane + 32 * j.
// One warp selects the top-k of one logit row.  ids/w receive the row's k outputs; hist (shared
// memory, or null) counts each pick.
// Variants (bias, renorm, scale): the selection runs over logit + bias[e] (bias fp32 [E] or
// null), the weights stay the unbiased softmax, renormalised over the picks or not, times scale.
template <typename Tin, int VPT>
__device__ __forceinline__ void topk_warp_row(const Tin* __restrict__ row, int E, int k, int32_t* __restrict__ ids,
                                              float* __restrict__ w, const float* __restrict__ bias = nullptr,
                                              bool renorm = true, float scale = 1.f, int* hist = nullptr) {
    const int lane = threadIdx.x & 31;
    float v[VPT];         // logits: the softmax
    uint32_t key[VPT];    // selection scores (logit + bias) as order-preserving integers; 0 once picked
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        const int e = lane + 32 * j;
        if (e < E) {
            float f = load_logit<Tin>(row + e);
            v[j] = (f != f) ? -INFINITY : f;  // NaN never wins a pick
            float sb = bias ? v[j] + __ldg(bias + e) : v[j];
            sb = (sb != sb) ? -INFINITY : sb + 0.f;  // + 0 folds -0 into +0: the two are equal scores
            const uint32_t u = __float_as_uint(sb);
            key[j] = (u & 0x80000000u) ? ~u : (u | 0x80000000u);  // -inf -> 0x007fffff, above 0
        } else {
            v[j] = -INFINITY;
            key[j] = 0u;  // padding is never a candidate
        }
    }
    // k rounds: the largest score (one warp max over the keys), then the lowest expert index
    // holding it (one warp min); the pick's key becomes 0, and a maximum of 0 means no candidate.
    for (int round = 0; round < k; ++round) {
        uint32_t bk = 0u;
#pragma unroll
        for (int j = 0; j < VPT; ++j) bk = max(bk, key[j]);
        const uint32_t gk = __reduce_max_sync(0xffffffffu, bk);
        if (gk == 0u) break;  // warp-uniform
        int cand = 0x7fffffff;
#pragma unroll
        for (int j = VPT - 1; j >= 0; --j)  // lane + 32 j grows with j: the last match kept is the lowest
            if (key[j] == gk) cand = lane + 32 * j;
        const int bi = __reduce_min_sync(0xffffffffu, cand);
#pragma unroll
        for (int j = 0; j < VPT; ++j)
            if (bi == lane + 32 * j) key[j] = 0u;
    }
    bool picked[VPT];
#pragma unroll
    for (int j = 0; j < VPT; ++j) picked[j] = key[j] == 0u && lane + 32 * j < E;
    float p[VPT];
    if (renorm) {
        // the softmax over all E renormalised over the picks is the softmax over the picked
        // logits alone: k exponentials, shifted by the largest picked logit
        float m = -INFINITY;
#pragma unroll
        for (int j = 0; j < VPT; ++j)
            if (picked[j]) m = fmaxf(m, v[j]);
        m = warp_max(m);
        float z = 0.f;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            p[j] = 0.f;
            if (picked[j] && m > -INFINITY) p[j] = expf(v[j] - m);  // a lane holds few picks
            z += p[j];
        }
        z = warp_sum(z);
        // denominator guard: a row with no finite picked logit spreads the weight evenly
        const float rz = (z > 0.f) ? 1.f / z : 0.f;
#pragma unroll
        for (int j = 0; j < VPT; ++j) p[j] = (z > 0.f) ? p[j] * rz : 1.f / k;
    } else {
        // fp32 softmax over all E logits
        float m = -INFINITY;
#pragma unroll
        for (int j = 0; j < VPT; ++j)
            if (lane + 32 * j < E) m = fmaxf(m, v[j]);
        m = warp_max(m);
        float z = 0.f;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            p[j] = (lane + 32 * j < E && m > -INFINITY) ? expf(v[j] - m) : 0.f;
            z += p[j];
        }
        z = warp_sum(z);
#pragma unroll
        for (int j = 0; j < VPT; ++j) p[j] = (z > 0.f) ? p[j] / z : 0.f;
    }
    // write the picks in ascending expert id: (j, lane) order
    int base = 0;
    const unsigned lt = lanemask_lt();
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        const unsigned b = __ballot_sync(0xffffffffu, picked[j]);
        if (picked[j]) {
            const int pos = base + __popc(b & lt);
            if (pos < k) {
                ids[pos] = lane + 32 * j;
                w[pos] = p[j] * scale;
                if (hist) atomicAdd(hist + lane + 32 * j, 1);  // the CTA's picks per expert (shared memory)
            }
        }
        base += __popc(b);
    }
}


// ------------------------------------------------------------------ dispatch pieces
// Walk a warp's slot run 32 at a time.  mode 0: count into hist; mode 1: scatter using hist
// as the running base (hist must hold the warp's starting position per expert).
// (ids_in_smem: the ids sit in this CTA's shared memory; otherwise they are read from global
// memory with coherent loads, since they may have been written by the same kernel)
__device__ __forceinline__ void warp_walk(const int32_t* ids, int begin, int end, int E,
                                          int* hist, int mode, int32_t* __restrict__ perm,
                                          int32_t* __restrict__ inv, int* status, bool ids_in_smem = false) {
    const int lane = threadIdx.x & 31;
    const unsigned lt = lanemask_lt();
    for (int base = begin; base < end; base += 32) {
        const int a = base + lane;
        int id = -1;
        if (a < end) {
            id = ids_in_smem ? ids[a] : __ldcg(ids + a);
            if (id < 0 || id >= E) {
                if (mode == 0) record_status(status, MOE_ERR_DEVICE_INDEX, a, id);
                id = -1;
            }
        }
        const unsigned peers = __match_any_sync(0xffffffffu, id);
        const int leader = __ffs(peers) - 1;
        if (mode == 0) {
            if (id >= 0 && lane == leader) hist[id] += __popc(peers);
        } else {
            int pos = -1;
            if (id >= 0) pos = hist[id] + __popc(peers & lt);
            __syncwarp();
            if (id >= 0 && lane == leader) hist[id] += __popc(peers);
            if (a < end) {
                if (id >= 0) perm[pos] = a;
                inv[a] = pos;
            }
        }
        __syncwarp();
    }
}

// Exclusive scan of v over threads 0..255 (v = 0 for threads >= n); returns the prefix and
// writes the total to *total.  Uses scratch[8 + 1].
__device__ __forceinline__ int cta_exclusive_scan_256(int v, int* scratch, int* total) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (threadIdx.x < 256 && lane == 31) scratch[w] = incl;
    __syncthreads();
    if (threadIdx.x == 0) {
        int run = 0;
        for (int i = 0; i < 8; ++i) {
            const int tmp = scratch[i];
            scratch[i] = run;
            run += tmp;
        }
        scratch[8] = run;
    }
    __syncthreads();
    const int res = (threadIdx.x < 256) ? scratch[w] + incl - v : 0;
    *total = scratch[8];
    __syncthreads();
    return res;
}

// After per-(warp or CTA) counts are known: counts, offsets, active list, and turns the
// count table cnt[rows][E] into starting positions.  Needs blockDim.x >= 256.
__device__ inline void finalize_plan(int* cnt, int rows, int E, int n, int32_t* counts, int32_t* offsets,
                              int32_t* active, int32_t* n_active, int* scratch) {
    const int e = threadIdx.x;
    int total = 0;
    if (e < E) {
        for (int r = 0; r < rows; ++r) {
            const int tmp = cnt[static_cast<size_t>(r) * E + e];
            cnt[static_cast<size_t>(r) * E + e] = total;
            total += tmp;
        }
    }
    int sum;
    const int off = cta_exclusive_scan_256(e < E ? total : 0, scratch, &sum);
    const int flag = (e < E && total > 0) ? 1 : 0;
    int nact;
    const int apos = cta_exclusive_scan_256(flag, scratch, &nact);
    if (e < E) {
        offsets[e] = off;
        if (counts) counts[e] = total;
        for (int r = 0; r < rows; ++r) cnt[static_cast<size_t>(r) * E + e] += off;
        if (flag) active[apos] = e;
    }
    if (threadIdx.x == 0) {
        offsets[E] = sum;
        *n_active = nact;
    }
    (void)n;
}

}  // namespace moe
