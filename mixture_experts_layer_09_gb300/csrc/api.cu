// api.cu -- the C ABI of include/moe.h: argument checks, workspace layout, kernel order.
//
// Nothing here computes a value of the layer; every step runs in the kernels of router.cu,
// dispatch.cu, gemv.cu, gemm_sm100.cu and combine.cu.  No call allocates device memory or
// synchronises, except moe_device_status, whose job is to read the status word.
#include <algorithm>
#include <new>

#include "common.cuh"
#include "internal.h"
#include "norm.h"
#include "quant.cuh"

using namespace moe;

namespace {

// Carves 256-byte-aligned pieces out of a workspace; with base == nullptr it only measures.
struct Carver {
    char* base;
    size_t off = kWsHead;  // status word and column counters
    explicit Carver(void* b) : base(static_cast<char*>(b)) {}
    template <typename T>
    T* take(size_t count) {
        T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
        off += align_up(count * sizeof(T) + (count == 0 ? 1 : 0), kWsAlign);
        return p;
    }
    size_t size() const { return off; }
};

struct Routing {
    float* logits;
    int32_t* ids;
    float* w;
    int32_t* counts;
    int32_t* offsets;
    int32_t* perm;
    int32_t* inv;
    int32_t* active;
    int32_t* n_active;
    void* disp_scratch;
    int* route_cnt;  // [CTAs][E]: per-CTA expert counts of the counted top-k (prefill layer)
};

struct GemvBufs {
    int16_t* xq; int2* xmeta;
    int16_t* hq; int2* hmeta;
    int16_t* sh_hq; int2* sh_hmeta;
    float* rows; float* sh_rows;      // ROWS mode (unweighted) / COMBINE mode (weighted slot terms)
};

struct GemmBufs {
    uint16_t* x16; uint16_t* h16; uint16_t* sh_h16;
    int* tiles; int* n_tiles;
    float* rows; float* sh_rows;
};

// Tokens per warp of the counted top-k: the fewest (1, 2, 4, ...) that keep its CTA count
// (kCountedWarps warps each) at most 64 -- every scatter CTA reads the whole count table -- and
// within the table's bounds.
int counted_ctas(int T, int tpw) { return (T + kCountedWarps * tpw - 1) / (kCountedWarps * tpw); }
int counted_tokens_per_warp(int T, int E) {
    int tpw = 1;
    while (tpw < (1 << 20) && (counted_ctas(T, tpw) > 64 || !dispatch_counted_supported(counted_ctas(T, tpw), E)))
        tpw *= 2;
    return tpw;
}

void carve_routing(Carver& c, int T, int E, int k, Routing& r) {
    const size_t n = static_cast<size_t>(T) * k;
    r.logits = c.take<float>(static_cast<size_t>(T) * (E + 1) * 4);  // up to 4 partial planes (K-split router)
    r.ids = c.take<int32_t>(n);
    r.w = c.take<float>(n);
    r.counts = c.take<int32_t>(E);
    r.offsets = c.take<int32_t>(E + 1);
    r.perm = c.take<int32_t>(n);
    r.inv = c.take<int32_t>(n);
    r.active = c.take<int32_t>(E);
    r.n_active = c.take<int32_t>(1);
    r.disp_scratch = c.take<char>(dispatch_scratch_bytes(static_cast<int>(n), E));
    const int tpw = counted_tokens_per_warp(T, E);
    r.route_cnt = c.take<int>(static_cast<size_t>(counted_ctas(T, tpw)) * E);
}

void carve_gemv(Carver& c, int T, int k, int H, int I, int I_sh, GemvBufs& b) {
    const size_t R = static_cast<size_t>(T) * k;
    b.xq = c.take<int16_t>(static_cast<size_t>(T) * act_row(H));
    b.xmeta = c.take<int2>(static_cast<size_t>(T) * act_gld(H));
    b.hq = c.take<int16_t>(R * act_row(I));
    b.hmeta = c.take<int2>(R * act_gld(I));
    const size_t Ts = I_sh > 0 ? static_cast<size_t>(T) : 0;
    const int Is = I_sh > 0 ? I_sh : 32;
    b.sh_hq = c.take<int16_t>(Ts * act_row(Is));
    b.sh_hmeta = c.take<int2>(Ts * act_gld(Is));
    b.rows = c.take<float>(R * H);
    b.sh_rows = c.take<float>(Ts * H);
}

void carve_gemm(Carver& c, int T, int k, int E, int H, int I, int I_sh, GemmBufs& b) {
    const size_t R = static_cast<size_t>(T) * k;
    const size_t Ts = I_sh > 0 ? static_cast<size_t>(T) : 0;
    b.x16 = c.take<uint16_t>((R + Ts) * H);
    b.h16 = c.take<uint16_t>(R * I);
    b.sh_h16 = c.take<uint16_t>(Ts * (I_sh > 0 ? I_sh : 0));
    b.tiles = c.take<int>(3 * static_cast<size_t>(gemm_ntile_max(static_cast<int>(R), E)));
    b.n_tiles = c.take<int>(1);
    b.rows = c.take<float>(R * H);
    b.sh_rows = c.take<float>(Ts * H);
}

int status_of(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The library runs only on compute capability 10.3 (sm_103a).
int check_device() {
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (major != 10 || minor != 3) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

int check_q4(const moe_q4& m) {
    if (!m.q || !m.s) return MOE_ERR_INVALID_ARG;
    if (!aligned16(m.q) || (reinterpret_cast<uintptr_t>(m.s) & 3u)) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

int check_experts(const moe_experts* W) {
    if (!W) return MOE_ERR_INVALID_ARG;
    if (W->E < 1 || W->E > MOE_MAX_E || W->H < 32 || W->I < 32 || W->H % 32 || W->I % 32) return MOE_ERR_INVALID_ARG;
    if (W->H > MOE_MAX_H) return MOE_ERR_INVALID_ARG;
    if (W->fmt != MOE_WFMT_INT4 && W->fmt != MOE_WFMT_MXFP4) return MOE_ERR_INVALID_ARG;
    int s;
    if ((s = check_q4(W->gate)) || (s = check_q4(W->up)) || (s = check_q4(W->down))) return s;
    return MOE_OK;
}

int check_shared(const moe_shared* sh) {
    if (!sh) return MOE_OK;
    if (sh->I_sh < 32 || sh->I_sh % 32) return MOE_ERR_INVALID_ARG;
    if (sh->fmt != MOE_WFMT_INT4 && sh->fmt != MOE_WFMT_MXFP4) return MOE_ERR_INVALID_ARG;
    int s;
    if ((s = check_q4(sh->gate)) || (s = check_q4(sh->up)) || (s = check_q4(sh->down))) return s;
    if (sh->g && !aligned16(sh->g)) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

// AUTO: the bandwidth arm while the batch puts at most a few rows on an expert (and on the
// shared expert, which takes every token), else the tensor arm -- the crossover measured by
// sweeping both arms over T.
int choose_arm(int arm, int T, int k, int E, int H, int I, int I_sh) {
    const bool gemm_ok = gemm_supported(H, I, I_sh);
    if (arm == MOE_ARM_GEMV) return MOE_ARM_GEMV;
    if (arm == MOE_ARM_GEMM) return gemm_ok ? MOE_ARM_GEMM : -1;
    if (arm != MOE_ARM_AUTO) return -1;
    const bool few_rows = static_cast<long long>(T) * k <= static_cast<long long>(MOE_AUTO_GEMV_ROWS_PER_EXPERT) * E &&
                          (I_sh <= 0 || T <= MOE_AUTO_GEMV_MAX_T_SHARED);
    if (few_rows || !gemm_ok) return MOE_ARM_GEMV;
    return MOE_ARM_GEMM;
}

cudaStream_t S(moe_stream_t s) { return static_cast<cudaStream_t>(s); }

// Builds the active-expert list from bucket offsets (for callers of moe_expert_mlp, whose
// dispatch may come from elsewhere).
__global__ void active_from_offsets_kernel(const int32_t* __restrict__ offsets, int E, int32_t* active,
                                           int32_t* n_active) {
    pdl_wait();
    pdl_trigger();
    __shared__ int warp_tot[8];
    const int e = threadIdx.x, lane = e & 31, w = e >> 5;
    const int f = (e < E && offsets[e + 1] > offsets[e]) ? 1 : 0;
    int incl = f;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) warp_tot[w] = incl;
    __syncthreads();
    int base = incl - f;
    for (int i = 0; i < w; ++i) base += warp_tot[i];
    if (f) active[base] = e;
    if (e == 255) *n_active = base + f;
}

// Expert MLP of every dispatched row: GEMV arm (rows or fused combine) or GEMM arm.
struct MlpCall {
    const uint16_t* x;
    int T, k;
    const moe_experts* W;
    const moe_shared* sh;
    const float* logits;  // nullptr unless a gated shared expert
    int logit_ld;
    const int32_t* offsets;
    const int32_t* perm;
    const int32_t* inv;
    const int32_t* active;
    const int32_t* n_active;
    const float* topk_w;
    const uint16_t* residual;
    float* rows_out;      // rows mode target (moe_expert_mlp) or nullptr
    float* y;             // layer mode target
    int* status;
    const NormOut* norm;  // layer mode: RMSNorm of y too, or nullptr
};

int run_gemv(const MlpCall& c, GemvBufs& b, bool x_quantized, cudaStream_t st) {
    const moe_experts* W = c.W;
    const int I_sh = c.sh ? c.sh->I_sh : 0;
    if (!x_quantized) {
        QuantArgs qx;
        qx.src0 = c.x; qx.src0_bf16 = 1; qx.rows0 = c.T; qx.K0 = W->H; qx.q0 = b.xq; qx.meta0 = b.xmeta;
        qx.gld0 = act_gld(W->H);
        if (launch_quantize(qx, st) != cudaSuccess) return MOE_ERR_CUDA;
    }
    GemvArgs p{};
    p.T = c.T; p.k = c.k; p.H = W->H; p.I = W->I;
    p.max_active = std::min(W->E, c.T * c.k);
    p.gate_q = W->gate.q; p.gate_s = W->gate.s; p.up_q = W->up.q; p.up_s = W->up.s;
    p.down_q = W->down.q; p.down_s = W->down.s;
    p.fp4_r = W->fmt == MOE_WFMT_MXFP4;
    p.fp4_s = c.sh && c.sh->fmt == MOE_WFMT_MXFP4;
    p.sh_I = I_sh;
    if (c.sh) {
        p.sh_gate_q = c.sh->gate.q; p.sh_gate_s = c.sh->gate.s; p.sh_up_q = c.sh->up.q; p.sh_up_s = c.sh->up.s;
        p.sh_down_q = c.sh->down.q; p.sh_down_s = c.sh->down.s;
        p.sh_gate_logit = c.sh->g ? c.logits + W->E : nullptr;
        p.logit_ld = c.logit_ld;
    }
    p.offsets = c.offsets; p.perm = c.perm; p.active = c.active; p.n_active = c.n_active; p.topk_w = c.topk_w;
    p.status = c.status;
    p.task_counter = reinterpret_cast<int*>(reinterpret_cast<char*>(c.status) + kWsTaskOffset);
    p.x_gld = act_gld(W->H); p.h_gld = act_gld(W->I); p.sh_gld = act_gld(I_sh > 0 ? I_sh : 32);
    p.xq = b.xq; p.xmeta = b.xmeta;
    p.hq = b.hq; p.hmeta = b.hmeta; p.sh_hq = b.sh_hq; p.sh_hmeta = b.sh_hmeta;
    if (!gemv_tensor_maps(p, W->E)) return MOE_ERR_CUDA;
    if (launch_gateup_gemv(p, st) != cudaSuccess) return MOE_ERR_CUDA;
    if (c.rows_out) {  // stage call: unweighted rows in dispatch order
        p.rows_out = c.rows_out;
        p.sh_rows_out = b.sh_rows;
        return launch_down_gemv(p, false, st) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
    }
    p.slot_term = b.rows;
    p.sh_term = b.sh_rows;
    p.col_counter = reinterpret_cast<int*>(reinterpret_cast<char*>(c.status) + kWsCounterOffset);
    p.residual = c.residual;
    p.y = c.y;
    if (launch_down_gemv(p, true, st) != cudaSuccess) return MOE_ERR_CUDA;
    if (!c.norm) return MOE_OK;
    return status_of(launch_rmsnorm(c.y, c.norm->gamma, c.T, W->H, c.norm->eps, c.norm->y_norm, st));
}

int run_gemm(const MlpCall& c, GemmBufs& b, cudaStream_t st, bool tiles_ready = false) {
    const moe_experts* W = c.W;
    GemmPlan p{};
    p.T = c.T; p.k = c.k; p.E = W->E; p.H = W->H; p.I = W->I;
    p.sh_I = c.sh ? c.sh->I_sh : 0;
    p.ntile_max = gemm_ntile_max(c.T * c.k, W->E);
    p.sh_tiles = (c.T + kGemmTileN - 1) / kGemmTileN;
    p.offsets = c.offsets; p.perm = c.perm; p.topk_w = c.topk_w;
    p.sh_gate_logit = (c.sh && c.sh->g) ? c.logits + W->E : nullptr;
    p.logit_ld = c.logit_ld;
    p.gate_q = W->gate.q; p.gate_s = W->gate.s; p.up_q = W->up.q; p.up_s = W->up.s;
    p.down_q = W->down.q; p.down_s = W->down.s;
    p.fp4_r = W->fmt == MOE_WFMT_MXFP4;
    p.fp4_s = c.sh && c.sh->fmt == MOE_WFMT_MXFP4;
    if (c.sh) {
        p.sh_gate_q = c.sh->gate.q; p.sh_gate_s = c.sh->gate.s; p.sh_up_q = c.sh->up.q; p.sh_up_s = c.sh->up.s;
        p.sh_down_q = c.sh->down.q; p.sh_down_s = c.sh->down.s;
    }
    p.x = c.x; p.x16 = b.x16; p.h16 = b.h16; p.sh_h16 = b.sh_h16; p.tiles = b.tiles; p.n_tiles = b.n_tiles;
    p.tiles_ready = tiles_ready ? 1 : 0;
    p.status = c.status;
    const bool rows_mode = c.rows_out != nullptr;
    p.rows_out = c.rows_out;
    p.slot_out = b.rows;
    p.sh_out = b.sh_rows;
    if (launch_gemm_arm(p, rows_mode, st) != cudaSuccess) return MOE_ERR_CUDA;
    if (!rows_mode) {
        const float* shr = c.sh ? b.sh_rows : nullptr;
        const cudaError_t e =
            c.norm ? launch_combine_norm(b.rows, c.inv, c.topk_w, true, shr, c.residual, c.T, c.k, W->H, c.y, *c.norm, st)
                   : launch_combine(b.rows, c.inv, c.topk_w, true, shr, c.residual, c.T, c.k, W->H, c.y, st);
        if (e != cudaSuccess) return MOE_ERR_CUDA;
    }
    return MOE_OK;
}

// The layer call, with the RMSNorm of its output when `norm` is set: the tensor arm's combine
// norms each row as it writes it.  On the GEMV arm the combine is folded into the down
// projection, whose column blocks finish in no fixed order; a row is complete only when the
// last block is, and one CTA norming every row then was slower than the norm's own launch
// (one CTA per row on as many SMs), so the norm follows as that launch.
int layer_forward(const uint16_t* x, const uint16_t* residual, const uint16_t* W_r, const moe_experts* W,
                  const moe_shared* sh, int T, int k, float* y, int32_t* topk_ids_out, float* topk_w_out, int arm,
                  void* ws, size_t ws_bytes, moe_stream_t stream, const NormOut* norm) {
    if (int s = check_experts(W)) return s;
    if (int s = check_shared(sh)) return s;
    if (T < 0 || k < 1 || k > MOE_MAX_K || k > W->E) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!x || !W_r || !y || !ws || !aligned16(x) || !aligned16(W_r) || !aligned16(y)) return MOE_ERR_INVALID_ARG;
    if (residual && (reinterpret_cast<uintptr_t>(residual) & 7u)) return MOE_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(ws) % kWsAlign) return MOE_ERR_INVALID_ARG;
    const int I_sh = sh ? sh->I_sh : 0;
    if (ws_bytes < moe_workspace_size(T, W->E, k, W->H, W->I, I_sh)) return MOE_ERR_INVALID_ARG;
    const int a = choose_arm(arm, T, k, W->E, W->H, W->I, I_sh);
    if (a < 0) return arm == MOE_ARM_AUTO || arm == MOE_ARM_GEMV || arm == MOE_ARM_GEMM ? MOE_ERR_UNSUPPORTED
                                                                                      : MOE_ERR_INVALID_ARG;
    if (int s = check_device()) return s;
    cudaStream_t st = S(stream);
    int* status = static_cast<int*>(ws);
    Carver c(ws);
    Routing r;
    carve_routing(c, T, W->E, k, r);
    int32_t* ids = topk_ids_out ? topk_ids_out : r.ids;
    float* w = topk_w_out ? topk_w_out : r.w;
    const uint16_t* g = sh ? sh->g : nullptr;
    const int ld = W->E + (g ? 1 : 0);
    MlpCall mc{};
    mc.x = x; mc.T = T; mc.k = k; mc.W = W; mc.sh = sh; mc.logits = r.logits; mc.logit_ld = ld;
    mc.offsets = r.offsets; mc.perm = r.perm; mc.inv = r.inv; mc.active = r.active; mc.n_active = r.n_active;
    mc.topk_w = w; mc.residual = residual; mc.rows_out = nullptr; mc.y = y; mc.status = status;
    mc.norm = norm;
    if (a == MOE_ARM_GEMV) {
        GemvBufs b;
        carve_gemv(c, T, k, W->H, W->I, I_sh, b);
        // decode batches: 3 launches -- logits + x quantisation + top-k + dispatch, gate/up, down + combine
        const bool fused_routing = T <= 32;
        DecodeRoute dr;
        if (fused_routing) {
            dr.k = k; dr.ids = ids; dr.w = w; dr.counts = r.counts; dr.offsets = r.offsets; dr.perm = r.perm;
            dr.inv = r.inv; dr.active = r.active; dr.n_active = r.n_active; dr.status = status;
            dr.done = reinterpret_cast<int*>(reinterpret_cast<char*>(status) + kWsRouteOffset);
        }
        if (launch_router_logits(x, W_r, g, T, W->H, W->E, r.logits, st, b.xq, b.xmeta, act_gld(W->H), status,
                                 fused_routing ? &dr : nullptr) != cudaSuccess)
            return MOE_ERR_CUDA;
        if (!fused_routing) {
            if (launch_router_topk(r.logits, false, ld, T, W->E, k, ids, w, st) != cudaSuccess) return MOE_ERR_CUDA;
            if (launch_dispatch(ids, T * k, W->E, r.counts, r.offsets, r.perm, r.inv, r.active, r.n_active,
                                r.disp_scratch, status, st) != cudaSuccess)
                return MOE_ERR_CUDA;
        }
        return run_gemv(mc, b, true, st);
    }
    GemmBufs b;
    carve_gemm(c, T, k, W->E, W->H, W->I, I_sh, b);
    // prefill routing: the top-k launch also counts each CTA's picks per expert (at most 64 CTAs,
    // so the count table always fits: 64 * E <= 16384 for E <= 256), and the dispatch is the
    // scatter alone, writing the tile list too (no count, scan or tile launches)
    const int tpw = counted_tokens_per_warp(T, W->E);
    const int rblk = counted_ctas(T, tpw);
    if (!dispatch_counted_supported(rblk, W->E)) return MOE_ERR_UNSUPPORTED;
    // tensor-core logits in up to 4 K ranges (more CTAs issuing copies), summed by the top-k
    int parts = 1;
    if (router_tc_supported(x, W_r, g, W->H, W->E)) {
        parts = router_tc_ksplit(W->H);
        if (launch_router_logits_tc(x, W_r, g, T, W->H, W->E, r.logits, status, st, parts) != cudaSuccess)
            return MOE_ERR_CUDA;
    } else if (launch_router_logits(x, W_r, g, T, W->H, W->E, r.logits, st, nullptr, nullptr, 0, status) !=
               cudaSuccess) {
        return MOE_ERR_CUDA;
    }
    if (launch_router_topk_counted(r.logits, ld, T, W->E, k, tpw, ids, w, r.route_cnt, st, parts) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (launch_dispatch_counted(ids, T * k, W->E, kCountedWarps * tpw * k, rblk, r.route_cnt, r.counts, r.offsets,
                                r.perm, r.inv, r.active, r.n_active, status, b.tiles, b.n_tiles, st) != cudaSuccess)
        return MOE_ERR_CUDA;
    return run_gemm(mc, b, st, true);
}

}  // namespace

extern "C" {

const char* moe_status_string(int status) {
    switch (status) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED: return "unsupported request";
        case MOE_ERR_CUDA: return "CUDA error";
        case MOE_ERR_DEVICE_TIMEOUT: return "device-side wait ran out";
        case MOE_ERR_DEVICE_INDEX: return "routed expert id out of range";
        case MOE_ERR_DEVICE_RANGE: return "MXFP4 scale exponent outside the supported range";
        default: return "unknown status";
    }
}

const char* moe_version(void) { return "moe-gb300 0.1 sm_103a"; }

int moe_router_logits(const uint16_t* x, const uint16_t* W_r, const uint16_t* g, int T, int H, int E, float* logits,
                      moe_stream_t stream) {
    if (T < 0 || H < 32 || H % 32 || E < 1 || E > MOE_MAX_E) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!x || !W_r || !logits || !aligned16(x) || !aligned16(W_r) || (g && !aligned16(g))) return MOE_ERR_INVALID_ARG;
    if (int s = check_device()) return s;
    return status_of(launch_router_logits(x, W_r, g, T, H, E, logits, S(stream)));
}

int moe_router_topk(const void* logits, int logits_is_bf16, int ld, int T, int E, int k, int32_t* topk_ids,
                    float* topk_w, moe_stream_t stream) {
    if (T < 0 || E < 1 || E > MOE_MAX_E || k < 1 || k > E || k > MOE_MAX_K || ld < E) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!logits || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
    if (int s = check_device()) return s;
    return status_of(launch_router_topk(logits, logits_is_bf16 != 0, ld, T, E, k, topk_ids, topk_w, S(stream)));
}

int moe_router_topk_v(const void* logits, int logits_is_bf16, int ld, int T, int E, int k, const float* sel_bias,
                      int renormalize, float scale, int32_t* topk_ids, float* topk_w, moe_stream_t stream) {
    if (T < 0 || E < 1 || E > MOE_MAX_E || k < 1 || k > E || k > MOE_MAX_K || ld < E) return MOE_ERR_INVALID_ARG;
    if (!(scale == scale) || scale == INFINITY || scale == -INFINITY) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!logits || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
    if (sel_bias && (reinterpret_cast<uintptr_t>(sel_bias) & 3u)) return MOE_ERR_INVALID_ARG;
    if (int s = check_device()) return s;
    return status_of(launch_router_topk(logits, logits_is_bf16 != 0, ld, T, E, k, topk_ids, topk_w, S(stream),
                                        sel_bias, renormalize != 0, scale));
}

size_t moe_dispatch_workspace_size(int T, int k, int E) {
    if (T < 0 || k < 1 || E < 1) return 0;
    return kWsHead + align_up(sizeof(int32_t) * (E + 1), kWsAlign) +
           dispatch_scratch_bytes(T * k, E);
}

int moe_dispatch(const int32_t* topk_ids, int T, int k, int E, int32_t* counts, int32_t* offsets, int32_t* perm,
                 int32_t* inv, void* ws, size_t ws_bytes, moe_stream_t stream) {
    if (T < 0 || k < 1 || k > MOE_MAX_K || E < 1 || E > MOE_MAX_E) return MOE_ERR_INVALID_ARG;
    if (!offsets || !ws) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!topk_ids || !perm || !inv)) return MOE_ERR_INVALID_ARG;
    if (ws_bytes < moe_dispatch_workspace_size(T, k, E)) return MOE_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(ws) % kWsAlign) return MOE_ERR_INVALID_ARG;
    if (int s = check_device()) return s;
    Carver c(ws);
    int32_t* active = c.take<int32_t>(E + 1);
    void* scratch = c.take<char>(dispatch_scratch_bytes(T * k, E));
    int* status = static_cast<int*>(ws);
    return status_of(launch_dispatch(topk_ids, T * k, E, counts, offsets, perm, inv, active, active + E, scratch,
                                     status, S(stream)));
}

size_t moe_expert_mlp_workspace_size(int T, int k, int E, int H, int I) {
    if (T < 0 || k < 1 || E < 1 || H < 32 || I < 32) return 0;
    Carver a(nullptr), b(nullptr);
    a.take<int32_t>(E + 1);
    b.take<int32_t>(E + 1);
    GemvBufs gv;
    GemmBufs gm;
    carve_gemv(a, T, k, H, I, 0, gv);
    carve_gemm(b, T, k, E, H, I, 0, gm);
    return std::max(a.size(), b.size());
}

int moe_expert_mlp(const uint16_t* x, int T, int k, const moe_experts* W, const int32_t* offsets, const int32_t* perm,
                   float* rows, int arm, void* ws, size_t ws_bytes, moe_stream_t stream) {
    if (int s = check_experts(W)) return s;
    if (T < 0 || k < 1 || k > MOE_MAX_K || k > W->E) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!x || !offsets || !perm || !rows || !ws || !aligned16(x) || !aligned16(rows)) return MOE_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(ws) % kWsAlign) return MOE_ERR_INVALID_ARG;
    if (ws_bytes < moe_expert_mlp_workspace_size(T, k, W->E, W->H, W->I)) return MOE_ERR_INVALID_ARG;
    const int a = choose_arm(arm, T, k, W->E, W->H, W->I, 0);
    if (a < 0) return arm == MOE_ARM_AUTO || arm == MOE_ARM_GEMV || arm == MOE_ARM_GEMM ? MOE_ERR_UNSUPPORTED
                                                                                      : MOE_ERR_INVALID_ARG;
    if (int s = check_device()) return s;
    cudaStream_t st = S(stream);
    Carver c(ws);
    int32_t* active = c.take<int32_t>(W->E + 1);
    {
        KernelScope ks_("active_from_offsets", st);
        if (launch_pdl(active_from_offsets_kernel, dim3(1), dim3(256), 0, st, offsets, W->E, active, active + W->E) !=
            cudaSuccess)
            return MOE_ERR_CUDA;
    }
    MlpCall mc{};
    mc.x = x; mc.T = T; mc.k = k; mc.W = W; mc.sh = nullptr; mc.offsets = offsets; mc.perm = perm;
    mc.active = active; mc.n_active = active + W->E; mc.rows_out = rows; mc.status = static_cast<int*>(ws);
    if (a == MOE_ARM_GEMV) {
        GemvBufs b;
        carve_gemv(c, T, k, W->H, W->I, 0, b);
        return run_gemv(mc, b, false, st);
    }
    GemmBufs b;
    carve_gemm(c, T, k, W->E, W->H, W->I, 0, b);
    return run_gemm(mc, b, st);
}

int moe_combine(const float* rows, const int32_t* inv, const float* topk_w, const float* shared,
                const uint16_t* residual, int T, int k, int H, float* y, moe_stream_t stream) {
    if (T < 0 || k < 1 || k > MOE_MAX_K || H < 32 || H % 32) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!rows || !inv || !topk_w || !y || !aligned16(rows) || !aligned16(y) || (shared && !aligned16(shared)) ||
        (residual && (reinterpret_cast<uintptr_t>(residual) & 7u)))
        return MOE_ERR_INVALID_ARG;
    if (int s = check_device()) return s;
    return status_of(launch_combine(rows, inv, topk_w, false, shared, residual, T, k, H, y, S(stream)));
}

size_t moe_workspace_size(int T, int E, int k, int H, int I, int I_sh) {
    if (T < 0 || E < 1 || k < 1 || H < 32 || I < 32) return 0;
    if (I_sh < 0) I_sh = 0;
    Carver a(nullptr), b(nullptr);
    Routing r;
    carve_routing(a, T, E, k, r);
    carve_routing(b, T, E, k, r);
    GemvBufs gv;
    GemmBufs gm;
    carve_gemv(a, T, k, H, I, I_sh, gv);
    carve_gemm(b, T, k, E, H, I, I_sh, gm);
    return std::max(a.size(), b.size());
}

int moe_layer_forward(const uint16_t* x, const uint16_t* residual, const uint16_t* W_r, const moe_experts* W,
                      const moe_shared* sh, int T, int k, float* y, int32_t* topk_ids_out, float* topk_w_out, int arm,
                      void* ws, size_t ws_bytes, moe_stream_t stream) {
    return layer_forward(x, residual, W_r, W, sh, T, k, y, topk_ids_out, topk_w_out, arm, ws, ws_bytes, stream,
                         nullptr);
}

int moe_rmsnorm(const float* y, const uint16_t* gamma, int T, int H, float eps, uint16_t* y_norm,
                moe_stream_t stream) {
    if (T < 0 || H < 32 || H > MOE_MAX_H || H % 32 || !(eps >= 0.f) || eps == INFINITY) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!y || !gamma || !y_norm || !aligned16(y) || (reinterpret_cast<uintptr_t>(gamma) & 7u) ||
        (reinterpret_cast<uintptr_t>(y_norm) & 7u))
        return MOE_ERR_INVALID_ARG;
    if (int s = check_device()) return s;
    return status_of(launch_rmsnorm(y, gamma, T, H, eps, y_norm, S(stream)));
}

int moe_layer_forward_norm(const uint16_t* x, const uint16_t* residual, const uint16_t* W_r, const moe_experts* W,
                           const moe_shared* sh, int T, int k, float* y, const uint16_t* norm_gamma, float eps,
                           uint16_t* y_norm, int32_t* topk_ids_out, float* topk_w_out, int arm, void* ws,
                           size_t ws_bytes, moe_stream_t stream) {
    if (int s = check_experts(W)) return s;
    if (!(eps >= 0.f) || eps == INFINITY) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!norm_gamma || !y_norm || (reinterpret_cast<uintptr_t>(norm_gamma) & 7u) ||
                  (reinterpret_cast<uintptr_t>(y_norm) & 7u)))
        return MOE_ERR_INVALID_ARG;
    const NormOut norm{norm_gamma, eps, y_norm};
    return layer_forward(x, residual, W_r, W, sh, T, k, y, topk_ids_out, topk_w_out, arm, ws, ws_bytes, stream,
                         &norm);
}

}  // extern "C"

namespace {
__global__ void write_test_hook_kernel(TestHook* hook, long long wait_limit, int withhold) {
    pdl_wait();
    pdl_trigger();
    hook->wait_limit = wait_limit;
    hook->withhold_copy = withhold;
    hook->pad = 0;
}
}  // namespace

extern "C" {

int moe_workspace_test_timeout(void* ws, size_t ws_bytes, long long wait_limit_cycles, moe_stream_t stream) {
    if (!ws || ws_bytes < kWsHead || wait_limit_cycles < 0) return MOE_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(ws) % kWsAlign) return MOE_ERR_INVALID_ARG;
    if (int s = check_device()) return s;
    cudaStream_t st = S(stream);
    TestHook* hook = reinterpret_cast<TestHook*>(static_cast<char*>(ws) + kWsTestHookOffset);
    KernelScope ks_("write_test_hook", st);
    return status_of(launch_pdl(write_test_hook_kernel, dim3(1), dim3(1), 0, st, hook, wait_limit_cycles, 1));
}

int moe_workspace_init(void* ws, size_t ws_bytes, moe_stream_t stream) {
    if (!ws || ws_bytes < kWsHead) return MOE_ERR_INVALID_ARG;
    return status_of(cudaMemsetAsync(ws, 0, kWsHead, S(stream)));
}

int moe_mxfp4_scales(const uint8_t* e8, size_t n, uint16_t* s, void* ws, size_t ws_bytes, moe_stream_t stream) {
    if (!e8 || !s || !ws || ws_bytes < kWsHead || (reinterpret_cast<uintptr_t>(s) & 1u)) return MOE_ERR_INVALID_ARG;
    if (n == 0) return MOE_OK;
    if (int st = check_device()) return st;
    return status_of(launch_mxfp4_scales(e8, n, s, static_cast<int*>(ws), S(stream)));
}

int moe_device_status(void* ws, size_t ws_bytes, int* status, moe_stream_t stream) {
    if (!ws || !status || ws_bytes < kWsHead) return MOE_ERR_INVALID_ARG;
    int host = 0;
    cudaStream_t st = S(stream);
    if (cudaMemcpyAsync(&host, ws, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaMemsetAsync(ws, 0, kWsAlign, st) != cudaSuccess) return MOE_ERR_CUDA;
    *status = host;
    return MOE_OK;
}

}  // extern "C"
