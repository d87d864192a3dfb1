// gemv.cu -- bandwidth arm of the expert MLP (decode batches): fused int4 GEMVs.
//
// The expert weights are int4 offset-binary (value = nibble - 8) with one fp16 scale per 32
// K-columns, uploaded in the CPU byte layout (colibri PR #418 "Vulkan backend: expert tier +
// dense + MLA attention on any Vulkan 1.2 GPU", Correctness and "Grouped scales in the Vulkan
// kernels": the scale is applied to the packed-word partial).  A lane streams one 16-byte
// chunk of a weight row = 32 nibbles = exactly one scale group, so the partial of a chunk is
//     sum_c (n_c - 8) * a_c  =  sum_c n_c * a_c  -  8 * sum_c a_c
// and the group scale multiplies that partial.  The activations a (hidden rows x, and the
// SwiGLU product h for the down projection) are first written as int16 with one power-of-two
// scale per 32 values, so sum_c n_c * a_c is an exact integer dot product (dp2a: two int16 by
// two 8-bit nibbles per instruction) and the only rounding is the activation's: bf16 hidden
// values within 2^7 of their group's largest magnitude convert exactly, smaller ones round at
// 2^-15 of that magnitude; fp32 h rounds at 2^-15 of its group's largest magnitude.
//
// Kernels:
//   quantize_rows    bf16 or fp32 rows -> int16 (dp2a order) + scale + integer sum per group
//   gateup_gemv      one warp per (active expert, row i): g = W_g x, u = W_u x for the
//                    expert's bucket, h = silu(g) * u (fp32)
//   down_gemv        one CTA per NR output rows; its warps cover (row, active expert) pairs;
//                    mode ROWS writes o per dispatched row; mode COMBINE keeps w * o per
//                    (token, slot) in shared memory and sums shared row, slots by j and the
//                    residual in that order (daScript PR #3988 "dasLLAMA vulkan: a MoE that
//                    fits the card ...", combine-folded residual commit).
// The shared expert, when present, is one more "expert" whose bucket is every token.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace moe {

// position of column j (0..7) of an 8-column word in the dp2a operand order
// [c0 c2 c4 c6 c1 c3 c5 c7]
__device__ __forceinline__ int dp2a_pos(int j) { return (j & 1) ? 4 + (j >> 1) : (j >> 1); }

// ------------------------------------------------------------------ activation quantisation
struct QuantSeg {
    const void* src;  // bf16 (is_bf16) or fp32 rows [rows][K]
    int is_bf16;
    int rows, K;
    int16_t* q;       // [rows][K], dp2a order within each 8-column word
    float* sc;        // [rows][K/32]
    int* sum;         // [rows][K/32]
};

__global__ void __launch_bounds__(256) quantize_rows_kernel(QuantSeg s0, QuantSeg s1) {
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
    const float amax = warp_max(fabsf(v));
    int q = 0;
    float scale = 1.f;
    if (amax > 0.f && amax <= 3.0e38f) {
        int ex;
        frexpf(amax, &ex);  // amax = m * 2^ex, m in [0.5, 1): |v| * 2^(15 - ex) < 2^15
        q = __float2int_rn(ldexpf(v, 15 - ex));
        q = max(-32767, min(32767, q));
        scale = ldexpf(1.f, ex - 15);
    }
    const int dst = grp * 32 + (lane & ~7) + dp2a_pos(lane & 7);
    s.q[static_cast<size_t>(row) * s.K + dst] = static_cast<int16_t>(q);
    const int qs = __reduce_add_sync(0xffffffffu, q);
    if (lane == 0) {
        s.sc[row * ng + grp] = scale;
        s.sum[row * ng + grp] = qs;
    }
}

cudaError_t launch_quantize(const QuantArgs& a, cudaStream_t st) {
    QuantSeg s0{a.src0, a.src0_bf16, a.rows0, a.K0, a.q0, a.sc0, a.sum0};
    QuantSeg s1{a.src1, a.src1_bf16, a.rows1, a.K1, a.q1, a.sc1, a.sum1};
    if (!a.src1) { s1.rows = 0; s1.K = 32; }
    const long warps = static_cast<long>(s0.rows) * (s0.K / 32) + static_cast<long>(s1.rows) * (s1.K / 32);
    if (warps == 0) return cudaSuccess;
    const long blocks = (warps + 7) / 8;
    {
        KernelScope ks_("quantize_rows", st);
        quantize_rows_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(s0, s1);
    }
    return cudaGetLastError();
}

// ------------------------------------------------------------------ int4 x int16 chunk dot
// w: 16 bytes = 4 words = 32 nibbles (columns 0..31 of a group);
// a: the group's 32 int16 activations in dp2a order (64 bytes).
__device__ __forceinline__ int dot_chunk(const uint4 w, const int16_t* __restrict__ a) {
    const uint4* ap = reinterpret_cast<const uint4*>(a);
    int acc = 0;
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const uint4 av = __ldg(ap + m);
        const uint32_t lo = ww[m] & 0x0F0F0F0Fu;
        const uint32_t hi = (ww[m] >> 4) & 0x0F0F0F0Fu;
        acc = __dp2a_lo(static_cast<int>(av.x), static_cast<int>(lo), acc);
        acc = __dp2a_hi(static_cast<int>(av.y), static_cast<int>(lo), acc);
        acc = __dp2a_lo(static_cast<int>(av.z), static_cast<int>(hi), acc);
        acc = __dp2a_hi(static_cast<int>(av.w), static_cast<int>(hi), acc);
    }
    return acc;
}

__device__ __forceinline__ float silu(float z) { return z / (1.f + expf(-z)); }

// ------------------------------------------------------------------ gate + up + SwiGLU
// Items: n_active * I routed rows, then I_sh shared rows.  CPL = 16-byte chunks per lane
// (ceil(H / 1024)).  TB = tokens per accumulation pass.
template <int CPL, int TB>
__global__ void __launch_bounds__(256) gateup_gemv_kernel(GemvArgs p) {
    const int lane = threadIdx.x & 31;
    const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int nw = (gridDim.x * blockDim.x) >> 5;
    const int n_act = *p.n_active;
    const long n_routed = static_cast<long>(n_act) * p.I;
    const long items = n_routed + (p.sh_I > 0 ? p.sh_I : 0);
    const int nch = p.H / 32;
    const int ng = nch;

    auto setup = [&](long it, const uint8_t*& qg, const uint8_t*& qu, const uint16_t*& sg, const uint16_t*& su) {
        if (it < n_routed) {
            const int e = p.active[it / p.I];
            const int i = static_cast<int>(it % p.I);
            const size_t row = static_cast<size_t>(e) * p.I + i;
            qg = p.gate_q + row * (p.H / 2);
            qu = p.up_q + row * (p.H / 2);
            sg = p.gate_s + row * ng;
            su = p.up_s + row * ng;
        } else {
            const size_t row = static_cast<size_t>(it - n_routed);
            qg = p.sh_gate_q + row * (p.H / 2);
            qu = p.sh_up_q + row * (p.H / 2);
            sg = p.sh_gate_s + row * ng;
            su = p.sh_up_s + row * ng;
        }
    };

    uint4 ng_buf[CPL], nu_buf[CPL];
    long it = gw;
    if (it < items) {
        const uint8_t *qg, *qu;
        const uint16_t *sg, *su;
        setup(it, qg, qu, sg, su);
#pragma unroll
        for (int j = 0; j < CPL; ++j) {
            const int c = lane + 32 * j;
            if (c < nch) {
                ng_buf[j] = ldg_stream(qg + static_cast<size_t>(c) * 16);
                nu_buf[j] = ldg_stream(qu + static_cast<size_t>(c) * 16);
            }
        }
    }
    for (; it < items; it += nw) {
        uint4 wg[CPL], wu[CPL];
#pragma unroll
        for (int j = 0; j < CPL; ++j) { wg[j] = ng_buf[j]; wu[j] = nu_buf[j]; }
        const uint8_t *qg, *qu;
        const uint16_t *sg, *su;
        setup(it, qg, qu, sg, su);
        float fsg[CPL], fsu[CPL];
#pragma unroll
        for (int j = 0; j < CPL; ++j) {
            const int c = lane + 32 * j;
            fsg[j] = (c < nch) ? __half2float(__ushort_as_half(__ldg(sg + c))) : 0.f;
            fsu[j] = (c < nch) ? __half2float(__ushort_as_half(__ldg(su + c))) : 0.f;
        }
        // prefetch the next item's chunks
        const long nit = it + nw;
        if (nit < items) {
            const uint8_t *qg2, *qu2;
            const uint16_t *sg2, *su2;
            setup(nit, qg2, qu2, sg2, su2);
#pragma unroll
            for (int j = 0; j < CPL; ++j) {
                const int c = lane + 32 * j;
                if (c < nch) {
                    ng_buf[j] = ldg_stream(qg2 + static_cast<size_t>(c) * 16);
                    nu_buf[j] = ldg_stream(qu2 + static_cast<size_t>(c) * 16);
                }
            }
        }
        // bucket of this item
        int rb, re, ldh, i;
        float* hout;
        const bool shared = it >= n_routed;
        if (!shared) {
            const int e = p.active[it / p.I];
            i = static_cast<int>(it % p.I);
            rb = p.offsets[e];
            re = p.offsets[e + 1];
            hout = p.h;
            ldh = p.I;
        } else {
            i = static_cast<int>(it - n_routed);
            rb = 0;
            re = p.T;
            hout = p.sh_h;
            ldh = p.sh_I;
        }
        for (int r0 = rb; r0 < re; r0 += TB) {
            float ag[TB], au[TB];
#pragma unroll
            for (int b = 0; b < TB; ++b) { ag[b] = 0.f; au[b] = 0.f; }
#pragma unroll
            for (int b = 0; b < TB; ++b) {
                if (r0 + b < re) {
                    const int t = shared ? (r0 + b) : (p.perm[r0 + b] / p.k);
                    const int16_t* xq = p.xq + static_cast<size_t>(t) * p.H;
                    const float* xs = p.xsc + static_cast<size_t>(t) * ng;
                    const int* xsum = p.xsum + static_cast<size_t>(t) * ng;
#pragma unroll
                    for (int j = 0; j < CPL; ++j) {
                        const int c = lane + 32 * j;
                        if (c < nch) {
                            const int16_t* a = xq + c * 32;
                            const int s8 = 8 * __ldg(xsum + c);
                            const float xsc = __ldg(xs + c);
                            const int dg = dot_chunk(wg[j], a) - s8;
                            const int du = dot_chunk(wu[j], a) - s8;
                            ag[b] = fmaf(static_cast<float>(dg), fsg[j] * xsc, ag[b]);
                            au[b] = fmaf(static_cast<float>(du), fsu[j] * xsc, au[b]);
                        }
                    }
                }
            }
#pragma unroll
            for (int b = 0; b < TB; ++b) {
                const float g = warp_sum(ag[b]);
                const float u = warp_sum(au[b]);
                if (lane == b && r0 + b < re) hout[static_cast<size_t>(r0 + b) * ldh + i] = silu(g) * u;
            }
        }
    }
}

// ------------------------------------------------------------------ down projection
constexpr int kDownNR = 4;        // output rows per CTA
constexpr int kDownWarps = 8;

template <int CPL, int TB, bool COMBINE>
__global__ void __launch_bounds__(kDownWarps * 32) down_gemv_kernel(GemvArgs p) {
    extern __shared__ float contrib[];  // COMBINE: [NR][T*k] slot terms, then [NR][T] shared terms
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int n0 = blockIdx.x * kDownNR;
    const int n_act = *p.n_active;
    const bool has_sh = p.sh_I > 0;
    const int items = kDownNR * (n_act + (has_sh ? 1 : 0));
    const int TK = p.T * p.k;
    float* slot_terms = contrib;
    float* sh_terms = contrib + kDownNR * TK;
    if (COMBINE) {
        for (int i = threadIdx.x; i < kDownNR * (TK + p.T); i += blockDim.x) contrib[i] = 0.f;
        __syncthreads();
    }

    auto setup = [&](int it, const uint8_t*& q, const uint16_t*& s, int& K, int& n) {
        const int rr = it % kDownNR;
        const int ai = it / kDownNR;
        n = n0 + rr;
        if (ai < n_act) {
            const int e = p.active[ai];
            K = p.I;
            const size_t row = static_cast<size_t>(e) * p.H + n;
            q = p.down_q + row * (K / 2);
            s = p.down_s + row * (K / 32);
        } else {
            K = p.sh_I;
            q = p.sh_down_q + static_cast<size_t>(n) * (K / 2);
            s = p.sh_down_s + static_cast<size_t>(n) * (K / 32);
        }
    };

    uint4 nbuf[CPL];
    int it = wid;
    if (it < items) {
        const uint8_t* q;
        const uint16_t* s;
        int K, n;
        setup(it, q, s, K, n);
        if (n < p.H) {
#pragma unroll
            for (int j = 0; j < CPL; ++j) {
                const int c = lane + 32 * j;
                if (c < K / 32) nbuf[j] = ldg_stream(q + static_cast<size_t>(c) * 16);
            }
        }
    }
    for (; it < items; it += kDownWarps) {
        uint4 w[CPL];
#pragma unroll
        for (int j = 0; j < CPL; ++j) w[j] = nbuf[j];
        const uint8_t* q;
        const uint16_t* s;
        int K, n;
        setup(it, q, s, K, n);
        const int nch = K / 32;
        const bool live = n < p.H;
        float fs[CPL];
#pragma unroll
        for (int j = 0; j < CPL; ++j) {
            const int c = lane + 32 * j;
            fs[j] = (live && c < nch) ? __half2float(__ushort_as_half(__ldg(s + c))) : 0.f;
        }
        const int nit = it + kDownWarps;
        if (nit < items) {
            const uint8_t* q2;
            const uint16_t* s2;
            int K2, n2;
            setup(nit, q2, s2, K2, n2);
            if (n2 < p.H) {
#pragma unroll
                for (int j = 0; j < CPL; ++j) {
                    const int c = lane + 32 * j;
                    if (c < K2 / 32) nbuf[j] = ldg_stream(q2 + static_cast<size_t>(c) * 16);
                }
            }
        }
        if (!live) continue;
        const int ai = it / kDownNR;
        const int rr = it % kDownNR;
        const bool shared = ai >= n_act;
        int rb, re;
        if (!shared) {
            const int e = p.active[ai];
            rb = p.offsets[e];
            re = p.offsets[e + 1];
        } else {
            rb = 0;
            re = p.T;
        }
        const int16_t* hq = shared ? p.sh_hq : p.hq;
        const float* hsc = shared ? p.sh_hsc : p.hsc;
        const int* hsum = shared ? p.sh_hsum : p.hsum;
        for (int r0 = rb; r0 < re; r0 += TB) {
            float acc[TB];
#pragma unroll
            for (int b = 0; b < TB; ++b) acc[b] = 0.f;
#pragma unroll
            for (int b = 0; b < TB; ++b) {
                if (r0 + b < re) {
                    const size_t r = static_cast<size_t>(r0 + b);
                    const int16_t* a = hq + r * K;
#pragma unroll
                    for (int j = 0; j < CPL; ++j) {
                        const int c = lane + 32 * j;
                        if (c < nch) {
                            const int d = dot_chunk(w[j], a + c * 32) - 8 * __ldg(hsum + r * nch + c);
                            acc[b] = fmaf(static_cast<float>(d), fs[j] * __ldg(hsc + r * nch + c), acc[b]);
                        }
                    }
                }
            }
#pragma unroll
            for (int b = 0; b < TB; ++b) {
                const float o = warp_sum(acc[b]);
                if (lane == b && r0 + b < re) {
                    const int r = r0 + b;
                    if (COMBINE) {
                        if (shared) {
                            float gate = 1.f;
                            if (p.sh_gate_logit) {
                                const float z = p.sh_gate_logit[static_cast<size_t>(r) * p.logit_ld];
                                gate = 1.f / (1.f + expf(-z));
                            }
                            sh_terms[rr * p.T + r] = gate * o;
                        } else {
                            const int a = p.perm[r];
                            slot_terms[rr * TK + a] = p.topk_w[a] * o;
                        }
                    } else if (shared) {
                        float gate = 1.f;
                        if (p.sh_gate_logit) {
                            const float z = p.sh_gate_logit[static_cast<size_t>(r) * p.logit_ld];
                            gate = 1.f / (1.f + expf(-z));
                        }
                        p.sh_rows_out[static_cast<size_t>(r) * p.H + n] = gate * o;
                    } else {
                        p.rows_out[static_cast<size_t>(r) * p.H + n] = o;
                    }
                }
            }
        }
    }
    if (!COMBINE) return;
    __syncthreads();
    // y[t][n] = shared term + slots in order j + residual
    for (int idx = threadIdx.x; idx < kDownNR * p.T; idx += blockDim.x) {
        const int rr = idx / p.T, t = idx % p.T;
        const int n = n0 + rr;
        if (n >= p.H) continue;
        float y = has_sh ? sh_terms[rr * p.T + t] : 0.f;
        for (int j = 0; j < p.k; ++j) y += slot_terms[rr * TK + t * p.k + j];
        if (p.residual) y += bf16_to_f32(p.residual[static_cast<size_t>(t) * p.H + n]);
        p.y[static_cast<size_t>(t) * p.H + n] = y;
    }
}

static int cpl_for(int K) {
    const int nch = K / 32;
    const int c = (nch + 31) / 32;
    if (c <= 1) return 1;
    if (c <= 2) return 2;
    if (c <= 4) return 4;
    if (c <= 8) return 8;
    return -1;
}

bool gemv_supported(int H, int I, int I_sh) {
    return cpl_for(H) > 0 && cpl_for(I) > 0 && (I_sh <= 0 || cpl_for(I_sh) > 0);
}

cudaError_t launch_gateup_gemv(const GemvArgs& p, int num_sms, cudaStream_t st) {
    const int cpl = cpl_for(p.H);
    // enough warps to cover every (expert, row) item of a full decode batch in one pass,
    // capped at 16 resident CTAs of 8 warps per SM
    long max_items = static_cast<long>(p.max_active) * p.I + (p.sh_I > 0 ? p.sh_I : 0);
    long blocks = (max_items + 7) / 8;
    blocks = std::min<long>(blocks, static_cast<long>(num_sms) * 8);
    if (blocks < 1) blocks = 1;
    const dim3 g(static_cast<unsigned>(blocks)), b(256);
    KernelScope ks_("gateup_gemv", st);
    switch (cpl) {
        case 1: gateup_gemv_kernel<1, 4><<<g, b, 0, st>>>(p); break;
        case 2: gateup_gemv_kernel<2, 4><<<g, b, 0, st>>>(p); break;
        case 4: gateup_gemv_kernel<4, 4><<<g, b, 0, st>>>(p); break;
        case 8: gateup_gemv_kernel<8, 2><<<g, b, 0, st>>>(p); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_down_gemv(const GemvArgs& p, bool combine, cudaStream_t st) {
    int cpl = cpl_for(p.I);
    if (p.sh_I > 0) cpl = std::max(cpl, cpl_for(p.sh_I));
    const dim3 g((p.H + kDownNR - 1) / kDownNR), b(kDownWarps * 32);
    const size_t smem = combine ? sizeof(float) * kDownNR * (static_cast<size_t>(p.T) * p.k + p.T) : 0;
    KernelScope ks_(combine ? "down_gemv_combine" : "down_gemv_rows", st);
#define MOE_DOWN_CASE(C)                                                              \
    case C:                                                                           \
        if (combine)                                                                  \
            down_gemv_kernel<C, 4, true><<<g, b, smem, st>>>(p);                      \
        else                                                                          \
            down_gemv_kernel<C, 4, false><<<g, b, smem, st>>>(p);                     \
        break;
    switch (cpl) {
        MOE_DOWN_CASE(1)
        MOE_DOWN_CASE(2)
        MOE_DOWN_CASE(4)
        MOE_DOWN_CASE(8)
        default: return cudaErrorInvalidValue;
    }
#undef MOE_DOWN_CASE
    return cudaGetLastError();
}

}  // namespace moe
