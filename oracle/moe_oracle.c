/*
 * moe_oracle.c -- plain fp64 CPU oracle of the routed Mixture-of-Experts layer.
 *
 * TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT (see moe_oracle.h).  Written for
 * a reader checking it against the pages by eye: one loop per definition, fp64
 * throughout, no blocking, fusion or reordering.  Independent rows (router
 * logits per token, expert rows, shared-expert tokens) may be spread over
 * worker threads (mo_set_threads); each row is still computed by the same
 * sequential loop, so the results do not depend on the thread count.
 *
 * Parity pins (tests/test_oracle_pins.py): brute-force full sort for top-k,
 * hand-decoded nibbles (int4 and MXFP4), closed forms of the MLP, the MXFP4 MLP against
 * its exact int4 twin, dispatch invariants, the
 * zero-weight invariance of the combine, and tests/golden fixtures.
 */
#define _POSIX_C_SOURCE 200809L
#include "moe_oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* ---- worker threads over independent rows (no arithmetic here) */
#define MO_MAX_THREADS 256
static int g_threads = 1;

void mo_set_threads(int n) { g_threads = n < 1 ? 1 : (n > MO_MAX_THREADS ? MO_MAX_THREADS : n); }
int mo_get_threads(void) { return g_threads; }

typedef int (*mo_row_fn)(void* ctx, long i);
struct mo_job {
    mo_row_fn fn;
    void* ctx;
    long n;
    int nthr, tid, rc;
};

/* Thread tid takes rows tid, tid + nthr, ... and stops at its first error. */
static void* mo_worker(void* arg) {
    struct mo_job* j = (struct mo_job*)arg;
    for (long i = j->tid; i < j->n; i += j->nthr) {
        int rc = j->fn(j->ctx, i);
        if (rc) {
            j->rc = rc;
            break;
        }
    }
    return NULL;
}

/* Runs fn(ctx, i) for i = 0 .. n-1; returns the first non-zero code in thread order. */
static int mo_for_rows(long n, mo_row_fn fn, void* ctx) {
    int nthr = g_threads;
    if (n < nthr) nthr = (int)(n > 0 ? n : 1);
    struct mo_job jobs[MO_MAX_THREADS];
    pthread_t th[MO_MAX_THREADS];
    int started[MO_MAX_THREADS];
    for (int t = 0; t < nthr; ++t) {
        jobs[t].fn = fn; jobs[t].ctx = ctx; jobs[t].n = n;
        jobs[t].nthr = nthr; jobs[t].tid = t; jobs[t].rc = 0;
        started[t] = t > 0 && pthread_create(&th[t], NULL, mo_worker, &jobs[t]) == 0;
    }
    for (int t = 0; t < nthr; ++t)
        if (!started[t]) mo_worker(&jobs[t]);  /* thread 0, or a thread that could not start */
    int rc = 0;
    for (int t = 0; t < nthr; ++t) {
        if (started[t]) pthread_join(th[t], NULL);
        if (!rc) rc = jobs[t].rc;
    }
    return rc;
}

/* bf16 is the top half of an IEEE binary32; widening is exact. */
double mo_bf16_to_f64(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* IEEE binary16, decoded field by field (normal, subnormal, inf/nan). */
double mo_f16_to_f64(uint16_t bits) {
    int sign = (bits >> 15) & 1;
    int ex = (bits >> 10) & 0x1F;
    int man = bits & 0x3FF;
    double v;
    if (ex == 0)
        v = ldexp((double)man, -24);              /* man/1024 * 2^-14 */
    else if (ex == 31)
        v = man ? NAN : INFINITY;
    else
        v = ldexp(1.0 + (double)man / 1024.0, ex - 15);
    return sign ? -v : v;
}

/* Every fp16 bit pattern decoded once by mo_f16_to_f64, when the library is
 * loaded (a lookup instead of a per-weight ldexp; the values are the same). */
static double g_f16_table[65536];
__attribute__((constructor)) static void fill_f16_table(void) {
    for (int b = 0; b < 65536; ++b) g_f16_table[b] = mo_f16_to_f64((uint16_t)b);
}
static double f16_value(uint16_t bits) { return g_f16_table[bits]; }

/* One weight element of an int4 matrix (colibri #418, "Correctness": int4 is
 * offset-binary, value = nibble - 8, in the CPU byte layout; "Grouped scales in
 * the Vulkan kernels": one scale per group of K-columns, here 32). */
static double weight_at(const uint8_t* q, const uint16_t* s, int K, int n, int c) {
    uint8_t byte = q[(size_t)n * (K / 2) + c / 2];
    int nib = (c & 1) ? (byte >> 4) : (byte & 0xF);
    return (double)(nib - 8) * f16_value(s[(size_t)n * (K / 32) + c / 32]);
}

int mo_dequant(const uint8_t* q, const uint16_t* s, int rows, int K, double* w) {
    if (!q || !s || !w || rows < 0 || K <= 0 || K % 32) return -1;
    for (int n = 0; n < rows; ++n)
        for (int c = 0; c < K; ++c)
            w[(size_t)n * K + c] = weight_at(q, s, K, n, c);
    return 0;
}

/* e2m1 (OCP Microscaling formats, FP4 E2M1), decoded field by field: sign bit 3, exponent
 * bits 2..1 with bias 1, mantissa bit 0; a zero exponent field is subnormal (m * 2^-1). */
double mo_e2m1_to_f64(int nibble) {
    int sign = (nibble >> 3) & 1;
    int ex = (nibble >> 1) & 3;
    int man = nibble & 1;
    double v = ex == 0 ? 0.5 * man : ldexp(1.0 + 0.5 * man, ex - 1);
    return sign ? -v : v;
}

/* ue8m0 (OCP Microscaling formats, E8M0 scale): 2^(e - 127); e = 255 is NaN. */
double mo_ue8m0_to_f64(uint8_t e) { return e == 255 ? NAN : ldexp(1.0, (int)e - 127); }

/* One weight element of an MXFP4 matrix (colibri #418, fmt=7: an e2m1 nibble times the
 * power-of-two scale of its 32-column group), in the int4 byte layout. */
static double weight_at_mxfp4(const uint8_t* q, const uint8_t* e8, int K, int n, int c) {
    uint8_t byte = q[(size_t)n * (K / 2) + c / 2];
    int nib = (c & 1) ? (byte >> 4) : (byte & 0xF);
    return mo_e2m1_to_f64(nib) * mo_ue8m0_to_f64(e8[(size_t)n * (K / 32) + c / 32]);
}

static int mxfp4_scales_finite(const uint8_t* e8, size_t n) {
    for (size_t i = 0; i < n; ++i)
        if (e8[i] == 255) return 0;
    return 1;
}

int mo_dequant_mxfp4(const uint8_t* q, const uint8_t* e8, int rows, int K, double* w) {
    if (!q || !e8 || !w || rows < 0 || K <= 0 || K % 32) return -1;
    if (!mxfp4_scales_finite(e8, (size_t)rows * (K / 32))) return -2;
    for (int n = 0; n < rows; ++n)
        for (int c = 0; c < K; ++c)
            w[(size_t)n * K + c] = weight_at_mxfp4(q, e8, K, n, c);
    return 0;
}

/* Weight element (n, c) of a matrix in format fmt; s is fp16 scales or ue8m0 exponents. */
static double weight_fmt(int fmt, const uint8_t* q, const void* s, int K, int n, int c) {
    return fmt == MO_FMT_MXFP4 ? weight_at_mxfp4(q, (const uint8_t*)s, K, n, c)
                               : weight_at(q, (const uint16_t*)s, K, n, c);
}

/* Bytes of one scale entry of format fmt. */
static size_t scale_bytes(int fmt) { return fmt == MO_FMT_MXFP4 ? 1 : 2; }

/* Router logits: one GEMV row per expert over the hidden row, and the shared
 * expert's gate logit as one more row "past the router's logits"
 * (dasLLAMA #3988, decode span and routed-block commits). */
struct logits_ctx {
    const uint16_t *x, *W_r, *g;
    int H, E;
    double* logits;
};

static int logits_token(void* vc, long t) {
    const struct logits_ctx* c = (const struct logits_ctx*)vc;
    int H = c->H, E = c->E, ld = E + (c->g ? 1 : 0);
    for (int e = 0; e < E; ++e) {
        double acc = 0.0;
        for (int h = 0; h < H; ++h)
            acc += mo_bf16_to_f64(c->x[(size_t)t * H + h]) * mo_bf16_to_f64(c->W_r[(size_t)e * H + h]);
        c->logits[(size_t)t * ld + e] = acc;
    }
    if (c->g) {
        double acc = 0.0;
        for (int h = 0; h < H; ++h)
            acc += mo_bf16_to_f64(c->x[(size_t)t * H + h]) * mo_bf16_to_f64(c->g[h]);
        c->logits[(size_t)t * ld + E] = acc;
    }
    return 0;
}

int mo_router_logits(const uint16_t* x, const uint16_t* W_r, const uint16_t* g,
                     int T, int H, int E, double* logits) {
    if (!x || !W_r || !logits || T < 0 || H <= 0 || E <= 0) return -1;
    struct logits_ctx c = {x, W_r, g, H, E, logits};
    return mo_for_rows(T, logits_token, &c);
}

/* Softmax top-k router (vllm.cpp #481, warp-router commit: softmax over the
 * row, pick k with a -inf mask, lowest index wins a tie; dasLLAMA #3988,
 * routed-block commit: per-row top-k "renormalized").  k rounds of argmax over
 * the unmasked experts with a strict '>' so the lowest index keeps a tie; the
 * picks are then written in ascending expert id.  Weights: the full softmax
 * over all E logits, renormalised over the k picks. */
int mo_router_topk(const double* logits, int ld, int T, int E, int k,
                   int32_t* ids, double* w) {
    if (!logits || !ids || !w || T < 0 || E <= 0 || ld < E || k < 1 || k > E) return -1;
    unsigned char* picked = (unsigned char*)malloc((size_t)E);
    double* p = (double*)malloc(sizeof(double) * (size_t)E);
    if (!picked || !p) { free(picked); free(p); return -1; }
    int rc = 0;
    for (int t = 0; t < T && rc == 0; ++t) {
        const double* l = logits + (size_t)t * ld;
        for (int e = 0; e < E; ++e)
            if (!isfinite(l[e])) rc = -2;
        if (rc) break;
        memset(picked, 0, (size_t)E);
        for (int round = 0; round < k; ++round) {
            int best = -1;
            for (int e = 0; e < E; ++e)
                if (!picked[e] && (best < 0 || l[e] > l[best])) best = e;
            picked[best] = 1;
        }
        double m = l[0];
        for (int e = 1; e < E; ++e)
            if (l[e] > m) m = l[e];
        double z = 0.0;
        for (int e = 0; e < E; ++e) z += exp(l[e] - m);
        for (int e = 0; e < E; ++e) p[e] = exp(l[e] - m) / z;
        double psel = 0.0;
        for (int e = 0; e < E; ++e)
            if (picked[e]) psel += p[e];
        int j = 0;
        for (int e = 0; e < E; ++e) {
            if (!picked[e]) continue;
            ids[(size_t)t * k + j] = e;
            w[(size_t)t * k + j] = p[e] / psel;
            ++j;
        }
    }
    free(picked);
    free(p);
    return rc;
}

/* Router variants: the definition written out step by step (see moe_oracle.h). */
int mo_router_topk_v(const double* logits, int ld, int T, int E, int k, const double* bias,
                     int renormalize, double scale, int32_t* ids, double* w) {
    if (!logits || !ids || !w || T < 0 || E <= 0 || ld < E || k < 1 || k > E) return -1;
    unsigned char* picked = (unsigned char*)malloc((size_t)E);
    double* sc = (double*)malloc(sizeof(double) * (size_t)E);
    double* p = (double*)malloc(sizeof(double) * (size_t)E);
    if (!picked || !sc || !p) { free(picked); free(sc); free(p); return -1; }
    int rc = 0;
    for (int t = 0; t < T && rc == 0; ++t) {
        const double* l = logits + (size_t)t * ld;
        for (int e = 0; e < E; ++e) {
            sc[e] = l[e] + (bias ? bias[e] : 0.0);
            if (!isfinite(l[e]) || !isfinite(sc[e])) rc = -2;
        }
        if (rc) break;
        /* selection: k rounds of argmax over the biased scores, strict '>' */
        memset(picked, 0, (size_t)E);
        for (int round = 0; round < k; ++round) {
            int best = -1;
            for (int e = 0; e < E; ++e)
                if (!picked[e] && (best < 0 || sc[e] > sc[best])) best = e;
            picked[best] = 1;
        }
        /* weights: softmax of the unbiased logits over all E */
        double m = l[0];
        for (int e = 1; e < E; ++e)
            if (l[e] > m) m = l[e];
        double z = 0.0;
        for (int e = 0; e < E; ++e) z += exp(l[e] - m);
        for (int e = 0; e < E; ++e) p[e] = exp(l[e] - m) / z;
        double psel = 0.0;
        for (int e = 0; e < E; ++e)
            if (picked[e]) psel += p[e];
        int q = 0;
        for (int e = 0; e < E; ++e) {
            if (!picked[e]) continue;
            ids[(size_t)t * k + q] = e;
            w[(size_t)t * k + q] = (renormalize ? p[e] / psel : p[e]) * scale;
            ++q;
        }
    }
    free(picked); free(sc); free(p);
    return rc;
}

/* Bucket schedule (dasLLAMA #3988, routed-block commit: thread e counts expert
 * e's slots, exclusive scans place the buckets, the slot map lands in slot
 * order).  counts[e] = #{slots a : ids[a] == e}; offsets = exclusive scan with
 * offsets[E] = T*k; perm lists, bucket by bucket, the slots a in ascending
 * order; inv[perm[r]] = r. */
int mo_dispatch(const int32_t* ids, int T, int k, int E, int32_t* counts,
                int32_t* offsets, int32_t* perm, int32_t* inv) {
    if (!ids || !counts || !offsets || !perm || !inv || T < 0 || k < 1 || E <= 0) return -1;
    int n = T * k;
    for (int a = 0; a < n; ++a)
        if (ids[a] < 0 || ids[a] >= E) return -1;
    for (int e = 0; e < E; ++e) {
        counts[e] = 0;
        for (int a = 0; a < n; ++a)
            if (ids[a] == e) ++counts[e];
    }
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    int r = 0;
    for (int e = 0; e < E; ++e)
        for (int a = 0; a < n; ++a)
            if (ids[a] == e) perm[r++] = a;
    for (int q = 0; q < n; ++q) inv[perm[q]] = q;
    return 0;
}

static double silu(double z) { return z / (1.0 + exp(-z)); }

/* The fused expert group "gate+up+silu->down" (colibri #418, "Summary"):
 * g = W_g x, u = W_u x, h = silu(g) * u, o = W_d h. */
int mo_expert_row_fmt(const uint16_t* x_row, int H, int I, int fmt,
                      const uint8_t* gq, const void* gs,
                      const uint8_t* uq, const void* us,
                      const uint8_t* dq, const void* ds, double* o) {
    if (!x_row || !gq || !gs || !uq || !us || !dq || !ds || !o) return -1;
    if (H <= 0 || I <= 0 || H % 32 || I % 32) return -1;
    if (fmt != MO_FMT_INT4 && fmt != MO_FMT_MXFP4) return -1;
    if (fmt == MO_FMT_MXFP4 &&
        (!mxfp4_scales_finite((const uint8_t*)gs, (size_t)I * (H / 32)) ||
         !mxfp4_scales_finite((const uint8_t*)us, (size_t)I * (H / 32)) ||
         !mxfp4_scales_finite((const uint8_t*)ds, (size_t)H * (I / 32))))
        return -2;
    double* h = (double*)malloc(sizeof(double) * (size_t)I);
    if (!h) return -1;
    for (int i = 0; i < I; ++i) {
        double g = 0.0, u = 0.0;
        for (int c = 0; c < H; ++c) {
            double xv = mo_bf16_to_f64(x_row[c]);
            g += weight_fmt(fmt, gq, gs, H, i, c) * xv;
            u += weight_fmt(fmt, uq, us, H, i, c) * xv;
        }
        h[i] = silu(g) * u;
    }
    for (int n = 0; n < H; ++n) {
        double acc = 0.0;
        for (int i = 0; i < I; ++i) acc += weight_fmt(fmt, dq, ds, I, n, i) * h[i];
        o[n] = acc;
    }
    free(h);
    return 0;
}

int mo_expert_row(const uint16_t* x_row, int H, int I,
                  const uint8_t* gq, const uint16_t* gs,
                  const uint8_t* uq, const uint16_t* us,
                  const uint8_t* dq, const uint16_t* ds, double* o) {
    return mo_expert_row_fmt(x_row, H, I, MO_FMT_INT4, gq, gs, uq, us, dq, ds, o);
}

struct mlp_ctx {
    const uint16_t* x;
    int H, I, E, k, fmt;
    const uint8_t *gate_q, *up_q, *down_q;
    const uint8_t *gs, *us, *ds;  /* scale arrays walked in bytes */
    size_t gq_sz, gs_sz, dq_sz, ds_sz;
    const int32_t *ids, *perm;
    const uint8_t* token_mask;
    double* rows;
};

/* Dispatched row r: a = perm[r], t = a / k, e = ids[a]; rows[r] = expert e on x[t]. */
static int mlp_row(void* vc, long r) {
    const struct mlp_ctx* c = (const struct mlp_ctx*)vc;
    int a = c->perm[r], t = a / c->k, e = c->ids[a];
    if (e < 0 || e >= c->E) return -1;
    if (c->token_mask && !c->token_mask[t]) return 0;
    return mo_expert_row_fmt(c->x + (size_t)t * c->H, c->H, c->I, c->fmt,
                             c->gate_q + e * c->gq_sz, c->gs + e * c->gs_sz,
                             c->up_q + e * c->gq_sz, c->us + e * c->gs_sz,
                             c->down_q + e * c->dq_sz, c->ds + e * c->ds_sz,
                             c->rows + (size_t)r * c->H);
}

int mo_expert_mlp_fmt(const uint16_t* x, int T, int H, int I, int E, int k, int fmt,
                      const uint8_t* gate_q, const void* gate_s,
                      const uint8_t* up_q, const void* up_s,
                      const uint8_t* down_q, const void* down_s,
                      const int32_t* ids, const int32_t* perm,
                      const uint8_t* token_mask, double* rows) {
    if (!x || !ids || !perm || !rows || T < 0 || E <= 0 || k < 1) return -1;
    if (!gate_s || !up_s || !down_s) return -1;
    struct mlp_ctx c;
    c.x = x; c.H = H; c.I = I; c.E = E; c.k = k; c.fmt = fmt;
    c.gate_q = gate_q; c.up_q = up_q; c.down_q = down_q;
    c.gs = (const uint8_t*)gate_s; c.us = (const uint8_t*)up_s; c.ds = (const uint8_t*)down_s;
    c.gq_sz = (size_t)I * (H / 2); c.gs_sz = (size_t)I * (H / 32) * scale_bytes(fmt);
    c.dq_sz = (size_t)H * (I / 2); c.ds_sz = (size_t)H * (I / 32) * scale_bytes(fmt);
    c.ids = ids; c.perm = perm; c.token_mask = token_mask; c.rows = rows;
    return mo_for_rows((long)T * k, mlp_row, &c);
}

int mo_expert_mlp(const uint16_t* x, int T, int H, int I, int E, int k,
                  const uint8_t* gate_q, const uint16_t* gate_s,
                  const uint8_t* up_q, const uint16_t* up_s,
                  const uint8_t* down_q, const uint16_t* down_s,
                  const int32_t* ids, const int32_t* perm,
                  const uint8_t* token_mask, double* rows) {
    return mo_expert_mlp_fmt(x, T, H, I, E, k, MO_FMT_INT4, gate_q, gate_s, up_q, up_s, down_q, down_s,
                             ids, perm, token_mask, rows);
}

/* Shared expert scaled by sigmoid of its gate logit; an ungated shared expert
 * adds at weight one (dasLLAMA #3988, decode span commit). */
struct shared_ctx {
    const uint16_t* x;
    int H, I_sh, fmt;
    const uint8_t *gate_q, *up_q, *down_q;
    const void *gate_s, *up_s, *down_s;
    const uint16_t* g;
    const uint8_t* token_mask;
    double* y_sh;
};

static int shared_token(void* vc, long t) {
    const struct shared_ctx* c = (const struct shared_ctx*)vc;
    int H = c->H;
    if (c->token_mask && !c->token_mask[t]) return 0;
    const uint16_t* xr = c->x + (size_t)t * H;
    int rc = mo_expert_row_fmt(xr, H, c->I_sh, c->fmt, c->gate_q, c->gate_s, c->up_q, c->up_s,
                               c->down_q, c->down_s, c->y_sh + (size_t)t * H);
    if (rc) return rc;
    double gate = 1.0;
    if (c->g) {
        double z = 0.0;
        for (int h = 0; h < H; ++h) z += mo_bf16_to_f64(xr[h]) * mo_bf16_to_f64(c->g[h]);
        gate = 1.0 / (1.0 + exp(-z));
    }
    for (int n = 0; n < H; ++n) c->y_sh[(size_t)t * H + n] *= gate;
    return 0;
}

int mo_shared_expert_fmt(const uint16_t* x, int T, int H, int I_sh, int fmt,
                         const uint8_t* gate_q, const void* gate_s,
                         const uint8_t* up_q, const void* up_s,
                         const uint8_t* down_q, const void* down_s,
                         const uint16_t* g, const uint8_t* token_mask, double* y_sh) {
    if (!x || !y_sh || T < 0) return -1;
    struct shared_ctx c = {x, H, I_sh, fmt, gate_q, up_q, down_q, gate_s, up_s, down_s,
                           g, token_mask, y_sh};
    return mo_for_rows(T, shared_token, &c);
}

int mo_shared_expert(const uint16_t* x, int T, int H, int I_sh,
                     const uint8_t* gate_q, const uint16_t* gate_s,
                     const uint8_t* up_q, const uint16_t* up_s,
                     const uint8_t* down_q, const uint16_t* down_s,
                     const uint16_t* g, const uint8_t* token_mask, double* y_sh) {
    return mo_shared_expert_fmt(x, T, H, I_sh, MO_FMT_INT4, gate_q, gate_s, up_q, up_s, down_q, down_s,
                                g, token_mask, y_sh);
}

/* Combine onto the residual (dasLLAMA #3988: the routed slots weighted by the
 * top-k weights, plus the gated shared row, onto the residual).  In fp64 the
 * summation order is immaterial; the pages' order (shared, slots, residual)
 * is kept anyway. */
int mo_combine(const double* rows, const int32_t* inv, const double* w,
               const double* shared, const uint16_t* residual,
               int T, int k, int H, const uint8_t* token_mask, double* y) {
    if (!rows || !inv || !w || !y || T < 0 || k < 1 || H <= 0) return -1;
    for (int t = 0; t < T; ++t) {
        if (token_mask && !token_mask[t]) continue;
        for (int n = 0; n < H; ++n) {
            double acc = shared ? shared[(size_t)t * H + n] : 0.0;
            for (int j = 0; j < k; ++j) {
                int a = t * k + j;
                acc += w[a] * rows[(size_t)inv[a] * H + n];
            }
            if (residual) acc += mo_bf16_to_f64(residual[(size_t)t * H + n]);
            y[(size_t)t * H + n] = acc;
        }
    }
    return 0;
}

int mo_layer_forward_fmt(const uint16_t* x, const uint16_t* residual,
                         const uint16_t* W_r, int T, int H, int I, int E, int k, int fmt_r,
                         const uint8_t* gate_q, const void* gate_s,
                         const uint8_t* up_q, const void* up_s,
                         const uint8_t* down_q, const void* down_s,
                         int I_sh, int fmt_s,
                         const uint8_t* sh_gate_q, const void* sh_gate_s,
                         const uint8_t* sh_up_q, const void* sh_up_s,
                         const uint8_t* sh_down_q, const void* sh_down_s,
                         const uint16_t* sh_g, const uint8_t* token_mask,
                         double* logits_out, int32_t* ids_out, double* w_out, double* y) {
    if (!x || !W_r || !y || T < 0 || k < 1 || k > E) return -1;
    size_t nslot = (size_t)T * k;
    double* logits = (double*)malloc(sizeof(double) * ((size_t)T * E + 1));
    int32_t* ids = (int32_t*)malloc(sizeof(int32_t) * (nslot + 1));
    double* w = (double*)malloc(sizeof(double) * (nslot + 1));
    int32_t* counts = (int32_t*)malloc(sizeof(int32_t) * (size_t)E);
    int32_t* offsets = (int32_t*)malloc(sizeof(int32_t) * ((size_t)E + 1));
    int32_t* perm = (int32_t*)malloc(sizeof(int32_t) * (nslot + 1));
    int32_t* inv = (int32_t*)malloc(sizeof(int32_t) * (nslot + 1));
    double* rows = (double*)calloc(nslot * (size_t)H + 1, sizeof(double));
    double* ysh = I_sh > 0 ? (double*)calloc((size_t)T * H + 1, sizeof(double)) : NULL;
    int rc = -1;
    if (!logits || !ids || !w || !counts || !offsets || !perm || !inv || !rows || (I_sh > 0 && !ysh))
        goto done;
    rc = mo_router_logits(x, W_r, NULL, T, H, E, logits);
    if (rc) goto done;
    /* the router consumes fp32 logits: round before selection */
    for (size_t i = 0; i < (size_t)T * E; ++i) logits[i] = (double)(float)logits[i];
    if (logits_out) memcpy(logits_out, logits, sizeof(double) * (size_t)T * E);
    rc = mo_router_topk(logits, E, T, E, k, ids, w);
    if (rc) goto done;
    rc = mo_dispatch(ids, T, k, E, counts, offsets, perm, inv);
    if (rc) goto done;
    rc = mo_expert_mlp_fmt(x, T, H, I, E, k, fmt_r, gate_q, gate_s, up_q, up_s, down_q, down_s,
                           ids, perm, token_mask, rows);
    if (rc) goto done;
    if (I_sh > 0) {
        rc = mo_shared_expert_fmt(x, T, H, I_sh, fmt_s, sh_gate_q, sh_gate_s, sh_up_q, sh_up_s,
                                  sh_down_q, sh_down_s, sh_g, token_mask, ysh);
        if (rc) goto done;
    }
    rc = mo_combine(rows, inv, w, ysh, residual, T, k, H, token_mask, y);
    if (rc) goto done;
    if (ids_out) memcpy(ids_out, ids, sizeof(int32_t) * nslot);
    if (w_out) memcpy(w_out, w, sizeof(double) * nslot);
done:
    free(logits); free(ids); free(w); free(counts); free(offsets);
    free(perm); free(inv); free(rows); free(ysh);
    return rc;
}

int mo_layer_forward(const uint16_t* x, const uint16_t* residual,
                     const uint16_t* W_r, int T, int H, int I, int E, int k,
                     const uint8_t* gate_q, const uint16_t* gate_s,
                     const uint8_t* up_q, const uint16_t* up_s,
                     const uint8_t* down_q, const uint16_t* down_s,
                     int I_sh,
                     const uint8_t* sh_gate_q, const uint16_t* sh_gate_s,
                     const uint8_t* sh_up_q, const uint16_t* sh_up_s,
                     const uint8_t* sh_down_q, const uint16_t* sh_down_s,
                     const uint16_t* sh_g, const uint8_t* token_mask,
                     double* logits_out, int32_t* ids_out, double* w_out, double* y) {
    return mo_layer_forward_fmt(x, residual, W_r, T, H, I, E, k, MO_FMT_INT4, gate_q, gate_s, up_q, up_s,
                                down_q, down_s, I_sh, MO_FMT_INT4, sh_gate_q, sh_gate_s, sh_up_q, sh_up_s,
                                sh_down_q, sh_down_s, sh_g, token_mask, logits_out, ids_out, w_out, y);
}

/* RMSNorm (see moe_oracle.h): the mean of squares in fp64, one division per row. */
int mo_rmsnorm(const double* y, const uint16_t* gamma, int T, int H, double eps, double* out) {
    if (!y || !gamma || !out || T < 0 || H <= 0 || !(eps >= 0.0)) return -1;
    for (int t = 0; t < T; ++t) {
        const double* r = y + (size_t)t * H;
        double ss = 0.0;
        for (int h = 0; h < H; ++h) ss += r[h] * r[h];
        const double inv = 1.0 / sqrt(ss / H + eps);
        for (int h = 0; h < H; ++h) out[(size_t)t * H + h] = r[h] * inv * mo_bf16_to_f64(gamma[h]);
    }
    return 0;
}
