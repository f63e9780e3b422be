/*
 * CPU oracle for the GLM MoE feed-forward sublayer forward pass.
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the tests, the smoke check and the
 * benchmark's CPU-baseline leg, never by the product path.  Plain loops in
 * the order the definitions state them, fp64 accumulation, OpenMP over
 * tokens (tokens are independent).  See moe_oracle.h for the step list and
 * the passages each step follows.
 */
#include "moe_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- storage access ------------------------------------------------------ */

/* Element i of a tensor stored as fp32 (dtype 0) or bf16 bit patterns (dtype 1). */
static inline float get(const void* p, int64_t i, int dtype) {
    if (dtype == 0) return ((const float*)p)[i];
    uint32_t bits = (uint32_t)((const uint16_t*)p)[i] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return f;
}

/* Round an fp32 value to the nearest bf16 value, ties to even (the rounding
 * torch uses for .to(torch.bfloat16)).  Inputs are finite in this oracle. */
static inline float round_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    u &= 0xffff0000u;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round a real value (given in fp64) to the nearest bf16 value, ties to even:
 * one rounding of the exact value, not two (fp64 -> fp32 -> bf16 could round
 * twice).  bf16 has fp32's exponent range and 8 significant bits. */
static inline float round_bf16_exact(double v) {
    if (v == 0.0 || !isfinite(v)) return (float)v;
    int e;
    frexp(v, &e);                                   /* |v| in [2^(e-1), 2^e) */
    double q = ldexp(1.0, e - 8);                   /* bf16 spacing in that binade */
    if (q < ldexp(1.0, -133)) q = ldexp(1.0, -133); /* subnormal range: fixed spacing */
    double m = v / q;                               /* exact: a power-of-two scaling */
    double r = nearbyint(m);                        /* ties to even in the default mode */
    return (float)(r * q);
}

static inline double silu(double z) { return z / (1.0 + exp(-z)); }

/* ---- step A: RMSNorm (GlmMoeDsaRMSNorm.forward) --------------------------- */

static void rmsnorm_row(const oracle_cfg* c, const void* x, int64_t row, const void* gain,
                        float* xn) {
    const int d = c->d;
    /* hidden_states.to(float32).pow(2).mean(-1): the exact mean, rounded to fp32 */
    double ss = 0.0;
    for (int j = 0; j < d; ++j) {
        double v = (double)get(x, row * d + j, c->dtype);
        ss += v * v;
    }
    float variance = (float)(ss / (double)d);
    /* torch.rsqrt(variance + eps): fp32 add, then 1/sqrt as two rounded fp32 ops */
    float denom = variance + c->eps;
    float r = 1.0f / sqrtf(denom);
    for (int j = 0; j < d; ++j) {
        float n = get(x, row * d + j, c->dtype) * r;      /* fp32 product */
        float g = get(gain, j, c->dtype);
        if (c->dtype == 1) {
            n = round_bf16(n);                             /* .to(input_dtype) */
            xn[j] = round_bf16(g * n);                     /* weight * hidden, bf16 result */
        } else {
            xn[j] = g * n;
        }
    }
}

int oracle_rmsnorm(const oracle_cfg* c, int64_t n, const void* x, const void* gain, float* xn) {
    if (!c || !x || !gain || !xn || n < 0) return 1;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < n; ++t) rmsnorm_row(c, x, t, gain, xn + t * c->d);
    return 0;
}

/* ---- steps B-D: router, selection, weights -------------------------------- */

/* Steps C-D for one token from its fp32 logits.
 * scratch: s [E], b [E], picked [E] (as char) */
static void select_row(const oracle_cfg* c, const float* logits, const float* bias,
                       const int32_t* forced, int32_t* idx, float* w, float* margin, float* s,
                       float* b, char* picked) {
    const int E = c->E, k = c->k;
    for (int e = 0; e < E; ++e) {
        s[e] = (float)(1.0 / (1.0 + exp(-(double)logits[e])));  /* sigmoid, rounded to fp32 */
        b[e] = s[e] + bias[e];                                    /* biased score, fp32 add */
        picked[e] = 0;
    }
    /* top-k of b: repeatedly take the largest remaining; on equal values the
     * first (lowest) index found wins because only a strictly larger value
     * replaces the current best. */
    for (int j = 0; j < k; ++j) {
        int best = -1;
        if (forced) {
            best = forced[j];
        } else {
            for (int e = 0; e < E; ++e) {
                if (picked[e]) continue;
                if (best < 0 || b[e] > b[best]) best = e;
            }
        }
        picked[best] = 1;
        idx[j] = best;
    }
    if (margin) {
        float next = -INFINITY;
        int any = 0;
        for (int e = 0; e < E; ++e)
            if (!picked[e] && (!any || b[e] > next)) { next = b[e]; any = 1; }
        margin[0] = any ? b[idx[k - 1]] - next : INFINITY;
    }
    /* weights: unbiased sigmoids of the chosen experts, renormalised, scaled */
    double ssum = 0.0;
    for (int j = 0; j < k; ++j) ssum += (double)s[idx[j]];
    for (int j = 0; j < k; ++j)
        w[j] = (float)((double)c->routed_scale * (double)s[idx[j]] / ssum);
}

/* Steps B-D for one token.  lbuf [E] receives the logits. */
static void route_row(const oracle_cfg* c, const float* xn, const void* Wr, const float* bias,
                      const int32_t* forced, float* lbuf, int32_t* idx, float* w,
                      float* margin, float* s, float* b, char* picked) {
    const int d = c->d, E = c->E;
    for (int e = 0; e < E; ++e) {
        double acc = 0.0;
        for (int j = 0; j < d; ++j) acc += (double)xn[j] * (double)get(Wr, (int64_t)e * d + j, c->dtype);
        lbuf[e] = (float)acc;                              /* fp32 router logit */
    }
    select_row(c, lbuf, bias, forced, idx, w, margin, s, b, picked);
}

int oracle_select(const oracle_cfg* c, int64_t n, const float* logits, const float* corr_bias,
                  int32_t* idx, float* w, float* margin) {
    if (!c || !logits || !corr_bias || !idx || !w || n < 0 || c->k < 1 || c->k > c->E) return 1;
    int failed = 0;
#pragma omp parallel
    {
        float* s = (float*)malloc(sizeof(float) * c->E);
        float* b = (float*)malloc(sizeof(float) * c->E);
        char* picked = (char*)malloc(c->E);
        if (!s || !b || !picked) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(static)
            for (int64_t t = 0; t < n; ++t)
                select_row(c, logits + t * c->E, corr_bias, NULL, idx + t * c->k, w + t * c->k,
                           margin ? margin + t : NULL, s, b, picked);
        }
        free(s); free(b); free(picked);
    }
    return failed ? 2 : 0;
}

int oracle_route(const oracle_cfg* c, int64_t n, const float* xn, const void* router_w,
                 const float* corr_bias, float* logits, int32_t* idx, float* w, float* margin) {
    if (!c || !xn || !router_w || !corr_bias || n < 0 || c->k < 1 || c->k > c->E) return 1;
    int failed = 0;
#pragma omp parallel
    {
        float* s = (float*)malloc(sizeof(float) * c->E);
        float* b = (float*)malloc(sizeof(float) * c->E);
        float* lb = (float*)malloc(sizeof(float) * c->E);
        char* picked = (char*)malloc(c->E);
        int32_t* idx_t = (int32_t*)malloc(sizeof(int32_t) * c->k);
        float* w_t = (float*)malloc(sizeof(float) * c->k);
        if (!s || !b || !lb || !picked || !idx_t || !w_t) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(static)
            for (int64_t t = 0; t < n; ++t) {
                route_row(c, xn + t * c->d, router_w, corr_bias, NULL, lb, idx_t, w_t,
                          margin ? margin + t : NULL, s, b, picked);
                for (int e = 0; e < c->E; ++e)
                    if (logits) logits[t * c->E + e] = lb[e];
                for (int j = 0; j < c->k; ++j) {
                    if (idx) idx[t * c->k + j] = idx_t[j];
                    if (w) w[t * c->k + j] = w_t[j];
                }
            }
        }
        free(s); free(b); free(lb); free(picked); free(idx_t); free(w_t);
    }
    return failed ? 2 : 0;
}

/* ---- steps E-I: experts, shared expert, combine --------------------------- */

/* One SwiGLU expert in the grouped layout: gu [d, 2I] (gate cols 0..I-1,
 * up cols I..2I-1), dn [I, d].  Adds w * y into acc [d].
 * scratch: g [I], u [I] (double) */
static void routed_expert(const oracle_cfg* c, const float* xn, const void* gu, const void* dn,
                          int64_t gu_off, int64_t dn_off, double wgt, double* acc,
                          double* g, double* u) {
    const int d = c->d, I = c->I;
    for (int i = 0; i < I; ++i) { g[i] = 0.0; u[i] = 0.0; }
    for (int j = 0; j < d; ++j) {
        double xj = (double)xn[j];
        int64_t rowb = gu_off + (int64_t)j * 2 * I;
        for (int i = 0; i < I; ++i) {
            g[i] += xj * (double)get(gu, rowb + i, c->dtype);
            u[i] += xj * (double)get(gu, rowb + I + i, c->dtype);
        }
    }
    for (int i = 0; i < I; ++i) g[i] = silu(g[i]) * u[i];  /* h */
    for (int i = 0; i < I; ++i) {
        double hw = wgt * g[i];
        int64_t rowb = dn_off + (int64_t)i * d;
        for (int o = 0; o < d; ++o) acc[o] += hw * (double)get(dn, rowb + o, c->dtype);
    }
}

/* Shared expert with nn.Linear weights: Gs, Us [Is, d], Ds [d, Is].  Adds sh into acc. */
static void shared_expert(const oracle_cfg* c, const float* xn, const void* Gs, const void* Us,
                          const void* Ds, double* acc, double* h) {
    const int d = c->d, Is = c->Is;
    for (int i = 0; i < Is; ++i) {
        double gs = 0.0, us = 0.0;
        for (int j = 0; j < d; ++j) {
            gs += (double)get(Gs, (int64_t)i * d + j, c->dtype) * (double)xn[j];
            us += (double)get(Us, (int64_t)i * d + j, c->dtype) * (double)xn[j];
        }
        h[i] = silu(gs) * us;
    }
    for (int o = 0; o < d; ++o) {
        double v = 0.0;
        for (int i = 0; i < Is; ++i) v += (double)get(Ds, (int64_t)o * Is + i, c->dtype) * h[i];
        acc[o] += v;
    }
}

int oracle_forward(const oracle_cfg* c, int64_t n, const int64_t* rows,
                   const void* x, const void* gain, const void* router_w, const float* corr_bias,
                   const void* gate_up, const void* down,
                   const void* shared_gate, const void* shared_up, const void* shared_down,
                   const int32_t* forced_idx,
                   float* out, int32_t* idx, float* w, float* margin, float* xn_out,
                   float* logits) {
    if (!c || !x || !gain || !router_w || !corr_bias || !gate_up || !down || !out || n < 0)
        return 1;
    if (c->k < 1 || c->k > c->E || c->d < 1 || c->I < 1 || c->Is < 0) return 1;
    if (c->Is > 0 && (!shared_gate || !shared_up || !shared_down)) return 1;
    const int d = c->d, E = c->E, I = c->I, k = c->k;
    int failed = 0;
#pragma omp parallel
    {
        int hmax = I > c->Is ? I : c->Is;
        float* xn = (float*)malloc(sizeof(float) * d);
        float* s = (float*)malloc(sizeof(float) * E);
        float* b = (float*)malloc(sizeof(float) * E);
        float* lb = (float*)malloc(sizeof(float) * E);
        char* picked = (char*)malloc(E);
        int32_t* sel = (int32_t*)malloc(sizeof(int32_t) * k);
        float* wt = (float*)malloc(sizeof(float) * k);
        double* acc = (double*)malloc(sizeof(double) * d);
        double* g = (double*)malloc(sizeof(double) * hmax);
        double* u = (double*)malloc(sizeof(double) * I);
        if (!xn || !s || !b || !lb || !picked || !sel || !wt || !acc || !g || !u) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t t = 0; t < n; ++t) {
                int64_t row = rows ? rows[t] : t;
                rmsnorm_row(c, x, row, gain, xn);
                route_row(c, xn, router_w, corr_bias, forced_idx ? forced_idx + t * k : NULL, lb,
                          sel, wt, margin ? margin + t : NULL, s, b, picked);
                if (logits) memcpy(logits + t * E, lb, sizeof(float) * E);
                for (int o = 0; o < d; ++o) acc[o] = 0.0;
                if (c->Is > 0) shared_expert(c, xn, shared_gate, shared_up, shared_down, acc, g);
                for (int j = 0; j < k; ++j) {
                    int e = sel[j];
                    routed_expert(c, xn, gate_up, down, (int64_t)e * d * 2 * I,
                                  (int64_t)e * I * d, (double)wt[j], acc, g, u);
                }
                for (int o = 0; o < d; ++o)
                    out[t * d + o] = (float)((double)get(x, row * d + o, c->dtype) + acc[o]);
                for (int j = 0; j < k; ++j) {
                    if (idx) idx[t * k + j] = sel[j];
                    if (w) w[t * k + j] = wt[j];
                }
                if (xn_out) memcpy(xn_out + t * d, xn, sizeof(float) * d);
            }
        }
        free(xn); free(s); free(b); free(lb); free(picked); free(sel); free(wt); free(acc); free(g); free(u);
    }
    return failed ? 2 : 0;
}

/* The dense feed-forward block of the first first_k_dense_replace decoder
 * layers (GLM-5 shared-expert page: GlmMoeDsaDecoderLayer.forward's second
 * half with GlmMoeDsaMLP as the mlp):
 *   out = x + down(silu(gate(xn)) * up(xn)),  xn = RMSNorm(x)  (step A),
 * with nn.Linear weights gate, up [Is, d] and down [d, Is]; c->Is is the
 * block's intermediate size, c->E, c->I and c->k are not used. */
int oracle_dense_forward(const oracle_cfg* c, int64_t n, const int64_t* rows, const void* x,
                         const void* gain, const void* gate, const void* up, const void* down,
                         float* out, float* xn_out) {
    if (!c || !x || !gain || !gate || !up || !down || !out || n < 0 || c->d < 1 || c->Is < 1)
        return 1;
    const int d = c->d;
    int failed = 0;
#pragma omp parallel
    {
        float* xn = (float*)malloc(sizeof(float) * d);
        double* acc = (double*)malloc(sizeof(double) * d);
        double* h = (double*)malloc(sizeof(double) * c->Is);
        if (!xn || !acc || !h) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t t = 0; t < n; ++t) {
                int64_t row = rows ? rows[t] : t;
                rmsnorm_row(c, x, row, gain, xn);
                for (int o = 0; o < d; ++o) acc[o] = 0.0;
                shared_expert(c, xn, gate, up, down, acc, h);
                for (int o = 0; o < d; ++o)
                    out[t * d + o] = (float)((double)get(x, row * d + o, c->dtype) + acc[o]);
                if (xn_out) memcpy(xn_out + t * d, xn, sizeof(float) * d);
            }
        }
        free(xn); free(acc); free(h);
    }
    return failed ? 2 : 0;
}

/* The query compression of GLM-5's sparse latent attention (GLM-5 "Query
 * latent" page, MLA __init__ and the query lines of its forward):
 *   c = q_a_proj(hidden)      nn.Linear(d -> rank, no bias, attention_bias is
 *                             false), its output in the input precision;
 *   q = q_a_layernorm(c)      GlmMoeDsaRMSNorm(rank), eps = c->eps (the page's
 *                             latent RMSNorms take the 1e-6 default).
 * w_qa is [rank, d] (nn.Linear [out, in]), gain [rank].  The Linear's output is
 * the exact sum rounded once to the storage dtype (bf16 or fp32); the RMSNorm
 * is step A's (rmsnorm_row) over the rank values of c.  c_out and q_out are
 * [n, rank] fp32 values (bf16-representable for dtype 1); c_out may be NULL. */
int oracle_q_latent(const oracle_cfg* c, int32_t rank, int64_t n, const int64_t* rows,
                    const void* hidden, const void* w_qa, const void* gain, float* c_out,
                    float* q_out) {
    if (!c || !hidden || !w_qa || !gain || !q_out || n < 0 || c->d < 1 || rank < 1) return 1;
    const int d = c->d;
    oracle_cfg cr = *c;       /* the norm runs over the rank features of c */
    cr.d = rank;
    int failed = 0;
#pragma omp parallel
    {
        float* cq = (float*)malloc(sizeof(float) * rank);
        uint16_t* cq16 = (uint16_t*)malloc(sizeof(uint16_t) * rank);
        if (!cq || !cq16) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (int64_t t = 0; t < n; ++t) {
                int64_t row = rows ? rows[t] : t;
                for (int r = 0; r < rank; ++r) {
                    double acc = 0.0;
                    for (int j = 0; j < d; ++j)
                        acc += (double)get(hidden, row * d + j, c->dtype) *
                               (double)get(w_qa, (int64_t)r * d + j, c->dtype);
                    cq[r] = c->dtype == 1 ? round_bf16_exact(acc) : (float)acc;
                }
                const void* cin = cq;
                if (c->dtype == 1) {          /* rmsnorm_row reads storage: bf16 bit patterns */
                    for (int r = 0; r < rank; ++r) {
                        uint32_t u;
                        memcpy(&u, &cq[r], sizeof u);
                        cq16[r] = (uint16_t)(u >> 16);
                    }
                    cin = cq16;
                }
                rmsnorm_row(&cr, cin, 0, gain, q_out + t * rank);
                if (c_out) memcpy(c_out + t * rank, cq, sizeof(float) * rank);
            }
        }
        free(cq); free(cq16);
    }
    return failed ? 2 : 0;
}

int64_t oracle_param_count(const oracle_cfg* c) {
    int64_t d = c->d, E = c->E, I = c->I, Is = c->Is;
    int64_t routed = E * d * 2 * I + E * I * d;       /* gate_and_up_projs + down_projs */
    int64_t shared = Is * d + Is * d + d * Is;         /* gate_proj, up_proj, down_proj */
    int64_t router = E * d + E;                        /* router weight + correction bias */
    return routed + shared + router;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
