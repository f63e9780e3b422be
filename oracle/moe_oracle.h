/*
 * CPU oracle for the GLM MoE feed-forward sublayer forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package's smoke check
 * and the benchmark's CPU-baseline leg may load or call this library.  The
 * product path never links it and shares no code, header or table with it.
 *
 * What it computes, per token t (tokens are independent):
 *   A  RMSNorm (GLM-5 shared-expert page, GlmMoeDsaRMSNorm.forward):
 *      ms = mean(x^2) in fp32; r = rsqrt(ms + eps); n = fp32(x * r);
 *      n is cast back to the input dtype, then xn = gain * n (rounded to the
 *      input dtype).
 *   B  router logits l[e] = sum_j xn[j] * Wr[e, j]        (fp32 result)
 *   C  s = sigmoid(l) (fp32); b = s + corr_bias; top-k of b, descending,
 *      ties to the lower expert index (the correction bias is a per-expert
 *      buffer: GLM-5 MoE block page, parameter accounting note)
 *   D  w_j = routed_scale * s[idx_j] / sum_i s[idx_i]
 *   E-G experts in the grouped native layout (NeMo GLM4-MoE state dict
 *      adapter page): gate = xn @ gate_up[e][:, 0:I], up = xn @
 *      gate_up[e][:, I:2I], h = silu(gate) * up, y = h @ down[e]
 *      (SwiGLU: GlmMoeDsaMLP.forward on the GLM-5 shared-expert page)
 *   H  shared expert with nn.Linear weights [out, in]:
 *      sh = Ds @ (silu(Gs @ xn) * (Us @ xn))
 *   I  out = x + sh + sum_j w_j * y_j   (GlmMoeDsaDecoderLayer.forward,
 *      second residual add)
 * and, for the dense layers, out = x + GlmMoeDsaMLP(xn) (oracle_dense_forward), and
 * the query compression of the attention (oracle_q_latent: q_a_layernorm(q_a_proj(h))).
 *
 * Precision: inputs are read exactly (bf16 bit patterns widened to fp32);
 * sums run in fp64 and are rounded to fp32 at the step boundaries above.
 * RMSNorm mirrors the page's fp32 steps and bf16 casts exactly, because the
 * routing decision depends on them.  Everything after routing is fp64.
 *
 * Every function here is pinned by the CPU tests (closed forms, brute-force
 * routing, the dense-SwiGLU reduction, invariants, and the GLM-5 parameter
 * count printed on the GLM-5 MoE block page).
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
    int32_t d;        /* hidden size */
    int32_t E;        /* routed experts */
    int32_t I;        /* routed expert intermediate size */
    int32_t Is;       /* shared expert intermediate size, 0 = no shared expert */
    int32_t k;        /* top_k */
    int32_t dtype;    /* storage of x, gain and weights: 0 = fp32, 1 = bf16 (uint16 bits) */
    float eps;        /* RMSNorm epsilon */
    float routed_scale;
} oracle_cfg;

/* Step A for n rows of x: xn [n, d] as fp32 values (bf16-representable when dtype = 1). */
int oracle_rmsnorm(const oracle_cfg* c, int64_t n, const void* x, const void* gain, float* xn);

/* Steps B-D given xn [n, d] (fp32 values).  Outputs (any may be NULL):
 * logits [n, E], idx [n, k], w [n, k], margin [n] = b_(k) - b_(k+1)
 * (+INF when k == E). */
int oracle_route(const oracle_cfg* c, int64_t n, const float* xn, const void* router_w,
                 const float* corr_bias, float* logits, int32_t* idx, float* w, float* margin);

/* Steps C-D given fp32 logits [n, E]: idx [n, k], w [n, k], margin [n] (may be NULL). */
int oracle_select(const oracle_cfg* c, int64_t n, const float* logits, const float* corr_bias,
                  int32_t* idx, float* w, float* margin);

/* The whole sublayer for the rows listed in `rows` (n of them; NULL = rows
 * 0..n-1 of x).  out [n, d] fp32.  Optional outputs may be NULL: idx [n,k],
 * w [n,k], margin [n], xn [n,d], logits [n,E].  When forced_idx [n,k] is not
 * NULL the listed experts replace the top-k selection (slot order as given);
 * their weights are still the renormalised unbiased sigmoids. */
int oracle_forward(const oracle_cfg* c, int64_t n, const int64_t* rows,
                   const void* x, const void* gain, const void* router_w, const float* corr_bias,
                   const void* gate_up, const void* down,
                   const void* shared_gate, const void* shared_up, const void* shared_down,
                   const int32_t* forced_idx,
                   float* out, int32_t* idx, float* w, float* margin, float* xn, float* logits);

/* The dense feed-forward block (GlmMoeDsaMLP with the residual), for the
 * rows listed in `rows` (NULL = rows 0..n-1 of x): out [n, d] fp32 =
 * x + down(silu(gate(xn)) * up(xn)), xn = step A.  gate, up [Is, d] and
 * down [d, Is] (nn.Linear); Is = c->Is >= 1.  xn [n, d] may be NULL. */
int oracle_dense_forward(const oracle_cfg* c, int64_t n, const int64_t* rows, const void* x,
                         const void* gain, const void* gate, const void* up, const void* down,
                         float* out, float* xn);

/* The query compression of GLM-5's sparse latent attention: c = q_a_proj(hidden)
 * (nn.Linear d -> rank, no bias, w_qa [rank, d], the exact sum rounded once to
 * the storage dtype) and q = q_a_layernorm(c) (step A over the rank values of
 * c, gain [rank], eps = c->eps), for the rows listed in `rows` (NULL = rows
 * 0..n-1 of hidden [*, d]).  c_out (may be NULL) and q_out are [n, rank] fp32. */
int oracle_q_latent(const oracle_cfg* c, int32_t rank, int64_t n, const int64_t* rows,
                    const void* hidden, const void* w_qa, const void* gain, float* c_out,
                    float* q_out);

/* Number of learned values and buffers the sublayer reads, RMSNorm gain excluded:
 * E*d*2I + E*I*d + 3*d*Is + E*d + E. */
int64_t oracle_param_count(const oracle_cfg* c);

/* Threads the OpenMP loops use. */
int oracle_num_threads(void);

#ifdef __cplusplus
}
#endif
#endif
