/*
 * moe.h — C ABI of the B300 (sm_103a) forward pass of the GLM MoE
 * feed-forward sublayer.
 *
 * The operation (per token t; tokens are independent):
 *   xn  = RMSNorm(x[t]) with one gain per feature: mean of squares in fp32,
 *         multiply by rsqrt(mean + eps), cast back to the input dtype, then
 *         multiply by the gain (GlmMoeDsaRMSNorm.forward, GLM-5 shared-expert
 *         page on OpenModelAtlas).
 *   l   = xn . router_w^T in fp32; s = sigmoid(l); b = s + corr_bias
 *         (the correction bias is a per-expert buffer: GLM-5 MoE block page,
 *         note under the parameter table).
 *   idx = the top_k experts by b, descending, ties to the lower index.
 *   w   = routed_scale * s[idx] / sum(s[idx]).
 *   y_e = SwiGLU expert in the grouped native layout (NeMo AutoModel
 *         GLM4-MoE state dict adapter page): gate = xn @ gate_up[e][:, :I],
 *         up = xn @ gate_up[e][:, I:], y_e = (silu(gate) * up) @ down[e]
 *         (SwiGLU: GlmMoeDsaMLP.forward).
 *   sh  = shared SwiGLU expert with nn.Linear weights [out, in]:
 *         shared_down @ (silu(shared_gate @ xn) * (shared_up @ xn)).
 *   out = x + sh + sum_j w_j * y_{idx_j}   (second residual add of
 *         GlmMoeDsaDecoderLayer.forward).
 *
 * Conventions for every entry point:
 *   - Tensor pointers are row-major and contiguous, in the dtype the handle
 *     was created with (fp32, or bf16 as 16-bit patterns), except corr_bias,
 *     which is always fp32.  "device" pointers must be CUDA device memory of
 *     the handle's device; "host" pointers ordinary host memory (pinned
 *     memory makes the copies asynchronous to the host).
 *   - The caller owns every tensor it passes and keeps it valid until the
 *     work queued on `stream` has finished.  The library owns only the
 *     workspace it allocates in moe_init and frees in moe_destroy.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).
 *   - Functions return a moe_status and never throw.  Argument errors are
 *     detected on the host before any work is queued.
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct moe_handle moe_handle;

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size, aliasing output */
    MOE_ERR_UNSUPPORTED = 2,  /* valid, but a shape this build does not handle */
    MOE_ERR_CUDA = 3,         /* a CUDA runtime/driver call or launch failed */
    MOE_ERR_OOM = 4,          /* workspace allocation failed in moe_init */
    MOE_ERR_TIMEOUT = 5,      /* a kernel's bounded wait expired (device error flag) */
    MOE_ERR_RANGE = 6         /* a weighted expert row exceeded the fp16 range (|v| > 65504) of the
                                 intermediate that carries it to the combine (device error flag) */
} moe_status;

typedef enum { MOE_DTYPE_FP32 = 0, MOE_DTYPE_BF16 = 1 } moe_dtype;

typedef struct {
    int32_t max_tokens;    /* largest T a forward may use (workspace sizing), >= 1 */
    int32_t hidden;        /* d */
    int32_t n_experts;     /* E, 1..1024; 0 makes a handle for moe_dense_forward only
                              (then inter, shared_inter and max_top_k must be 0) */
    int32_t inter;         /* I, routed expert intermediate size */
    int32_t shared_inter;  /* Is, shared expert intermediate size; 0 = no shared expert */
    int32_t max_top_k;     /* largest top_k a forward may use, 1..min(E, 32) */
    int32_t dtype;         /* moe_dtype of x, weights and out */
    float eps;             /* RMSNorm epsilon (the pages' default: 1e-6) */
    int32_t device;        /* CUDA device ordinal */
    int32_t gemm_path;     /* 0 = automatic (tensor cores for bf16); 1 = force the
                              CUDA-core (FFMA) expert kernels (the fp32 path) */
    int32_t dense_inter;   /* largest intermediate size moe_dense_forward may use;
                              0 = the handle has no dense workspace */
} moe_config;

/* Creates a handle on cfg->device and allocates its workspace for
 * max_tokens * max_top_k routed rows (and max_tokens * dense_inter values
 * for moe_dense_forward).  bf16 handles on the tensor-core path need hidden,
 * inter, shared_inter and dense_inter to be multiples of 64; the CUDA-core
 * path needs hidden, inter, shared_inter and dense_inter <= 12288
 * (MOE_ERR_UNSUPPORTED otherwise).  *out is set only on MOE_OK. */
MOE_API moe_status moe_init(const moe_config* cfg, moe_handle** out);

/* One forward pass of the sublayer over T tokens (0 <= T <= max_tokens),
 * queued on `stream`; asynchronous, no host synchronisation, no allocation.
 * All pointers are device pointers:
 *   x           [T, d]          input hidden states (the residual)
 *   norm_w      [d]             RMSNorm gain
 *   router_w    [E, d]          router weight (logits = xn . router_w^T)
 *   corr_bias   [E]  fp32       per-expert correction bias (selection only)
 *   gate_up     [E, d, 2I]      grouped gate|up projections: columns 0..I-1
 *                               are the gate, I..2I-1 the up projection
 *   down        [E, I, d]       grouped down projections
 *   shared_gate [Is, d], shared_up [Is, d], shared_down [d, Is]
 *                               shared expert (nn.Linear [out, in]); may be
 *                               NULL when the handle has shared_inter == 0
 *   top_k       1..max_top_k;  routed_scale: factor on the renormalised weights
 *   out         [T, d]          must not overlap any input
 * x, out and the weight tensors must be 16-byte aligned.  T == 0 queues
 * nothing and reads no pointer (any may be NULL).  A device-side timeout is
 * reported by moe_sync_status. */
MOE_API moe_status moe_forward(moe_handle* h, int32_t T, const void* x, const void* norm_w,
                       const void* router_w, const float* corr_bias, const void* gate_up,
                       const void* down, const void* shared_gate, const void* shared_up,
                       const void* shared_down, int32_t top_k, float routed_scale, void* out,
                       void* stream);

/* moe_forward with x and out in HOST memory (the weights stay device
 * pointers): copies x into the handle's device staging buffer, runs the
 * forward, copies the result back into `out` and synchronises `stream`.
 * Returns MOE_ERR_TIMEOUT if a kernel's bounded wait expired. */
MOE_API moe_status moe_forward_host(moe_handle* h, int32_t T, const void* x_host, const void* norm_w,
                            const void* router_w, const float* corr_bias, const void* gate_up,
                            const void* down, const void* shared_gate, const void* shared_up,
                            const void* shared_down, int32_t top_k, float routed_scale,
                            void* out_host, void* stream);

/* Pipelined form of moe_forward_host for a stream of batches: queues the
 * H2D copy of x (on an internal copy stream), the forward (on `stream`) and
 * the D2H copy of the result (on a second copy stream) and returns without
 * waiting, so one batch's copies overlap the neighbouring batches' forwards.
 * Two staging slots alternate between calls; events keep each slot from being
 * overwritten before its previous forward and copy-out are done.  The caller
 * keeps x_host and out_host valid and unread until moe_forward_host_wait
 * returns; x_host/out_host should be pinned (pageable memory works but does
 * not overlap).  Same argument checks as moe_forward_host.  Not for
 * concurrent calls on one handle from several threads. */
MOE_API moe_status moe_forward_host_async(moe_handle* h, int32_t T, const void* x_host, const void* norm_w,
                                  const void* router_w, const float* corr_bias, const void* gate_up,
                                  const void* down, const void* shared_gate, const void* shared_up,
                                  const void* shared_down, int32_t top_k, float routed_scale,
                                  void* out_host, void* stream);

/* Waits for every moe_forward_host_async call queued on this handle (their
 * results are then in the callers' out_host buffers) and reports the device
 * error flag like moe_sync_status. */
MOE_API moe_status moe_forward_host_wait(moe_handle* h);

/* The dense feed-forward block of the first first_k_dense_replace decoder
 * layers (GlmMoeDsaDecoderLayer.forward's second half with GlmMoeDsaMLP as
 * the mlp, GLM-5 shared-expert page on OpenModelAtlas), per token:
 *   out = x + down_w @ (silu(gate_w @ xn) * (up_w @ xn)),  xn = RMSNorm(x)
 * with the same RMSNorm as moe_forward and nn.Linear weights:
 *   x [T, d], norm_w [d], gate_w [inter, d], up_w [inter, d],
 *   down_w [d, inter], out [T, d]   (device pointers, 16-byte aligned;
 *   out must not overlap any input)
 * 1 <= inter <= cfg.dense_inter, 0 <= T <= max_tokens (T == 0 queues
 * nothing and reads no pointer).  The residual is added to the down
 * projection's fp32 accumulator and rounded once.  Asynchronous on `stream`,
 * no allocation, no host synchronisation; a device-side timeout is reported
 * by moe_sync_status.  It reuses the handle's RMSNorm buffer (MOE_T_XN),
 * which then holds the dense block's values; the per-stage times of moe_read_stats cover
 * moe_forward only (the launch count includes both). */
MOE_API moe_status moe_dense_forward(moe_handle* h, int32_t T, const void* x, const void* norm_w,
                             const void* gate_w, const void* up_w, const void* down_w,
                             int32_t inter, void* out, void* stream);

/* The query compression of GLM-5's sparse latent attention (GLM-5 "Query
 * latent" page on OpenModelAtlas: the MLA __init__ builds q_a_proj =
 * nn.Linear(hidden_size, q_lora_rank, bias=attention_bias) with
 * attention_bias false, and q_a_layernorm = GlmMoeDsaRMSNorm(q_lora_rank);
 * its forward computes q_resid = q_a_layernorm(q_a_proj(hidden_states))):
 *   c_out = hidden @ w_qa^T      the query latent, rounded once to the handle dtype
 *   q_out = RMSNorm(c_out)       with gain q_norm_w and the handle's eps (the
 *                                page's latent norms take the 1e-6 default)
 * Device pointers, row-major, 16-byte aligned, owned by the caller:
 *   hidden [T, d] (d = cfg.hidden: the attention input, already normalised),
 *   w_qa [q_rank, d] (nn.Linear [out, in]), q_norm_w [q_rank],
 *   c_out [T, q_rank], q_out [T, q_rank]; the outputs must not overlap the
 *   inputs or each other (MOE_ERR_INVALID_ARG).
 * q_rank >= 1 (a multiple of 64 on the tensor-core path, else
 * MOE_ERR_UNSUPPORTED); any T >= 0 (T == 0 queues nothing).  Any handle
 * whose hidden size is d serves; small batches (T <= 128, T <= max_tokens
 * and q_rank <= d) use its split-K buffer.  Asynchronous on `stream`, no
 * allocation, no host synchronisation; a device-side timeout is reported by
 * moe_sync_status. */
MOE_API moe_status moe_q_latent(moe_handle* h, int32_t T, int32_t q_rank, const void* hidden,
                        const void* w_qa, const void* q_norm_w, void* c_out, void* q_out,
                        void* stream);

/* Routing of the last forward on this handle, copied (device to device, on
 * `stream`) into caller buffers; any pointer may be NULL:
 *   idx [T, top_k] int32 expert ids in slot order, w [T, top_k] fp32 weights,
 *   counts [E] int32 tokens routed to each expert. */
MOE_API moe_status moe_get_routing(moe_handle* h, int32_t* idx, float* w, int32_t* counts,
                           void* stream);

/* Intermediates of the last forward, for stage-by-stage testing. */
typedef enum {
    MOE_T_XN = 0,       /* [T, d] RMSNorm output, handle dtype */
    MOE_T_LOGITS = 1,   /* [T, E] fp32 router logits */
    MOE_T_OFFSETS = 2,  /* [E + 1] int32 first permuted row of each expert */
    MOE_T_POS = 3,      /* [T, top_k] int32 permuted row of each (token, slot) */
    MOE_T_ROW_TOK = 4,  /* [T * top_k] int32 token of each permuted row */
    MOE_T_H = 5,        /* [T * top_k, I] routed SwiGLU activations, handle dtype */
    MOE_T_YP = 6        /* [T * top_k, d] weighted expert rows w * expert(xn), permuted
                           order: fp16 on the tensor-core path, else the handle dtype */
} moe_tensor;

/* Copies intermediate `which` of the last forward into dst (device memory
 * of dst_bytes bytes) on `stream`.  MOE_ERR_INVALID_ARG if dst_bytes is
 * smaller than the tensor. */
MOE_API moe_status moe_get_intermediate(moe_handle* h, moe_tensor which, void* dst, size_t dst_bytes,
                                void* stream);

/* Synchronises `stream`, then reads and clears the handle's device error
 * flag: MOE_ERR_TIMEOUT if a kernel gave up a bounded wait since the last
 * call, MOE_ERR_RANGE if a weighted expert row overflowed its fp16
 * intermediate (that forward's output holds infinities), MOE_ERR_CUDA on an
 * asynchronous CUDA error, else MOE_OK. */
MOE_API moe_status moe_sync_status(moe_handle* h, void* stream);

/* Self-test of failure detection (no counterpart in the paper): queues on
 * `stream` one wait on a device barrier that nothing completes, bounded like
 * every wait of the library's tensor-core kernels.  After timeout_us
 * microseconds (1 .. 1,000,000) the wait gives up and sets the handle's
 * device error flag, so the next moe_sync_status returns MOE_ERR_TIMEOUT and
 * clears it.  Nothing faults or hangs, and the context stays usable: it is
 * the path a kernel takes when a copy or a peer never arrives. */
MOE_API moe_status moe_selftest_wait_timeout(moe_handle* h, uint32_t timeout_us, void* stream);

/* Counters of the forwards run since the last moe_read_stats. */
#define MOE_MAX_STAGES 16
typedef struct {
    int32_t forwards;                /* forwards counted */
    int32_t launches;                /* kernels those forwards launched */
    int32_t n_stages;                /* stages of the forward (entries of stage_ms in use) */
    float stage_ms[MOE_MAX_STAGES];  /* summed GPU time per stage, from CUDA events recorded on
                                        the forward's stream while profiling is on; else 0.
                                        Stages: 0 RMSNorm (fused with the router on the
                                        CUDA-core path), 1 router logits, 2 top-k, 3 scan,
                                        4 scatter, 5 row gather, 6 gate|up + SwiGLU (routed and
                                        shared), 7 down + routing weight (routed and shared),
                                        8 combine + residual.  Batches of at most 32 tokens
                                        (and 256 experts) on the tensor-core path route in one
                                        kernel, counted in stage 2; stages 3 and 4 are then
                                        empty, and so is 5 when that kernel gathered the rows. */
} moe_stats;

/* Turns per-stage CUDA-event timing on (enable != 0) or off.  Recording
 * events does not synchronise; after 256 profiled forwards without a
 * moe_read_stats call, the next forward waits for the oldest one. */
MOE_API moe_status moe_set_profiling(moe_handle* h, int32_t enable);

/* Synchronises the device, returns the counters accumulated since the last
 * call, and resets them. */
MOE_API moe_status moe_read_stats(moe_handle* h, moe_stats* out);

/* Frees the workspace (synchronises the device first).  NULL is a no-op. */
MOE_API moe_status moe_destroy(moe_handle* h);

/* Routing of a batch from given router logits, with no allocation of any
 * kind.  It has no counterpart in the paper.  It is there for callers that
 * cannot call cudaMalloc: a serving engine that reserved all device memory
 * for its own pool up front, or code that must not let a cudaMalloc or
 * cudaFree synchronise the device in the middle of its work.
 *
 * It runs the routing part of moe_forward on the calling thread's current
 * device: s = sigmoid(logits), top_k experts by s + corr_bias (ties to the lower
 * index), w = routed_scale * s / sum(s), the expert histogram, its
 * exclusive scan and the stable scatter.  Given the logits moe_forward
 * used (MOE_T_LOGITS), every output equals moe_forward's bit for bit.
 * All pointers are device memory of the current device, 4-byte aligned,
 * owned by the caller:
 *   logits  [T, E] fp32 in;  corr_bias [E] fp32 in
 *   idx [T, top_k] int32, w [T, top_k] fp32      experts and weights, slot order
 *   counts [E] int32, offsets [E + 1] int32      tokens per expert, first row of each
 *   pos [T, top_k] int32                         permuted row of each (token, slot)
 *   row_tok [T * top_k] int32, row_w [T * top_k] fp32   token and weight of each row
 * Its scratch (per-chunk histograms) is a 1 MB static device array that
 * every GPU loading the library holds until the process exits; the limit
 * is ceil(T / 128) * E <= 131072 (e.g. T = 65536 with E = 256), beyond
 * which it returns MOE_ERR_UNSUPPORTED before queueing anything.  Every
 * call on a device shares that array, which keeps the last call's
 * contents: calls that overlap on the GPU (other streams, other threads)
 * race, so serialise them.  The first call on each device looks up the
 * array's device address (cudaGetSymbolAddress); make that first call
 * before any stream capture.  1 <= E <= 1024, 1 <= top_k <= min(E, 32),
 * T >= 0 (T == 0 queues nothing); MOE_ERR_INVALID_ARG for other values,
 * null/misaligned pointers, or an output that overlaps an input or another
 * output.  Asynchronous on `stream`. */
MOE_API moe_status moe_route_static(int32_t T, int32_t E, int32_t top_k, float routed_scale,
                            const float* logits, const float* corr_bias, int32_t* idx, float* w,
                            int32_t* counts, int32_t* offsets, int32_t* pos, int32_t* row_tok,
                            float* row_w, void* stream);

/* Packs HF per-expert nn.Linear weights into the grouped native layout that
 * moe_forward reads (NeMo AutoModel GLM4-MoE state dict adapter page:
 * experts.{E}.gate_proj / up_proj / down_proj are grouped into
 * gate_and_up_projs [n_experts, dim, 2*moe_inter_dim] and down_projs
 * [n_experts, moe_inter_dim, dim]).  Device pointers, row-major:
 *   gate, up [E, I, d], down [E, d, I]   the E experts' HF tensors, stacked
 *   gate_up [E, d, 2I]   gate_up[e][j][i] = gate[e][i][j],
 *                        gate_up[e][j][I + i] = up[e][i][j]
 *   down_projs [E, I, d] down_projs[e][i][o] = down[e][o][i]
 * A caller holding the experts as separate tensors calls once per expert
 * with E = 1 and the outputs advanced by e experts.  elem_bytes is 2 (bf16)
 * or 4 (fp32); the copy is exact.  Either output may be NULL to skip it (its
 * inputs are then not read).  Pointers 4-byte aligned; outputs must not
 * overlap the inputs or each other (MOE_ERR_INVALID_ARG).  E == 0 queues
 * nothing; E > 65535, or odd d or I with 2-byte elements, give
 * MOE_ERR_UNSUPPORTED.  No handle, no allocation; asynchronous on `stream`
 * (the calling thread's current device). */
MOE_API moe_status moe_pack_experts(int32_t E, int32_t d, int32_t I, int32_t elem_bytes,
                            const void* gate, const void* up, const void* down, void* gate_up,
                            void* down_projs, void* stream);

/* Static description of a status code. */
MOE_API const char* moe_status_string(moe_status s);

#ifdef __cplusplus
}
#endif
#endif /* MOE_B300_H */
