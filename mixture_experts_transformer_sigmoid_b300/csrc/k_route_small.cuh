// Routing of a small batch (decode) in one block: the router's split-K logit
// sum, the sigmoid scores and the top-k selection with its weights, the
// expert histogram and its scan, the stable scatter into per-expert rows and,
// when the rows are few, the row gather.  The separate kernels that do this
// for large batches (router_reduce, topk, scan, scatter, gather) are each a
// chain of dependent memory round trips that a few tokens cannot fill; here
// the whole chain runs in shared memory.
//
// The results are bit for bit those of the separate kernels: the logits come
// from the same compensated sum (reduce_logit_pair), the scores from
// router_score, the slots and weights from warp_select_topk (one warp per
// token, as in topk_kernel), and the rows of an expert are ordered by token,
// as in scatter_kernel.
#pragma once
#include <cuda_bf16.h>
#include <cstdint>

#include "k_route.cuh"
#include "k_router_tc.cuh"
#include "ptx.cuh"

namespace moe {

constexpr int RS_THREADS = 1024;
constexpr int RS_MAX_T = 32;                 // tokens (a bit mask per expert)
constexpr int RS_MAX_TE = 8192;              // T * E scores kept in shared memory
constexpr int RS_MAX_E = 256;                // experts per lane of the top-k warps <= 8
constexpr int RS_MAX_K = 32;                 // one slot per lane
// router partials the block adds itself (more are summed by router_reduce_kernel first)
constexpr int RS_MAX_PAIRS = 49152;
// rows gathered by the block itself (more go to gather_rows_kernel)
constexpr size_t RS_GATHER_MAX_BYTES = 128 * 1024;

struct RouteSmallArgs {
    const float2* part;   // router (hi, lo) partials [ksplit][T][E]
    int ksplit;           // ranges to add (1: one pair per logit, added as is)
    const float* bias;    // [E]
    float* logits;        // [T][E] out
    int T, E, k;
    float routed_scale;
    int* idx;             // [T][k] out
    float* w;             // [T][k] out
    int* counts;          // [E] out
    int* offsets;         // [E + 1] out
    int* pos;             // [T][k] out
    int* row_tok;         // [T k] out
    float* row_w;         // [T k] out
    const void* xn;       // [T][d]; with xp non-null the rows are gathered here
    void* xp;             // [T k][d] out, or nullptr
    int row_bytes;        // d * element size (a multiple of 16)
};

// Dynamic shared memory of one launch (bytes).
__host__ __device__ constexpr size_t route_small_smem(int T, int E, int k) {
    return sizeof(float) * (2 * static_cast<size_t>(T) * E      // scores, keys
                            + 3 * static_cast<size_t>(T) * k    // slot experts, weights, row -> token
                            + 2 * static_cast<size_t>(E) + 1    // token masks, offsets
                            + 32);                              // warp totals
}

// EPL = experts per lane (ceil(E / 32)) of the top-k warps.
template <int EPL>
__global__ void __launch_bounds__(RS_THREADS) route_small_kernel(const RouteSmallArgs a) {
    grid_dep_wait();
    extern __shared__ float rs_smem[];
    const int T = a.T, E = a.E, k = a.k;
    const int n = T * E, P = T * k;
    float* sc = rs_smem;                                        // [T][E] sigmoid scores
    float* key = sc + n;                                        // [T][E] selection keys
    int* slot_e = reinterpret_cast<int*>(key + n);              // [P] expert of each slot
    float* wsl = reinterpret_cast<float*>(slot_e + P);          // [P] weight of each slot
    int* rtok = reinterpret_cast<int*>(wsl + P);                // [P] token of each row
    uint32_t* mask = reinterpret_cast<uint32_t*>(rtok + P);     // [E] tokens that chose e
    int* offs = reinterpret_cast<int*>(mask + E);               // [E + 1]
    int* wtot = offs + E + 1;                                   // [32]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    // logits, scores and keys
    for (int i = tid; i < n; i += blockDim.x) {
        const float2 pv = a.ksplit > 1 ? reduce_logit_pair(a.part, a.ksplit, n, i) : a.part[i];
        const float l = __fadd_rn(pv.x, pv.y);
        a.logits[i] = l;
        router_score(l, a.bias[i % E], sc[i], key[i]);
    }
    for (int e = tid; e < E; e += blockDim.x) mask[e] = 0u;
    __syncthreads();

    // top-k: one warp per token (warp_select_topk, as topk_kernel)
    for (int t = warp; t < T; t += blockDim.x >> 5) {
        float bv[EPL], sv[EPL];
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = lane + 32 * i;
            bv[i] = e < E ? key[t * E + e] : 0.f;
            sv[i] = e < E ? sc[t * E + e] : 0.f;
        }
        int my_e;
        float my_w;
        warp_select_topk<EPL>(bv, sv, E, k, a.routed_scale, lane, my_e, my_w);
        if (lane < k) {
            const int q = t * k + lane;
            a.idx[q] = my_e;
            a.w[q] = my_w;
            slot_e[q] = my_e;
            wsl[q] = my_w;
            atomicOr(&mask[my_e], 1u << t);
        }
    }
    __syncthreads();

    // histogram and its exclusive scan (one thread per expert)
    const int c = tid < E ? __popc(mask[tid]) : 0;
    int incl = c;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += u;
    }
    if (lane == 31) wtot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int v = lane < static_cast<int>(blockDim.x >> 5) ? wtot[lane] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, v, off);
            if (lane >= off) v += u;
        }
        wtot[lane] = v;
    }
    __syncthreads();
    const int excl = incl - c + (warp > 0 ? wtot[warp - 1] : 0);
    if (tid < E) {
        a.counts[tid] = c;
        a.offsets[tid] = excl;
        offs[tid] = excl;
        if (tid == E - 1) a.offsets[E] = excl + c;
    }
    __syncthreads();

    // stable scatter: rows of expert e ordered by token
    for (int q = tid; q < P; q += blockDim.x) {
        const int t = q / k;
        const int e = slot_e[q];
        const int row = offs[e] + __popc(mask[e] & ((1u << t) - 1u));
        a.pos[q] = row;
        a.row_tok[row] = t;
        a.row_w[row] = wsl[q];
        rtok[row] = t;
    }
    if (a.xp == nullptr) return;
    __syncthreads();

    // xp[row] = xn[row_tok[row]], 16-byte vectors, four loads in flight per thread
    const int nvec = a.row_bytes / 16;
    const int total = P * nvec;
    const int4* src = static_cast<const int4*>(a.xn);
    int4* dst = static_cast<int4*>(a.xp);
    constexpr int U = 4;
    for (int v0 = tid; v0 < total; v0 += U * blockDim.x) {
        int4 r[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int v = v0 + u * blockDim.x;
            if (v < total) {
                const int row = v / nvec;
                r[u] = src[static_cast<size_t>(rtok[row]) * nvec + (v - row * nvec)];
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int v = v0 + u * blockDim.x;
            if (v < total) dst[v] = r[u];
        }
    }
}

}  // namespace moe
