// CUDA-core kernels of the MoE sublayer: RMSNorm, router logits (FFMA
// path), per-token top-k, the expert histogram / scan / stable scatter that
// build the permuted row index, the row gather, the deterministic combine,
// and the FFMA expert kernels used for fp32 storage.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "numeric.cuh"
#include "ptx.cuh"

namespace moe {

constexpr int CHUNK_TOKENS = 128;  // tokens per histogram chunk (topk and scatter agree on it)

// ------------------------------------------------------------ element I/O
template <typename T> struct Elem;
template <> struct Elem<float> {
    static constexpr int V = 4;  // elements per 16-byte vector
    __device__ static float to_f(float v) { return v; }
    __device__ static float from_f(float v) { return v; }
    // RMSNorm's cast back to the input dtype is the identity for fp32
    __device__ static float round_io(float v) { return v; }
};
template <> struct Elem<__nv_bfloat16> {
    static constexpr int V = 8;
    __device__ static float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
    __device__ static __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
    __device__ static float round_io(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }
};
template <> struct Elem<__half> {   // the weighted expert rows of the tensor-core path
    static constexpr int V = 8;
    __device__ static float to_f(__half v) { return __half2float(v); }
    __device__ static __half from_f(float v) { return __float2half_rn(v); }
};

template <typename T>
__device__ __forceinline__ void unpack_vec(const int4& raw, float (&f)[Elem<T>::V]) {
    const T* e = reinterpret_cast<const T*>(&raw);
#pragma unroll
    for (int i = 0; i < Elem<T>::V; ++i) f[i] = Elem<T>::to_f(e[i]);
}
template <typename T>
__device__ __forceinline__ void load_vec(const T* p, float (&f)[Elem<T>::V]) {
    unpack_vec<T>(*reinterpret_cast<const int4*>(p), f);
}
template <typename T>
__device__ __forceinline__ void store_vec(T* p, const float (&f)[Elem<T>::V]) {
    int4 raw;
    T* e = reinterpret_cast<T*>(&raw);
#pragma unroll
    for (int i = 0; i < Elem<T>::V; ++i) e[i] = Elem<T>::from_f(f[i]);
    *reinterpret_cast<int4*>(p) = raw;
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + __expf(-z)); }

// --------------------------------------------------------------- RMSNorm
// Block-wide sum of (hi, lo) pairs; every thread receives the total.
__device__ __forceinline__ void block_sum_pair(float& hi, float& lo, float2* red) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        float oh = __shfl_xor_sync(0xffffffffu, hi, off);
        float ol = __shfl_xor_sync(0xffffffffu, lo, off);
        float s, e;
        two_sum_f(hi, oh, s, e);
        hi = s;
        lo = __fadd_rn(__fadd_rn(lo, ol), e);
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    if (lane == 0) red[warp] = make_float2(hi, lo);
    __syncthreads();
    if (warp == 0) {
        float2 v = lane < nw ? red[lane] : make_float2(0.f, 0.f);
        hi = v.x;
        lo = v.y;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            float oh = __shfl_xor_sync(0xffffffffu, hi, off);
            float ol = __shfl_xor_sync(0xffffffffu, lo, off);
            float s, e;
            two_sum_f(hi, oh, s, e);
            hi = s;
            lo = __fadd_rn(__fadd_rn(lo, ol), e);
        }
        if (lane == 0) red[32] = make_float2(hi, lo);
    }
    __syncthreads();
    hi = red[32].x;
    lo = red[32].y;
}

// Reciprocal RMS of one row (GlmMoeDsaRMSNorm.forward): the mean of squares
// is accumulated with compensated fp32 sums (squares split exactly with an
// FMA), so it equals the exact mean rounded to fp32 except in vanishingly
// rare cases; then rsqrt(mean + eps) as an fp32 add, sqrt and divide, each
// correctly rounded.
template <typename T>
__device__ __forceinline__ float row_rrms(const T* xr, int d, float eps, float2* red) {
    constexpr int V = Elem<T>::V;
    float hi = 0.f, lo = 0.f;
    for (int v = threadIdx.x; v < d / V; v += blockDim.x) {
        float f[V];
        load_vec<T>(xr + v * V, f);
#pragma unroll
        for (int i = 0; i < V; ++i) {
            float p = __fmul_rn(f[i], f[i]);
            float pe = fmaf(f[i], f[i], -p);  // exact low part of the square
            float s, e;
            two_sum_f(hi, p, s, e);
            hi = s;
            lo = __fadd_rn(lo, __fadd_rn(e, pe));
        }
    }
    block_sum_pair(hi, lo, red);
    const float ms = mean_of_pair(hi, lo, d);
    return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, eps)));
}

// xn = gain * cast(x * r): one block per token.  Rows of up to
// RMS_REG_VECS vectors per thread stay in registers between the reduction
// and the scaling (x is read once); longer rows are read twice.
constexpr int RMS_REG_VECS = 4;

template <typename T>
__global__ void rmsnorm_kernel(const T* __restrict__ x, const T* __restrict__ gain,
                               T* __restrict__ xn, int d, float eps) {
    grid_dep_wait();
    __shared__ float2 red[33];
    constexpr int V = Elem<T>::V;
    const size_t t = blockIdx.x;
    const T* xr = x + t * d;
    const int nvec = d / V;
    if (nvec > RMS_REG_VECS * static_cast<int>(blockDim.x)) {
        const float r = row_rrms<T>(xr, d, eps, red);
        for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
            float f[V], g[V];
            load_vec<T>(xr + v * V, f);
            load_vec<T>(gain + v * V, g);
#pragma unroll
            for (int i = 0; i < V; ++i) f[i] = __fmul_rn(g[i], Elem<T>::round_io(__fmul_rn(f[i], r)));
            store_vec<T>(xn + t * d + v * V, f);
        }
        return;
    }
    // the gain's vectors are loaded with the row's, so that the scaling after
    // the reduction waits for no second round trip to memory
    float f[RMS_REG_VECS][V];
    int4 graw[RMS_REG_VECS];
#pragma unroll
    for (int j = 0; j < RMS_REG_VECS; ++j) {
        const int v = threadIdx.x + j * blockDim.x;
        if (v < nvec) {
            load_vec<T>(xr + v * V, f[j]);
            graw[j] = *reinterpret_cast<const int4*>(gain + v * V);
        }
    }
    // the same compensated sum of squares as row_rrms, over the registers
    float hi = 0.f, lo = 0.f;
#pragma unroll
    for (int j = 0; j < RMS_REG_VECS; ++j) {
        if (threadIdx.x + j * blockDim.x >= nvec) continue;
#pragma unroll
        for (int i = 0; i < V; ++i) {
            const float p = __fmul_rn(f[j][i], f[j][i]);
            const float pe = fmaf(f[j][i], f[j][i], -p);
            float s, e;
            two_sum_f(hi, p, s, e);
            hi = s;
            lo = __fadd_rn(lo, __fadd_rn(e, pe));
        }
    }
    block_sum_pair(hi, lo, red);
    const float ms = mean_of_pair(hi, lo, d);
    const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, eps)));
#pragma unroll
    for (int j = 0; j < RMS_REG_VECS; ++j) {
        const int v = threadIdx.x + j * blockDim.x;
        if (v >= nvec) continue;
        float g[V];
        unpack_vec<T>(graw[j], g);
#pragma unroll
        for (int i = 0; i < V; ++i) f[j][i] = __fmul_rn(g[i], Elem<T>::round_io(__fmul_rn(f[j][i], r)));
        store_vec<T>(xn + t * d + v * V, f[j]);
    }
}

// One 16-byte vector of the RMSNorm output: gain * cast(x * r), each
// product rounded as the storage dtype's is.  For bf16 the gain product is
// one packed bf16 multiply: the product of two bf16 values is exact in fp32,
// so rounding it once to bf16 gives what the fp32 multiply and the store's
// rounding give.
template <typename T>
__device__ __forceinline__ int4 rms_scale_vec(const int4& raw, const int4& graw, float r) {
    constexpr int V = Elem<T>::V;
    float f[V], g[V];
    unpack_vec<T>(raw, f);
    unpack_vec<T>(graw, g);
#pragma unroll
    for (int i = 0; i < V; ++i) f[i] = __fmul_rn(g[i], Elem<T>::round_io(__fmul_rn(f[i], r)));
    int4 out;
    store_vec<T>(reinterpret_cast<T*>(&out), f);
    return out;
}
template <>
__device__ __forceinline__ int4 rms_scale_vec<__nv_bfloat16>(const int4& raw, const int4& graw, float r) {
    const __nv_bfloat162* xv = reinterpret_cast<const __nv_bfloat162*>(&raw);
    const __nv_bfloat162* gv = reinterpret_cast<const __nv_bfloat162*>(&graw);
    int4 out;
    __nv_bfloat162* ov = reinterpret_cast<__nv_bfloat162*>(&out);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 xf = __bfloat1622float2(xv[i]);
        ov[i] = __hmul2(gv[i], __floats2bfloat162_rn(__fmul_rn(xf.x, r), __fmul_rn(xf.y, r)));
    }
    return out;
}

// The same RMSNorm with a warp per token and the rows staged in shared
// memory.  Each warp owns RMSB_NBUF row buffers, filled by untiled bulk
// copies (cp.async.bulk) that complete on one mbarrier per buffer; a buffer
// is refilled with the warp's next row as soon as its row is scaled.  The
// scaling pass reads the row from shared memory instead of again from L2,
// and the block holds the gain row in shared memory too.  With 12 KB rows,
// sixteen warps of one buffer (39.8 us for 8192 x 6144 bf16) measured faster
// than eight warps of two (43.0 us): the kernel is bound by the issue of its
// dependent arithmetic more than by the copies' latency, and more warps hide
// more of it (eight vectors in flight per lane instead of four did not).
// The warps loop over tokens (stride: all warps of the grid).  Per lane the
// arithmetic is that of a warp reading the row itself: vectors lane,
// lane + 32, ... in order
// (four at a time, for independent instructions), each vector's V squares
// by an FMA chain (at most V roundings, a relative error below V * 2^-24 of
// the vector's sum), the vectors added with a compensated sum, then a shuffle
// reduction.  The waits are bounded: a copy that has not landed after
// RMS_WAIT_NS sets the timeout bit of the device error flag, and the warp
// waits (again bounded) for its copies in flight before it returns.
// Shared memory: RMSB_NBUF barriers per warp (RMSB_WARPS_MAX slots), the
// gain row, then RMSB_NBUF row buffers per warp.  Rows 16-byte aligned (d *
// sizeof(T) a multiple of 16).
constexpr int RMSB_WARPS_MAX = 16;
constexpr int RMSB_NBUF = 1;
constexpr int RMSB_U = 4;                          // vectors per lane in flight
constexpr size_t RMSB_BAR_BYTES = (8 * RMSB_NBUF * RMSB_WARPS_MAX + 15) / 16 * 16;
constexpr uint64_t RMS_WAIT_NS = 2000000000ull;   // 2 s
constexpr uint64_t RMS_DRAIN_NS = 100000000ull;   // 100 ms

__host__ __device__ constexpr size_t rmsb_smem(int warps, size_t row_bytes) {
    return RMSB_BAR_BYTES + static_cast<size_t>(1 + RMSB_NBUF * warps) * row_bytes;
}

// Untiled bulk copy of `bytes` from global to shared memory, completing on
// `bar` as that many transaction bytes (16-byte aligned addresses, bytes a
// multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

template <typename T>
__global__ void __launch_bounds__(32 * RMSB_WARPS_MAX)
    rmsnorm_bulk_kernel(const T* __restrict__ x, const T* __restrict__ gain, T* __restrict__ xn, int n_tok, int d,
                        float eps, int* __restrict__ err) {
    extern __shared__ __align__(16) uint8_t rms_smem[];
    constexpr int V = Elem<T>::V;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int stride = gridDim.x * (blockDim.x >> 5);
    const uint32_t row_bytes = static_cast<uint32_t>(d) * sizeof(T);
    const int nvec = d / V;
    uint64_t* bar = reinterpret_cast<uint64_t*>(rms_smem) + RMSB_NBUF * warp;
    int4* gs = reinterpret_cast<int4*>(rms_smem + RMSB_BAR_BYTES);
    uint8_t* buf = rms_smem + RMSB_BAR_BYTES + static_cast<size_t>(1 + RMSB_NBUF * warp) * row_bytes;
    int t = blockIdx.x * (blockDim.x >> 5) + warp;
    // the gain is a weight (no kernel before this one writes it)
    for (int v = threadIdx.x; v < nvec; v += blockDim.x) gs[v] = reinterpret_cast<const int4*>(gain)[v];
    if (lane == 0) {
        for (int b = 0; b < RMSB_NBUF; ++b) mbar_init(&bar[b], 1);
        fence_mbarrier_init();
    }
    __syncthreads();
    grid_dep_wait();
    if (lane == 0) {
        for (int b = 0; b < RMSB_NBUF; ++b) {
            const int tb = t + b * stride;
            if (tb < n_tok) {
                mbar_arrive_expect_tx(&bar[b], row_bytes);
                bulk_load(buf + b * row_bytes, x + static_cast<size_t>(tb) * d, row_bytes, &bar[b]);
            }
        }
    }
    int j = 0;
    for (; t < n_tok; ++j, t += stride) {
        const int b = j % RMSB_NBUF;
        const int4* row = reinterpret_cast<const int4*>(buf + b * row_bytes);
        // every lane observes the phase, which makes the copied bytes visible to it
        const bool landed = mbar_wait(&bar[b], (j / RMSB_NBUF) & 1, nullptr, RMS_WAIT_NS);
        if (!__all_sync(0xffffffffu, landed)) break;
        float hi = 0.f, lo = 0.f;
        for (int v0 = lane; v0 < nvec; v0 += 32 * RMSB_U) {
            float c[RMSB_U];
#pragma unroll
            for (int u = 0; u < RMSB_U; ++u) {
                c[u] = 0.f;
                const int v = v0 + 32 * u;
                if (v < nvec) {
                    const int4 raw = row[v];
                    const T* e = reinterpret_cast<const T*>(&raw);
#pragma unroll
                    for (int i = 0; i < V; ++i) {
                        const float f = Elem<T>::to_f(e[i]);
                        c[u] = fmaf(f, f, c[u]);
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < RMSB_U; ++u) {
                if (v0 + 32 * u >= nvec) break;
                float s, er;
                two_sum_f(hi, c[u], s, er);
                hi = s;
                lo = __fadd_rn(lo, er);
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float oh = __shfl_xor_sync(0xffffffffu, hi, off);
            const float ol = __shfl_xor_sync(0xffffffffu, lo, off);
            float s, er;
            two_sum_f(hi, oh, s, er);
            hi = s;
            lo = __fadd_rn(__fadd_rn(lo, ol), er);
        }
        const float ms = mean_of_pair(hi, lo, d);
        const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, eps)));
        int4* out = reinterpret_cast<int4*>(xn + static_cast<size_t>(t) * d);
        for (int v0 = lane; v0 < nvec; v0 += 32 * RMSB_U) {
#pragma unroll
            for (int u = 0; u < RMSB_U; ++u) {
                const int v = v0 + 32 * u;
                if (v < nvec) out[v] = rms_scale_vec<T>(row[v], gs[v], r);
            }
        }
        // the buffer is refilled by the async proxy after every lane's reads
        __syncwarp();
        const int tn = t + RMSB_NBUF * stride;
        if (lane == 0 && tn < n_tok) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_arrive_expect_tx(&bar[b], row_bytes);
            bulk_load(buf + b * row_bytes, x + static_cast<size_t>(tn) * d, row_bytes, &bar[b]);
        }
    }
    if (t < n_tok && lane == 0) {
        // gave up on row j: report it, then wait for this warp's copies still
        // in flight (rows j .. j + RMSB_NBUF - 1) before its shared memory is
        // released
        atomicOr(err, 1);
        for (int i = 0; i < RMSB_NBUF && t + i * stride < n_tok; ++i)
            mbar_wait(&bar[(j + i) % RMSB_NBUF], ((j + i) / RMSB_NBUF) & 1, nullptr, RMS_DRAIN_NS);
    }
}

// RMSNorm fused with the router logits on CUDA cores (fp32 accumulation):
// one block per token; the normalised row stays in shared memory and each
// warp takes experts e = warp, warp + nwarps, ... with 16-byte loads of the
// router weight and a warp-shuffle reduction.  The logits are written as
// (value, 0) pairs, the format the top-k kernel reads.  Dynamic smem: d floats.
template <typename T>
__global__ void rmsnorm_router_kernel(const T* __restrict__ x, const T* __restrict__ gain,
                                      const T* __restrict__ router_w, T* __restrict__ xn,
                                      float2* __restrict__ part, int d, int E, float eps) {
    extern __shared__ float xs[];
    __shared__ float2 red[33];
    constexpr int V = Elem<T>::V;
    const size_t t = blockIdx.x;
    const T* xr = x + t * d;
    const float r = row_rrms<T>(xr, d, eps, red);
    for (int v = threadIdx.x; v < d / V; v += blockDim.x) {
        float f[V], g[V];
        load_vec<T>(xr + v * V, f);
        load_vec<T>(gain + v * V, g);
#pragma unroll
        for (int i = 0; i < V; ++i) {
            f[i] = __fmul_rn(g[i], Elem<T>::round_io(__fmul_rn(f[i], r)));
            f[i] = Elem<T>::round_io(f[i]);
            xs[v * V + i] = f[i];
        }
        store_vec<T>(xn + t * d + v * V, f);
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    for (int e = warp; e < E; e += nw) {
        const T* wr = router_w + static_cast<size_t>(e) * d;
        float acc = 0.f;
        for (int v = lane; v < d / V; v += 32) {
            float w[V];
            load_vec<T>(wr + v * V, w);
#pragma unroll
            for (int i = 0; i < V; ++i) acc = fmaf(xs[v * V + i], w[i], acc);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == 0) part[t * E + e] = make_float2(acc, 0.f);
    }
}

// ------------------------------------------------------------------ top-k
// Where the top-k kernel reads a token's logits from: the router's (hi, lo)
// partial-sum pair, rounded once here (and recorded in `logits` for
// inspection), or plain fp32 logits given by the caller.  load() only reads,
// so that a lane's loads of all its experts are in flight together; record()
// writes afterwards.
struct LogitsFromPairs {
    const float2* __restrict__ part;
    float* __restrict__ logits;
    __device__ float load(size_t i) const {
        const float2 pv = part[i];
        return __fadd_rn(pv.x, pv.y);   // the (hi, lo) pair, rounded once
    }
    __device__ void record(size_t i, float l) const { logits[i] = l; }
};
struct LogitsPlain {
    const float* __restrict__ logits;
    __device__ float load(size_t i) const { return logits[i]; }
    __device__ void record(size_t, float) const {}
};

// The routing score of one logit: s = sigmoid(l) and the selection key
// b = s + correction bias, a NaN key ranking last (keeps the order total).
// Both top-k kernels call this, so they take the same decisions.
__device__ __forceinline__ void router_score(float l, float bias_e, float& s, float& b) {
    s = __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-l)));
    const float bb = __fadd_rn(s, bias_e);
    b = (bb == bb) ? bb : -INFINITY;
}

// Top-k of one token by one warp: k rounds of a warp argmax on (key bv
// descending, expert index ascending) over the experts lane + 32 i held in
// bv / sv (keys / sigmoid scores).  Slot j's expert and weight end up in lane
// j: w_j = routed_scale * s_j / (s_0 + ... + s_{k-1}), the sum taken in slot
// order.  Lanes j >= k get expert 0 and weight 0.
// Each (key, expert) is packed into one 64-bit integer whose order is that
// order: the key's bits mapped to an unsigned integer of the same order (after
// -0 is made +0, so that the two tie as floats do) above the expert index
// subtracted from 2^32 - 1.  A round's warp argmax is then a 64-bit max over
// five shuffle levels, and one more shuffle fetches the winner's score from
// the lane that holds it.  Keys are never NaN (router_score ranks NaN last as
// -inf, whose mapped key is 0x007FFFFF); an expert already taken, or past E,
// gets the key 0, below every real key.  Only the 32-bit keys are kept (the
// 64-bit values would not fit the registers of a 1024-thread block).
template <int EPL>
__device__ __forceinline__ void warp_select_topk(const float (&bv)[EPL], const float (&sv)[EPL], int E, int k,
                                                 float routed_scale, int lane, int& my_e, float& my_w) {
    uint32_t key[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        const uint32_t u = __float_as_uint(__fadd_rn(bv[i], 0.0f));
        key[i] = e < E ? ((u & 0x80000000u) ? ~u : (u | 0x80000000u)) : 0u;
    }
    my_e = 0;
    float my_s = 0.f;
    for (int j = 0; j < k; ++j) {
        // candidate of this lane: the best expert it still holds (every
        // unselected expert is a candidate, so a winner always exists: k <= E)
        uint64_t cand = 0ull;
        float cs = 0.f;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const uint64_t v = (static_cast<uint64_t>(key[i]) << 32) |
                               (0xFFFFFFFFu - static_cast<uint32_t>(lane + 32 * i));
            if (v > cand) { cand = v; cs = sv[i]; }
        }
        uint64_t win = cand;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const uint64_t o = __shfl_xor_sync(0xffffffffu, win, off);
            win = o > win ? o : win;
        }
        const int we = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(win));
        const float ws = __shfl_sync(0xffffffffu, cs, we & 31);
        if ((we & 31) == lane) {
#pragma unroll
            for (int i = 0; i < EPL; ++i)
                if (i == (we >> 5)) key[i] = 0u;
        }
        if (lane == j) { my_e = we; my_s = ws; }
    }
    float ssum = 0.f;
    for (int j = 0; j < k; ++j) ssum = __fadd_rn(ssum, __shfl_sync(0xffffffffu, my_s, j));
    my_w = lane < k ? __fdiv_rn(__fmul_rn(routed_scale, my_s), ssum) : 0.f;
}

// One warp per token.  s = sigmoid(l), b = s + bias; k rounds of a warp
// argmax on (b descending, expert index ascending); slot j's expert and
// sigmoid end up in lane j.  w_j = routed_scale * s_j / sum_i s_i.  Blocks
// cover CHUNK_TOKENS / split tokens of a histogram chunk (split blocks per
// chunk, so that small batches still spread over the SMs); each counts its
// tokens' experts in shared memory and adds the counts to its chunk's
// histogram in global memory (zeroed before the launch when split > 1;
// integer adds, so the result does not depend on their order).
// EPL = experts per lane (ceil(E / 32)).  The selection does not depend on
// where the logits came from: given the same fp32 logits, both sources take
// the same decisions and give the same weights bit for bit.
template <int EPL, typename Src>
__global__ void topk_kernel(const Src src, const float* __restrict__ bias, int T, int E, int k,
                            float routed_scale, int* __restrict__ idx_out, float* __restrict__ w_out,
                            int* __restrict__ chunk_cnt, int split) {
    grid_dep_wait();
    extern __shared__ int cnt[];  // [E]
    for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    const int chunk = blockIdx.x / split;
    const int sub_tokens = CHUNK_TOKENS / split;
    const int first = chunk * CHUNK_TOKENS + (blockIdx.x - chunk * split) * sub_tokens;
    for (int tl = warp; tl < sub_tokens; tl += nw) {
        const int t = first + tl;
        if (t >= T) break;
        float bv[EPL], sv[EPL], lv[EPL];
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = lane + 32 * i;
            lv[i] = e < E ? src.load(static_cast<size_t>(t) * E + e) : 0.f;
        }
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = lane + 32 * i;
            if (e < E) {
                const float l = lv[i];
                src.record(static_cast<size_t>(t) * E + e, l);
                router_score(l, bias[e], sv[i], bv[i]);
            } else {
                sv[i] = 0.f;
                bv[i] = 0.f;
            }
        }
        int my_e;
        float my_w;
        warp_select_topk<EPL>(bv, sv, E, k, routed_scale, lane, my_e, my_w);
        if (lane < k) {
            idx_out[static_cast<size_t>(t) * k + lane] = my_e;
            w_out[static_cast<size_t>(t) * k + lane] = my_w;
            atomicAdd(&cnt[my_e], 1);
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        if (split == 1)
            chunk_cnt[static_cast<size_t>(chunk) * E + e] = cnt[e];
        else if (cnt[e] != 0)
            atomicAdd(&chunk_cnt[static_cast<size_t>(chunk) * E + e], cnt[e]);
    }
}

// --------------------------------------------------- histogram scan (1 block)
// counts[e] = sum over chunks; offsets = exclusive scan of counts (offsets[E]
// = T*k); chunk_base[c][e] = offsets[e] + rows of expert e in chunks < c.
__global__ void scan_kernel(const int* __restrict__ chunk_cnt, int n_chunks, int E,
                            int* __restrict__ counts, int* __restrict__ offsets,
                            int* __restrict__ chunk_base) {
    grid_dep_wait();
    __shared__ int warp_tot[32];
    const int e = threadIdx.x;  // blockDim.x >= E, multiple of 32
    int total = 0;
    if (e < E)
        for (int c = 0; c < n_chunks; ++c) total += chunk_cnt[static_cast<size_t>(c) * E + e];
    const int lane = e & 31, warp = e >> 5;
    int incl = total;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += u;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int v = lane < (blockDim.x >> 5) ? warp_tot[lane] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, v, off);
            if (lane >= off) v += u;
        }
        warp_tot[lane] = v;  // inclusive scan of warp totals
    }
    __syncthreads();
    const int excl = incl - total + (warp > 0 ? warp_tot[warp - 1] : 0);
    if (e < E) {
        counts[e] = total;
        offsets[e] = excl;
        if (e == E - 1) offsets[E] = excl + total;
        int run = excl;
        for (int c = 0; c < n_chunks; ++c) {
            chunk_base[static_cast<size_t>(c) * E + e] = run;
            run += chunk_cnt[static_cast<size_t>(c) * E + e];
        }
    }
}

// ---------------------------------------------------------- stable scatter
// One block (CHUNK_TOKENS threads) per chunk.  The row of (token t, slot j)
// is chunk_base[c][e] + (number of earlier tokens of the chunk routed to e),
// so rows of each expert are ordered by token.  Dynamic smem: E * 4 words.
__global__ void scatter_kernel(const int* __restrict__ idx, const float* __restrict__ w, int T,
                               int E, int k, const int* __restrict__ chunk_base,
                               int* __restrict__ pos, int* __restrict__ row_tok,
                               float* __restrict__ row_w) {
    grid_dep_wait();
    extern __shared__ uint32_t mask[];  // [E][CHUNK_TOKENS / 32]
    constexpr int WORDS = CHUNK_TOKENS / 32;
    for (int i = threadIdx.x; i < E * WORDS; i += blockDim.x) mask[i] = 0u;
    __syncthreads();
    const int tl = threadIdx.x;
    const int t = blockIdx.x * CHUNK_TOKENS + tl;
    const bool valid = t < T;
    if (valid)
        for (int j = 0; j < k; ++j)
            atomicOr(&mask[idx[static_cast<size_t>(t) * k + j] * WORDS + (tl >> 5)],
                     1u << (tl & 31));
    __syncthreads();
    if (!valid) return;
    for (int j = 0; j < k; ++j) {
        const int e = idx[static_cast<size_t>(t) * k + j];
        int rank = __popc(mask[e * WORDS + (tl >> 5)] & ((1u << (tl & 31)) - 1u));
        for (int wi = 0; wi < (tl >> 5); ++wi) rank += __popc(mask[e * WORDS + wi]);
        const int row = chunk_base[static_cast<size_t>(blockIdx.x) * E + e] + rank;
        pos[static_cast<size_t>(t) * k + j] = row;
        row_tok[row] = t;
        row_w[row] = w[static_cast<size_t>(t) * k + j];
    }
}

// xp[pos[t, j]] = xn[t] for every slot j: one warp per token, so each xn row
// is read from memory once (a row-by-row gather re-reads it k times, and the
// stream of writes evicts it from L2 in between).  16-byte vectors, eight in
// flight per lane.  Rows outside [0, P) are skipped.
template <typename T>
__global__ void gather_tokens_kernel(const T* __restrict__ xn, const int* __restrict__ pos,
                                     T* __restrict__ xp, int n_tok, int k, int d, int P) {
    grid_dep_wait();
    const int lane = threadIdx.x & 31;
    const int nvec = d * static_cast<int>(sizeof(T)) / 16;
    constexpr int U = 8;
    for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < n_tok;
         t += (gridDim.x * blockDim.x) >> 5) {
        const int4* src = reinterpret_cast<const int4*>(xn + static_cast<size_t>(t) * d);
        int rows[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) rows[j] = j < k ? pos[static_cast<size_t>(t) * k + j] : -1;
        for (int v0 = 0; v0 < nvec; v0 += 32 * U) {
            int4 r[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int v = v0 + u * 32 + lane;
                if (v < nvec) r[u] = __ldg(src + v);
            }
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                if (j >= k) break;
                const int row = rows[j];
                if (row < 0 || row >= P) continue;
                int4* dst = reinterpret_cast<int4*>(xp + static_cast<size_t>(row) * d);
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int v = v0 + u * 32 + lane;
                    if (v < nvec) dst[v] = r[u];
                }
            }
        }
    }
}

// xp[row] = xn[row_tok[row]]: one warp per row, 16-byte vectors.  The token
// index is clamped into [0, n_tok) so that no input can make it read out of range.
template <typename T>
__global__ void gather_rows_kernel(const T* __restrict__ xn, const int* __restrict__ row_tok,
                                   T* __restrict__ xp, int P, int d, int n_tok) {
    grid_dep_wait();
    const int lane = threadIdx.x & 31;
    const int nvec = d * static_cast<int>(sizeof(T)) / 16;
    for (int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; row < P;
         row += (gridDim.x * blockDim.x) >> 5) {
        const int t = min(max(row_tok[row], 0), n_tok - 1);
        const int4* src = reinterpret_cast<const int4*>(xn + static_cast<size_t>(t) * d);
        int4* dst = reinterpret_cast<int4*>(xp + static_cast<size_t>(row) * d);
        // eight 16-byte loads in flight per lane before the stores
        constexpr int U = 8;
        int v = lane;
        for (; v + 32 * (U - 1) < nvec; v += 32 * U) {
            int4 r[U];
#pragma unroll
            for (int u = 0; u < U; ++u) r[u] = __ldg(src + v + 32 * u);
#pragma unroll
            for (int u = 0; u < U; ++u) dst[v + 32 * u] = r[u];
        }
        for (; v < nvec; v += 32) dst[v] = __ldg(src + v);
    }
}

// out[t] = x[t] + sh[t] + sum_j yp[pos[t, j]] in fp32, slots in order, one
// rounding at the end (yp rows already carry their routing weight).  On the
// tensor-core path the shared expert's output sh is fp32 (ST) and the
// weighted rows yp fp16 (YT); elsewhere both are the handle dtype.  Block
// (t, y) covers token t's vectors y * blockDim.x + threadIdx.x, ... (small
// batches split a row over several blocks so that its loads run in parallel).
// The slots' rows are loaded COMBINE_U at a time before they are added (with
// k a run-time count, a load-add loop kept one row load in flight per thread).
constexpr int COMBINE_U = 8;
template <typename T, typename YT = T, typename ST = T>
__global__ void combine_kernel(const T* __restrict__ x, const ST* __restrict__ sh,
                               const YT* __restrict__ yp, const int* __restrict__ pos, int d, int k,
                               T* __restrict__ out) {
    grid_dep_wait();
    constexpr int V = Elem<T>::V;
    const size_t t = blockIdx.x;
    for (int v = blockIdx.y * blockDim.x + threadIdx.x; v < d / V; v += gridDim.y * blockDim.x) {
        float acc[V], tmp[V];
        load_vec<T>(x + t * d + v * V, acc);
        if (sh != nullptr) {
            if constexpr (Elem<ST>::V == V) {
                load_vec<ST>(sh + t * d + v * V, tmp);
            } else {   // fp32 sh beside 16-bit x: two 16-byte loads per vector
                static_assert(V == 2 * Elem<ST>::V, "vector widths");
                float lo[Elem<ST>::V], hi[Elem<ST>::V];
                load_vec<ST>(sh + t * d + v * V, lo);
                load_vec<ST>(sh + t * d + v * V + Elem<ST>::V, hi);
#pragma unroll
                for (int i = 0; i < Elem<ST>::V; ++i) { tmp[i] = lo[i]; tmp[Elem<ST>::V + i] = hi[i]; }
            }
#pragma unroll
            for (int i = 0; i < V; ++i) acc[i] += tmp[i];
        }
        static_assert(Elem<YT>::V == V, "one 16-byte vector of yp per vector of out");
        for (int j0 = 0; j0 < k; j0 += COMBINE_U) {
            int4 raw[COMBINE_U];
#pragma unroll
            for (int u = 0; u < COMBINE_U; ++u)
                if (j0 + u < k)
                    raw[u] = *reinterpret_cast<const int4*>(
                        yp + static_cast<size_t>(pos[t * k + j0 + u]) * d + v * V);
#pragma unroll
            for (int u = 0; u < COMBINE_U; ++u) {
                if (j0 + u >= k) break;
                unpack_vec<YT>(raw[u], tmp);
#pragma unroll
                for (int i = 0; i < V; ++i) acc[i] += tmp[i];
            }
        }
        store_vec<T>(out + t * d + v * V, acc);
    }
}

// Split-K dense down projection: out = res + sum over the k-ranges of the fp32
// partials part[s][i] (s in order, then the residual), rounded once.  n (the
// element count) is a multiple of 4; part, res and out are 16-byte aligned.
template <typename T>
__global__ void splitk_residual_kernel(const float* __restrict__ part, int nsplit, size_t stride,
                                       const T* __restrict__ res, T* __restrict__ out, size_t n) {
    grid_dep_wait();
    for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n / 4;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        float4 acc = reinterpret_cast<const float4*>(part)[i];
        for (int sp = 1; sp < nsplit; ++sp) {
            const float4 v = reinterpret_cast<const float4*>(part + sp * stride)[i];
            acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
        }
        float r[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) r[j] = Elem<T>::to_f(res[4 * i + j]);
        out[4 * i + 0] = Elem<T>::from_f(acc.x + r[0]);
        out[4 * i + 1] = Elem<T>::from_f(acc.y + r[1]);
        out[4 * i + 2] = Elem<T>::from_f(acc.z + r[2]);
        out[4 * i + 3] = Elem<T>::from_f(acc.w + r[3]);
    }
}

// The dense block's split gate|up projection: h[t, f] = silu(g) * u with g
// and u the sums, in k-range order, of the fp32 partials part[s][t][f] and
// part[s][t][F + f], rounded once to the storage dtype (the same SwiGLU
// arithmetic as the GEMM epilogue).  Four features per thread; F is a
// multiple of 4.
template <typename T>
__global__ void splitk_swiglu_kernel(const float* __restrict__ part, int nsplit, int n_tok, int F,
                                     T* __restrict__ h) {
    grid_dep_wait();
    const size_t stride = static_cast<size_t>(n_tok) * 2 * F;
    const size_t n4 = static_cast<size_t>(n_tok) * F / 4;
    for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const size_t t = i / (F / 4), f = (i - t * (F / 4)) * 4;
        const float* g0 = part + t * 2 * F + f;
        float4 g = *reinterpret_cast<const float4*>(g0);
        float4 u = *reinterpret_cast<const float4*>(g0 + F);
        for (int sp = 1; sp < nsplit; ++sp) {
            const float4 gs = *reinterpret_cast<const float4*>(g0 + sp * stride);
            const float4 us = *reinterpret_cast<const float4*>(g0 + sp * stride + F);
            g.x += gs.x; g.y += gs.y; g.z += gs.z; g.w += gs.w;
            u.x += us.x; u.y += us.y; u.z += us.z; u.w += us.w;
        }
        T* o = h + t * F + f;
        o[0] = Elem<T>::from_f(g.x / (1.0f + __expf(-g.x)) * u.x);
        o[1] = Elem<T>::from_f(g.y / (1.0f + __expf(-g.y)) * u.y);
        o[2] = Elem<T>::from_f(g.z / (1.0f + __expf(-g.z)) * u.z);
        o[3] = Elem<T>::from_f(g.w / (1.0f + __expf(-g.w)) * u.w);
    }
}

// The query compression's split-K epilogue, one block per token: c = the sum
// of the k-range partials part[s][t] (s in order) rounded once to the
// storage dtype (the Linear's output), then q = gain * cast(c * r) with r the
// reciprocal RMS of the rounded c (GlmMoeDsaRMSNorm, the same arithmetic as
// rmsnorm_kernel).  Both passes run over 16-byte vectors; the second re-reads
// c from memory it just wrote (L2).  rank is a multiple of the vector width.
template <typename T>
__global__ void splitk_rmsnorm_kernel(const float* __restrict__ part, int nsplit, size_t stride, int rank,
                                      const T* __restrict__ gain, float eps, T* __restrict__ c_out,
                                      T* __restrict__ q_out) {
    grid_dep_wait();
    __shared__ float2 red[33];
    constexpr int V = Elem<T>::V;
    const size_t t = blockIdx.x;
    const float* pr = part + t * rank;
    T* cr = c_out + t * rank;
    float hi = 0.f, lo = 0.f;
    for (int v = threadIdx.x; v < rank / V; v += blockDim.x) {
        float a[V];
#pragma unroll
        for (int i = 0; i < V; i += 4) {
            const float4 p4 = *reinterpret_cast<const float4*>(pr + v * V + i);
            a[i] = p4.x; a[i + 1] = p4.y; a[i + 2] = p4.z; a[i + 3] = p4.w;
        }
        for (int sp = 1; sp < nsplit; ++sp) {
#pragma unroll
            for (int i = 0; i < V; i += 4) {
                const float4 p4 = *reinterpret_cast<const float4*>(pr + sp * stride + v * V + i);
                a[i] += p4.x; a[i + 1] += p4.y; a[i + 2] += p4.z; a[i + 3] += p4.w;
            }
        }
#pragma unroll
        for (int i = 0; i < V; ++i) {
            a[i] = Elem<T>::round_io(a[i]);
            const float sq = __fmul_rn(a[i], a[i]);
            const float sqe = fmaf(a[i], a[i], -sq);
            float s2, e2;
            two_sum_f(hi, sq, s2, e2);
            hi = s2;
            lo = __fadd_rn(lo, __fadd_rn(e2, sqe));
        }
        store_vec<T>(cr + v * V, a);
    }
    block_sum_pair(hi, lo, red);   // its barriers also order the c stores before the reads below
    const float ms = mean_of_pair(hi, lo, rank);
    const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, eps)));
    for (int v = threadIdx.x; v < rank / V; v += blockDim.x) {
        float f[V], g[V];
        load_vec<T>(cr + v * V, f);
        load_vec<T>(gain + v * V, g);
#pragma unroll
        for (int i = 0; i < V; ++i) f[i] = __fmul_rn(g[i], Elem<T>::round_io(__fmul_rn(f[i], r)));
        store_vec<T>(q_out + t * rank + v * V, f);
    }
}

// ------------------------------------------------- FFMA expert kernels (fp32)
// Expert of a permuted row: the last e with offsets[e] <= row.
__device__ __forceinline__ int expert_of_row(const int* offsets, int E, int row) {
    int lo = 0, hi = E;  // offsets[lo] <= row < offsets[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (offsets[mid] <= row) lo = mid; else hi = mid;
    }
    return lo;
}

// h[row, i] = silu(xp[row] . gate_up[e][:, i]) * (xp[row] . gate_up[e][:, I + i]).
// grid (P, ceil(I / blockDim)); dynamic smem: d floats.
template <typename T>
__global__ void simt_gate_up_kernel(const T* __restrict__ xp, const T* __restrict__ gate_up,
                                    const int* __restrict__ offsets, int E, int d, int I,
                                    T* __restrict__ h) {
    extern __shared__ float rowv[];
    const int row = blockIdx.x;
    const int e = expert_of_row(offsets, E, row);
    for (int j = threadIdx.x; j < d; j += blockDim.x)
        rowv[j] = Elem<T>::to_f(xp[static_cast<size_t>(row) * d + j]);
    __syncthreads();
    const int i = blockIdx.y * blockDim.x + threadIdx.x;
    if (i >= I) return;
    const T* w = gate_up + static_cast<size_t>(e) * d * 2 * I;
    float g = 0.f, u = 0.f;
    for (int j = 0; j < d; ++j) {
        g = fmaf(rowv[j], Elem<T>::to_f(w[static_cast<size_t>(j) * 2 * I + i]), g);
        u = fmaf(rowv[j], Elem<T>::to_f(w[static_cast<size_t>(j) * 2 * I + I + i]), u);
    }
    h[static_cast<size_t>(row) * I + i] = Elem<T>::from_f(silu_f(g) * u);
}

// yp[row, o] = row_w[row] * (h[row] . down[e][:, o]).  grid (P, ceil(d / blockDim)).
template <typename T>
__global__ void simt_down_kernel(const T* __restrict__ h, const T* __restrict__ down,
                                 const int* __restrict__ offsets, const float* __restrict__ row_w,
                                 int E, int I, int d, T* __restrict__ yp) {
    extern __shared__ float rowv[];
    const int row = blockIdx.x;
    const int e = expert_of_row(offsets, E, row);
    for (int i = threadIdx.x; i < I; i += blockDim.x)
        rowv[i] = Elem<T>::to_f(h[static_cast<size_t>(row) * I + i]);
    __syncthreads();
    const int o = blockIdx.y * blockDim.x + threadIdx.x;
    if (o >= d) return;
    const T* w = down + static_cast<size_t>(e) * I * d;
    float acc = 0.f;
    for (int i = 0; i < I; ++i) acc = fmaf(rowv[i], Elem<T>::to_f(w[static_cast<size_t>(i) * d + o]), acc);
    yp[static_cast<size_t>(row) * d + o] = Elem<T>::from_f(acc * row_w[row]);
}

// Shared expert, nn.Linear weights: hs[t, i] = silu(Gs[i] . xn[t]) * (Us[i] . xn[t]).
template <typename T>
__global__ void simt_shared_gate_up_kernel(const T* __restrict__ xn, const T* __restrict__ Gs,
                                           const T* __restrict__ Us, int d, int Is,
                                           T* __restrict__ hs) {
    extern __shared__ float rowv[];
    const int t = blockIdx.x;
    for (int j = threadIdx.x; j < d; j += blockDim.x)
        rowv[j] = Elem<T>::to_f(xn[static_cast<size_t>(t) * d + j]);
    __syncthreads();
    const int i = blockIdx.y * blockDim.x + threadIdx.x;
    if (i >= Is) return;
    float g = 0.f, u = 0.f;
    for (int j = 0; j < d; ++j) {
        g = fmaf(Elem<T>::to_f(Gs[static_cast<size_t>(i) * d + j]), rowv[j], g);
        u = fmaf(Elem<T>::to_f(Us[static_cast<size_t>(i) * d + j]), rowv[j], u);
    }
    hs[static_cast<size_t>(t) * Is + i] = Elem<T>::from_f(silu_f(g) * u);
}

// sh[t, o] = Ds[o] . hs[t], plus res[t, o] when res is not null (the dense
// block's residual, added in fp32 before the one rounding).
template <typename T>
__global__ void simt_shared_down_kernel(const T* __restrict__ hs, const T* __restrict__ Ds,
                                        int Is, int d, T* __restrict__ sh,
                                        const T* __restrict__ res = nullptr) {
    extern __shared__ float rowv[];
    const int t = blockIdx.x;
    for (int i = threadIdx.x; i < Is; i += blockDim.x)
        rowv[i] = Elem<T>::to_f(hs[static_cast<size_t>(t) * Is + i]);
    __syncthreads();
    const int o = blockIdx.y * blockDim.x + threadIdx.x;
    if (o >= d) return;
    float acc = 0.f;
    for (int i = 0; i < Is; ++i) acc = fmaf(Elem<T>::to_f(Ds[static_cast<size_t>(o) * Is + i]), rowv[i], acc);
    const size_t at = static_cast<size_t>(t) * d + o;
    if (res != nullptr) acc += Elem<T>::to_f(res[at]);
    sh[at] = Elem<T>::from_f(acc);
}

}  // namespace moe
