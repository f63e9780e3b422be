// Router logits l[t, e] = xn[t] . router_w[e] on the tcgen05 tensor cores,
// with an accumulation exact enough for the top-k decision.
//
// A tensor-core accumulation chained over the whole hidden size (hundreds of
// MMAs into one fp32 accumulator) carries a rounding error that grows with
// the chain and can exceed the top-k margins the routing must resolve
// (biased-score gaps down to 1e-5).  So every RT_CHAIN k-blocks of 64 (16
// MMAs) start a fresh accumulator in tensor memory, and the epilogue warps
// add the chain results into a compensated (hi, lo) fp32 pair with an
// error-free two-sum.  The bf16 x bf16 products themselves are exact; the
// rounding error of a chain grows with its length (about 1e-6 for 4 MMAs,
// 1e-4 for 384), so short chains keep the logits within a few 1e-6.
//
// Tile: 128 experts (M, router_w rows, K-major) x BN tokens (N, xn rows,
// K-major), BN = 64 for decode-sized batches and 128 above.  An MMA of N = 128
// costs the tensor core about as long as one of N = 64 (its fixed cost per
// instruction dominates below N of about 138), so the wider tile does twice
// the work per MMA, and a GLM-5 prefill batch (8192 tokens, 256 experts) is
// one wave of 128 tiles; batches of at most 64 tokens keep the narrower tile
// (its epilogue has half the columns to read).  Split-K: a tile may cover only
// a range of k-blocks (small T fills the GPU that way); each range writes its
// own (hi, lo) partials and router_reduce_kernel adds the ranges in a fixed
// order.
//
// Warps: 0 TMA producer, 1 TMEM allocation + MMA issue, then BN / 8 epilogue
// warps (BN / 32 per TMEM lane quarter, each taking 32 token columns, in loads
// of 8 columns: at 576 threads a thread has at most 96 registers, and its 32
// (hi, lo) sums must stay in them).
#pragma once
#include <cuda.h>
#include <cstdint>

#include "numeric.cuh"
#include "ptx.cuh"

namespace moe {

constexpr int RT_BN_MAX = 128;      // tokens per tile, the wider of the two tiles
constexpr int RT_CHAIN = 4;         // k-blocks accumulated in tensor memory per epilogue read
constexpr int RT_STAGES = 6;
constexpr int RT_NACC = 4;          // BN-column accumulators between MMA and epilogue
constexpr uint32_t RT_BOX = 64 * 64 * 2;

template <int BN>
struct RtCfg {
    static_assert(BN == 64 || BN == 128, "BN");
    static constexpr int EPI_WARPS = BN / 8;
    static constexpr int THREADS = 64 + 32 * EPI_WARPS;
    // A: 2 boxes (128 experts), B: one box of BN rows (BN tokens)
    static constexpr uint32_t STAGE_BYTES = 2 * RT_BOX + BN * 128;
    static constexpr uint32_t SMEM = 1024 + RT_STAGES * STAGE_BYTES + (2 * RT_STAGES + 2 * RT_NACC + 1) * 8 + 32;
};
constexpr uint64_t RT_TIMEOUT_NS = 2000000000ull;
constexpr uint64_t RT_DRAIN_NS = 100000000ull;

struct RouterParams {
    CUtensorMap a;       // router_w [E, d]
    CUtensorMap b;       // xn [T, d]
    int T, E, d;
    int ksplit;          // k-block ranges per tile
    int kb_per_split;    // k-blocks per range (the last range may have fewer)
    float2* part;        // [ksplit][T][E] (hi, lo) partial sums
    int* err;
};

struct RouterTile {
    int t0, e0, s, kb0, nkb;
};

template <int BN>
__device__ __forceinline__ bool router_tile(const RouterParams& p, int L, RouterTile& rt) {
    const int n_tt = (p.T + BN - 1) / BN;
    const int n_et = (p.E + 127) / 128;
    if (L >= n_tt * n_et * p.ksplit) return false;
    rt.s = L % p.ksplit;
    const int r = L / p.ksplit;
    rt.e0 = (r % n_et) * 128;
    rt.t0 = (r / n_et) * BN;
    const int nkb_total = p.d / 64;
    rt.kb0 = rt.s * p.kb_per_split;
    rt.nkb = min(p.kb_per_split, nkb_total - rt.kb0);
    return true;
}

template <int BN>
__global__ void __launch_bounds__(RtCfg<BN>::THREADS, 1) router_tc_kernel(const __grid_constant__ RouterParams p) {
    using C = RtCfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + RT_STAGES * C::STAGE_BYTES);
    uint64_t* empty = full + RT_STAGES;
    uint64_t* tfull = empty + RT_STAGES;
    uint64_t* tempty = tfull + RT_NACC;
    uint64_t* drain = tempty + RT_NACC;
    uint32_t* misc = reinterpret_cast<uint32_t*>(drain + 1);
    uint32_t* tmem_holder = misc;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < RT_STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < RT_NACC; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], C::EPI_WARPS);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbarrier_init();
        tma_prefetch_desc(&p.a);
        tma_prefetch_desc(&p.b);
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, RT_NACC * BN);
        tmem_relinquish();
    }
    grid_dep_wait();   // xn comes from the previous kernel
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0, issued = 0;
            uint32_t phase = 0;
            bool ok = true;
            RouterTile rt;
            for (int L = blockIdx.x; ok && router_tile<BN>(p, L, rt); L += gridDim.x) {
                for (int kb = rt.kb0; kb < rt.kb0 + rt.nkb; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, RT_TIMEOUT_NS)) {
                        ok = false;
                        break;
                    }
                    uint8_t* dst = smem + stage * C::STAGE_BYTES;
                    mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
                    tma_load_2d_nohint(dst, &p.a, &full[stage], kb * 64, rt.e0);
                    tma_load_2d_nohint(dst + RT_BOX, &p.a, &full[stage], kb * 64, rt.e0 + 64);
                    tma_load_2d_nohint(dst + 2 * RT_BOX, &p.b, &full[stage], kb * 64, rt.t0);
                    ++issued;
                    if (++stage == RT_STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok) {
                const int n = issued < RT_STAGES ? issued : RT_STAGES;
                int s = stage;
                uint32_t ph = phase;
                for (int i = 0; i < n; ++i) {
                    if (--s < 0) { s = RT_STAGES - 1; ph ^= 1u; }
                    mbar_wait(&full[s], ph, nullptr, RT_DRAIN_NS);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(128, BN, 0, 0);
            int stage = 0;
            uint32_t phase = 0;
            uint32_t g = 0;  // k-blocks issued by this CTA (selects the accumulator)
            bool ok = true;
            RouterTile rt;
            for (int L = blockIdx.x; ok && router_tile<BN>(p, L, rt); L += gridDim.x) {
                for (int kb = 0; kb < rt.nkb; ++kb) {
                    const uint32_t slot = g % RT_NACC;
                    const bool first = kb % RT_CHAIN == 0;
                    const bool last = kb % RT_CHAIN == RT_CHAIN - 1 || kb == rt.nkb - 1;
                    if ((first && !mbar_wait(&tempty[slot], ((g / RT_NACC) & 1u) ^ 1u, abort_flag,
                                             RT_TIMEOUT_NS)) ||
                        !mbar_wait(&full[stage], phase, abort_flag, RT_TIMEOUT_NS)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(smem + stage * C::STAGE_BYTES);
                    const uint32_t b_addr = a_addr + 2 * RT_BOX;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc_mma_bf16(tmem_base + slot * BN, sdesc_sw128(a_addr + kk * 32, 16, 1024),
                                    sdesc_sw128(b_addr + kk * 32, 16, 1024), idesc,
                                    (first && kk == 0) ? 0u : 1u);
                    tc_commit(&empty[stage]);
                    if (last) {
                        tc_commit(&tfull[slot]);
                        ++g;
                    }
                    if (++stage == RT_STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            tc_commit(drain);
            mbar_wait(drain, 0, nullptr, ok ? RT_TIMEOUT_NS : RT_DRAIN_NS);
        }
    } else {
        const int q = warp & 3;              // TMEM lane quarter
        const int half = (warp - 2) >> 2;    // token columns [32 half, 32 half + 32), half = 0..3
        uint32_t g = 0;
        bool ok = true;
        RouterTile rt;
        for (int L = blockIdx.x; ok && router_tile<BN>(p, L, rt); L += gridDim.x) {
            float hi[32], lo[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) { hi[c] = 0.f; lo[c] = 0.f; }
            for (int kb = 0; kb < rt.nkb; kb += RT_CHAIN, ++g) {
                const uint32_t slot = g % RT_NACC;
                int good = 1;
                if (lane == 0) good = mbar_wait(&tfull[slot], (g / RT_NACC) & 1u, abort_flag, RT_TIMEOUT_NS) ? 1 : 0;
                good = __shfl_sync(0xffffffffu, good, 0);
                if (!good) { ok = false; break; }
                tc_fence_after();
                const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + slot * BN + half * 32;
#pragma unroll
                for (int h2 = 0; h2 < 4; ++h2) {
                    uint32_t v[8];
                    tmem_ld_32x32b_x8(taddr + h2 * 8, v);
                    tmem_ld_wait();
                    if (h2 == 3) {
                        tc_fence_before();
                        if (lane == 0) mbar_arrive(&tempty[slot]);
                    }
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        float s, e;
                        two_sum_f(hi[h2 * 8 + c], __uint_as_float(v[c]), s, e);
                        hi[h2 * 8 + c] = s;
                        lo[h2 * 8 + c] = __fadd_rn(lo[h2 * 8 + c], e);
                    }
                }
            }
            if (!ok) break;
            const int e = rt.e0 + q * 32 + lane;
            if (e < p.E) {
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const int t = rt.t0 + half * 32 + c;
                    if (t < p.T)
                        p.part[(static_cast<size_t>(rt.s) * p.T + t) * p.E + e] = make_float2(hi[c], lo[c]);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, RT_NACC * BN);
    if (threadIdx.x == 0 && *abort_flag) atomicOr(p.err, 1);
}

// The compensated sum of logit i's ksplit (hi, lo) pairs, in range order,
// as the single pair (l, 0); eight ranges' loads are in flight at a time.
__device__ __forceinline__ float2 reduce_logit_pair(const float2* __restrict__ part, int ksplit, size_t n,
                                                    size_t i) {
    float hi = 0.f, lo = 0.f;
    for (int s0 = 0; s0 < ksplit; s0 += 8) {
        float2 pv[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (s0 + j < ksplit) pv[j] = part[static_cast<size_t>(s0 + j) * n + i];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (s0 + j >= ksplit) break;
            float s2, e2;
            two_sum_f(hi, pv[j].x, s2, e2);
            hi = s2;
            lo = __fadd_rn(lo, __fadd_rn(e2, pv[j].y));
        }
    }
    return make_float2(__fadd_rn(hi, lo), 0.f);
}

// Adds the ksplit (hi, lo) partial pairs of each logit in range order with a
// compensated fp32 sum and stores the result as the single pair (l, 0) of
// range 0.  Each thread owns one (t, e) across all ranges, so it may
// overwrite range 0 in place.
__global__ void router_reduce_kernel(float2* __restrict__ part, int ksplit, size_t n) {
    grid_dep_wait();
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<size_t>(gridDim.x) * blockDim.x)
        part[i] = reduce_logit_pair(part, ksplit, n, i);
}

}  // namespace moe
