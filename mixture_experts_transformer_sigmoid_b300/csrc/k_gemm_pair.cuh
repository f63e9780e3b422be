// Grouped GEMM on CTA pairs (tcgen05.mma.cta_group::2), for batches large
// enough that each expert gets tens to hundreds of tokens.
//
// Same orientation and segments as tc_gemm_kernel (k_gemm_tc.cuh): weight
// features on the MMA's M side, tokens on N.  Two CTAs of a cluster work on
// one 256 x N tile: each holds 128 weight rows (its A half) and N/2 of the
// tile's tokens (its B half); the tensor cores of the pair exchange the B
// halves, and each CTA's tensor memory receives its 128 rows of D over all
// N columns.  Compared with one CTA per 128 x 256 tile, a CTA stages half
// the token bytes per k-block (32 KB stages instead of 48 KB), so the ring
// is 6 deep instead of 4, and each token tile is read from L2 by half as
// many CTAs.
//
// Roles.  Lane 0 of warp 0 of each CTA loads its own A and B halves (one
// TMA copy each per k-block); both CTAs' copies count on the leader's (rank
// 0) `full` barrier, so the leader's MMA warp sees one barrier per stage.
// The leader's warp 1 issues every MMA from one elected lane and commits to
// the `empty` and `tfull` barriers of both CTAs at once (multicast).  Warps
// 2-5 of each CTA drain its own tensor memory; all eight epilogue warps
// arrive on the leader's `tempty` barrier.  Every wait is bounded; a CTA
// that gives up sets the device error flag, and both CTAs still meet at the
// final cluster barrier before tensor memory is freed.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "k_gemm_tc.cuh"
#include "ptx.cuh"

namespace moe {

constexpr int PR_BN = 256;                           // tokens per tile (MMA N, both CTAs)
constexpr int PR_STAGES = 6;
constexpr uint32_t PR_A_BYTES = 2 * TC_BOX_BYTES;    // 128 weight rows x 64 k
constexpr uint32_t PR_B_BYTES = 2 * TC_BOX_BYTES;    // up to 128 token rows x 64 k
constexpr uint32_t PR_STAGE_BYTES = PR_A_BYTES + PR_B_BYTES;

struct PrSmem {
    static constexpr uint32_t RING = PR_STAGES * PR_STAGE_BYTES;
    static constexpr uint32_t BARS = (2 * PR_STAGES + 5) * 8;
    // epilogue staging: SwiGLU gate and up as [32 tokens][65] fp32 each; the
    // weighted epilogue uses 4 warps x [32 tokens][33] fp32
    static constexpr uint32_t XBUF = 2 * 32 * 65 * 4 + 256;
    static constexpr int MAX_E = 1024;
    static constexpr uint32_t PREFIX = (MAX_E + 4) * 4;
    static constexpr uint32_t MISC = 32;
    static constexpr uint32_t TOTAL = 1024 + RING + BARS + MISC + PREFIX + XBUF;
};

// How a CTA's 128 A rows arrive, one k-block at a time (16 KB either way).
enum PairAKind {
    PA_TWO_2D = 0,      // two 64-row boxes of K-major maps: a0 at row f0, a1 at row f0 + a_foff1
    PA_ONE_2D = 1,      // one 128-row box of the K-major map a0 at row f0
    PA_HALVES_4D = 2,   // grouped gate|up: 4-D map {feature, k, half, expert}, both halves at f0
    PA_CHUNKS_4D = 3    // grouped down: 4-D map {feature, k, 64-feature chunk, expert}, chunks f0/64 and f0/64 + 1
};

// Position of a CTA's producer in its sequence of (tile, k-block) loads, with
// the coordinates of the CTA's half of the tile.  Every tile runs over its
// segment's whole K: segments given to this kernel are never split over
// k-ranges (TcSeg::k_split is for the single-CTA kernel).
struct PairCursor {
    int L, kb, nkb;
    int f0;      // first feature of this CTA's A rows
    int r0;      // first token row of this CTA's B half
    int nb;      // B bytes this CTA loads per k-block, in 8 KB units (one 64- or 128-row box)
    bool valid;
    TileInfo ti;

    __device__ void set_tile(const TcParams& p, const int* prefix, uint32_t rank) {
        valid = decode_tile(p, prefix, L, PR_BN, ti);
        if (!valid) return;
        const TcSeg& sg = p.seg[ti.seg];
        const int half = ((ti.rows + 15) & ~15) >> 1;  // MMA N / 2
        nb = half > 64 ? 2 : 1;
        f0 = ti.ftile * sg.a_fstride + static_cast<int>(rank) * sg.a_rank_off;
        r0 = ti.row0 + static_cast<int>(rank) * half;
        nkb = sg.K / TC_BK;
        kb = 0;
    }
    __device__ void start(const TcParams& p, const int* prefix, int first, uint32_t rank) {
        L = first;
        set_tile(p, prefix, rank);
    }
    __device__ void advance(const TcParams& p, const int* prefix, int stride, uint32_t rank) {
        if (++kb < nkb) return;
        L += stride;
        set_tile(p, prefix, rank);
    }
};

// a8 (+)= the eight bf16 values of v, widened to fp32 (set: a8 = v).
__device__ __forceinline__ void add_bf16x8(const uint4 v, float (&a8)[8], bool set) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[j]));
        a8[2 * j] = set ? f.x : a8[2 * j] + f.x;
        a8[2 * j + 1] = set ? f.y : a8[2 * j + 1] + f.y;
    }
}


// Launched with a cluster dimension of 2 (cudaLaunchKernelEx).
template <int EPI>
__global__ void __launch_bounds__(TC_THREADS, 1) tc_gemm_pair_kernel(const __grid_constant__ TcParams p) {
    using S = PrSmem;
    static_assert(S::TOTAL <= 232448, "shared memory");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint8_t* sA = smem;                               // PR_STAGES x 16 KB
    uint8_t* sB = smem + PR_STAGES * PR_A_BYTES;      // PR_STAGES x 16 KB
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::RING);
    uint64_t* empty = full + PR_STAGES;
    uint64_t* tfull = empty + PR_STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + S::RING + S::BARS);
    uint32_t* tmem_holder = misc;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
    volatile int* epi_ok = reinterpret_cast<volatile int*>(misc + 2);
    int* prefix = reinterpret_cast<int*>(smem + S::RING + S::BARS + S::MISC);
    float* xbuf = reinterpret_cast<float*>(smem + S::RING + S::BARS + S::MISC + S::PREFIX);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int pair = static_cast<int>(cluster_id_x());
    const int n_pairs = static_cast<int>(n_clusters_x());

    if (threadIdx.x == 0) {
        for (int s = 0; s < PR_STAGES; ++s) {
            mbar_init(&full[s], 1);    // the leader's expect_tx; bytes of both CTAs
            mbar_init(&empty[s], 1);   // the leader's multicast commit
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 8);  // four epilogue warps in each CTA
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbarrier_init();
        for (int s = 0; s < p.n_segs; ++s) {
            tma_prefetch_desc(&p.a0[s]);
            tma_prefetch_desc(&p.a1[s]);
            tma_prefetch_desc(&p.b[s]);
            tma_prefetch_desc(&p.b128[s]);
        }
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_holder, 2 * PR_BN);
        tmem_relinquish_pair();
    }
    // barriers and tensor memory are set up before the wait for the previous
    // kernel, which writes the offsets and every operand except the weights
    grid_dep_wait();
    if (warp == 2) {
        bool any_grouped = false;
        for (int s = 0; s < p.n_segs; ++s) any_grouped |= (p.seg[s].grouped != 0);
        if (any_grouped) {
            tile_prefix(p.offsets, p.E, PR_BN, prefix, lane);
        }
    }
    tc_fence_before();
    cluster_sync_all();   // barriers of both CTAs initialised, tensor memory allocated
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer (both CTAs)
        // One A load (16 KB) and one B load (8 or 16 KB) per k-block: the TMA
        // unit's cost grows with the number of copies, not only their bytes.
        // A single lane waits and issues: it is usually ahead and really
        // waits, and a whole warp polling the ring's barriers slows the
        // barrier traffic the MMA warp and the copies depend on.
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            PairCursor ld;
            ld.start(p, prefix, pair, rank);
            while (ld.valid) {
                if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, TC_TIMEOUT_NS)) {
                    ok = false;
                    break;
                }
                const uint32_t bar = mapa_shared(smem_u32(&full[stage]), 0);
                if (leader) mbar_arrive_expect_tx(&full[stage], 2u * (PR_A_BYTES + ld.nb * TC_BOX_BYTES));
                uint8_t* a_dst = sA + stage * PR_A_BYTES;
                uint8_t* b_dst = sB + stage * PR_B_BYTES;
                const int sgi = ld.ti.seg;
                const TcSeg& sg = p.seg[sgi];
                const int k0 = ld.kb * TC_BK;
                switch (sg.a_kind) {
                    case PA_TWO_2D:
                        tma_load_2d_pair(a_dst, &p.a0[sgi], bar, k0, ld.f0);
                        tma_load_2d_pair(a_dst + TC_BOX_BYTES, &p.a1[sgi], bar, k0, ld.f0 + sg.a_foff1);
                        break;
                    case PA_ONE_2D:
                        tma_load_2d_pair(a_dst, &p.a0[sgi], bar, k0, ld.f0);
                        break;
                    case PA_HALVES_4D:
                        tma_load_4d_pair(a_dst, &p.a0[sgi], bar, ld.f0, k0, 0, ld.ti.grp);
                        break;
                    default:
                        tma_load_4d_pair(a_dst, &p.a0[sgi], bar, 0, k0, ld.f0 >> 6, ld.ti.grp);
                        break;
                }
                tma_load_2d_pair(b_dst, ld.nb == 2 ? &p.b128[sgi] : &p.b[sgi], bar, k0, ld.r0);
                if (++stage == PR_STAGES) { stage = 0; phase ^= 1u; }
                ld.advance(p, prefix, n_pairs, rank);
            }
            if (!ok) {
                // let copies already issued land before the CTA moves on
                const uint64_t t0 = globaltimer_ns();
                while (globaltimer_ns() - t0 < 2000000ull) {}
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (leader only)
        // The whole warp runs the loop and the barrier waits (warp-uniform
        // control flow and operands); one elected lane issues each MMA and
        // commit.  Issuing from a single diverged lane measured slower.
        if (leader) {
            // Shared-memory descriptors are built once: the start address is the
            // low field (address >> 4, below 2^14 for any shared address), and
            // another ring stage or k-step of 16 is an add on it.
            const uint64_t a_desc_mn = sdesc_sw128(smem_u32(sA), TC_BOX_BYTES, 1024);
            const uint64_t a_desc_k = sdesc_sw128(smem_u32(sA), 16, 1024);
            const uint64_t b_desc0 = sdesc_sw128(smem_u32(sB), 16, 1024);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int L = pair; ok; L += n_pairs) {
                TileInfo ti;
                if (!decode_tile(p, prefix, L, PR_BN, ti)) break;
                const TcSeg& sg = p.seg[ti.seg];
                const int n = (ti.rows + 15) & ~15;
                const int a_mn = sg.grouped;
                const uint32_t idesc = idesc_bf16_f32(2 * TC_BM, n, a_mn, 0);
                // one lane polls a barrier that is not ready; the warp takes its result
                int got = 1;
                if (lane == 0) got = mbar_wait_cluster(&tempty[acc], acc_phase ^ 1u, abort_flag, TC_TIMEOUT_NS);
                ok = __shfl_sync(0xffffffffu, got, 0) != 0;
                if (!ok) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * PR_BN);
                const int nkb = sg.K / TC_BK;
                // MN-major A (grouped weights): 64-feature x 8-k atoms of 1 KB, the two
                // 64-feature boxes 8 KB apart, a k-step of 16 moves two atoms (2 KB).
                // K-major A and B: 8-row x 128-byte atoms, a k-step of 16 moves 32
                // bytes inside the swizzled row.  The peer's halves sit at the same
                // shared-memory offsets.
                const uint64_t a_desc0 = a_mn ? a_desc_mn : a_desc_k;
                const uint64_t a_kstep = a_mn ? (2048 >> 4) : (32 >> 4);
                // Stage operands arrive by TMA and are read by the MMAs, both in the
                // async proxy, ordered by the full barrier: no tcgen05 fence per stage.
                // The try_wait of the next stage starts before this stage's MMAs, so
                // its round trip overlaps their issue.
                uint32_t ready = __all_sync(0xffffffffu, mbar_try_wait(&full[stage], phase)) ? 1u : 0u;
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!ready) {
                        int got = 1;
                        if (lane == 0) got = mbar_wait(&full[stage], phase, abort_flag, TC_TIMEOUT_NS);
                        if (!__shfl_sync(0xffffffffu, got, 0)) {
                            ok = false;
                            break;
                        }
                    }
                    const int next = stage + 1 == PR_STAGES ? 0 : stage + 1;
                    const uint32_t next_phase = stage + 1 == PR_STAGES ? phase ^ 1u : phase;
                    const uint64_t ad = a_desc0 + static_cast<uint64_t>(stage) * (PR_A_BYTES >> 4);
                    const uint64_t bd = b_desc0 + static_cast<uint64_t>(stage) * (PR_B_BYTES >> 4);
                    ready = __all_sync(0xffffffffu,
                                       mma4_pair_commit_trywait_warp(d_tmem, ad, bd, a_kstep, 32 >> 4, idesc,
                                                                     kb > 0 ? 1u : 0u, &empty[stage], 0x3,
                                                                     &full[next], next_phase) != 0u)
                                ? 1u : 0u;
                    stage = next;
                    phase = next_phase;
                }
                if (!ok) break;
                tc_commit_pair_warp(&tfull[acc], 0x3);
                if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
            }
            // wait until every MMA issued by this warp has completed
            tc_commit_pair_warp(drain, 0x1);
            if (lane == 0) mbar_wait(drain, 0, nullptr, ok ? TC_TIMEOUT_NS : TC_DRAIN_NS);
            __syncwarp();
        }
    } else {
        // ------------------------------------------------ epilogue (warps 2-5, both CTAs)
        const int q = warp & 3;
        const int et = threadIdx.x - 64;
        const uint32_t tempty_leader0 = mapa_shared(smem_u32(&tempty[0]), 0);
        const uint32_t tempty_leader1 = mapa_shared(smem_u32(&tempty[1]), 0);
        int acc = 0;
        uint32_t acc_phase = 0;
        int it = 0;
        for (int L = pair;; L += n_pairs, ++it) {
            TileInfo ti;
            if (!decode_tile(p, prefix, L, PR_BN, ti)) break;
            if (et == 0)
                epi_ok[it & 1] = mbar_wait(&tfull[acc], acc_phase, abort_flag, TC_TIMEOUT_NS) ? 1 : 0;
            named_bar_sync(1, 128);
            if (!epi_ok[it & 1]) break;
            tc_fence_after();
            const TcSeg& sg = p.seg[ti.seg];
            const int fbase = ti.ftile * sg.a_fstride + static_cast<int>(rank) * sg.a_rank_off;
            const uint32_t t_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                    static_cast<uint32_t>(acc * PR_BN);
            for (int c0 = 0; c0 < ti.rows; c0 += 32) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(t_base + c0, v);
                tmem_ld_wait();
                const int cmax = min(32, ti.rows - c0);
                __nv_bfloat16* out = static_cast<__nv_bfloat16*>(sg.out);
                if constexpr (EPI == EPI_SWIGLU) {
                    // lanes 0-63 of tensor memory hold gate, 64-127 up, for the same 64
                    // features: stage both as [token][feature], then each warp takes 8
                    // tokens and writes 8 features of one token per 16-byte store
                    float* gs = xbuf;
                    float* us = xbuf + 32 * 65;
                    float* dst = q < 2 ? gs : us;
                    const int f = (q & 1) * 32 + lane;
#pragma unroll
                    for (int c = 0; c < 32; ++c) dst[c * 65 + f] = __uint_as_float(v[c]);
                    named_bar_sync(2, 128);
                    const int t = (warp - 2) * 8 + (lane >> 2);   // token of this lane (bank = t + 8 * sub)
#pragma unroll
                    for (int pass = 0; pass < 2; ++pass) {
                        const int sub = pass * 4 + (lane & 3);     // 8-feature chunk of the 64
                        const int col = fbase + sub * 8;
                        if (t < cmax && col < sg.F) {
                            uint32_t pk[4];
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const float g0 = gs[t * 65 + sub * 8 + 2 * j], g1 = gs[t * 65 + sub * 8 + 2 * j + 1];
                                const float u0 = us[t * 65 + sub * 8 + 2 * j], u1 = us[t * 65 + sub * 8 + 2 * j + 1];
                                const float h0 = g0 / (1.0f + __expf(-g0)) * u0;
                                const float h1 = g1 / (1.0f + __expf(-g1)) * u1;
                                const __nv_bfloat162 hb = __floats2bfloat162_rn(h0, h1);
                                pk[j] = *reinterpret_cast<const uint32_t*>(&hb);
                            }
                            *reinterpret_cast<uint4*>(out + static_cast<size_t>(ti.row0 + c0 + t) * sg.ld_out + col) =
                                make_uint4(pk[0], pk[1], pk[2], pk[3]);
                        }
                    }
                    named_bar_sync(2, 128);
                } else {
                    // stage this warp's 32 features x 32 tokens, then write 8 features of
                    // one token per 16-byte store (two for fp32 output): scaled by that
                    // token's routing weight (EPI_WEIGHTED) or added to 8 residual values
                    // read with one 16-byte load (EPI_RESIDUAL)
                    static_assert(EPI == EPI_WEIGHTED || EPI == EPI_RESIDUAL, "epilogue");
                    float* stg = xbuf + q * (32 * 33);
#pragma unroll
                    for (int c = 0; c < 32; ++c) stg[c * 33 + lane] = __uint_as_float(v[c]);
                    __syncwarp();
                    const int sub = lane & 3;
                    const int col = fbase + q * 32 + sub * 8;
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const int t = r * 8 + (lane >> 2);       // bank = t + 8 * sub: conflict-free
                        if (t < cmax && col < sg.F) {
                            const int row = ti.row0 + c0 + t;
                            uint32_t pk[4];
                            if constexpr (EPI == EPI_WEIGHTED) {
                                const float wv = sg.row_w ? sg.row_w[row] : 1.0f;
                                if (sg.out_kind == OUT_F32) {
                                    float* o32 = static_cast<float*>(sg.out) + static_cast<size_t>(row) * sg.ld_out + col;
                                    const float* sp = stg + t * 33 + sub * 8;
                                    *reinterpret_cast<float4*>(o32) = make_float4(sp[0] * wv, sp[1] * wv, sp[2] * wv, sp[3] * wv);
                                    *reinterpret_cast<float4*>(o32 + 4) = make_float4(sp[4] * wv, sp[5] * wv, sp[6] * wv, sp[7] * wv);
                                    continue;
                                }
                                if (sg.out_kind == OUT_F16) {
                                    float amax = 0.f;
#pragma unroll
                                    for (int j = 0; j < 4; ++j) {
                                        const float y0 = stg[t * 33 + sub * 8 + 2 * j] * wv;
                                        const float y1 = stg[t * 33 + sub * 8 + 2 * j + 1] * wv;
                                        amax = fmaxf(amax, fmaxf(fabsf(y0), fabsf(y1)));
                                        const __half2 hh = __floats2half2_rn(y0, y1);
                                        pk[j] = *reinterpret_cast<const uint32_t*>(&hh);
                                    }
                                    if (!(amax <= 65504.0f)) atomicOr(p.err, DEVERR_RANGE);
                                } else {
#pragma unroll
                                    for (int j = 0; j < 4; ++j) {
                                        const __nv_bfloat162 hb = __floats2bfloat162_rn(
                                            stg[t * 33 + sub * 8 + 2 * j] * wv, stg[t * 33 + sub * 8 + 2 * j + 1] * wv);
                                        pk[j] = *reinterpret_cast<const uint32_t*>(&hb);
                                    }
                                }
                            } else {
                                const uint4 r4 = *reinterpret_cast<const uint4*>(
                                    static_cast<const __nv_bfloat16*>(sg.res) + static_cast<size_t>(row) * sg.ld_out + col);
                                float a8[8];
                                add_bf16x8(r4, a8, true);
#pragma unroll
                                for (int j = 0; j < 8; ++j) a8[j] += stg[t * 33 + sub * 8 + j];
#pragma unroll
                                for (int j = 0; j < 4; ++j) {
                                    const __nv_bfloat162 hb = __floats2bfloat162_rn(a8[2 * j], a8[2 * j + 1]);
                                    pk[j] = *reinterpret_cast<const uint32_t*>(&hb);
                                }
                            }
                            *reinterpret_cast<uint4*>(out + static_cast<size_t>(row) * sg.ld_out + col) =
                                make_uint4(pk[0], pk[1], pk[2], pk[3]);
                        }
                    }
                    __syncwarp();
                }
            }
            tc_fence_before();
            if (lane == 0) mbar_arrive_cluster(acc == 0 ? tempty_leader0 : tempty_leader1);
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        }
    }

    tc_fence_before();
    cluster_sync_all();   // no CTA frees tensor memory or exits while its peer may still signal it
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem_base, 2 * PR_BN);
    if (threadIdx.x == 0 && *abort_flag) atomicOr(p.err, DEVERR_TIMEOUT);
}

}  // namespace moe
