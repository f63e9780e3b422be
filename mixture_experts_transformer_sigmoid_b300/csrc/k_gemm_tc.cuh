// Grouped GEMM on the 5th-generation tensor cores (tcgen05, TMEM, TMA).
//
// Orientation ("swap-AB"): the MMA's M side (128 rows) holds 128 features
// of a weight matrix and its N side holds up to BN tokens, so D = W^T X^T
// lands in tensor memory as [feature lane, token column].  Tokens are the
// ragged dimension of an MoE (each expert gets a different count), and N can
// be any multiple of 16 up to 256, so an expert's tail tile wastes at most 15
// columns instead of up to 127 rows.
//
// One launch runs up to two "segments" of tiles:
//   grouped segment: the routed experts; expert e owns permuted rows
//     [offsets[e], offsets[e+1]) of the B matrix; its weights are read
//     MN-major from the grouped layout ([E, K, F] with F contiguous) through
//     a 3-D tensor map with the expert index as the outer coordinate.
//   dense segment: one group of n_rows rows (the shared expert); its
//     weights are nn.Linear [F, K] rows, read K-major.
// The A tile is two 64-row TMA boxes (rows 0-63 and 64-127 of the MMA's M);
// for the gate|up launch they are the gate and the up rows of the same 64
// features, so the SwiGLU can be applied in the epilogue.
//
// Warp roles (192 threads, one CTA per SM, persistent over a static tile
// order): warp 0 issues TMA loads into a STAGES-deep shared-memory ring,
// warp 1 allocates tensor memory and issues the MMAs (one thread), warps 2-5
// read the fp32 accumulators back from tensor memory (each warp may only
// touch the 32 TMEM lanes of its quarter, warp % 4) and run the epilogue.
// Two accumulators in tensor memory let the epilogue of one tile overlap the
// MMAs of the next.  Every wait is bounded: on a timeout the kernel sets a
// device error flag, drains its in-flight copies and MMAs, frees tensor
// memory and returns.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "ptx.cuh"

namespace moe {

constexpr int TC_BM = 128;                     // MMA M
constexpr int TC_BK = 64;                      // k per stage: one 128-byte swizzle row of bf16
constexpr int TC_UMMA_K = 16;                  // k per tcgen05.mma (kind::f16)
constexpr uint32_t TC_BOX_BYTES = 64 * 64 * 2;  // one 64 x 64 bf16 TMA box
constexpr uint32_t TC_A_BYTES = 2 * TC_BOX_BYTES;
constexpr int TC_THREADS = 192;
constexpr uint64_t TC_TIMEOUT_NS = 2000000000ull;   // 2 s
constexpr uint64_t TC_DRAIN_NS = 100000000ull;      // 100 ms
constexpr int DEVERR_TIMEOUT = 1;
constexpr int DEVERR_RANGE = 2;     // an fp16 output overflowed (|v| > 65504)

// SWIGLU: out = silu(gate) * up, from the gate and up halves of the A rows.
// WEIGHTED: out = row_w[row] * acc (row_w null: acc), stored as the
//   segment's out_kind says: bf16, fp16 (an overflow sets DEVERR_RANGE) or fp32.
// RESIDUAL: out = res[row, col] + acc, added in fp32 and rounded once.
// PARTIAL: fp32 acc of one k-range of a split dense segment, to
//   out[k-range][row][col] (single-CTA kernel; the ranges are added later).
//   With partial_halves set (a gate|up segment: A rows 64-127 are the up rows
//   of the same features as rows 0-63), the second half goes to columns
//   F + col, so a row of the partials holds all gates, then all ups.
enum EpiKind { EPI_SWIGLU = 1, EPI_WEIGHTED = 2, EPI_RESIDUAL = 3, EPI_PARTIAL = 4 };
enum OutKind { OUT_BF16 = 0, OUT_F16 = 1, OUT_F32 = 2 };

struct TcSeg {
    int grouped;          // 1: expert groups from offsets[]; 0: one group of n_rows rows
    int n_rows;           // dense segment: rows of B
    int K;                // reduction length, multiple of 64
    int a_fstride;        // first feature of feature tile f: f * a_fstride
    int a_foff1;          // feature offset of the second A box (rows 64..127)
    int n_ftiles;         // feature tiles per group
    int F;                // features that exist (stores are guarded by it)
    int ld_out;           // output row stride in elements
    void* out;            // bf16 output [rows, ld_out]
    const float* row_w;   // weighted epilogue: per-row factor; null means 1
    int a_rank_off;       // CTA-pair kernel: feature offset of the second CTA's rows
    int a_kind;           // CTA-pair kernel: how a0 delivers the 128 A rows (PairAKind)
    const void* res;      // residual epilogue: bf16 [rows, ld_out], indexed like out
    int f_group;          // dense segment: feature tiles per tile group (0: all of them)
    int k_split;          // dense segment, single-CTA kernel: k-ranges per tile (0 or 1: none)
    int out_kind;         // weighted epilogue: OutKind of `out`
    int partial_halves;   // partial epilogue: rows 64-127 of A are a second half (see EPI_PARTIAL)
};

struct TcParams {
    CUtensorMap a0[2];    // per segment: map of the first A box
    CUtensorMap a1[2];    // per segment: map of the second A box
    CUtensorMap b[2];     // per segment: map of B ([rows, K], K contiguous)
    CUtensorMap b128[2];  // CTA-pair kernel: the same B with 128-row boxes
    TcSeg seg[2];
    int n_segs;
    int E;                // groups of the grouped segment
    const int* offsets;   // [E + 1] first row of each group
    int* err;             // device error flag
};

struct TileInfo {
    int seg, grp, row0, rows, ftile;
    int ks, kb0, nkb;     // k-range of the tile: its index and k-blocks [kb0, kb0 + nkb)
};

// prefix[e] = token tiles (of BN rows) of the groups before e, for e = 0..E,
// computed by one warp.  Each lane loads its groups' offsets for eight
// 32-group blocks at once, so a launch pays about one round trip to memory
// for E <= 256 instead of one per block.
__device__ __forceinline__ void tile_prefix(const int* offsets, int E, int BN, int* prefix, int lane) {
    constexpr int U = 8;
    int run = 0;
    for (int base = 0; base < E; base += 32 * U) {
        int lo[U], hi[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int e = base + 32 * u + lane;
            lo[u] = e < E ? offsets[e] : 0;
            hi[u] = e < E ? offsets[e + 1] : 0;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int e = base + 32 * u + lane;
            int v = (hi[u] - lo[u] + BN - 1) / BN;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int w = __shfl_up_sync(0xffffffffu, v, off);
                if (lane >= off) v += w;
            }
            if (e < E) prefix[e + 1] = run + v;
            run += __shfl_sync(0xffffffffu, v, 31);
        }
    }
    if (lane == 0) prefix[0] = 0;
}

// Linear tile id -> (segment, group, first row, rows, feature tile).  Tiles
// are ordered segment-major, then token tile, then feature tile, so CTAs that
// run at the same time share the B tile and the L2 lines of the same expert.
// A group of m rows is split evenly into ceil(m / BN) token tiles (e.g. 300
// rows as 150 + 150, not 256 + 44): the same weight traffic, but no MMA with
// a small N, whose fixed cost per instruction would dominate.
// A dense segment whose weights do not fit in L2 orders its tiles in groups
// of f_group feature tiles, token tile-major inside a group: the CTAs that
// run together then share a few weight tiles and a few token tiles, and each
// group's weights are read from DRAM once (token tile-major over all feature
// tiles would stream every weight once per token tile).
// A split dense segment (k_split > 1) repeats its tiles once per k-range,
// k-range-major; the ranges split the k-blocks evenly.
__device__ __forceinline__ bool decode_tile(const TcParams& p, const int* prefix, int L, int BN,
                                            TileInfo& ti) {
    for (int s = 0; s < p.n_segs; ++s) {
        const TcSeg& sg = p.seg[s];
        const int ntok = sg.grouped ? prefix[p.E] : (sg.n_rows + BN - 1) / BN;
        const int nsplit = (!sg.grouped && sg.k_split > 1) ? sg.k_split : 1;
        const int per_split = ntok * sg.n_ftiles;
        const int cnt = per_split * nsplit;
        if (L < cnt) {
            const int ks = L / per_split;
            L -= ks * per_split;
            const int nkb_all = sg.K / TC_BK;
            ti.ks = ks;
            ti.kb0 = static_cast<int>(static_cast<int64_t>(ks) * nkb_all / nsplit);
            ti.nkb = static_cast<int>(static_cast<int64_t>(ks + 1) * nkb_all / nsplit) - ti.kb0;
            int tt = L / sg.n_ftiles;
            ti.ftile = L - tt * sg.n_ftiles;
            ti.seg = s;
            if (!sg.grouped && sg.f_group > 0 && sg.f_group < sg.n_ftiles) {
                const int per_group = sg.f_group * ntok;
                const int g = L / per_group;
                const int f_first = g * sg.f_group;
                const int gf = min(sg.f_group, sg.n_ftiles - f_first);
                const int within = L - g * per_group;
                tt = within / gf;
                ti.ftile = f_first + (within - tt * gf);
            }
            if (sg.grouped) {
                int lo = 0, hi = p.E;  // prefix[lo] <= tt < prefix[hi]
                while (hi - lo > 1) {
                    const int mid = (lo + hi) >> 1;
                    if (prefix[mid] <= tt) lo = mid; else hi = mid;
                }
                ti.grp = lo;
                const int m = p.offsets[lo + 1] - p.offsets[lo];
                const int ntt = prefix[lo + 1] - prefix[lo];
                const int j = tt - prefix[lo];
                ti.row0 = p.offsets[lo] + static_cast<int>(static_cast<int64_t>(j) * m / ntt);
                ti.rows = p.offsets[lo] + static_cast<int>(static_cast<int64_t>(j + 1) * m / ntt) - ti.row0;
            } else {
                const int m = sg.n_rows;
                ti.grp = 0;
                ti.row0 = static_cast<int>(static_cast<int64_t>(tt) * m / ntok);
                ti.rows = static_cast<int>(static_cast<int64_t>(tt + 1) * m / ntok) - ti.row0;
            }
            return true;
        }
        L -= cnt;
    }
    return false;
}

template <int BN, int STAGES>
struct TcSmem {
    static constexpr uint32_t B_BYTES = BN * TC_BK * 2;
    static constexpr uint32_t STAGE_BYTES = TC_A_BYTES + B_BYTES;
    static constexpr uint32_t RING = STAGES * STAGE_BYTES;
    static constexpr uint32_t BARS = (2 * STAGES + 5) * 8;
    static constexpr uint32_t XBUF = 64 * 33 * 4;  // SwiGLU exchange of up values
    static constexpr int MAX_E = 1024;
    static constexpr uint32_t PREFIX = (MAX_E + 4) * 4;
    static constexpr uint32_t MISC = 32;
    static constexpr uint32_t TOTAL = 1024 + RING + BARS + MISC + PREFIX + XBUF;
};

template <int BN, int STAGES, int EPI>
__global__ void __launch_bounds__(TC_THREADS, 1) tc_gemm_kernel(const __grid_constant__ TcParams p) {
    using S = TcSmem<BN, STAGES>;
    static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "BN");
    static_assert(S::TOTAL <= 232448, "shared memory");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint8_t* sA = smem;                              // STAGES x 16 KB
    uint8_t* sB = smem + STAGES * TC_A_BYTES;        // STAGES x B_BYTES
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::RING);
    uint64_t* empty = full + STAGES;
    uint64_t* tfull = empty + STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + S::RING + S::BARS);
    uint32_t* tmem_holder = misc;                    // misc[0]
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
    volatile int* epi_ok = reinterpret_cast<volatile int*>(misc + 2);  // misc[2..3]
    int* prefix = reinterpret_cast<int*>(smem + S::RING + S::BARS + S::MISC);
    float* xbuf = reinterpret_cast<float*>(smem + S::RING + S::BARS + S::MISC + S::PREFIX);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 4);  // one arrival per epilogue warp
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbarrier_init();
        for (int s = 0; s < p.n_segs; ++s) {
            tma_prefetch_desc(&p.a0[s]);
            tma_prefetch_desc(&p.a1[s]);
            tma_prefetch_desc(&p.b[s]);
        }
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, 2 * BN);
        tmem_relinquish();
    }
    // barriers and tensor memory are set up before the wait for the previous
    // kernel, which writes the offsets and every operand except the weights
    grid_dep_wait();
    if (warp == 2) {
        // prefix[e] = token tiles of groups < e (grouped segment)
        bool any_grouped = false;
        for (int s = 0; s < p.n_segs; ++s) any_grouped |= (p.seg[s].grouped != 0);
        if (any_grouped) {
            tile_prefix(p.offsets, p.E, BN, prefix, lane);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int issued = 0;
            bool ok = true;
            for (int L = blockIdx.x; ok; L += gridDim.x) {
                TileInfo ti;
                if (!decode_tile(p, prefix, L, BN, ti)) break;
                const TcSeg& sg = p.seg[ti.seg];
                const CUtensorMap* ma0 = &p.a0[ti.seg];
                const CUtensorMap* ma1 = &p.a1[ti.seg];
                const CUtensorMap* mb = &p.b[ti.seg];
                const int nb = (ti.rows + 63) >> 6;
                const int f0 = ti.ftile * sg.a_fstride;
                for (int kb = ti.kb0; kb < ti.kb0 + ti.nkb; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, TC_TIMEOUT_NS)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[stage], TC_A_BYTES + nb * TC_BOX_BYTES);
                    uint8_t* a_dst = sA + stage * TC_A_BYTES;
                    uint8_t* b_dst = sB + stage * S::B_BYTES;
                    const int k0 = kb * TC_BK;
                    if (sg.grouped) {
                        tma_load_3d_nohint(a_dst, ma0, &full[stage], f0, k0, ti.grp);
                        tma_load_3d_nohint(a_dst + TC_BOX_BYTES, ma1, &full[stage], f0 + sg.a_foff1,
                                           k0, ti.grp);
                    } else {
                        tma_load_2d_nohint(a_dst, ma0, &full[stage], k0, f0);
                        tma_load_2d_nohint(a_dst + TC_BOX_BYTES, ma1, &full[stage], k0,
                                           f0 + sg.a_foff1);
                    }
                    for (int j = 0; j < nb; ++j)
                        tma_load_2d_nohint(b_dst + j * TC_BOX_BYTES, mb, &full[stage], k0,
                                           ti.row0 + j * 64);
                    ++issued;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok) {
                // drain: wait for the copies still in flight before the CTA exits
                const int n = issued < STAGES ? issued : STAGES;
                int s = stage;
                uint32_t ph = phase;
                for (int i = 0; i < n; ++i) {
                    if (--s < 0) { s = STAGES - 1; ph ^= 1u; }
                    mbar_wait(&full[s], ph, nullptr, TC_DRAIN_NS);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int L = blockIdx.x; ok; L += gridDim.x) {
                TileInfo ti;
                if (!decode_tile(p, prefix, L, BN, ti)) break;
                const TcSeg& sg = p.seg[ti.seg];
                const int n = (ti.rows + 15) & ~15;
                const int a_mn = sg.grouped;  // grouped weights are MN-major, dense ones K-major
                const uint32_t idesc = idesc_bf16_f32(TC_BM, n, a_mn, 0);
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, TC_TIMEOUT_NS)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int kb = 0; kb < ti.nkb; ++kb) {
                    if (!mbar_wait(&full[stage], phase, abort_flag, TC_TIMEOUT_NS)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(sA + stage * TC_A_BYTES);
                    const uint32_t b_addr = smem_u32(sB + stage * S::B_BYTES);
#pragma unroll
                    for (int kk = 0; kk < TC_BK / TC_UMMA_K; ++kk) {
                        // MN-major A: 64-feature x 8-k swizzle atoms of 1 KB; the two
                        // 64-feature boxes are 8 KB apart (leading byte offset), 8-k
                        // groups 1 KB apart (stride byte offset); a k-step of 16 moves
                        // two atoms.  K-major: 8-row x 128-byte atoms, 1 KB apart; a
                        // k-step of 16 moves 32 bytes inside the swizzled row.
                        const uint64_t ad = a_mn ? sdesc_sw128(a_addr + kk * 2048, TC_BOX_BYTES, 1024)
                                                 : sdesc_sw128(a_addr + kk * 32, 16, 1024);
                        const uint64_t bd = sdesc_sw128(b_addr + kk * 32, 16, 1024);
                        tc_mma_bf16(d_tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
                    }
                    tc_commit(&empty[stage]);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                tc_commit(&tfull[acc]);
                if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
            }
            // wait until every MMA issued by this thread has completed
            tc_commit(drain);
            mbar_wait(drain, 0, nullptr, ok ? TC_TIMEOUT_NS : TC_DRAIN_NS);
        }
    } else {
        // ------------------------------------------------ epilogue (warps 2-5)
        const int q = warp & 3;  // TMEM lane quarter
        const int et = threadIdx.x - 64;
        int acc = 0;
        uint32_t acc_phase = 0;
        int it = 0;
        for (int L = blockIdx.x;; L += gridDim.x, ++it) {
            TileInfo ti;
            if (!decode_tile(p, prefix, L, BN, ti)) break;
            if (et == 0) epi_ok[it & 1] = mbar_wait(&tfull[acc], acc_phase, abort_flag, TC_TIMEOUT_NS) ? 1 : 0;
            named_bar_sync(1, 128);
            if (!epi_ok[it & 1]) break;
            tc_fence_after();
            const TcSeg& sg = p.seg[ti.seg];
            const uint32_t t_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                    static_cast<uint32_t>(acc * BN);
            for (int c0 = 0; c0 < ti.rows; c0 += 32) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(t_base + c0, v);
                tmem_ld_wait();
                if constexpr (EPI == EPI_SWIGLU) {
                    // lanes 0-63 hold gate, 64-127 up, for the same 64 features
                    if (q >= 2) {
#pragma unroll
                        for (int c = 0; c < 32; ++c) xbuf[((q - 2) * 32 + lane) * 33 + c] = __uint_as_float(v[c]);
                    }
                    named_bar_sync(2, 128);
                    if (q < 2) {
                        const int col = ti.ftile * sg.a_fstride + q * 32 + lane;
                        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(sg.out);
                        if (col < sg.F) {
                            const int cmax = min(32, ti.rows - c0);
#pragma unroll
                            for (int c = 0; c < 32; ++c) {
                                if (c >= cmax) break;
                                const float g = __uint_as_float(v[c]);
                                const float u = xbuf[(q * 32 + lane) * 33 + c];
                                const float hv = g / (1.0f + __expf(-g)) * u;
                                out[static_cast<size_t>(ti.row0 + c0 + c) * sg.ld_out + col] =
                                    __float2bfloat16_rn(hv);
                            }
                        }
                    }
                    named_bar_sync(2, 128);
                } else if constexpr (EPI == EPI_WEIGHTED) {
                    const int col = ti.ftile * sg.a_fstride + q * 32 + lane;
                    if (col < sg.F) {
                        const int cmax = min(32, ti.rows - c0);
                        float amax = 0.f;
#pragma unroll
                        for (int c = 0; c < 32; ++c) {
                            if (c >= cmax) break;
                            const int row = ti.row0 + c0 + c;
                            const float wv = sg.row_w ? sg.row_w[row] : 1.0f;
                            const float y = __uint_as_float(v[c]) * wv;
                            const size_t at = static_cast<size_t>(row) * sg.ld_out + col;
                            if (sg.out_kind == OUT_F16) {
                                static_cast<__half*>(sg.out)[at] = __float2half_rn(y);
                                amax = fmaxf(amax, fabsf(y));
                            } else if (sg.out_kind == OUT_F32) {
                                static_cast<float*>(sg.out)[at] = y;
                            } else {
                                static_cast<__nv_bfloat16*>(sg.out)[at] = __float2bfloat16_rn(y);
                            }
                        }
                        if (!(amax <= 65504.0f)) atomicOr(p.err, DEVERR_RANGE);
                    }
                } else if constexpr (EPI == EPI_PARTIAL) {
                    const int fq = sg.partial_halves ? (q & 1) : q;
                    const int col = ti.ftile * sg.a_fstride + fq * 32 + lane;
                    const int coff = (sg.partial_halves && q >= 2) ? sg.F : 0;
                    float* part = static_cast<float*>(sg.out) +
                                  static_cast<size_t>(ti.ks) * sg.n_rows * sg.ld_out;
                    if (col < sg.F) {
                        const int cmax = min(32, ti.rows - c0);
#pragma unroll
                        for (int c = 0; c < 32; ++c) {
                            if (c >= cmax) break;
                            part[static_cast<size_t>(ti.row0 + c0 + c) * sg.ld_out + coff + col] = __uint_as_float(v[c]);
                        }
                    }
                } else if constexpr (EPI == EPI_RESIDUAL) {
                    const int col = ti.ftile * sg.a_fstride + q * 32 + lane;
                    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(sg.out);
                    const __nv_bfloat16* res = static_cast<const __nv_bfloat16*>(sg.res);
                    if (col < sg.F) {
                        const int cmax = min(32, ti.rows - c0);
#pragma unroll
                        for (int c = 0; c < 32; ++c) {
                            if (c >= cmax) break;
                            const int row = ti.row0 + c0 + c;
                            const size_t at = static_cast<size_t>(row) * sg.ld_out + col;
                            out[at] = __float2bfloat16_rn(__bfloat162float(res[at]) + __uint_as_float(v[c]));
                        }
                    }
                }
            }
            tc_fence_before();
            if (lane == 0) mbar_arrive(&tempty[acc]);
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, 2 * BN);
    if (threadIdx.x == 0 && *abort_flag) atomicOr(p.err, DEVERR_TIMEOUT);
}

// Self-test of the bounded waits above: one thread waits on an mbarrier that
// nothing arrives at, with the same wait helper, gives up after timeout_ns
// as a kernel whose producer or peer stalled would, and sets the device
// error flag.  Nothing faults and nothing hangs.
__global__ void wait_timeout_selftest_kernel(int* err, uint64_t timeout_ns) {
    __shared__ uint64_t bar;
    __shared__ volatile int abort_flag;
    if (threadIdx.x != 0) return;
    abort_flag = 0;
    mbar_init(&bar, 1);
    fence_mbarrier_init();
    if (!mbar_wait(&bar, 0, &abort_flag, timeout_ns)) atomicOr(err, DEVERR_TIMEOUT);
}

}  // namespace moe
