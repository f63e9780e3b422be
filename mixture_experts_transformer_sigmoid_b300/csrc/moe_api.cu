// Host side of the C ABI declared in include/moe.h: argument validation,
// workspace, TMA tensor-map encoding and the launch sequence of one forward.
//
// bf16 forward on one stream (no host synchronisation):
//   rmsnorm -> router logits (tcgen05, split accumulation) -> top-k + chunk histograms ->
//   scan -> stable scatter -> row gather -> gate|up grouped GEMM with SwiGLU
//   epilogue (routed experts + shared expert in one launch) -> down grouped
//   GEMM with routing-weight epilogue (routed + shared in one launch) ->
//   combine with the residual.
// fp32 storage (and gemm_path = 1) runs the same routing kernels with the
// router fused into RMSNorm and the expert contractions on CUDA cores.
//
// Dense feed-forward block (moe_dense_forward): rmsnorm -> gate|up GEMM with
// SwiGLU epilogue -> down GEMM with the residual added in its epilogue, on
// the same two GEMM kernels (one dense segment each).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>
#include <type_traits>
#include <vector>

#include "k_gemm_pair.cuh"
#include "k_gemm_tc.cuh"
#include "k_pack.cuh"
#include "k_route.cuh"
#include "k_router_tc.cuh"
#include "k_route_small.cuh"
#include "moe.h"

using namespace moe;

// Launches a kernel on st with programmatic stream serialization: its blocks
// may be scheduled once the kernel before it has exited, while that kernel's
// memory operations are still being flushed.  Every kernel launched this way
// calls grid_dep_wait before it touches global memory that an earlier kernel
// writes or reads.  Errors are returned and also left for cudaGetLastError.
template <typename... KArgs, typename... Args>
cudaError_t launch_dep(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

struct moe_handle {
    moe_config cfg;
    int es;            // bytes per stored element
    bool tc;           // tensor-core expert/router path
    int num_sms;
    int64_t P_max;     // max_tokens * max_top_k
    int n_chunks_max;
    // workspace
    void* xn = nullptr;
    float* logits = nullptr;
    float2* part = nullptr;   // router (hi, lo) partial sums [ksplit][T][E]
    int* topk_idx = nullptr;
    float* topk_w = nullptr;
    int* chunk_cnt = nullptr;
    int* chunk_base = nullptr;
    int* counts = nullptr;
    int* offsets = nullptr;
    int* pos = nullptr;
    int* row_tok = nullptr;
    float* row_w = nullptr;
    void* xp = nullptr;
    void* h = nullptr;
    void* yp = nullptr;
    void* hs = nullptr;
    void* sh = nullptr;
    void* hd = nullptr;       // dense block activations [max_tokens, dense_inter]
    float* dpart = nullptr;   // split-K partials of the dense down projection [DENSE_SPLIT_MAX][DENSE_SPLIT_MAX_T][d]
    float* gpart = nullptr;   // split-K partials of the dense gate|up projection [DENSE_GU_SPLIT_MAX][DENSE_SPLIT_MAX_T][2 dense_inter]
    void* x_stage = nullptr;
    void* out_stage = nullptr;
    // pipelined host I/O (moe_forward_host_async): a second staging slot, copy
    // streams and the events that order each slot's reuse
    void* x_stage2 = nullptr;
    void* out_stage2 = nullptr;
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t ev_in[2] = {}, ev_done[2] = {}, ev_out[2] = {};
    int async_slot = 0;
    int* err = nullptr;
    int last_T = 0;
    int last_k = 0;
    // counters and per-stage profiling (ring of event sets, one per forward)
    static constexpr int NSTAGE = 9;
    static constexpr int RING = 256;
    int64_t launches = 0;
    int forwards = 0;
    bool profiling = false;
    std::vector<cudaEvent_t> ev;  // RING x (NSTAGE + 1)
    int ring_head = 0, ring_pending = 0;
    double stage_ms[NSTAGE] = {};
    cudaEvent_t* cur = nullptr;   // event set of the forward being queued, or null
};

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode;
}

// bf16 tensor [outer][inner] (inner contiguous), 64 x box_rows boxes, 128-byte swizzle.
bool map_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_rows = 64) {
    auto enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
// bf16 tensor [groups][mid][inner], 64 x 64 x 1 boxes, 128-byte swizzle.
bool map_3d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t mid, uint64_t groups) {
    auto enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {inner, mid, groups};
    cuuint64_t strides[2] = {inner * 2, inner * mid * 2};
    cuuint32_t box[3] = {64, 64, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Grouped bf16 weights read as two 64-feature x 64-k boxes per copy: a 4-D
// view {feature (f_extent, contiguous), k (k_extent rows, k_stride bytes),
// chunk (n_chunks, chunk_stride bytes), group (groups, group_stride bytes)},
// box {64, 64, 2, 1}.  The copy lands as chunk 0 then chunk 1, each 64 k
// rows of 128 swizzled bytes: the layout of two separate 64 x 64 boxes.
bool map_4d_chunks(CUtensorMap* m, const void* base, uint64_t f_extent, uint64_t k_extent,
                   uint64_t k_stride, uint64_t n_chunks, uint64_t chunk_stride, uint64_t groups,
                   uint64_t group_stride) {
    auto enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[4] = {f_extent, k_extent, n_chunks, groups};
    cuuint64_t strides[3] = {k_stride, chunk_stride, group_stride};
    cuuint32_t box[4] = {64, 64, 2, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + nb && b0 < a0 + na;
}

void free_ws(moe_handle* h) {
    void* ptrs[] = {h->xn, h->logits, h->part, h->topk_idx, h->topk_w, h->chunk_cnt, h->chunk_base,
                    h->counts, h->offsets, h->pos, h->row_tok, h->row_w, h->xp, h->h, h->yp,
                    h->hs, h->sh, h->hd, h->dpart, h->gpart, h->x_stage, h->out_stage, h->x_stage2,
                    h->out_stage2, h->err};
    for (void* p : ptrs)
        if (p) cudaFree(p);
}

// Adds the stage times of the oldest pending profiled forward.
bool fold_oldest(moe_handle* h) {
    const int slot = (h->ring_head - h->ring_pending + moe_handle::RING) % moe_handle::RING;
    cudaEvent_t* e = &h->ev[static_cast<size_t>(slot) * (moe_handle::NSTAGE + 1)];
    if (cudaEventSynchronize(e[moe_handle::NSTAGE]) != cudaSuccess) return false;
    for (int i = 0; i < moe_handle::NSTAGE; ++i) {
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, e[i], e[i + 1]) != cudaSuccess) return false;
        h->stage_ms[i] += ms;
    }
    --h->ring_pending;
    return true;
}

// Records the boundary before stage i (i == NSTAGE: end of the forward).
inline void mark(moe_handle* h, int i, cudaStream_t st) {
    if (h->cur) cudaEventRecord(h->cur[i], st);
}

template <int BN, int STAGES, int EPI>
cudaError_t launch_tc(const TcParams& prm, int grid, cudaStream_t st) {
    using S = TcSmem<BN, STAGES>;
    static bool attr_set[64] = {};  // per instantiation and device, before the first launch
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        e = cudaFuncSetAttribute(tc_gemm_kernel<BN, STAGES, EPI>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, S::TOTAL);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    return launch_dep(tc_gemm_kernel<BN, STAGES, EPI>, grid, TC_THREADS, S::TOTAL, st, prm);
}

// Upper bound of the tiles a launch can have (the exact count depends on
// the routing, which stays on the device).
int tile_bound(const TcParams& prm, int BN, int P) {
    int64_t n = 0;
    for (int s = 0; s < prm.n_segs; ++s) {
        const TcSeg& sg = prm.seg[s];
        const int64_t ntok = sg.grouped ? (static_cast<int64_t>(P) + BN - 1) / BN + prm.E
                                        : (static_cast<int64_t>(sg.n_rows) + BN - 1) / BN;
        n += ntok * sg.n_ftiles * (!sg.grouped && sg.k_split > 1 ? sg.k_split : 1);
    }
    return static_cast<int>(std::min<int64_t>(n, 1 << 30));
}

// Tile groups of a dense segment (TcSeg::f_group): weights that fit in L2
// with room to spare keep one group (plain token tile-major order); larger
// ones are cut into groups of about 48 MB of weight rows.
#ifndef MOE_DENSE_GROUP_MB
#define MOE_DENSE_GROUP_MB 48
#endif
// Split-K of the dense down projection for decode-sized batches on the
// single-CTA kernel: with T <= DENSE_SPLIT_MAX_T tokens it has only
// ceil(T / 64) * ceil(d / 128) tiles (48 at d = 6144), too few to stream its
// weights with every SM; up to DENSE_SPLIT_MAX k-ranges bring the tile count
// near the SM count.
constexpr int DENSE_SPLIT_MAX = 8;
constexpr int DENSE_SPLIT_MAX_T = 128;

int dense_down_split(int Tn, int d, int Id, int num_sms) {
    if (Tn > DENSE_SPLIT_MAX_T) return 1;
    const int tiles = ((Tn + 63) / 64) * ((d + 127) / 128);
    return std::max(1, std::min({Id / 64, DENSE_SPLIT_MAX, num_sms / tiles}));
}

// Split-K of the dense gate|up projection for decode-sized batches: its
// ceil(T / 64) * I / 64 tiles (192 at I = 12288) are 1.3 waves; k-ranges (at
// most DENSE_GU_SPLIT_MAX) are chosen for the fullest last wave, and their
// fp32 partials (gates, then ups) are added by splitk_swiglu_kernel.
constexpr int DENSE_GU_SPLIT_MAX = 4;

int dense_gate_up_split(int Tn, int d, int Id, int num_sms) {
    if (Tn > DENSE_SPLIT_MAX_T) return 1;
    const int tiles = ((Tn + 63) / 64) * (Id / 64);
    int best = 1;
    double best_eff = 0.0;
    for (int ks = 1; ks <= std::min(DENSE_GU_SPLIT_MAX, d / 64); ++ks) {
        const double waves = static_cast<double>(tiles) * ks / num_sms;
        const double eff = waves / std::ceil(waves);   // busy fraction of the SMs over the launch
        if (eff > best_eff + 0.02) { best_eff = eff; best = ks; }
    }
    return best;
}

void set_dense_groups(TcSeg& sg, int weight_rows_per_ftile) {
    const double ftile_bytes = 2.0 * weight_rows_per_ftile * sg.K;
    if (ftile_bytes * sg.n_ftiles <= 64.0 * (1 << 20)) {
        sg.f_group = 0;
        return;
    }
    sg.f_group = std::max(1, static_cast<int>(MOE_DENSE_GROUP_MB * double(1 << 20) / ftile_bytes));
}

// CTA-pair grouped GEMM: as many clusters of two as the device keeps
// resident at once (the tile schedule is static, so every launched cluster
// must run from the start), at most one per tile.
template <int EPI>
cudaError_t launch_pair(const TcParams& prm, int P, int num_sms, cudaStream_t st) {
    static int max_clusters[64] = {};  // per device, found before the first launch
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 64) return cudaErrorInvalidDevice;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // as launch_dep
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(TC_THREADS, 1, 1);
    cfg.dynamicSmemBytes = PrSmem::TOTAL;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (max_clusters[dev] == 0) {
        e = cudaFuncSetAttribute(tc_gemm_pair_kernel<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 PrSmem::TOTAL);
        if (e != cudaSuccess) return e;
        cfg.gridDim = dim3(std::max(2, num_sms / 2 * 2), 1, 1);
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, tc_gemm_pair_kernel<EPI>, &cfg);
        if (e != cudaSuccess) return e;
        if (n < 1) return cudaErrorInvalidConfiguration;
        max_clusters[dev] = n;
    }
    const int clusters = std::max(1, std::min(max_clusters[dev], tile_bound(prm, PR_BN, P)));
    cfg.gridDim = dim3(2 * clusters, 1, 1);
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, tc_gemm_pair_kernel<EPI>, prm);
}

template <int EPI>
cudaError_t run_tc(const TcParams& prm, bool pair, int P, int num_sms, cudaStream_t st) {
    if (pair) return launch_pair<EPI>(prm, P, num_sms, st);
    const int grid = std::max(1, std::min(num_sms, tile_bound(prm, 64, P)));
    return launch_tc<64, 8, EPI>(prm, grid, st);
}

// Top-k from either logit source (LogitsFromPairs / LogitsPlain).  A chunk
// of 128 tokens (one histogram) is split over up to 4 blocks until the grid
// covers the SMs; each block takes as many warps as its registers allow, up
// to one per token.
template <int EPL, typename Src>
void launch_topk_e(const Src& src, const float* bias, int T, int E, int k, float scale, int* idx,
                   float* w, int* chunk_cnt, int num_sms, cudaStream_t st) {
    const int n_chunks = (T + CHUNK_TOKENS - 1) / CHUNK_TOKENS;
    int split = 1;
    while (split < 4 && n_chunks * split * 2 <= num_sms) split *= 2;
    static int threads[64] = {};  // per device, found before the first launch
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev >= 64) dev = 0;
    if (threads[dev] == 0) {
        cudaFuncAttributes fa;
        int tmax = 512;
        if (cudaFuncGetAttributes(&fa, topk_kernel<EPL, Src>) == cudaSuccess)
            tmax = std::min(1024, fa.maxThreadsPerBlock) / 32 * 32;
        threads[dev] = std::max(32, tmax);
    }
    const int nthreads = std::min(threads[dev], 32 * (CHUNK_TOKENS / split));
    if (split > 1) cudaMemsetAsync(chunk_cnt, 0, static_cast<size_t>(n_chunks) * E * sizeof(int), st);
    launch_dep(topk_kernel<EPL, Src>, n_chunks * split, nthreads, E * sizeof(int), st,
               src, bias, T, E, k, scale, idx, w, chunk_cnt, split);
}

template <typename Src>
void launch_topk(const Src& src, const float* bias, int T, int E, int k, float scale, int* idx, float* w,
                 int* chunk_cnt, int num_sms, cudaStream_t st) {
#define MOE_TOPK(EPL) launch_topk_e<EPL>(src, bias, T, E, k, scale, idx, w, chunk_cnt, num_sms, st)
    if (E <= 32) MOE_TOPK(1);
    else if (E <= 64) MOE_TOPK(2);
    else if (E <= 128) MOE_TOPK(4);
    else if (E <= 256) MOE_TOPK(8);
    else if (E <= 512) MOE_TOPK(16);
    else MOE_TOPK(32);
#undef MOE_TOPK
}

// Router logits on the tensor cores.  Split-K is chosen so that small
// batches still spread over the SMs; the ranges are then added by
// router_reduce_kernel, or, when defer is given and the partials are few
// enough for one block to read, left to the fused small-batch routing kernel
// (*defer = the number of ranges it must add; 1 when nothing is left).
// Returns the number of launches (0 on error).
// The router launch for a token tile width BN (see router_tc_kernel).
template <int BN>
cudaError_t launch_router_bn(const RouterParams& rp, int grid, cudaStream_t st) {
    using C = RtCfg<BN>;
    static bool attr_set[64] = {};   // per tile width and device, before the first launch
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        e = cudaFuncSetAttribute(router_tc_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    return launch_dep(router_tc_kernel<BN>, grid, C::THREADS, C::SMEM, st, rp);
}

int launch_router_tc(moe_handle* h, const void* router_w, const void* xn, int T, cudaStream_t st,
                     int* defer = nullptr) {
    const int d = h->cfg.hidden, E = h->cfg.n_experts;
    const int BN = T > 64 ? 128 : 64;   // tokens per router tile
    RouterParams rp;
    std::memset(&rp, 0, sizeof rp);
    if (!map_2d(&rp.a, router_w, d, E) || !map_2d(&rp.b, xn, d, T, BN)) return 0;
    const int nkb = d / 64;
    const int tiles0 = ((T + BN - 1) / BN) * ((E + 127) / 128);
    int ks = std::max(1, std::min(h->num_sms / tiles0, nkb / 4));   // at most one wave
    const int kbps = (nkb + ks - 1) / ks;
    ks = (nkb + kbps - 1) / kbps;
    rp.T = T;
    rp.E = E;
    rp.d = d;
    rp.ksplit = ks;
    rp.kb_per_split = kbps;
    rp.part = h->part;
    rp.err = h->err;
    const int grid = std::min(h->num_sms, tiles0 * ks);
    if ((BN == 128 ? launch_router_bn<128>(rp, grid, st) : launch_router_bn<64>(rp, grid, st)) != cudaSuccess)
        return 0;
    if (defer != nullptr) *defer = 1;
    if (ks == 1) return cudaGetLastError() == cudaSuccess ? 1 : 0;
    const size_t n = static_cast<size_t>(T) * E;
    if (defer != nullptr && n * ks <= static_cast<size_t>(RS_MAX_PAIRS)) {
        *defer = ks;
        return cudaGetLastError() == cudaSuccess ? 1 : 0;
    }
    launch_dep(router_reduce_kernel, static_cast<int>(std::min<size_t>((n + 255) / 256, 4 * h->num_sms)), 256, 0, st,
               h->part, ks, n);
    return cudaGetLastError() == cudaSuccess ? 2 : 0;
}

// RMSNorm of Tn rows of d elements.  From 8 tokens per SM up, a warp per
// token with the rows staged in shared memory (rmsnorm_bulk_kernel: as many
// warps per block, up to RMSB_WARPS_MAX, as fit RMSB_NBUF row buffers each
// next to the gain row in RMSB_SMEM_BUDGET; as many blocks as are resident
// at once, each warp looping over tokens); smaller batches, and rows too long
// for one such warp, a block per token.
constexpr size_t RMSB_SMEM_BUDGET = 216 * 1024;

template <typename T>
cudaError_t launch_rmsnorm(moe_handle* h, const T* x, const T* gain, T* xn, int Tn, int d, float eps,
                           cudaStream_t st) {
    const size_t row_bytes = static_cast<size_t>(d) * sizeof(T);
    const size_t fixed = rmsb_smem(0, row_bytes);   // barriers and the gain row
    const int warps = fixed >= RMSB_SMEM_BUDGET
                          ? 0
                          : static_cast<int>(std::min<size_t>(RMSB_WARPS_MAX,
                                                              (RMSB_SMEM_BUDGET - fixed) / (RMSB_NBUF * row_bytes)));
    if (Tn < 8 * h->num_sms || warps < 1)
        return launch_dep(rmsnorm_kernel<T>, Tn, 256, 0, st, x, gain, xn, d, eps);
    static bool attr_set[64] = {};   // per device: the budget as the kernel's shared-memory limit
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        e = cudaFuncSetAttribute(rmsnorm_bulk_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(RMSB_SMEM_BUDGET));
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    const size_t smem = rmsb_smem(warps, row_bytes);
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, rmsnorm_bulk_kernel<T>, 32 * warps, smem);
    if (e != cudaSuccess) return e;
    const int blocks = std::min(std::max(per_sm, 1) * h->num_sms, (Tn + warps - 1) / warps);
    return launch_dep(rmsnorm_bulk_kernel<T>, blocks, 32 * warps, smem, st, x, gain, xn, Tn, d, eps, h->err);
}

// The fused small-batch routing block, instantiated for the experts per lane.
template <int EPL>
cudaError_t launch_route_small_e(const RouteSmallArgs& ra, cudaStream_t st) {
    // the largest shared memory any batch it takes can need, set once per device
    constexpr size_t SMEM_MAX = route_small_smem(RS_MAX_T, RS_MAX_TE / RS_MAX_T, RS_MAX_K) +
                                sizeof(float) * 2 * RS_MAX_E;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        e = cudaFuncSetAttribute(route_small_kernel<EPL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(SMEM_MAX));
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    const size_t smem = route_small_smem(ra.T, ra.E, ra.k);
    if (smem > SMEM_MAX) return cudaErrorInvalidValue;
    return launch_dep(route_small_kernel<EPL>, 1, RS_THREADS, smem, st, ra);
}

cudaError_t launch_route_small(const RouteSmallArgs& ra, cudaStream_t st) {
    if (ra.E <= 32) return launch_route_small_e<1>(ra, st);
    if (ra.E <= 64) return launch_route_small_e<2>(ra, st);
    if (ra.E <= 128) return launch_route_small_e<4>(ra, st);
    return launch_route_small_e<8>(ra, st);   // E <= RS_MAX_E = 256
}

// Grid of the combine: a block per token, and for batches too small to fill
// the SMs each row split over several blocks of 256 vectors.
dim3 combine_grid(int Tn, int nvec, int num_sms) {
    const int split = Tn >= 4 * num_sms ? 1 : std::max(1, (nvec + 255) / 256);
    return dim3(Tn, split, 1);
}

struct FwdArgs {
    int T;
    const void *x, *norm_w, *router_w;
    const float* bias;
    const void *gate_up, *down, *sg, *su, *sd;
    int k;
    float scale;
    void* out;
};

template <typename T>
moe_status forward_simt_or_routing(moe_handle* h, const FwdArgs& a, cudaStream_t st) {
    const moe_config& c = h->cfg;
    const int d = c.hidden, E = c.n_experts, I = c.inter, Is = c.shared_inter;
    const int Tn = a.T, k = a.k, P = Tn * k;
    const int n_chunks = (Tn + CHUNK_TOKENS - 1) / CHUNK_TOKENS;
    const T* x = static_cast<const T*>(a.x);
    T* xn = static_cast<T*>(h->xn);
    // decode-sized batches route in one block (route_small_kernel)
    const bool small = h->tc && Tn <= RS_MAX_T && Tn * E <= RS_MAX_TE && E <= RS_MAX_E && k <= RS_MAX_K;
    int ks_left = 1;

    // A+B: RMSNorm and router logits
    mark(h, 0, st);
    if (h->tc) {
        if (launch_rmsnorm(h, x, static_cast<const T*>(a.norm_w), xn, Tn, d, c.eps, st) != cudaSuccess)
            return MOE_ERR_CUDA;
        mark(h, 1, st);
        const int n_router = launch_router_tc(h, a.router_w, xn, Tn, st, small ? &ks_left : nullptr);
        if (n_router == 0) return MOE_ERR_CUDA;
        h->launches += 1 + n_router;
    } else {
        rmsnorm_router_kernel<T><<<Tn, 256, d * sizeof(float), st>>>(
            x, static_cast<const T*>(a.norm_w), static_cast<const T*>(a.router_w), xn, h->part, d,
            E, c.eps);
        mark(h, 1, st);
        h->launches += 1;
    }
    // C+D: top-k, weights, chunk histograms; E: scan, scatter, gather
    mark(h, 2, st);
    bool gathered = false;
    if (small) {
        // one block from the logit partials to the permuted rows; the rows are
        // gathered there too when they are few
        RouteSmallArgs ra;
        ra.part = h->part;
        ra.ksplit = ks_left;
        ra.bias = a.bias;
        ra.logits = h->logits;
        ra.T = Tn;
        ra.E = E;
        ra.k = k;
        ra.routed_scale = a.scale;
        ra.idx = h->topk_idx;
        ra.w = h->topk_w;
        ra.counts = h->counts;
        ra.offsets = h->offsets;
        ra.pos = h->pos;
        ra.row_tok = h->row_tok;
        ra.row_w = h->row_w;
        ra.xn = xn;
        gathered = static_cast<size_t>(P) * d * sizeof(T) <= RS_GATHER_MAX_BYTES;
        ra.xp = gathered ? h->xp : nullptr;
        ra.row_bytes = d * static_cast<int>(sizeof(T));
        if (launch_route_small(ra, st) != cudaSuccess) return MOE_ERR_CUDA;
        mark(h, 3, st);
        mark(h, 4, st);
        mark(h, 5, st);
        h->launches += 1;
    } else {
        launch_topk(LogitsFromPairs{h->part, h->logits}, a.bias, Tn, E, k, a.scale, h->topk_idx, h->topk_w,
                    h->chunk_cnt, h->num_sms, st);
        mark(h, 3, st);
        launch_dep(scan_kernel, 1, std::max(32, (E + 31) / 32 * 32), 0, st,
                   h->chunk_cnt, n_chunks, E, h->counts, h->offsets, h->chunk_base);
        mark(h, 4, st);
        launch_dep(scatter_kernel, n_chunks, CHUNK_TOKENS, E * (CHUNK_TOKENS / 32) * sizeof(uint32_t), st,
                   h->topk_idx, h->topk_w, Tn, E, k, h->chunk_base, h->pos, h->row_tok, h->row_w);
        mark(h, 5, st);
        h->launches += 3;
    }
    // CTA pairs (256 x 256 tiles) once experts average 64 tokens or more; below
    // that the single-CTA kernel with 64-token tiles wastes less.
    const bool pair = h->tc && P >= 64 * E;
    if (!gathered) {
        if (Tn >= 8 * h->num_sms)   // a warp per token: each xn row read once
            launch_dep(gather_tokens_kernel<T>, std::min(8 * h->num_sms, (Tn + 7) / 8), 256, 0, st,
                       xn, h->pos, static_cast<T*>(h->xp), Tn, k, d, P);
        else                        // few tokens: a warp per row spreads the copy over more SMs
            launch_dep(gather_rows_kernel<T>, std::min(4 * h->num_sms, (P + 7) / 8), 256, 0, st,
                       xn, h->row_tok, static_cast<T*>(h->xp), P, d, Tn);
        h->launches += 1;
    }
    mark(h, 6, st);

    T* hbuf = static_cast<T*>(h->h);
    T* yp = static_cast<T*>(h->yp);
    T* hs = static_cast<T*>(h->hs);
    T* sh = Is > 0 ? static_cast<T*>(h->sh) : nullptr;
    if (h->tc) {
        auto fail = [&]() { return MOE_ERR_CUDA; };
        // F+H(gate|up): routed + shared gate|up with the SwiGLU epilogue, one launch
        TcParams g1;
        std::memset(&g1, 0, sizeof g1);
        g1.E = E;
        g1.offsets = h->offsets;
        g1.err = h->err;
        g1.n_segs = Is > 0 ? 2 : 1;
        const uint64_t I2 = 2ull * I;
        if (pair) {
            // gate and up halves of 64 features in one copy: {f < I, k, half (stride I), expert}
            if (!map_4d_chunks(&g1.a0[0], a.gate_up, I, d, I2 * 2, 2, uint64_t(I) * 2, E, d * I2 * 2) ||
                !map_2d(&g1.b[0], h->xp, d, P) || !map_2d(&g1.b128[0], h->xp, d, P, 128))
                return fail();
            g1.seg[0] = TcSeg{1, 0, d, 128, I, (I + 127) / 128, I, I, hbuf, nullptr, 64, PA_HALVES_4D};
        } else {
            if (!map_3d(&g1.a0[0], a.gate_up, I2, d, E) || !map_3d(&g1.a1[0], a.gate_up, I2, d, E) ||
                !map_2d(&g1.b[0], h->xp, d, P))
                return fail();
            g1.seg[0] = TcSeg{1, 0, d, 64, I, I / 64, I, I, hbuf, nullptr, 0, 0};
        }
        if (Is > 0) {
            if (!map_2d(&g1.a0[1], a.sg, d, Is) || !map_2d(&g1.a1[1], a.su, d, Is) ||
                !map_2d(&g1.b[1], xn, d, Tn) || !map_2d(&g1.b128[1], xn, d, Tn, 128))
                return fail();
            g1.seg[1] = pair ? TcSeg{0, Tn, d, 128, 0, (Is + 127) / 128, Is, Is, hs, nullptr, 64, PA_TWO_2D}
                             : TcSeg{0, Tn, d, 64, 0, Is / 64, Is, Is, hs, nullptr, 0, 0};
            set_dense_groups(g1.seg[1], pair ? 256 : 128);
        }
        if (run_tc<EPI_SWIGLU>(g1, pair, P, h->num_sms, st) != cudaSuccess) return fail();
        mark(h, 7, st);
        // G+H(down): routed down projection with the routing weight -> yp (fp16),
        // and the shared expert's down projection -> sh (fp32), one launch
        TcParams g2;
        std::memset(&g2, 0, sizeof g2);
        g2.E = E;
        g2.offsets = h->offsets;
        g2.err = h->err;
        g2.n_segs = Is > 0 ? 2 : 1;
        if (pair) {
            // two consecutive 64-feature chunks in one copy: {f < 64, k, chunk (stride 128 B), expert}
            if (!map_4d_chunks(&g2.a0[0], a.down, 64, I, uint64_t(d) * 2, d / 64, 128, E,
                               uint64_t(I) * d * 2) ||
                !map_2d(&g2.b[0], hbuf, I, P) || !map_2d(&g2.b128[0], hbuf, I, P, 128))
                return fail();
            g2.seg[0] = TcSeg{1, 0, I, 256, 64, (d + 255) / 256, d, d, yp, h->row_w, 128, PA_CHUNKS_4D};
        } else {
            if (!map_3d(&g2.a0[0], a.down, d, I, E) || !map_3d(&g2.a1[0], a.down, d, I, E) ||
                !map_2d(&g2.b[0], hbuf, I, P))
                return fail();
            g2.seg[0] = TcSeg{1, 0, I, 128, 64, (d + 127) / 128, d, d, yp, h->row_w, 0, 0};
        }
        // the weighted rows go to the combine in fp16: the same bytes as bf16,
        // with 3 more significand bits (an overflow is reported as MOE_ERR_RANGE)
        g2.seg[0].out_kind = OUT_F16;
        if (Is > 0) {
            if (pair) {
                // 128 consecutive nn.Linear rows of the shared down projection in one copy
                if (!map_2d(&g2.a0[1], a.sd, Is, d, 128) || !map_2d(&g2.b[1], hs, Is, Tn) ||
                    !map_2d(&g2.b128[1], hs, Is, Tn, 128))
                    return fail();
                g2.seg[1] = TcSeg{0, Tn, Is, 256, 64, (d + 255) / 256, d, d, h->sh, nullptr, 128, PA_ONE_2D};
                set_dense_groups(g2.seg[1], 256);
            } else {
                if (!map_2d(&g2.a0[1], a.sd, Is, d) || !map_2d(&g2.a1[1], a.sd, Is, d) ||
                    !map_2d(&g2.b[1], hs, Is, Tn))
                    return fail();
                g2.seg[1] = TcSeg{0, Tn, Is, 128, 64, (d + 127) / 128, d, d, h->sh, nullptr, 0, 0};
                set_dense_groups(g2.seg[1], 128);
            }
            // the shared expert's output reaches the combine in fp32, never rounded on its own
            g2.seg[1].out_kind = OUT_F32;
        }
        if (run_tc<EPI_WEIGHTED>(g2, pair, P, h->num_sms, st) != cudaSuccess) return fail();
        h->launches += 2;
        // I: combine with the residual
        mark(h, 8, st);
        if constexpr (std::is_same<T, __nv_bfloat16>::value)   // the tensor-core path stores bf16
            launch_dep(combine_kernel<T, __half, float>, combine_grid(Tn, d / Elem<T>::V, h->num_sms), 256, 0, st,
                       x, Is > 0 ? static_cast<const float*>(h->sh) : nullptr,
                       static_cast<const __half*>(h->yp), h->pos, d, k, static_cast<T*>(a.out));
        h->launches += 1;
        mark(h, moe_handle::NSTAGE, st);
        return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
    } else {
        const T* gu = static_cast<const T*>(a.gate_up);
        const T* dn = static_cast<const T*>(a.down);
        simt_gate_up_kernel<T><<<dim3(P, (I + 127) / 128), 128, d * sizeof(float), st>>>(
            static_cast<const T*>(h->xp), gu, h->offsets, E, d, I, hbuf);
        if (Is > 0)
            simt_shared_gate_up_kernel<T><<<dim3(Tn, (Is + 127) / 128), 128, d * sizeof(float), st>>>(
                xn, static_cast<const T*>(a.sg), static_cast<const T*>(a.su), d, Is, hs);
        mark(h, 7, st);
        simt_down_kernel<T><<<dim3(P, (d + 127) / 128), 128, I * sizeof(float), st>>>(
            hbuf, dn, h->offsets, h->row_w, E, I, d, yp);
        if (Is > 0)
            simt_shared_down_kernel<T><<<dim3(Tn, (d + 127) / 128), 128, Is * sizeof(float), st>>>(
                hs, static_cast<const T*>(a.sd), Is, d, sh);
        h->launches += Is > 0 ? 4 : 2;
    }
    // I: combine with the residual
    mark(h, 8, st);
    launch_dep(combine_kernel<T>, combine_grid(Tn, d / Elem<T>::V, h->num_sms), 256, 0, st,
               x, sh, yp, h->pos, d, k, static_cast<T*>(a.out));
    h->launches += 1;
    mark(h, moe_handle::NSTAGE, st);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// Dense feed-forward block: RMSNorm, then gate|up with the SwiGLU epilogue
// into hd, then down with the residual added to the fp32 result before its
// one rounding (in the GEMM epilogue, or in the CUDA-core down kernel).
template <typename T>
moe_status dense_impl(moe_handle* h, int Tn, const void* x_, const void* norm_w, const void* gw,
                      const void* uw, const void* dw, int Id, void* out, cudaStream_t st) {
    const moe_config& c = h->cfg;
    const int d = c.hidden;
    const T* x = static_cast<const T*>(x_);
    T* xn = static_cast<T*>(h->xn);
    T* hd = static_cast<T*>(h->hd);
    if (launch_rmsnorm(h, x, static_cast<const T*>(norm_w), xn, Tn, d, c.eps, st) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (h->tc) {
        // CTA pairs (256 x 256 tiles) from two 64-token tiles up
        const bool pair = Tn >= 128;
        TcParams g1;
        std::memset(&g1, 0, sizeof g1);
        g1.E = 1;
        g1.offsets = h->offsets;
        g1.err = h->err;
        g1.n_segs = 1;
        if (!map_2d(&g1.a0[0], gw, d, Id) || !map_2d(&g1.a1[0], uw, d, Id) || !map_2d(&g1.b[0], xn, d, Tn) ||
            !map_2d(&g1.b128[0], xn, d, Tn, 128))
            return MOE_ERR_CUDA;
        g1.seg[0] = pair ? TcSeg{0, Tn, d, 128, 0, (Id + 127) / 128, Id, Id, hd, nullptr, 64, PA_TWO_2D, nullptr}
                         : TcSeg{0, Tn, d, 64, 0, Id / 64, Id, Id, hd, nullptr, 0, 0, nullptr};
        set_dense_groups(g1.seg[0], pair ? 256 : 128);
        const int ks1 = (pair || h->gpart == nullptr) ? 1 : dense_gate_up_split(Tn, d, Id, h->num_sms);
        if (ks1 > 1) {
            // k-ranges of fp32 partials [ks1][Tn][gates | ups], then SwiGLU of their sums
            g1.seg[0].out = h->gpart;
            g1.seg[0].ld_out = 2 * Id;
            g1.seg[0].k_split = ks1;
            g1.seg[0].partial_halves = 1;
            const int grid = std::max(1, std::min(h->num_sms, tile_bound(g1, 64, Tn)));
            if (launch_tc<64, 8, EPI_PARTIAL>(g1, grid, st) != cudaSuccess) return MOE_ERR_CUDA;
            const size_t n4 = static_cast<size_t>(Tn) * Id / 4;
            launch_dep(splitk_swiglu_kernel<T>,
                       static_cast<int>(std::min<size_t>((n4 + 255) / 256, 4 * h->num_sms)), 256, 0, st,
                       h->gpart, ks1, Tn, Id, hd);
            h->launches += 1;
        } else if (run_tc<EPI_SWIGLU>(g1, pair, Tn, h->num_sms, st) != cudaSuccess) {
            return MOE_ERR_CUDA;
        }
        TcParams g2;
        std::memset(&g2, 0, sizeof g2);
        g2.E = 1;
        g2.offsets = h->offsets;
        g2.err = h->err;
        g2.n_segs = 1;
        if (pair) {
            if (!map_2d(&g2.a0[0], dw, Id, d, 128) || !map_2d(&g2.b[0], hd, Id, Tn) ||
                !map_2d(&g2.b128[0], hd, Id, Tn, 128))
                return MOE_ERR_CUDA;
            g2.seg[0] = TcSeg{0, Tn, Id, 256, 64, (d + 255) / 256, d, d, out, nullptr, 128, PA_ONE_2D, x};
            set_dense_groups(g2.seg[0], 256);
        } else {
            if (!map_2d(&g2.a0[0], dw, Id, d) || !map_2d(&g2.a1[0], dw, Id, d) || !map_2d(&g2.b[0], hd, Id, Tn))
                return MOE_ERR_CUDA;
            g2.seg[0] = TcSeg{0, Tn, Id, 128, 64, (d + 127) / 128, d, d, out, nullptr, 0, 0, x};
            set_dense_groups(g2.seg[0], 128);
        }
        const int ks = pair ? 1 : dense_down_split(Tn, d, Id, h->num_sms);
        if (ks > 1) {
            // k-ranges of fp32 partials [ks][Tn][d], then their sum in order plus the residual
            g2.seg[0].out = h->dpart;
            g2.seg[0].res = nullptr;
            g2.seg[0].k_split = ks;
            const int grid = std::max(1, std::min(h->num_sms, tile_bound(g2, 64, Tn)));
            if (launch_tc<64, 8, EPI_PARTIAL>(g2, grid, st) != cudaSuccess) return MOE_ERR_CUDA;
            const size_t n = static_cast<size_t>(Tn) * d;
            launch_dep(splitk_residual_kernel<T>,
                       static_cast<int>(std::min<size_t>((n / 4 + 255) / 256, 4 * h->num_sms)), 256, 0, st,
                       h->dpart, ks, n, x, static_cast<T*>(out), n);
            h->launches += 4;
        } else {
            if (run_tc<EPI_RESIDUAL>(g2, pair, Tn, h->num_sms, st) != cudaSuccess) return MOE_ERR_CUDA;
            h->launches += 3;
        }
    } else {
        simt_shared_gate_up_kernel<T><<<dim3(Tn, (Id + 127) / 128), 128, d * sizeof(float), st>>>(
            xn, static_cast<const T*>(gw), static_cast<const T*>(uw), d, Id, hd);
        simt_shared_down_kernel<T><<<dim3(Tn, (d + 127) / 128), 128, Id * sizeof(float), st>>>(
            hd, static_cast<const T*>(dw), Id, d, static_cast<T*>(out), x);
        h->launches += 3;
    }
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// Query compression of the sparse latent attention: c = hidden · w_qaᵀ (the
// Linear's output, rounded once to the storage dtype), q = RMSNorm(c).
// Prefill-sized batches run the CTA-pair GEMM with a plain epilogue, then the
// RMSNorm over the rank features of c.  Small batches run the single-CTA GEMM
// split over k-ranges (enough tiles to stream w_qa with every SM) and one
// kernel that adds the partials, rounds c and normalises it.
template <typename T>
moe_status q_latent_impl(moe_handle* h, int Tn, int rank, const void* hidden, const void* w_qa,
                         const void* gain, void* c_out, void* q_out, cudaStream_t st) {
    const moe_config& c = h->cfg;
    const int d = c.hidden;
    T* cq = static_cast<T*>(c_out);
    auto norm = [&]() {
        return launch_rmsnorm(h, static_cast<const T*>(cq), static_cast<const T*>(gain), static_cast<T*>(q_out), Tn,
                              rank, c.eps, st);
    };
    if (!h->tc) {
        simt_shared_down_kernel<T><<<dim3(Tn, (rank + 127) / 128), 128, d * sizeof(float), st>>>(
            static_cast<const T*>(hidden), static_cast<const T*>(w_qa), d, rank, cq);
        if (norm() != cudaSuccess) return MOE_ERR_CUDA;
        h->launches += 2;
        return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
    }
    TcParams g;
    std::memset(&g, 0, sizeof g);
    g.E = 1;
    g.offsets = h->offsets;
    g.err = h->err;
    g.n_segs = 1;
    const int tiles_pair = ((Tn + 255) / 256) * ((rank + 255) / 256);
    const bool pair = Tn >= 128 && 2 * tiles_pair >= h->num_sms;
    if (pair) {
        if (!map_2d(&g.a0[0], w_qa, d, rank, 128) || !map_2d(&g.b[0], hidden, d, Tn) ||
            !map_2d(&g.b128[0], hidden, d, Tn, 128))
            return MOE_ERR_CUDA;
        g.seg[0] = TcSeg{0, Tn, d, 256, 64, (rank + 255) / 256, rank, rank, c_out, nullptr, 128, PA_ONE_2D};
        set_dense_groups(g.seg[0], 256);
        if (run_tc<EPI_WEIGHTED>(g, true, Tn, h->num_sms, st) != cudaSuccess) return MOE_ERR_CUDA;
        if (norm() != cudaSuccess) return MOE_ERR_CUDA;
        h->launches += 2;
        return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
    }
    if (!map_2d(&g.a0[0], w_qa, d, rank) || !map_2d(&g.a1[0], w_qa, d, rank) || !map_2d(&g.b[0], hidden, d, Tn))
        return MOE_ERR_CUDA;
    g.seg[0] = TcSeg{0, Tn, d, 128, 64, (rank + 127) / 128, rank, rank, c_out, nullptr, 0, 0};
    set_dense_groups(g.seg[0], 128);
    const int tiles = ((Tn + 63) / 64) * ((rank + 127) / 128);
    // the split-K partials [ks][Tn][rank] must fit the handle's buffer [8][min(T, 128)][d]
    const int ks = Tn <= std::min(c.max_tokens, DENSE_SPLIT_MAX_T) && rank <= d
                       ? std::max(1, std::min({d / 64, DENSE_SPLIT_MAX, h->num_sms / tiles}))
                       : 1;
    const int grid_cap = h->num_sms;
    if (ks > 1) {
        g.seg[0].out = h->dpart;
        g.seg[0].k_split = ks;
        const int grid = std::max(1, std::min(grid_cap, tile_bound(g, 64, Tn)));
        if (launch_tc<64, 8, EPI_PARTIAL>(g, grid, st) != cudaSuccess) return MOE_ERR_CUDA;
        launch_dep(splitk_rmsnorm_kernel<T>, Tn, 256, 0, st,
                   h->dpart, ks, static_cast<size_t>(Tn) * rank, rank, static_cast<const T*>(gain), c.eps, cq,
                   static_cast<T*>(q_out));
    } else {
        if (run_tc<EPI_WEIGHTED>(g, false, Tn, h->num_sms, st) != cudaSuccess) return MOE_ERR_CUDA;
        if (norm() != cudaSuccess) return MOE_ERR_CUDA;
    }
    h->launches += 2;
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status validate_forward(moe_handle* h, const FwdArgs& a, bool host_io) {
    if (!h) return MOE_ERR_INVALID_ARG;
    const moe_config& c = h->cfg;
    if (a.T < 0 || a.T > c.max_tokens) return MOE_ERR_INVALID_ARG;
    if (a.k < 1 || a.k > c.max_top_k || a.k > c.n_experts) return MOE_ERR_INVALID_ARG;
    if (!std::isfinite(a.scale)) return MOE_ERR_INVALID_ARG;
    if (a.T == 0) return MOE_OK;  // nothing is read or written
    if (!a.x || !a.norm_w || !a.router_w || !a.bias || !a.gate_up || !a.down || !a.out)
        return MOE_ERR_INVALID_ARG;
    if (c.shared_inter > 0 && (!a.sg || !a.su || !a.sd)) return MOE_ERR_INVALID_ARG;
    const void* vec_ptrs[] = {a.x, a.norm_w, a.router_w, a.gate_up, a.down, a.out};
    for (const void* p : vec_ptrs)
        if (!aligned16(p)) return MOE_ERR_INVALID_ARG;
    if (c.shared_inter > 0 && (!aligned16(a.sg) || !aligned16(a.su) || !aligned16(a.sd)))
        return MOE_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(a.bias) & 3u) != 0) return MOE_ERR_INVALID_ARG;
    if (!host_io) {
        const size_t es = h->es, d = c.hidden, E = c.n_experts, I = c.inter, Is = c.shared_inter;
        const size_t out_b = static_cast<size_t>(a.T) * d * es;
        const struct { const void* p; size_t n; } ins[] = {
            {a.x, out_b},         {a.norm_w, d * es},        {a.router_w, E * d * es},
            {a.bias, E * 4},      {a.gate_up, E * d * 2 * I * es}, {a.down, E * I * d * es},
            {a.sg, Is * d * es},  {a.su, Is * d * es},       {a.sd, d * Is * es}};
        for (const auto& in : ins)
            if (overlaps(a.out, out_b, in.p, in.n)) return MOE_ERR_INVALID_ARG;
    }
    return MOE_OK;
}

moe_status forward_impl(moe_handle* h, const FwdArgs& a, cudaStream_t st) {
    if (cudaSetDevice(h->cfg.device) != cudaSuccess) return MOE_ERR_CUDA;
    h->last_T = a.T;
    h->last_k = a.k;
    h->forwards += 1;
    if (a.T == 0) return MOE_OK;
    h->cur = nullptr;
    if (h->profiling) {
        if (h->ring_pending == moe_handle::RING && !fold_oldest(h)) return MOE_ERR_CUDA;
        h->cur = &h->ev[static_cast<size_t>(h->ring_head) * (moe_handle::NSTAGE + 1)];
    }
    moe_status s = h->cfg.dtype == MOE_DTYPE_BF16 ? forward_simt_or_routing<__nv_bfloat16>(h, a, st)
                                                   : forward_simt_or_routing<float>(h, a, st);
    if (h->cur) {
        if (s == MOE_OK) {
            h->ring_head = (h->ring_head + 1) % moe_handle::RING;
            h->ring_pending += 1;
        }
        h->cur = nullptr;
    }
    return s;
}

}  // namespace

// ------------------------------------------- routing without allocation
// Scratch of moe_route_static: the per-chunk expert histograms and their
// running bases, [ceil(T / 128)][E] each.  It lives in the module's static
// device memory, so the entry point never allocates; every GPU that loads
// the library holds these 1 MB until the process exits.  All calls on a
// device share it, so calls that overlap on the GPU race.  Every cell a
// call reads is written earlier in the same call, so nothing needs clearing
// between calls.
constexpr int ROUTE_STATIC_MAX_CELLS = 131072;  // ceil(T / 128) * E, per array
static __device__ __align__(256) int g_route_scratch[2 * ROUTE_STATIC_MAX_CELLS];

namespace {
std::mutex g_route_scratch_mu;
int* g_route_scratch_dev[64] = {};  // device address of g_route_scratch, per device

// The symbol's device address on device `dev` (the current device).  In
// host code g_route_scratch names a host-side stand-in, not device memory,
// so kernels must be given this address instead.
int* route_scratch(int dev) {
    std::lock_guard<std::mutex> lock(g_route_scratch_mu);
    if (g_route_scratch_dev[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess) return nullptr;
        g_route_scratch_dev[dev] = static_cast<int*>(p);
    }
    return g_route_scratch_dev[dev];
}

}  // namespace

extern "C" {

moe_status moe_route_static(int32_t T, int32_t E, int32_t top_k, float routed_scale,
                            const float* logits, const float* corr_bias, int32_t* idx, float* w,
                            int32_t* counts, int32_t* offsets, int32_t* pos, int32_t* row_tok,
                            float* row_w, void* stream) {
    if (T < 0 || E < 1 || E > 1024 || top_k < 1 || top_k > 32 || top_k > E ||
        !std::isfinite(routed_scale))
        return MOE_ERR_INVALID_ARG;
    const int64_t n_chunks = (static_cast<int64_t>(T) + CHUNK_TOKENS - 1) / CHUNK_TOKENS;
    if (n_chunks * E > ROUTE_STATIC_MAX_CELLS) return MOE_ERR_UNSUPPORTED;
    if (T == 0) return MOE_OK;
    const void* ptrs[] = {logits, corr_bias, idx, w, counts, offsets, pos, row_tok, row_w};
    for (const void* p : ptrs)
        if (p == nullptr || (reinterpret_cast<uintptr_t>(p) & 3u) != 0) return MOE_ERR_INVALID_ARG;
    // no output may overlap an input or another output
    const size_t Tk = static_cast<size_t>(T) * top_k * 4, Eb = static_cast<size_t>(E) * 4;
    const struct { const void* p; size_t n; } bufs[] = {
        {logits, static_cast<size_t>(T) * Eb}, {corr_bias, Eb}, {idx, Tk}, {w, Tk}, {counts, Eb},
        {offsets, Eb + 4}, {pos, Tk}, {row_tok, Tk}, {row_w, Tk}};
    constexpr int n_bufs = sizeof(bufs) / sizeof(bufs[0]);
    for (int o = 2; o < n_bufs; ++o)
        for (int i = 0; i < n_bufs; ++i)
            if (i != o && overlaps(bufs[o].p, bufs[o].n, bufs[i].p, bufs[i].n)) return MOE_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
    int* scratch = route_scratch(dev);
    if (scratch == nullptr) return MOE_ERR_CUDA;
    int* chunk_cnt = scratch;
    int* chunk_base = scratch + ROUTE_STATIC_MAX_CELLS;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int nch = static_cast<int>(n_chunks);
    int n_sms = 148;
    if (cudaDeviceGetAttribute(&n_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return MOE_ERR_CUDA;
    launch_topk(LogitsPlain{logits}, corr_bias, T, E, top_k, routed_scale, idx, w, chunk_cnt, n_sms, st);
    launch_dep(scan_kernel, 1, std::max(32, (E + 31) / 32 * 32), 0, st,
               chunk_cnt, nch, E, counts, offsets, chunk_base);
    launch_dep(scatter_kernel, nch, CHUNK_TOKENS, E * (CHUNK_TOKENS / 32) * sizeof(uint32_t), st,
               idx, w, T, E, top_k, chunk_base, pos, row_tok, row_w);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_pack_experts(int32_t E, int32_t d, int32_t I, int32_t elem_bytes, const void* gate,
                            const void* up, const void* down, void* gate_up, void* down_projs,
                            void* stream) {
    if (E < 0 || d < 1 || I < 1 || (elem_bytes != 2 && elem_bytes != 4)) return MOE_ERR_INVALID_ARG;
    if (E > 65535 || (elem_bytes == 2 && (d % 2 != 0 || I % 2 != 0))) return MOE_ERR_UNSUPPORTED;
    if (E == 0 || (gate_up == nullptr && down_projs == nullptr)) return MOE_OK;
    auto word_aligned = [](const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 3u) == 0; };
    if (gate_up != nullptr && (!word_aligned(gate) || !word_aligned(up) || !word_aligned(gate_up)))
        return MOE_ERR_INVALID_ARG;
    if (down_projs != nullptr && (!word_aligned(down) || !word_aligned(down_projs))) return MOE_ERR_INVALID_ARG;
    const size_t n = static_cast<size_t>(E) * d * I * elem_bytes;   // bytes of each HF stack
    const struct { const void* p; size_t n; } ins[] = {{gate, n}, {up, n}, {down, n}};
    for (const auto& in : ins) {
        if (in.p == nullptr) continue;
        if (gate_up != nullptr && overlaps(gate_up, 2 * n, in.p, in.n)) return MOE_ERR_INVALID_ARG;
        if (down_projs != nullptr && overlaps(down_projs, n, in.p, in.n)) return MOE_ERR_INVALID_ARG;
    }
    if (gate_up != nullptr && down_projs != nullptr && overlaps(gate_up, 2 * n, down_projs, n))
        return MOE_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const uint64_t dI = static_cast<uint64_t>(d) * I;
    // out[b][c][col_off + r] = in[b][r][c] over R x C inputs
    auto launch = [&](const void* in, int R, int C, void* out, int out_ld, int col_off) {
        const dim3 grid((C + PACK_TILE - 1) / PACK_TILE, (R + PACK_TILE - 1) / PACK_TILE, E);
        const uint64_t out_bstride = static_cast<uint64_t>(C) * out_ld;
        if (elem_bytes == 2)
            pack_transpose_b16_kernel<<<grid, PACK_THREADS, 0, st>>>(
                static_cast<const uint32_t*>(in), R, C, dI / 2, static_cast<uint32_t*>(out), out_ld, col_off,
                out_bstride / 2);
        else
            pack_transpose_b32_kernel<<<grid, PACK_THREADS, 0, st>>>(
                static_cast<const uint32_t*>(in), R, C, dI, static_cast<uint32_t*>(out), out_ld, col_off,
                out_bstride);
    };
    if (gate_up != nullptr) {
        launch(gate, I, d, gate_up, 2 * I, 0);   // gate_and_up[e][j][i]     = gate[e][i][j]
        launch(up, I, d, gate_up, 2 * I, I);     // gate_and_up[e][j][I + i] = up[e][i][j]
    }
    if (down_projs != nullptr) launch(down, d, I, down_projs, d, 0);   // down_projs[e][i][o] = down[e][o][i]
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

const char* moe_status_string(moe_status s) {
    switch (s) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED: return "unsupported shape or configuration";
        case MOE_ERR_CUDA: return "CUDA error";
        case MOE_ERR_OOM: return "out of device memory";
        case MOE_ERR_TIMEOUT: return "device-side wait timed out";
        case MOE_ERR_RANGE: return "a weighted expert row exceeded the fp16 range of its intermediate";
    }
    return "unknown status";
}

moe_status moe_init(const moe_config* cfg, moe_handle** out) {
    if (!cfg || !out) return MOE_ERR_INVALID_ARG;
    const moe_config c = *cfg;
    const bool dense_only = c.n_experts == 0;
    const bool sizes_ok =
        dense_only ? (c.inter == 0 && c.shared_inter == 0 && c.max_top_k == 0 && c.dense_inter >= 1)
                   : (c.n_experts <= 1024 && c.inter >= 1 && c.shared_inter >= 0 && c.max_top_k >= 1 &&
                      c.max_top_k <= 32 && c.max_top_k <= c.n_experts && c.dense_inter >= 0);
    if (c.max_tokens < 1 || c.hidden < 1 || c.n_experts < 0 || !sizes_ok ||
        (c.dtype != MOE_DTYPE_FP32 && c.dtype != MOE_DTYPE_BF16) || !(c.eps >= 0.0f) ||
        !std::isfinite(c.eps) || c.device < 0 || (c.gemm_path != 0 && c.gemm_path != 1))
        return MOE_ERR_INVALID_ARG;
    const int es = c.dtype == MOE_DTYPE_BF16 ? 2 : 4;
    const int vec = 16 / es;  // 16-byte vectors in RMSNorm, gather and combine
    if (c.hidden % vec != 0 || c.inter % vec != 0 || c.shared_inter % vec != 0 || c.dense_inter % vec != 0)
        return MOE_ERR_UNSUPPORTED;
    const bool tc = c.dtype == MOE_DTYPE_BF16 && c.gemm_path == 0;
    if (tc && (c.hidden % 64 != 0 || c.inter % 64 != 0 || c.shared_inter % 64 != 0 || c.dense_inter % 64 != 0))
        return MOE_ERR_UNSUPPORTED;
    // the CUDA-core contractions stage one input row of fp32 in 48 KB of shared memory
    constexpr int FFMA_MAX_K = 48 * 1024 / 4;
    if (!tc && (c.hidden > FFMA_MAX_K || c.inter > FFMA_MAX_K || c.shared_inter > FFMA_MAX_K ||
                c.dense_inter > FFMA_MAX_K))
        return MOE_ERR_UNSUPPORTED;
    const int64_t P_max = static_cast<int64_t>(c.max_tokens) * c.max_top_k;
    if (P_max > (int64_t(1) << 31) - 1) return MOE_ERR_UNSUPPORTED;

    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || c.device >= ndev) return MOE_ERR_CUDA;
    if (cudaSetDevice(c.device) != cudaSuccess) return MOE_ERR_CUDA;
    if (tc && !encoder()) return MOE_ERR_CUDA;

    moe_handle* h = new (std::nothrow) moe_handle();
    if (!h) return MOE_ERR_OOM;
    h->cfg = c;
    h->es = es;
    h->tc = tc;
    h->P_max = P_max;
    h->n_chunks_max = (c.max_tokens + CHUNK_TOKENS - 1) / CHUNK_TOKENS;
    if (cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, c.device) != cudaSuccess) {
        delete h;
        return MOE_ERR_CUDA;
    }
    const size_t T = c.max_tokens, d = c.hidden, E = c.n_experts, I = c.inter, Is = c.shared_inter;
    const size_t P = P_max, k = c.max_top_k, nch = h->n_chunks_max;
    bool ok = true;
    auto alloc = [&](auto** p, size_t bytes) {
        if (!ok) return;
        void* q = nullptr;
        if (cudaMalloc(&q, std::max<size_t>(bytes, 256)) != cudaSuccess) ok = false;
        *p = static_cast<std::remove_reference_t<decltype(*p)>>(q);
    };
    alloc(&h->xn, T * d * es);
    alloc(&h->logits, T * E * 4);
    // router partials: the split-K choice (ksplit <= SMs / token tiles of BN <= RT_BN_MAX
    // tokens) keeps ksplit * T below T + RT_BN_MAX * (number of SMs)
    alloc(&h->part, (T + static_cast<size_t>(RT_BN_MAX) * h->num_sms) * E * sizeof(float2));
    alloc(&h->topk_idx, T * k * 4);
    alloc(&h->topk_w, T * k * 4);
    alloc(&h->chunk_cnt, nch * E * 4);
    alloc(&h->chunk_base, nch * E * 4);
    alloc(&h->counts, E * 4);
    alloc(&h->offsets, (E + 1) * 4);
    alloc(&h->pos, T * k * 4);
    alloc(&h->row_tok, P * 4);
    alloc(&h->row_w, P * 4);
    alloc(&h->xp, P * d * es);
    alloc(&h->h, P * I * es);
    alloc(&h->yp, P * d * es);
    alloc(&h->hs, T * std::max<size_t>(Is, 1) * es);
    alloc(&h->sh, T * d * (tc ? 4 : es));   // the tensor-core path keeps the shared expert's output in fp32
    if (c.dense_inter > 0) {
        alloc(&h->hd, T * static_cast<size_t>(c.dense_inter) * es);
        if (tc)
            alloc(&h->gpart, static_cast<size_t>(DENSE_GU_SPLIT_MAX) * std::min<size_t>(T, DENSE_SPLIT_MAX_T) * 2 *
                                 static_cast<size_t>(c.dense_inter) * 4);
    }
    // split-K partials of the dense down projection and of the query compression
    if (tc) alloc(&h->dpart, static_cast<size_t>(DENSE_SPLIT_MAX) * std::min<size_t>(T, DENSE_SPLIT_MAX_T) * d * 4);
    if (!dense_only) {   // host-I/O staging of moe_forward_host(_async)
        alloc(&h->x_stage, T * d * es);
        alloc(&h->out_stage, T * d * es);
        alloc(&h->x_stage2, T * d * es);
        alloc(&h->out_stage2, T * d * es);
    }
    alloc(&h->err, 4);
    if (ok && cudaMemset(h->err, 0, 4) != cudaSuccess) ok = false;
    if (!ok) {
        cudaGetLastError();
        free_ws(h);
        delete h;
        return MOE_ERR_OOM;
    }
    bool ev_ok = cudaStreamCreateWithFlags(&h->h2d, cudaStreamNonBlocking) == cudaSuccess &&
                 cudaStreamCreateWithFlags(&h->d2h, cudaStreamNonBlocking) == cudaSuccess;
    for (int i = 0; i < 2 && ev_ok; ++i)
        ev_ok = cudaEventCreateWithFlags(&h->ev_in[i], cudaEventDisableTiming) == cudaSuccess &&
                cudaEventCreateWithFlags(&h->ev_done[i], cudaEventDisableTiming) == cudaSuccess &&
                cudaEventCreateWithFlags(&h->ev_out[i], cudaEventDisableTiming) == cudaSuccess;
    if (!ev_ok) {
        cudaGetLastError();
        moe_destroy(h);
        return MOE_ERR_CUDA;
    }
    *out = h;
    return MOE_OK;
}

moe_status moe_forward(moe_handle* h, int32_t T, const void* x, const void* norm_w,
                       const void* router_w, const float* corr_bias, const void* gate_up,
                       const void* down, const void* shared_gate, const void* shared_up,
                       const void* shared_down, int32_t top_k, float routed_scale, void* out,
                       void* stream) {
    FwdArgs a{T, x, norm_w, router_w, corr_bias, gate_up, down, shared_gate, shared_up,
              shared_down, top_k, routed_scale, out};
    moe_status s = validate_forward(h, a, false);
    if (s != MOE_OK) return s;
    return forward_impl(h, a, static_cast<cudaStream_t>(stream));
}

moe_status moe_dense_forward(moe_handle* h, int32_t T, const void* x, const void* norm_w,
                             const void* gate_w, const void* up_w, const void* down_w,
                             int32_t inter, void* out, void* stream) {
    if (!h) return MOE_ERR_INVALID_ARG;
    const moe_config& c = h->cfg;
    if (T < 0 || T > c.max_tokens || inter < 1 || inter > c.dense_inter) return MOE_ERR_INVALID_ARG;
    if (inter % (h->tc ? 64 : 16 / h->es) != 0) return MOE_ERR_UNSUPPORTED;
    if (T == 0) return MOE_OK;  // nothing is read or written
    const void* ptrs[] = {x, norm_w, gate_w, up_w, down_w, out};
    for (const void* p : ptrs)
        if (p == nullptr || !aligned16(p)) return MOE_ERR_INVALID_ARG;
    const size_t es = h->es, d = c.hidden, Id = inter;
    const size_t out_b = static_cast<size_t>(T) * d * es;
    const struct { const void* p; size_t n; } ins[] = {
        {x, out_b}, {norm_w, d * es}, {gate_w, Id * d * es}, {up_w, Id * d * es}, {down_w, d * Id * es}};
    for (const auto& in : ins)
        if (overlaps(out, out_b, in.p, in.n)) return MOE_ERR_INVALID_ARG;
    if (cudaSetDevice(c.device) != cudaSuccess) return MOE_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return c.dtype == MOE_DTYPE_BF16
               ? dense_impl<__nv_bfloat16>(h, T, x, norm_w, gate_w, up_w, down_w, inter, out, st)
               : dense_impl<float>(h, T, x, norm_w, gate_w, up_w, down_w, inter, out, st);
}

moe_status moe_q_latent(moe_handle* h, int32_t T, int32_t q_rank, const void* hidden, const void* w_qa,
                        const void* q_norm_w, void* c_out, void* q_out, void* stream) {
    if (!h) return MOE_ERR_INVALID_ARG;
    const moe_config& c = h->cfg;
    if (T < 0 || q_rank < 1) return MOE_ERR_INVALID_ARG;
    if (q_rank % (h->tc ? 64 : 16 / h->es) != 0) return MOE_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(T) * std::max(q_rank, c.hidden) > (int64_t(1) << 31) - 1) return MOE_ERR_UNSUPPORTED;
    if (T == 0) return MOE_OK;  // nothing is read or written
    const void* ptrs[] = {hidden, w_qa, q_norm_w, c_out, q_out};
    for (const void* p : ptrs)
        if (p == nullptr || !aligned16(p)) return MOE_ERR_INVALID_ARG;
    const size_t es = h->es, d = c.hidden, R = q_rank;
    const size_t nc = static_cast<size_t>(T) * R * es;
    const struct { const void* p; size_t n; } bufs[] = {
        {hidden, static_cast<size_t>(T) * d * es}, {w_qa, R * d * es}, {q_norm_w, R * es}};
    for (const auto& in : bufs)
        if (overlaps(c_out, nc, in.p, in.n) || overlaps(q_out, nc, in.p, in.n)) return MOE_ERR_INVALID_ARG;
    if (overlaps(c_out, nc, q_out, nc)) return MOE_ERR_INVALID_ARG;
    if (cudaSetDevice(c.device) != cudaSuccess) return MOE_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return c.dtype == MOE_DTYPE_BF16
               ? q_latent_impl<__nv_bfloat16>(h, T, q_rank, hidden, w_qa, q_norm_w, c_out, q_out, st)
               : q_latent_impl<float>(h, T, q_rank, hidden, w_qa, q_norm_w, c_out, q_out, st);
}

moe_status moe_forward_host(moe_handle* h, int32_t T, const void* x_host, const void* norm_w,
                            const void* router_w, const float* corr_bias, const void* gate_up,
                            const void* down, const void* shared_gate, const void* shared_up,
                            const void* shared_down, int32_t top_k, float routed_scale,
                            void* out_host, void* stream) {
    FwdArgs a{T, x_host, norm_w, router_w, corr_bias, gate_up, down, shared_gate, shared_up,
              shared_down, top_k, routed_scale, out_host};
    moe_status s = validate_forward(h, a, true);
    if (s != MOE_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaSetDevice(h->cfg.device) != cudaSuccess) return MOE_ERR_CUDA;
    const size_t bytes = static_cast<size_t>(T) * h->cfg.hidden * h->es;
    if (bytes && cudaMemcpyAsync(h->x_stage, x_host, bytes, cudaMemcpyHostToDevice, st) != cudaSuccess)
        return MOE_ERR_CUDA;
    a.x = h->x_stage;
    a.out = h->out_stage;
    s = forward_impl(h, a, st);
    if (s != MOE_OK) return s;
    if (bytes && cudaMemcpyAsync(out_host, h->out_stage, bytes, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return MOE_ERR_CUDA;
    return moe_sync_status(h, stream);
}

moe_status moe_forward_host_async(moe_handle* h, int32_t T, const void* x_host, const void* norm_w,
                                  const void* router_w, const float* corr_bias, const void* gate_up,
                                  const void* down, const void* shared_gate, const void* shared_up,
                                  const void* shared_down, int32_t top_k, float routed_scale,
                                  void* out_host, void* stream) {
    FwdArgs a{T, x_host, norm_w, router_w, corr_bias, gate_up, down, shared_gate, shared_up,
              shared_down, top_k, routed_scale, out_host};
    moe_status s = validate_forward(h, a, true);
    if (s != MOE_OK) return s;
    if (cudaSetDevice(h->cfg.device) != cudaSuccess) return MOE_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int slot = h->async_slot;
    void* xs = slot == 0 ? h->x_stage : h->x_stage2;
    void* os = slot == 0 ? h->out_stage : h->out_stage2;
    const size_t bytes = static_cast<size_t>(T) * h->cfg.hidden * h->es;
    // H2D once the slot's previous forward has read its input
    if (cudaStreamWaitEvent(h->h2d, h->ev_done[slot], 0) != cudaSuccess ||
        (bytes && cudaMemcpyAsync(xs, x_host, bytes, cudaMemcpyHostToDevice, h->h2d) != cudaSuccess) ||
        cudaEventRecord(h->ev_in[slot], h->h2d) != cudaSuccess)
        return MOE_ERR_CUDA;
    // the forward once its input is in and the slot's previous output copied out
    if (cudaStreamWaitEvent(st, h->ev_in[slot], 0) != cudaSuccess ||
        cudaStreamWaitEvent(st, h->ev_out[slot], 0) != cudaSuccess)
        return MOE_ERR_CUDA;
    a.x = xs;
    a.out = os;
    s = forward_impl(h, a, st);
    if (s != MOE_OK) return s;
    if (cudaEventRecord(h->ev_done[slot], st) != cudaSuccess) return MOE_ERR_CUDA;
    // D2H once the forward is done
    if (cudaStreamWaitEvent(h->d2h, h->ev_done[slot], 0) != cudaSuccess ||
        (bytes && cudaMemcpyAsync(out_host, os, bytes, cudaMemcpyDeviceToHost, h->d2h) != cudaSuccess) ||
        cudaEventRecord(h->ev_out[slot], h->d2h) != cudaSuccess)
        return MOE_ERR_CUDA;
    h->async_slot = slot ^ 1;
    return MOE_OK;
}

moe_status moe_forward_host_wait(moe_handle* h) {
    if (!h) return MOE_ERR_INVALID_ARG;
    if (cudaSetDevice(h->cfg.device) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(h->h2d) != cudaSuccess || cudaStreamSynchronize(h->d2h) != cudaSuccess)
        return MOE_ERR_CUDA;
    return moe_sync_status(h, h->d2h);
}

moe_status moe_get_routing(moe_handle* h, int32_t* idx, float* w, int32_t* counts, void* stream) {
    if (!h) return MOE_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaSetDevice(h->cfg.device) != cudaSuccess) return MOE_ERR_CUDA;
    const size_t pairs = static_cast<size_t>(h->last_T) * h->last_k;
    if (idx && pairs &&
        cudaMemcpyAsync(idx, h->topk_idx, pairs * 4, cudaMemcpyDeviceToDevice, st) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (w && pairs &&
        cudaMemcpyAsync(w, h->topk_w, pairs * 4, cudaMemcpyDeviceToDevice, st) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (counts) {
        cudaError_t e = h->last_T > 0
                            ? cudaMemcpyAsync(counts, h->counts, h->cfg.n_experts * 4,
                                              cudaMemcpyDeviceToDevice, st)
                            : cudaMemsetAsync(counts, 0, h->cfg.n_experts * 4, st);
        if (e != cudaSuccess) return MOE_ERR_CUDA;
    }
    return MOE_OK;
}

moe_status moe_get_intermediate(moe_handle* h, moe_tensor which, void* dst, size_t dst_bytes,
                                void* stream) {
    if (!h || !dst) return MOE_ERR_INVALID_ARG;
    const size_t T = h->last_T, k = h->last_k, d = h->cfg.hidden, E = h->cfg.n_experts;
    const void* src = nullptr;
    size_t bytes = 0;
    switch (which) {
        case MOE_T_XN: src = h->xn; bytes = T * d * h->es; break;
        case MOE_T_LOGITS: src = h->logits; bytes = T * E * 4; break;
        case MOE_T_OFFSETS: src = h->offsets; bytes = (E + 1) * 4; break;
        case MOE_T_POS: src = h->pos; bytes = T * k * 4; break;
        case MOE_T_ROW_TOK: src = h->row_tok; bytes = T * k * 4; break;
        case MOE_T_H: src = h->h; bytes = T * k * h->cfg.inter * h->es; break;
        case MOE_T_YP: src = h->yp; bytes = T * k * d * h->es; break;
        default: return MOE_ERR_INVALID_ARG;
    }
    if (dst_bytes < bytes) return MOE_ERR_INVALID_ARG;
    if (cudaSetDevice(h->cfg.device) != cudaSuccess) return MOE_ERR_CUDA;
    if (bytes && cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice,
                                 static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

moe_status moe_sync_status(moe_handle* h, void* stream) {
    if (!h) return MOE_ERR_INVALID_ARG;
    if (cudaSetDevice(h->cfg.device) != cudaSuccess) return MOE_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
    int flag = 0;
    if (cudaMemcpy(&flag, h->err, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
    if (flag != 0) {
        if (cudaMemset(h->err, 0, 4) != cudaSuccess) return MOE_ERR_CUDA;
        return (flag & DEVERR_TIMEOUT) ? MOE_ERR_TIMEOUT : MOE_ERR_RANGE;
    }
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_selftest_wait_timeout(moe_handle* h, uint32_t timeout_us, void* stream) {
    if (!h || timeout_us < 1 || timeout_us > 1000000) return MOE_ERR_INVALID_ARG;
    if (cudaSetDevice(h->cfg.device) != cudaSuccess) return MOE_ERR_CUDA;
    wait_timeout_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        h->err, static_cast<uint64_t>(timeout_us) * 1000u);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_set_profiling(moe_handle* h, int32_t enable) {
    if (!h) return MOE_ERR_INVALID_ARG;
    if (cudaSetDevice(h->cfg.device) != cudaSuccess) return MOE_ERR_CUDA;
    if (enable && h->ev.empty()) {
        h->ev.resize(static_cast<size_t>(moe_handle::RING) * (moe_handle::NSTAGE + 1));
        for (auto& e : h->ev)
            if (cudaEventCreate(&e) != cudaSuccess) return MOE_ERR_CUDA;
    }
    h->profiling = enable != 0;
    return MOE_OK;
}

moe_status moe_read_stats(moe_handle* h, moe_stats* out) {
    if (!h || !out) return MOE_ERR_INVALID_ARG;
    if (cudaSetDevice(h->cfg.device) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
    while (h->ring_pending > 0)
        if (!fold_oldest(h)) return MOE_ERR_CUDA;
    std::memset(out, 0, sizeof *out);
    out->forwards = h->forwards;
    out->launches = static_cast<int32_t>(h->launches);
    out->n_stages = moe_handle::NSTAGE;
    for (int i = 0; i < moe_handle::NSTAGE; ++i) out->stage_ms[i] = static_cast<float>(h->stage_ms[i]);
    h->forwards = 0;
    h->launches = 0;
    for (double& v : h->stage_ms) v = 0.0;
    return MOE_OK;
}

moe_status moe_destroy(moe_handle* h) {
    if (!h) return MOE_OK;
    cudaSetDevice(h->cfg.device);
    cudaDeviceSynchronize();
    for (auto& e : h->ev) cudaEventDestroy(e);
    for (int i = 0; i < 2; ++i) {
        if (h->ev_in[i]) cudaEventDestroy(h->ev_in[i]);
        if (h->ev_done[i]) cudaEventDestroy(h->ev_done[i]);
        if (h->ev_out[i]) cudaEventDestroy(h->ev_out[i]);
    }
    if (h->h2d) cudaStreamDestroy(h->h2d);
    if (h->d2h) cudaStreamDestroy(h->d2h);
    free_ws(h);
    delete h;
    return MOE_OK;
}

}  // extern "C"
