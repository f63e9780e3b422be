// Packing of HF per-expert nn.Linear weights into the grouped native layout
// (NeMo AutoModel GLM4-MoE state dict adapter page, Glm4MoeStateDictAdapter:
// experts.{E}.gate_proj / up_proj / down_proj -> gate_and_up_projs
// [n_experts, dim, 2*moe_inter_dim] and down_projs [n_experts,
// moe_inter_dim, dim]).  Each output is a batched transpose written at a
// column offset of a wider row:
//   out[b][c][col_off + r] = in[b][r][c],  r < R, c < C.
// HBM-bound: one read and one write of every element, both through 128-byte
// coalesced rows, the transpose done in shared memory.
#pragma once
#include <cstdint>

namespace moe {

constexpr int PACK_TILE = 64;       // elements per tile side
constexpr int PACK_THREADS = 256;

// 2-byte elements, handled as 32-bit words.  A thread loads one word (two
// elements of a row) from each of two consecutive rows and transposes the
// 2 x 2 block with byte permutes; the two words it gets are two elements of
// two consecutive output rows.  The shared-memory tile holds the output
// rows as words, each row rotated by its row-pair index so that both the
// stores (one word per output row pair) and the row reads hit 32 banks.
// R, C, out_ld and col_off are even (whole words).
__global__ void __launch_bounds__(PACK_THREADS) pack_transpose_b16_kernel(
    const uint32_t* __restrict__ in, int R, int C, uint64_t in_bstride_w, uint32_t* __restrict__ out,
    int out_ld, int col_off, uint64_t out_bstride_w) {
    __shared__ uint32_t S[PACK_TILE][PACK_TILE / 2];
    const int r0 = blockIdx.y * PACK_TILE, c0 = blockIdx.x * PACK_TILE;
    const int Cw = C >> 1, ldw = out_ld >> 1, Rw = R >> 1;
    const uint32_t* src = in + blockIdx.z * in_bstride_w;
    uint32_t* dst = out + blockIdx.z * out_bstride_w;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int cw = (c0 >> 1) + lane;    // input word column: elements c0 + 2 lane, + 1
#pragma unroll
    for (int i = 0; i < PACK_TILE / 2 / (PACK_THREADS / 32); ++i) {
        const int rp = wid + (PACK_THREADS / 32) * i;   // row pair inside the tile
        const int r = r0 + 2 * rp;
        uint32_t w0 = 0, w1 = 0;
        if (cw < Cw && r < R) {
            w0 = src[static_cast<uint64_t>(r) * Cw + cw];
            w1 = src[static_cast<uint64_t>(r + 1) * Cw + cw];   // R is even: r + 1 < R
        }
        const int col = (rp + lane) & 31;
        S[2 * lane][col] = __byte_perm(w0, w1, 0x5410);       // (in[r][c], in[r+1][c])
        S[2 * lane + 1][col] = __byte_perm(w0, w1, 0x7632);   // (in[r][c+1], in[r+1][c+1])
    }
    __syncthreads();
    const int rw = (r0 >> 1) + lane;    // output word: elements r0 + 2 lane, + 1
#pragma unroll
    for (int j = 0; j < PACK_TILE / (PACK_THREADS / 32); ++j) {
        const int cc = wid + (PACK_THREADS / 32) * j;   // output row inside the tile
        const int c = c0 + cc;
        if (c < C && rw < Rw)
            dst[static_cast<uint64_t>(c) * ldw + (col_off >> 1) + rw] = S[cc][(lane + (cc >> 1)) & 31];
    }
}

// 4-byte elements: a 64 x 64 tile with one word of padding per row.
__global__ void __launch_bounds__(PACK_THREADS) pack_transpose_b32_kernel(
    const uint32_t* __restrict__ in, int R, int C, uint64_t in_bstride, uint32_t* __restrict__ out,
    int out_ld, int col_off, uint64_t out_bstride) {
    __shared__ uint32_t S[PACK_TILE][PACK_TILE + 1];
    const int r0 = blockIdx.y * PACK_TILE, c0 = blockIdx.x * PACK_TILE;
    const uint32_t* src = in + blockIdx.z * in_bstride;
    uint32_t* dst = out + blockIdx.z * out_bstride;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    for (int i = wid; i < PACK_TILE * 2; i += PACK_THREADS / 32) {
        const int rr = i >> 1, cc = (i & 1) * 32 + lane;
        if (r0 + rr < R && c0 + cc < C) S[rr][cc] = src[static_cast<uint64_t>(r0 + rr) * C + c0 + cc];
    }
    __syncthreads();
    for (int i = wid; i < PACK_TILE * 2; i += PACK_THREADS / 32) {
        const int cc = i >> 1, rr = (i & 1) * 32 + lane;
        if (r0 + rr < R && c0 + cc < C)
            dst[static_cast<uint64_t>(c0 + cc) * out_ld + col_off + r0 + rr] = S[rr][cc];
    }
}

}  // namespace moe
