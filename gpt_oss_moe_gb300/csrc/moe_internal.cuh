// Internal declarations shared by the kernels and the C-ABI host code:
// workspace layout, kernel parameter blocks and launch helpers.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace moe {

constexpr int kRouterTokens = 32;      // tokens per router / permutation block
constexpr int kMaxExperts = 256;
constexpr int kMaxTopK = 8;
constexpr int kBlockK = 64;            // K elements per pipeline stage (128 B of bf16)
constexpr int kWeightTileRows = 128;   // MMA M: weight rows per tile
constexpr int kMaxTokenTile = 256;     // MMA N upper bound

// Status region: word 0 is the device status word (MOE_DEV_* bits),
// word 1 the number of GEMM token tiles written by the permutation kernel.
constexpr int kStatusWord = 0;
constexpr int kNumTilesWord = 1;

struct WsLayout {
    size_t status, topk_ids, topk_w, blk_cnt, offsets, sorted_assign, assign_row;
    size_t tiles, x_perm, h, out_acc, total;
    int max_tiles;
};

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

inline WsLayout ws_layout(long long T, int H, int I, int E, int k) {
    WsLayout L{};
    const size_t R = static_cast<size_t>(T) * k;
    const size_t nb = (static_cast<size_t>(T) + kRouterTokens - 1) / kRouterTokens;
    L.max_tiles = static_cast<int>(R / 16 + (R < static_cast<size_t>(E) ? R : E) + 1);
    size_t o = 0;
    auto take = [&](size_t bytes) {
        size_t at = o;
        o = align_up(o + bytes, 256);
        return at;
    };
    L.status = take(256);
    L.topk_ids = take(R * 4);
    L.topk_w = take(R * 4);
    L.blk_cnt = take(nb * E * 4);
    L.offsets = take((E + 1) * 4);
    L.sorted_assign = take(R * 4);
    L.assign_row = take(R * 4);
    L.tiles = take(static_cast<size_t>(L.max_tiles) * 16);
    L.x_perm = take(R * H * 2);
    L.h = take(R * I * 2);
    L.out_acc = take(static_cast<size_t>(T) * H * 4);
    L.total = o;
    return L;
}

// ------------------------------------------------------------ router (K1)

struct RouterParams {
    const __nv_bfloat16* x;      // [T, H]
    const __nv_bfloat16* wr;     // [E, H]
    const __nv_bfloat16* br;     // [E]
    int T, H, E, top_k;
    int32_t* topk_ids;           // [T, k]
    float* topk_w;               // [T, k]
    int32_t* blk_cnt;            // [nblocks, E]
    float* zero_out;             // [T, H] fp32 rows to clear, or null
    int32_t* status;
};

// ------------------------------------------------------------ permutation (K2)

struct PermuteParams {
    const int32_t* topk_ids;     // [T, k]
    const int32_t* blk_cnt;      // [nblocks, E]
    const __nv_bfloat16* x;      // [T, H]
    int T, H, E, top_k, nblocks;
    int token_tile;              // rows of tokens per GEMM tile
    int32_t* offsets;            // [E+1]
    int32_t* sorted_assign;      // [T*k]
    int32_t* assign_row;         // [T*k]
    int4* tiles;                 // (expert, first row, rows, 0)
    int max_tiles;
    __nv_bfloat16* x_perm;       // [T*k, H] or null (no gather)
    int32_t* status;
};

// ------------------------------------------------------------ grouped GEMM

enum EpilogueKind { kEpiGlu = 0, kEpiCombine = 1 };

struct GemmParams {
    const int4* tiles;           // token tiles from the permutation kernel
    const int32_t* num_tiles;    // device count of tiles
    int n_wblocks;               // weight-row blocks of 128 per expert
    int k_blocks;                // K / 64
    int w_rows;                  // weight rows per expert (2I or H)
    int token_box;               // token rows per TMA box (= MMA N bound)
    int stages;
    int tmem_cols;               // allocated TMEM columns (2 accumulators)
    int num_experts;             // E (tile bounds check)
    int rows_total;              // T * k (tile bounds check)
    const __nv_bfloat16* bias;   // [E, w_rows]
    // kEpiGlu: h[row, w_rows/2] bf16
    __nv_bfloat16* h;
    // kEpiCombine: out[t, w_rows] += w * y
    float* out;
    const int32_t* sorted_assign;
    const float* topk_w;
    int top_k;
    int32_t* status;
};

// Shared memory used by one GEMM CTA (bytes, excluding the 1 KB alignment slack).
inline size_t gemm_smem_bytes(int stages, int token_box) {
    size_t a = static_cast<size_t>(kWeightTileRows) * kBlockK * 2;
    size_t b = static_cast<size_t>(token_box) * kBlockK * 2;
    size_t meta = static_cast<size_t>(token_box) * 8;
    size_t bars = 256;
    return stages * (a + b) + meta + bars;
}

// Kernel launchers (defined next to each kernel).
cudaError_t launch_router(const RouterParams& p, cudaStream_t s);
cudaError_t launch_permute(const PermuteParams& p, cudaStream_t s, bool pdl);
cudaError_t launch_gemm(int epi, const GemmParams& p, const CUtensorMap* tmap_w,
                        const CUtensorMap* tmap_x, int grid, size_t smem,
                        cudaStream_t s, bool pdl);
cudaError_t launch_to_bf16(const float* in, __nv_bfloat16* out, size_t n, cudaStream_t s,
                           bool pdl);

}  // namespace moe
