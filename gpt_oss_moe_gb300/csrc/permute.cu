// Expert permutation on the device, with no host synchronisation (xserv
// docs/19-gpt-oss-moe.md, "Phase 19: gpt-oss-20b", §2 "MoE 前向": topk_ids
// stay on the GPU and the host never waits for them).
//
// The T*k assignments a = t*k + j are placed in rows sorted by
// (expert, a) ascending -- a stable counting sort.  The router kernel already
// counted, per block of 32 tokens, how many assignments go to each expert
// (blk_cnt[b][e]).  Block b of this kernel (the same 32 tokens):
//   1. sums blk_cnt over all blocks (per-expert totals) and over the blocks
//      before b (its per-expert base inside each expert's segment);
//   2. scans the totals into expert offsets;
//   3. ranks its own assignments per expert in order of a (warp match), so
//      row(a) = offsets[e] + base_b[e] + rank;
//   4. copies the activation row of each assignment into x_perm[row], the
//      contiguous per-expert operand of the gate_up GEMM.
// Block 0 also writes the expert offsets and the GEMM token-tile list
// (expert, first row, rows), each expert's rows split into near-equal tiles
// of at most token_tile rows whose sizes are multiples of 16 except the last.
#include "moe_internal.cuh"
#include "ptx.cuh"
#include "../../include/moe.h"

namespace moe {
namespace {

constexpr int kThreads = 256;

// Exclusive scan of vals[0..n) (n <= 256) by warp 0; writes out[0..n] with
// out[n] = total.  Caller synchronises before and after.
__device__ __forceinline__ void warp0_exclusive_scan(const int* vals, int* out, int n) {
    const int lane = threadIdx.x & 31;
    int local[8];
    int sum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int idx = lane * 8 + i;
        local[i] = idx < n ? vals[idx] : 0;
        sum += local[i];
    }
    int incl = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
    }
    int run = incl - sum;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int idx = lane * 8 + i;
        if (idx < n) out[idx] = run;
        run += local[i];
    }
    const int all = __shfl_sync(0xffffffffu, incl, 31);
    if (lane == 0) out[n] = all;
}

__global__ void __launch_bounds__(kThreads) permute_kernel(const PermuteParams p) {
    __shared__ int total[kMaxExperts];
    __shared__ int offs[kMaxExperts + 1];
    __shared__ int base[kMaxExperts];
    __shared__ int running[kMaxExperts];
    __shared__ int tcount[kMaxExperts];
    __shared__ int toff[kMaxExperts + 1];
    __shared__ int rows_s[kRouterTokens * kMaxTopK];

    pdl_wait();                 // routing results of the previous kernel
    pdl_launch_dependents();    // the GEMM may start its prologue

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int E = p.E, k = p.top_k, b = blockIdx.x;

    if (tid < E) {
        int pre = 0, tot = 0;
        for (int bb = 0; bb < p.nblocks; ++bb) {
            const int c = p.blk_cnt[static_cast<size_t>(bb) * E + tid];
            pre += bb < b ? c : 0;
            tot += c;
        }
        total[tid] = tot;
        base[tid] = pre;
        running[tid] = 0;
    }
    __syncthreads();
    if (warp == 0) warp0_exclusive_scan(total, offs, E);
    __syncthreads();
    if (tid < E) base[tid] += offs[tid];

    if (b == 0) {
        // expert offsets and the token-tile list
        if (tid <= E) p.offsets[tid] = offs[tid];
        if (tid < E) tcount[tid] = (total[tid] + p.token_tile - 1) / p.token_tile;
        __syncthreads();
        if (warp == 0) warp0_exclusive_scan(tcount, toff, E);
        __syncthreads();
        if (tid < E && total[tid] > 0) {
            const int m = total[tid], nt = tcount[tid];
            const int per = ((m + nt - 1) / nt + 15) / 16 * 16;
            for (int i = 0; i < nt; ++i) {
                const int slot = toff[tid] + i;
                if (slot < p.max_tiles) {
                    p.tiles[slot] = make_int4(tid, offs[tid] + i * per, min(per, m - i * per), 0);
                } else {
                    atomicOr(p.status + kStatusWord, MOE_DEV_BAD_TILE);
                }
            }
        }
        if (tid == 0) p.status[kNumTilesWord] = min(toff[E], p.max_tiles);
    }
    __syncthreads();

    // Stable ranks of this block's assignments (warp 0, 32 at a time).
    const int a0 = b * kRouterTokens * k;
    const int a1 = min(p.T, (b + 1) * kRouterTokens) * k;
    if (warp == 0) {
        for (int ab = a0; ab < a1; ab += 32) {
            const int a = ab + lane;
            const bool valid = a < a1;
            int e = valid ? p.topk_ids[a] : -1;
            const bool good = valid && e >= 0 && e < E;
            if (valid && !good) {
                atomicOr(p.status + kStatusWord, MOE_DEV_BAD_EXPERT_ID);
            }
            if (!good) e = -1 - lane;   // unique per lane: never matches a real expert
            const unsigned peers = __match_any_sync(0xffffffffu, e);
            const int rank = __popc(peers & ((1u << lane) - 1u));
            const int r0 = good ? running[e] : 0;
            __syncwarp();
            if (good && rank == 0) running[e] = r0 + __popc(peers);
            __syncwarp();
            const int row = good ? base[e] + r0 + rank : -1;
            if (valid) {
                if (good) p.sorted_assign[row] = a;
                p.assign_row[a] = row;
                rows_s[a - a0] = row;
            }
        }
    }
    __syncthreads();

    // Gather the activation rows: x_perm[row(a)] = x[a / k].
    if (p.x_perm) {
        const int n = a1 - a0;
        const int vec_per_row = p.H / 8;
        const int total_vec = n * vec_per_row;
        for (int i = tid; i < total_vec; i += kThreads) {
            const int la = i / vec_per_row, v = i - la * vec_per_row;
            const int row = rows_s[la];
            if (row < 0) continue;
            const int t = (a0 + la) / k;
            const uint4 val = reinterpret_cast<const uint4*>(p.x + static_cast<size_t>(t) * p.H)[v];
            reinterpret_cast<uint4*>(p.x_perm + static_cast<size_t>(row) * p.H)[v] = val;
        }
    }
}

}  // namespace

cudaError_t launch_permute(const PermuteParams& p, cudaStream_t s, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.nblocks);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, permute_kernel, p);
}

}  // namespace moe
