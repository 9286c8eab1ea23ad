// Router Linear + bias, top-k selection and softmax over the selected logits,
// the per-expert counts and the expert offsets / GEMM tile list, in one
// launch (xserv docs/19-gpt-oss-moe.md, "Phase 19: gpt-oss-20b": §1 table
// "MoE" row -- the router is a plain Linear [2880 -> 32] with bias; §2
// "MoE 前向" -- router GEMV then topk_softmax on the GPU, ids stay there).
//
// Grid (token blocks of 32, expert groups of 32, K slices).  CTA (b, g, q)
// computes the logits of tokens [32b, 32b+32) for experts [32g, 32g+32) over
// the q-th slice of the hidden dimension, as an fp32-accumulated bf16
// contraction on the tensor cores (mma.sync m16n8k16; the router is ~0.1% of
// the layer's flops, far too small for a TMEM pipeline).  A producer warp
// streams 64-wide K chunks of x and Wr through a TMA ring (128-byte
// swizzle); each of the four compute warps owns every fourth chunk, so four
// independent MMA chains run at once, and their partial sums are added in
// warp order.  Slicing K spreads a small batch's loads over many SMs (one
// CTA streams only ~40 GB/s).
// Results are merged by atomic tickets -- no CTA ever waits for another:
//   * the last K slice of (b, g) to finish adds the slices' partials in
//     slice order (the same order every run);
//   * with more than one expert group, the last group of block b gathers the
//     block's full logit rows;
//   * that CTA selects the top k per token -- one lane per token: each
//     compute warp scans a quarter of the experts into per-lane sorted
//     lists (strict > so equal logits keep the lower expert index), warp 0
//     merges the four lists in expert order -- computes the softmax over the
//     k selected logits (max-subtracted, expf) and counts the assignments
//     per expert, storing the block's counts and adding them to per-expert
//     totals;
//   * the last token block scans the totals into expert offsets and writes
//     the GEMM token-tile list.
// Every ticket counter (and the totals) is reset by the CTA that takes the
// last ticket, so the counters are zero between calls.
//
// Tails: rows past T and experts past E are zero-filled by TMA and masked
// out of the selection; a CTA leaves early only as a whole, right after a
// barrier (the failure mode of §4).  Every wait is bounded.
#include <cfloat>
#include <climits>

#include "moe_internal.cuh"
#include "ptx.cuh"
#include "trace.cuh"
#include "../../include/moe.h"

namespace moe {
namespace {

MOE_TRACE_ARRAY(g_trace_router, 1);

constexpr int kComputeWarps = 4;
constexpr int kThreads = (kComputeWarps + 1) * 32;   // + one producer warp
// Ring depth: a multiple of kComputeWarps, so chunk c and chunk c + S (same
// slot) always belong to the same compute warp.  Each slot then has a single
// consumer that takes its phases in order, and a parity wait can never be
// satisfied by a phase two behind.  One CTA streams ~40 GB/s, so 8 x 8 KB in
// flight covers the latency.
constexpr int kMaxStages = 8;
constexpr int kGroup = 32;                            // experts per CTA
constexpr uint32_t kTileBytes = kRouterTokens * kBlockK * 2;   // 4 KB (x or w tile)
constexpr uint32_t kStageBytes = 2 * kTileBytes;
constexpr int kPartStride = kGroup + 1;                // padded row of partial logits
// logits of the top-k CTA: [32][E + 1] floats, E <= 256
constexpr uint32_t kLogitsBytes = kRouterTokens * (kMaxExperts + 1) * 4;
constexpr uint32_t kPartialBytes = kComputeWarps * kRouterTokens * kPartStride * 4;

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                            uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4],
                                               uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Byte offset of the 16-byte chunk `c` (0..7) of row `r` in a tile written
// by TMA with the 128-byte swizzle (rows of 128 B, 1024-byte aligned tile).
__device__ __forceinline__ uint32_t swz(int r, int c) {
    return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ int warp_inclusive_scan(int v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += o;
    }
    return v;
}

// Exclusive scan of vals[0..n) (n <= 256) by one warp; out[0..n] with
// out[n] = total.
__device__ __forceinline__ void warp_exclusive_scan256(const int* vals, int* out, int n) {
    const int lane = threadIdx.x & 31;
    int local[8];
    int sum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int idx = lane * 8 + i;
        local[i] = idx < n ? vals[idx] : 0;
        sum += local[i];
    }
    const int incl = warp_inclusive_scan(sum);
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

// Inserts (v, e) into a top-K list sorted by value, descending.  Candidates
// arrive in increasing expert order, and an equal value never displaces an
// entry (strict >), so equal logits keep the lower expert index first.
template <int K>
__device__ __forceinline__ void topk_insert(float (&bv)[K], int (&be)[K], float v, int e) {
#pragma unroll
    for (int s = K - 1; s > 0; --s) {
        if (v > bv[s - 1]) {
            bv[s] = bv[s - 1];
            be[s] = be[s - 1];
        } else if (v > bv[s]) {
            bv[s] = v;
            be[s] = e;
        }
    }
    if (v > bv[0]) {
        bv[0] = v;
        be[0] = e;
    }
}

// Top-K selection and softmax for the token block, one lane per token.
// Compute warp w scans experts [wE/4, (w+1)E/4) of all 32 tokens (logit +
// bias; NaN counts as the lowest value) into a per-lane list; warp 0 then
// merges the four lists in warp order -- lower expert ranges first, each list
// in rank order -- so ties still resolve to the lower expert index.  The
// softmax runs over the K selected logits, max-subtracted, summed in rank
// order.  cand: [kComputeWarps][32][K] values then indices (scratch smem).
template <int K>
__device__ void topk_block(const RouterParams& p, const float* logits, int ls, const float* bias_s,
                           float* cand, int t0, int* hist, int* ids_s) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = p.E;
    float* cv = cand;
    int* ce = reinterpret_cast<int*>(cand + kComputeWarps * kRouterTokens * K);
    if (warp < kComputeWarps) {
        float bv[K];
        int be[K];
#pragma unroll
        for (int s = 0; s < K; ++s) {
            bv[s] = -INFINITY;
            be[s] = INT_MAX;
        }
        const int e_lo = E * warp / kComputeWarps, e_hi = E * (warp + 1) / kComputeWarps;
        const float* row = logits + lane * ls;
        for (int e = e_lo; e < e_hi; ++e) {
            float v = row[e] + bias_s[e];
            if (!(v == v)) v = -FLT_MAX;
            topk_insert<K>(bv, be, v, e);
        }
#pragma unroll
        for (int s = 0; s < K; ++s) {
            cv[(warp * kRouterTokens + lane) * K + s] = bv[s];
            ce[(warp * kRouterTokens + lane) * K + s] = be[s];
        }
    }
    __syncthreads();
    if (warp != 0) return;
    float bv[K];
    int be[K];
#pragma unroll
    for (int s = 0; s < K; ++s) {
        bv[s] = -INFINITY;
        be[s] = INT_MAX;
    }
    for (int w = 0; w < kComputeWarps; ++w) {
#pragma unroll
        for (int s = 0; s < K; ++s) {
            const int e = ce[(w * kRouterTokens + lane) * K + s];
            if (e != INT_MAX) topk_insert<K>(bv, be, cv[(w * kRouterTokens + lane) * K + s], e);
        }
    }
    const int t = t0 + lane;
    if (t >= p.T) return;
    float ex[K];
    float denom = 0.f;
#pragma unroll
    for (int s = 0; s < K; ++s) {
        ex[s] = expf(bv[s] - bv[0]);
        denom += ex[s];
    }
#pragma unroll
    for (int s = 0; s < K; ++s) {
        // test fault (inject & 1): token 0's first id is written out of range
        // after it was counted, as a corrupted id would arrive
        const bool bad = (p.inject & 1) && t == 0 && s == 0 && p.E < kMaxExperts;
        p.topk_ids[static_cast<size_t>(t) * K + s] = bad ? p.E : be[s];
        // (small batches: kept for the permutation made by the last CTA)
        if (p.small_perm) ids_s[t * K + s] = bad ? p.E : be[s];
        p.topk_w[static_cast<size_t>(t) * K + s] = ex[s] / denom;
        atomicAdd(&hist[be[s]], 1);
    }
}

// Top-K selection and softmax for a block of at most kThreads / 32 valid
// tokens, one warp per token: lane l holds experts l, l + 32, ...; each of
// the K rounds takes the warp's best remaining (logit descending, expert
// ascending, NaN as the lowest value), so the selection, its order and the
// softmax are those of topk_block.  With few tokens this is a few dozen
// dependent instructions instead of a scan over every expert by one lane.
template <int K>
__device__ void topk_warp(const RouterParams& p, const float* logits, int ls, const float* bias_s,
                          int t0, int n_valid, int* hist, int* ids_s) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp >= n_valid) return;
    const int E = p.E;
    constexpr int kPerLane = kMaxExperts / 32;
    float v[kPerLane];
    const float* row = logits + warp * ls;
#pragma unroll
    for (int j = 0; j < kPerLane; ++j) {
        const int e = lane + 32 * j;
        float x = -INFINITY;                 // not an expert: never selected
        if (e < E) {
            x = row[e] + bias_s[e];
            if (!(x == x)) x = -FLT_MAX;
        }
        v[j] = x;
    }
    float bv[K];
    int be[K];
#pragma unroll
    for (int s = 0; s < K; ++s) {
        // this lane's best remaining candidate (lower expert first on ties)
        float mv = -INFINITY;
        int me = INT_MAX;
#pragma unroll
        for (int j = 0; j < kPerLane; ++j)
            if (v[j] > mv) {
                mv = v[j];
                me = lane + 32 * j;
            }
        // the warp's best
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, mv, d);
            const int oe = __shfl_xor_sync(0xffffffffu, me, d);
            if (ov > mv || (ov == mv && oe < me)) {
                mv = ov;
                me = oe;
            }
        }
        bv[s] = mv;
        be[s] = me;
        // the winner's lane retires it
#pragma unroll
        for (int j = 0; j < kPerLane; ++j)
            if (lane + 32 * j == me) v[j] = -INFINITY;
    }
    if (lane != 0) return;
    const int t = t0 + warp;
    float ex[K];
    float denom = 0.f;
#pragma unroll
    for (int s = 0; s < K; ++s) {
        ex[s] = expf(bv[s] - bv[0]);
        denom += ex[s];
    }
#pragma unroll
    for (int s = 0; s < K; ++s) {
        // test fault (inject & 1): as in topk_block
        const bool bad = (p.inject & 1) && t == 0 && s == 0 && p.E < kMaxExperts;
        p.topk_ids[static_cast<size_t>(t) * K + s] = bad ? p.E : be[s];
        // (small batches: kept for the permutation made by the last CTA)
        if (p.small_perm) ids_s[t * K + s] = bad ? p.E : be[s];
        p.topk_w[static_cast<size_t>(t) * K + s] = ex[s] / denom;
        atomicAdd(&hist[be[s]], 1);
    }
}

// Last CTA of the grid: expert totals (summed by every token block's
// atomics; with a single token block, that block's own counts, already in
// total_s), expert offsets, GEMM token tiles.  The per-block prefixes that
// place each block's rows are left to the permutation kernel, whose CTAs
// sum the earlier blocks' counts in parallel: done here by one CTA, that
// scan took 14 us at T = 4096 and 37 us at E = 128, T = 8192.
// ids_s: the routed ids of all tokens (small_perm; this block's already
// there, the others' loaded here).
template <int kNT = kThreads>
__device__ void finish_routing(const RouterParams& p, int* total_s, int* offs_s, int* tcnt_s,
                               int* toff_s, int* ids_s) {
    constexpr int kThreads = kNT;              // the calling kernel's block size
    const int tid = threadIdx.x, warp = tid >> 5;
    const int E = p.E;
    if (p.nblocks > 1) {
        int32_t* totals = p.counters + kExpertTotalsOffset;
        for (int e = tid; e < E; e += kThreads) {
            total_s[e] = __ldcg(totals + e);
            totals[e] = 0;   // zero for the next call
        }
    }
    __syncthreads();
    if (warp == 0) warp_exclusive_scan256(total_s, offs_s, E);
    __syncthreads();
    for (int e = tid; e <= E; e += kThreads) p.offsets[e] = offs_s[e];
    // token tiles of the local experts only (expert-parallel form)
    for (int e = tid; e < E; e += kThreads)
        tcnt_s[e] = e >= p.ex_lo && e < p.ex_lo + p.ex_n
                        ? (total_s[e] + p.token_tile - 1) / p.token_tile : 0;
    __syncthreads();
    if (warp == 0) warp_exclusive_scan256(tcnt_s, toff_s, E);
    __syncthreads();
    for (int e = tid; e < E; e += kThreads) {
        const int m = total_s[e];
        const int nt = tcnt_s[e];
        if (m == 0 || nt == 0) continue;
        const int per = ((m + nt - 1) / nt + 15) / 16 * 16;
        for (int i = 0; i < nt; ++i) {
            const int slot = toff_s[e] + i;
            if (slot < p.max_tiles &&
                MOE_BOUNDS(offs_s[e] + i * per + min(per, m - i * per) <= p.T * p.top_k,
                           p.status + kStatusWord))
                p.tiles[slot] =
                    make_int4(e - p.ex_lo, offs_s[e] + i * per, min(per, m - i * per), 0);
            else
                atomicOr(p.status + kStatusWord, MOE_DEV_BAD_TILE);
        }
    }
    // test fault (inject & 2): the first tile names an expert the GEMMs do
    // not hold
    __syncthreads();
    if (tid == 0) {
        if ((p.inject & 2) && toff_s[E] > 0) p.tiles[0] = make_int4(p.ex_n, 0, 1, 0);
        p.status[kNumTilesWord] = min(toff_s[E], p.max_tiles);
        p.status[kGridCounterWord] = 0;   // ready for the next call
    }
    if (p.small_perm) {
        // Small batches: the stable permutation is made here (the
        // permutation kernel is not launched).  Rows are sorted by (expert,
        // a): warp 0 ranks 32 assignments at a time against a running count
        // per expert, as the permutation kernel does per token block.  The
        // ids come from shared memory: this block's own (ids_s, kept by the
        // top-k), the other token blocks' loaded from global memory by every
        // thread at once (their writes were made visible before the ticket
        // that chose this CTA).
        int* running = tcnt_s;                 // free now
        const int R = p.T * p.top_k;
        // this CTA's token block (the last to finish, not necessarily the
        // last block) holds assignments [own0, own1)
        const int own0 = static_cast<int>(blockIdx.x) * kRouterTokens * p.top_k;
        const int own1 = min(R, own0 + kRouterTokens * p.top_k);
        for (int e = tid; e < E; e += kThreads) running[e] = 0;
        for (int a = tid; a < R; a += kThreads)
            if (a < own0 || a >= own1) ids_s[a] = __ldcg(p.topk_ids + a);
        __syncthreads();
        if (warp == 0) {
            const int lane = tid & 31;
            for (int ab = 0; ab < R; ab += 32) {
                const int a = ab + lane;
                const bool valid = a < R;
                int e = valid ? ids_s[a] : -1;
                const bool good = valid && e >= 0 && e < E;
                if (valid && !good) atomicOr(p.status + kStatusWord, MOE_DEV_BAD_EXPERT_ID);
                if (!good) e = -1 - lane;       // unique per lane: never a real expert
                const unsigned peers = __match_any_sync(0xffffffffu, e);
                const int rank = __popc(peers & ((1u << lane) - 1u));
                const int r0 = good ? running[e] : 0;
                __syncwarp();
                if (good && rank == 0) running[e] = r0 + __popc(peers);
                __syncwarp();
                int row = good ? offs_s[e] + r0 + rank : -1;
                if (good && (row < 0 || row >= R)) {
                    atomicOr(p.status + kStatusWord, MOE_DEV_BAD_TILE);
                    row = -1;
                }
                if (valid) {
                    if (row >= 0) p.sorted_assign[row] = a;
                    p.assign_row[a] = row;
                }
            }
        }
    }
}

__global__ void __launch_bounds__(kThreads)
    router_topk_kernel(const RouterParams p, const __grid_constant__ CUtensorMap tmap_x,
                       const __grid_constant__ CUtensorMap tmap_wr) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int S = p.stages;
    const size_t ring_bytes = static_cast<size_t>(S) * kStageBytes;
    const size_t region = ring_bytes > kLogitsBytes ? ring_bytes : kLogitsBytes;
    uint8_t* ring = smem;                                                   // [S][x | w]
    float* logits = reinterpret_cast<float*>(smem);                         // after the loop
    float* partial = reinterpret_cast<float*>(smem + region);               // [4][32][33]
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + region + kPartialBytes);
    uint64_t* empty = full + kMaxStages;
    int* hist = reinterpret_cast<int*>(empty + kMaxStages);                 // [256]
    int* scan_a = hist + kMaxExperts;                                       // [257]
    int* scan_b = scan_a + kMaxExperts + 1;                                 // [256]
    int* scan_c = scan_b + kMaxExperts;                                     // [257]
    volatile int* flag = scan_c + kMaxExperts + 1;                          // [4]
    float* bias_s = reinterpret_cast<float*>(scan_c + kMaxExperts + 5);      // [256]
    int* ids_s = reinterpret_cast<int*>(bias_s + kMaxExperts);              // [256] (small_perm)

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = blockIdx.x, g = blockIdx.y, q = blockIdx.z;
    const int t0 = b * kRouterTokens;
    const int E = p.E;
    const int nchunks = p.H / kBlockK;
    const int per = (nchunks + p.ksplit - 1) / p.ksplit;
    const int c_begin = q * per;
    const int nc = min(nchunks, c_begin + per) - c_begin;   // chunks of this slice

    // Inputs, workspace and counters may be written by the kernel launched
    // before this one (a previous call's last kernel, or the caller's): wait
    // for it before the first global access.  The permutation kernel may
    // launch now: it waits for this grid to complete.
    const int trace_cta = (b * p.egroups + g) * p.ksplit + q;
    if (tid == 0) MOE_TRACE_POINT(g_trace_router, 0, trace_cta, 0);
    pdl_wait();
    pdl_launch_dependents();
    if (tid == 0) MOE_TRACE_POINT(g_trace_router, 0, trace_cta, 1);
    // a slot would be shared by two consumer warps: refuse (the host never
    // asks for this); the CTA still takes part in its cluster's barriers
    const bool bad_cfg = nc > S && S % kComputeWarps != 0;
    if (bad_cfg && tid == 0) atomicOr(p.status + kStatusWord, MOE_DEV_BAD_TILE);
    for (int e = tid; e < kMaxExperts; e += kThreads) {
        hist[e] = 0;
        bias_s[e] = e < E ? __bfloat162float(p.br[e]) : 0.f;
    }
    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(full + s), 1);
            mbar_init(smem_u32(empty + s), 1);
        }
        flag[0] = bad_cfg ? 1 : 0;
        flag[1] = 0;
        flag[2] = 0;
        flag[3] = 0;
        mbar_fence_init();
    }
    __syncthreads();

    float acc[2][4][4];
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[m][j][r] = 0.f;

    if (bad_cfg) {
        // nothing loaded or computed
    } else if (warp == kComputeWarps) {
        // ---------------- producer: one lane issues every chunk's two loads
        if (lane == 0) {
            tma_prefetch_desc(&tmap_x);
            tma_prefetch_desc(&tmap_wr);
            const uint64_t pol_x = policy_evict_first();
            const uint64_t pol_w = policy_evict_last();
            int issued = 0;
            for (; issued < nc; ++issued) {
                const int c = issued, s = c % S;
                if (c >= S &&
                    !mbar_wait(smem_u32(empty + s), static_cast<uint32_t>(c / S - 1) & 1u, flag)) {
                    flag[0] = 1;
                    break;
                }
                const uint32_t bar = smem_u32(full + s);
                uint8_t* st = ring + static_cast<size_t>(s) * kStageBytes;
                const int k0 = (c_begin + c) * kBlockK;
                mbar_arrive_expect_tx(bar, kStageBytes);
                tma_load_2d(smem_u32(st), &tmap_x, bar, k0, t0, pol_x);
                tma_load_2d(smem_u32(st + kTileBytes), &tmap_wr, bar, k0, g * kGroup, pol_w);
            }
            // Every issued load must land before the CTA may leave (bounded).
            for (int c = issued - S > 0 ? issued - S : 0; c < issued; ++c)
                mbar_wait(smem_u32(full + c % S), static_cast<uint32_t>(c / S) & 1u, nullptr);
        }
    } else {
        // ---------------- compute warp w: chunks w, w+4, w+8, ... of the slice
        for (int c = warp; c < nc; c += kComputeWarps) {
            const int s = c % S;
            if (!mbar_wait(smem_u32(full + s), static_cast<uint32_t>(c / S) & 1u, flag)) {
                flag[0] = 1;
                break;
            }
            const uint8_t* xs = ring + static_cast<size_t>(s) * kStageBytes;
            const uint8_t* ws = xs + kTileBytes;
#pragma unroll
            for (int ks = 0; ks < kBlockK / 16; ++ks) {
                uint32_t a[2][4], bw[4][2];
                const int mi = lane >> 3, r = lane & 7;
#pragma unroll
                for (int m = 0; m < 2; ++m)
                    ldmatrix_x4(smem_u32(xs + swz(m * 16 + (mi & 1) * 8 + r, ks * 2 + (mi >> 1))),
                                a[m][0], a[m][1], a[m][2], a[m][3]);
                // B fragments of n-tiles (2h, 2h+1): rows n*8 + (lane & 7)
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    ldmatrix_x4(smem_u32(ws + swz((2 * h + (mi >> 1)) * 8 + r, ks * 2 + (mi & 1))),
                                bw[2 * h][0], bw[2 * h][1], bw[2 * h + 1][0], bw[2 * h + 1][1]);
#pragma unroll
                for (int j = 0; j < 4; ++j)
#pragma unroll
                    for (int m = 0; m < 2; ++m) mma_bf16_16816(acc[m][j], a[m], bw[j][0], bw[j][1]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(empty + s));
        }
        // Partial logits of this warp -> smem [warp][token][expert].
        const int gq = lane >> 2, cq = lane & 3;
        float* pw = partial + warp * kRouterTokens * kPartStride;
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int col = j * 8 + 2 * cq, row = m * 16 + gq;
                pw[row * kPartStride + col] = acc[m][j][0];
                pw[row * kPartStride + col + 1] = acc[m][j][1];
                pw[(row + 8) * kPartStride + col] = acc[m][j][2];
                pw[(row + 8) * kPartStride + col + 1] = acc[m][j][3];
            }
    }
    __syncthreads();
    if (tid == 0) MOE_TRACE_POINT(g_trace_router, 0, trace_cta, 2);
    if (flag[0]) {
        if (tid == 0 && !bad_cfg) atomicOr(p.status + kStatusWord, MOE_DEV_WAIT_TIMEOUT);
        // block-uniform (flag read after the barrier); the K slices of a
        // cluster must all reach its barriers, so they carry on (with
        // meaningless logits: the status word reports the failure)
        if (p.ksplit == 1) return;
    }

    // This slice's 32 x 32 block: the warp partials added in warp order.
    // `blk` lives in the partial buffer's warp-0 slot.
    float* blk = partial;
    for (int i = tid; i < kRouterTokens * kGroup; i += kThreads) {
        const int row = i / kGroup, col = i - row * kGroup;
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < kComputeWarps; ++w)
            v += partial[(w * kRouterTokens + row) * kPartStride + col];
        blk[row * kPartStride + col] = v;   // only this thread reads this slot
    }
    __syncthreads();

    const int pair = b * p.egroups + g;
    if (p.ksplit > 1) {
        // The K slices of (b, g) form one thread-block cluster.  Once every
        // slice is done with its ring (first cluster barrier), slices 1..
        // store their blocks into slot q of slice 0's ring region (remote
        // shared-memory stores); after the second barrier slice 0 adds the
        // slots in slice order and the others leave.  (Measured on GB300 at
        // 20b T=1: the former merge through global memory and a ticket took
        // ~4 us from the last slice's loads to the summed block.)
        float* slots = reinterpret_cast<float*>(ring);   // [ksplit][32][32], slice 0
        const uint32_t rank = cluster_ctarank();
        cluster_sync();
        if (tid == 0) MOE_TRACE_POINT(g_trace_router, 0, trace_cta, 6);
        if (rank != 0) {
            const uint32_t dst = mapa_shared(smem_u32(slots + rank * kRouterTokens * kGroup), 0);
            for (int i = tid; i < kRouterTokens * kGroup; i += kThreads)
                st_shared_cluster_f32(dst + 4u * static_cast<uint32_t>(i),
                                      blk[(i / kGroup) * kPartStride + (i % kGroup)]);
        }
        cluster_sync();
        if (tid == 0) MOE_TRACE_POINT(g_trace_router, 0, trace_cta, 7);
        if (rank != 0) return;   // CTA-uniform
        for (int i = tid; i < kRouterTokens * kGroup; i += kThreads) {
            const int row = i / kGroup, col = i - row * kGroup;
            float v = blk[row * kPartStride + col];
            for (int q2 = 1; q2 < p.ksplit; ++q2) v += slots[q2 * kRouterTokens * kGroup + i];
            blk[row * kPartStride + col] = v;   // only this thread reads this slot
        }
        __syncthreads();
    }

    // Full logit rows of the token block in smem: logits[token][expert].
    const int ls = E + 1;
    if (p.egroups == 1) {
        for (int i = tid; i < kRouterTokens * E; i += kThreads) {
            const int row = i / E, col = i - row * E;
            logits[row * ls + col] = blk[row * kPartStride + col];
        }
    } else {
        // The last expert group of block b gathers the block's rows.
        const int g0 = g * kGroup;
        for (int i = tid; i < kRouterTokens * kGroup; i += kThreads) {
            const int row = i / kGroup, col = i - row * kGroup;
            if (g0 + col < E)
                p.logits[(static_cast<size_t>(b) * kRouterTokens + row) * E + g0 + col] =
                    blk[row * kPartStride + col];
        }
        __threadfence();
        __syncthreads();
        int* gcount = p.counters + kPairSlots + b;
        if (tid == 0) {
            const int ticket = atomicAdd(gcount, 1);
            flag[2] = (ticket == p.egroups - 1);
            if (flag[2]) *gcount = 0;
        }
        __syncthreads();
        if (!flag[2]) return;   // block-uniform
        __threadfence();
        const float* rows = p.logits + static_cast<size_t>(b) * kRouterTokens * E;
        for (int i0 = 0; i0 < kRouterTokens * E; i0 += 8 * kThreads) {
            float v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int i = i0 + u * kThreads + tid;
                v[u] = i < kRouterTokens * E ? __ldcg(rows + i) : 0.f;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int i = i0 + u * kThreads + tid;
                if (i < kRouterTokens * E) logits[(i / E) * ls + (i % E)] = v[u];
            }
        }
    }
    __syncthreads();

    // Top-k + softmax, one lane per token (the partial buffer is free now).
    if (tid == 0) MOE_TRACE_POINT(g_trace_router, 0, trace_cta, 3);
    const int n_valid = min(kRouterTokens, p.T - t0);
    if (n_valid <= kThreads / 32) {
        switch (p.top_k) {
            case 1: topk_warp<1>(p, logits, ls, bias_s, t0, n_valid, hist, ids_s); break;
            case 2: topk_warp<2>(p, logits, ls, bias_s, t0, n_valid, hist, ids_s); break;
            case 3: topk_warp<3>(p, logits, ls, bias_s, t0, n_valid, hist, ids_s); break;
            case 4: topk_warp<4>(p, logits, ls, bias_s, t0, n_valid, hist, ids_s); break;
            case 5: topk_warp<5>(p, logits, ls, bias_s, t0, n_valid, hist, ids_s); break;
            case 6: topk_warp<6>(p, logits, ls, bias_s, t0, n_valid, hist, ids_s); break;
            case 7: topk_warp<7>(p, logits, ls, bias_s, t0, n_valid, hist, ids_s); break;
            default: topk_warp<8>(p, logits, ls, bias_s, t0, n_valid, hist, ids_s); break;
        }
    } else {
        switch (p.top_k) {
            case 1: topk_block<1>(p, logits, ls, bias_s, partial, t0, hist, ids_s); break;
            case 2: topk_block<2>(p, logits, ls, bias_s, partial, t0, hist, ids_s); break;
            case 3: topk_block<3>(p, logits, ls, bias_s, partial, t0, hist, ids_s); break;
            case 4: topk_block<4>(p, logits, ls, bias_s, partial, t0, hist, ids_s); break;
            case 5: topk_block<5>(p, logits, ls, bias_s, partial, t0, hist, ids_s); break;
            case 6: topk_block<6>(p, logits, ls, bias_s, partial, t0, hist, ids_s); break;
            case 7: topk_block<7>(p, logits, ls, bias_s, partial, t0, hist, ids_s); break;
            default: topk_block<8>(p, logits, ls, bias_s, partial, t0, hist, ids_s); break;
        }
    }
    __syncthreads();
    for (int e = tid; e < E; e += kThreads) {
        p.blk_cnt[static_cast<size_t>(e) * p.nblocks + b] = hist[e];
        if (p.nblocks > 1 && hist[e] != 0)
            atomicAdd(p.counters + kExpertTotalsOffset + e, hist[e]);
    }

    if (p.nblocks > 1) {
        // The last token block finishes the routing tables.
        __threadfence();
        __syncthreads();
        if (tid == 0) {
            const int ticket = atomicAdd(p.status + kGridCounterWord, 1);
            flag[3] = (ticket == p.nblocks - 1);
        }
        __syncthreads();
        if (!flag[3]) return;   // block-uniform
        __threadfence();
    } else {
        __syncthreads();
    }
    if (tid == 0) MOE_TRACE_POINT(g_trace_router, 0, trace_cta, 4);
    finish_routing(p, hist, scan_a, scan_b, scan_c, ids_s);
    if (tid == 0) MOE_TRACE_POINT(g_trace_router, 0, trace_cta, 5);
}

}  // namespace

// ------------------------------------------------------------ tiny batches
//
// Batches of at most kTinyTokens tokens: one CTA of kTinyThreads threads
// does the whole routing -- the logits, the top k (a warp per token), the
// expert offsets, the GEMM tiles and, on the small-batch path, the stable
// permutation -- with no ticket or merge between CTAs.  Measured on GB300 at
// gpt-oss-20b, T = 1: the multi-CTA router spent ~11 us from its dependency
// wait to the finished tables, mostly in hand-offs between its phases.
//
// The token rows are copied to shared memory first, by every thread at once
// (read in the dot-product loop, each load waited for in turn, they cost
// ~5 us of dependent L2 round trips at T = 1).  When the router matrix also
// fits (gpt-oss-20b: 32 x 2880 bf16, 184 KB) it is copied there by bulk
// copies issued before the dependency wait, so its load overlaps the kernel
// before this one (the weights are not written by it), and the logits are
// an mma.sync contraction: warp w takes the 16-wide K steps w, w + 16, ...
// of every 16-expert tile, and the warps' partial tiles are added in warp
// order.  Otherwise warp w computes the logits of experts 2w, 2w + 1, then
// 2w + 32, ... with fp32 FMAs over its lanes' shares of both rows (every
// load of a pass issued before the first multiply) and a warp reduction.
// Either way the order is fixed (the same logits every run); the other
// routers' orders differ, as any two sum orders may, in the last bits.
constexpr int kTinyThreads = 512;
constexpr int kTinyTokens = 8;
constexpr size_t kTinySmemMax = 224 * 1024;
// Batches of up to kTinyGridMaxT tokens whose router matrix can be staged
// next to four token rows: a grid of CTAs of kTinyGridTokens tokens each,
// every CTA staging the whole matrix before the wait; their counts are
// added by the last CTA to finish (an atomic ticket), which then finishes
// the tables as the single CTA does.
constexpr int kTinyGridTokens = 4;
constexpr int kTinyGridMaxT = 64;
static_assert(64 * (kTinyGridMaxT / kTinyGridTokens) <= kMaxTokenBlocks,
              "the grid's per-CTA counts must fit the token-block ticket area");

// Rows in shared memory are H * 2 + 16 bytes apart, so that the eight rows
// an ldmatrix reads at one column fall in different banks.
size_t router_tiny_row_bytes(int H) { return static_cast<size_t>(H) * 2 + 16; }
size_t router_tiny_base_bytes() {
    return kTinyTokens * kMaxExperts * 4 + (6 * kMaxExperts + 2) * 4;
}
// the token rows and one zero row
size_t router_tiny_x_bytes(int T, int H) { return static_cast<size_t>(T + 1) * router_tiny_row_bytes(H); }
// the warps' partial logits [16 warps][64 experts][8 tokens] fp32 (they
// alias the staged matrix once it has been read, when it is large enough)
constexpr size_t kTinyRedBytes = 16 * 64 * kTinyTokens * 4;
// bytes of the staged router matrix (0: read from global memory)
size_t router_tiny_stage_bytes(int T, int H, int E) {
    const size_t b = static_cast<size_t>(E) * router_tiny_row_bytes(H);
    const size_t red = b >= kTinyRedBytes ? 0 : kTinyRedBytes;
    return (H % 16 == 0 &&
            b + red + router_tiny_x_bytes(T, H) + router_tiny_base_bytes() <= kTinySmemMax)
               ? b + red : 0;
}

__global__ void __launch_bounds__(kTinyThreads, 1)
    router_tiny_kernel(const RouterParams p, const __nv_bfloat16* __restrict__ x,
                       const __nv_bfloat16* __restrict__ wr, uint32_t wstage, int tb) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t wbar;
    __shared__ int last_cta;
    // this CTA's tokens: [t0, t0 + T) of the batch (tb per CTA)
    const int t0 = static_cast<int>(blockIdx.x) * tb;
    const int T = min(tb, p.T - t0), H = p.H, E = p.E;
    const uint32_t rs = static_cast<uint32_t>(H) * 2u + 16u;               // padded row bytes
    uint8_t* w_s = smem_raw;                                                // [E][rs], staged
    uint8_t* x_s = smem_raw + wstage;                                       // [T + 1][rs]
    float* logits = reinterpret_cast<float*>(x_s + static_cast<size_t>(T + 1) * rs);
    int* hist = reinterpret_cast<int*>(logits + kTinyTokens * kMaxExperts);  // [256]
    int* scan_a = hist + kMaxExperts;                                        // [257]
    int* scan_b = scan_a + kMaxExperts + 1;                                  // [256]
    int* scan_c = scan_b + kMaxExperts;                                      // [257]
    int* ids_s = scan_c + kMaxExperts + 1;                                   // [256]
    float* bias_s = reinterpret_cast<float*>(ids_s + kMaxExperts);           // [256]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) MOE_TRACE_POINT(g_trace_router, 0, blockIdx.x, 0);
    if (wstage && tid == 0) {
        // the router matrix, one bulk copy per expert row (16-byte multiples)
        mbar_init(smem_u32(&wbar), 1);
        mbar_fence_init();
        const uint32_t row_bytes = static_cast<uint32_t>(H) * 2u;
        mbar_arrive_expect_tx(smem_u32(&wbar), row_bytes * static_cast<uint32_t>(E));
        for (int e = 0; e < E; ++e)
            bulk_load(smem_u32(w_s) + static_cast<uint32_t>(e) * rs,
                      wr + static_cast<size_t>(e) * H, row_bytes, smem_u32(&wbar));
    }
    // token rows, workspace and counters may be written by the kernel before
    pdl_wait();
    pdl_launch_dependents();
    if (tid == 0) MOE_TRACE_POINT(g_trace_router, 0, blockIdx.x, 1);

    const int hv = H / 8;                                   // 16-byte vectors per row
    const uint4* xg = reinterpret_cast<const uint4*>(x) + static_cast<size_t>(t0) * hv;
    for (int e = tid; e < kMaxExperts; e += kTinyThreads) {
        hist[e] = 0;
        bias_s[e] = e < E ? __bfloat162float(p.br[e]) : 0.f;
    }
    // token rows t < T, then a zero row (the operand rows past T or E)
    for (int i = tid; i < (T + 1) * hv; i += kTinyThreads) {
        const int t = i / hv, v = i - t * hv;
        *reinterpret_cast<uint4*>(x_s + t * rs + v * 16) =
            t < T ? __ldg(xg + i) : make_uint4(0u, 0u, 0u, 0u);
    }
    __syncthreads();
    // the staged matrix has landed (a bounded wait; if it gives up, the
    // logits are computed from global memory instead and the status word
    // reports the timeout)
    bool staged = wstage != 0;
    if (staged) {
        staged = __syncthreads_and(mbar_wait(smem_u32(&wbar), 0, nullptr) ? 1 : 0) != 0;
        if (!staged && tid == 0) atomicOr(p.status, MOE_DEV_WAIT_TIMEOUT);
    }
    if (tid == 0) MOE_TRACE_POINT(g_trace_router, 0, blockIdx.x, 2);
    constexpr int kWarps = kTinyThreads / 32;
    if (staged) {
        // logits on the tensor cores: D[expert][token] += W[expert][k] x[token][k]
        // (mma.sync m16n8k16, bf16 in, fp32 accumulation).  Warp w takes
        // the 16-wide K steps w, w + 16, ... for every 16-expert tile; the
        // warps' partial tiles are then added in warp order.
        const int nmt = (E + 15) / 16;                      // <= 4
        const int nks = H / 16;
        const uint8_t* zrow = x_s + static_cast<size_t>(T) * rs;
        float d[4][4];
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
            for (int i = 0; i < 4; ++i) d[mt][i] = 0.f;
        // this lane's ldmatrix rows: B (token lane % 8, k half (lane / 8) % 2),
        // A (expert 16 mt + lane % 16, k half lane / 16)
        const int bn = lane & 7, bk = (lane >> 3) & 1;
        const uint32_t b_row = smem_u32(bn < T ? x_s + static_cast<size_t>(bn) * rs : zrow) + 16u * bk;
        uint32_t a_row[4];
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
            const int e = 16 * mt + (lane & 15);
            a_row[mt] = smem_u32(e < E ? w_s + static_cast<size_t>(e) * rs : zrow) + 16u * (lane >> 4);
        }
        for (int ks = warp; ks < nks; ks += kWarps) {
            uint32_t b0, b1, b2, b3;
            ldmatrix_x4(b_row + 32u * ks, b0, b1, b2, b3);   // (b2, b3: lanes 16-31's rows, unused)
#pragma unroll
            for (int mt = 0; mt < 4; ++mt) {
                if (mt >= nmt) break;
                uint32_t a[4];
                ldmatrix_x4(a_row[mt] + 32u * ks, a[0], a[1], a[2], a[3]);
                mma_bf16_16816(d[mt], a, b0, b1);
            }
        }
        __syncthreads();                                    // every warp is done with w_s
        // partials [warp][expert 0..63][token 0..7]
        float* red = reinterpret_cast<float*>(w_s);
        const int g = lane >> 2, q = lane & 3;
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
            if (mt >= nmt) break;
            float* rw = red + (warp * 64 + 16 * mt) * kTinyTokens;
            rw[g * kTinyTokens + 2 * q] = d[mt][0];
            rw[g * kTinyTokens + 2 * q + 1] = d[mt][1];
            rw[(g + 8) * kTinyTokens + 2 * q] = d[mt][2];
            rw[(g + 8) * kTinyTokens + 2 * q + 1] = d[mt][3];
        }
        __syncthreads();
        for (int i = tid; i < E * T; i += kTinyThreads) {
            const int t = i / E, e = i - t * E;
            float v = 0.f;
#pragma unroll 4
            for (int w = 0; w < kWarps; ++w) v += red[(w * 64 + e) * kTinyTokens + t];
            logits[t * E + e] = v;
        }
    } else {
    const uint4* wbase = reinterpret_cast<const uint4*>(wr);

    // logits from global memory: warp w takes experts 2w, 2w + 1, then
    // 2w + 2 * warps, ...  Lane l sums vectors l, l + 32, ... of both rows:
    // every load of a row pass is issued before the first multiply
    // (predicated, no early exit).
    constexpr int kBatch = 6;                               // loads per row per lane and pass
    const auto row_pass = [&](const uint4* w0row, const uint4* w1row, int v0, float (&acc)[2][kTinyTokens]) {
        uint4 w[2][kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int v = v0 + u * 32 + lane;
            const bool in = v < hv;
            w[0][u] = in ? w0row[v] : make_uint4(0u, 0u, 0u, 0u);
            w[1][u] = in && w1row ? w1row[v] : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int t = 0; t < kTinyTokens; ++t) {
            if (t >= T) break;
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int v = v0 + u * 32 + lane;
                const uint4 xv = v < hv ? *reinterpret_cast<const uint4*>(x_s + t * rs + v * 16)
                                        : make_uint4(0u, 0u, 0u, 0u);
                const uint32_t xx[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const uint32_t ww[4] = {w[r][u].x, w[r][u].y, w[r][u].z, w[r][u].w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        acc[r][t] = fmaf(__uint_as_float(ww[q] << 16),
                                         __uint_as_float(xx[q] << 16), acc[r][t]);
                        acc[r][t] = fmaf(__uint_as_float(ww[q] & 0xFFFF0000u),
                                         __uint_as_float(xx[q] & 0xFFFF0000u), acc[r][t]);
                    }
                }
            }
        }
    };
    for (int e0 = 2 * warp; e0 < E; e0 += 2 * kWarps) {
        float acc[2][kTinyTokens];
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
            for (int t = 0; t < kTinyTokens; ++t) acc[r][t] = 0.f;
        const uint4* w0row = wbase + static_cast<size_t>(e0) * hv;
        const uint4* w1row = e0 + 1 < E ? w0row + hv : nullptr;
        for (int v0 = 0; v0 < hv; v0 += 32 * kBatch) row_pass(w0row, w1row, v0, acc);
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
            for (int t = 0; t < kTinyTokens; ++t) {
                if (t >= T) break;
                float v = acc[r][t];
#pragma unroll
                for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
                if (lane == 0 && e0 + r < E) logits[t * E + e0 + r] = v;
            }
    }
    }
    if (tid == 0) MOE_TRACE_POINT(g_trace_router, 0, blockIdx.x, 6);
    __syncthreads();
    if (tid == 0) MOE_TRACE_POINT(g_trace_router, 0, blockIdx.x, 3);

    switch (p.top_k) {
        case 1: topk_warp<1>(p, logits, E, bias_s, t0, T, hist, ids_s); break;
        case 2: topk_warp<2>(p, logits, E, bias_s, t0, T, hist, ids_s); break;
        case 3: topk_warp<3>(p, logits, E, bias_s, t0, T, hist, ids_s); break;
        case 4: topk_warp<4>(p, logits, E, bias_s, t0, T, hist, ids_s); break;
        case 5: topk_warp<5>(p, logits, E, bias_s, t0, T, hist, ids_s); break;
        case 6: topk_warp<6>(p, logits, E, bias_s, t0, T, hist, ids_s); break;
        case 7: topk_warp<7>(p, logits, E, bias_s, t0, T, hist, ids_s); break;
        default: topk_warp<8>(p, logits, E, bias_s, t0, T, hist, ids_s); break;
    }
    __syncthreads();
    if (gridDim.x > 1) {
        // This CTA's counts per expert and the totals; the last CTA to take a
        // ticket adds the counts per 32-token block for the permutation
        // kernel and finishes the tables.  The counts go to [E][CTAs] ints of
        // the completion-counter block that the multi-block router keeps its
        // per-token-block tickets in (unused by this router, zero between
        // calls: the last CTA clears what it read).
        const int nb = static_cast<int>(gridDim.x);
        int32_t* cnt = p.counters + kPairSlots;
        for (int e = tid; e < E; e += kTinyThreads) {
            cnt[e * nb + blockIdx.x] = hist[e];
            if (hist[e] != 0) atomicAdd(p.counters + kExpertTotalsOffset + e, hist[e]);
        }
        __threadfence();
        __syncthreads();
        if (tid == 0) last_cta = atomicAdd(p.status + kGridCounterWord, 1) == nb - 1;
        __syncthreads();
        if (!last_cta) return;   // block-uniform
        __threadfence();
        const int R = p.T * p.top_k;
        if (p.small_perm) {
            // every token's ids (this CTA's own among them) from global memory
            for (int a = tid; a < R; a += kTinyThreads) ids_s[a] = __ldcg(p.topk_ids + a);
        } else {
            const int nb32 = (p.T + kRouterTokens - 1) / kRouterTokens;
            const int per32 = kRouterTokens / tb;      // router CTAs per 32-token block
            for (int i = tid; i < E * nb32; i += kTinyThreads) {
                const int e = i / nb32, b = i - e * nb32;
                int c_sum = 0;
                for (int c = b * per32; c < min(nb, (b + 1) * per32); ++c)
                    c_sum += __ldcg(cnt + e * nb + c);
                p.blk_cnt[e * nb32 + b] = c_sum;
            }
        }
        __syncthreads();
        for (int i = tid; i < E * nb; i += kTinyThreads) cnt[i] = 0;
    } else if (!p.small_perm) {
        // one CTA, one 32-token block: its counts for the permutation kernel
        for (int e = tid; e < E; e += kTinyThreads) p.blk_cnt[e] = hist[e];
    }
    if (tid == 0) MOE_TRACE_POINT(g_trace_router, 0, blockIdx.x, 4);
    finish_routing<kTinyThreads>(p, hist, scan_a, scan_b, scan_c, ids_s);
    if (tid == 0) MOE_TRACE_POINT(g_trace_router, 0, blockIdx.x, 5);
}

size_t router_tiny_smem_bytes(int T, int H, int E) {
    return router_tiny_stage_bytes(T, H, E) + router_tiny_x_bytes(T, H) + router_tiny_base_bytes();
}

// (one SM reads the whole router matrix: with 128 experts, 737 KB at
// H = 2880, the multi-block router measured faster at T = 8)
// tokens per CTA of the single-block router for a batch of T (0: not used)
int router_tiny_tokens_per_cta(int T, int H, int E) {
    // (one SM reads the whole matrix: with 128 experts, 737 KB at H = 2880,
    // it wins at T <= 2 -- 120b shape, T = 1: 59.3 -> 57.9 us per layer --
    // and the multi-block router at T = 8)
    if (T < 1 || E > (T <= 2 ? 128 : 64) || H % 8 != 0) return 0;
    if (T <= kTinyTokens)
        return router_tiny_x_bytes(T, H) + router_tiny_base_bytes() <= kTinySmemMax ? T : 0;
    // larger batches only with the router matrix staged
    if (T <= kTinyGridMaxT && router_tiny_stage_bytes(kTinyGridTokens, H, E) > 0)
        return kTinyGridTokens;
    return 0;
}

bool router_tiny_fits(int T, int H, int E) { return router_tiny_tokens_per_cta(T, H, E) > 0; }

cudaError_t launch_router_tiny(const RouterParams& p, const void* x, const void* wr,
                               cudaStream_t s, bool pdl) {
    const int tb = router_tiny_tokens_per_cta(p.T, p.H, p.E);
    const int nb = tb > 0 ? (p.T + tb - 1) / tb : 0;
    if (tb == 0 || p.nblocks != nb) return cudaErrorInvalidValue;
    const uint32_t wstage = static_cast<uint32_t>(router_tiny_stage_bytes(tb, p.H, p.E));
    const size_t smem = router_tiny_smem_bytes(tb, p.H, p.E);
    cudaError_t err = cudaFuncSetAttribute(router_tiny_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(nb);
    cfg.blockDim = dim3(kTinyThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, router_tiny_kernel, p,
                              static_cast<const __nv_bfloat16*>(x),
                              static_cast<const __nv_bfloat16*>(wr), wstage, tb);
}

size_t router_stage_bytes() { return kStageBytes; }

size_t trace_copy_router(unsigned long long* dst, size_t cap) {
    MOE_TRACE_COPY(g_trace_router, dst, cap);
}

// Shared memory for `stages` ring slots (at least the top-k logits), the
// warp partials, barriers and scan buffers, plus 1 KB alignment slack.
size_t router_smem_bytes(int stages) {
    const size_t ring = static_cast<size_t>(stages) * kStageBytes;
    return 1024 + (ring > kLogitsBytes ? ring : kLogitsBytes) + kPartialBytes +
           2 * kMaxStages * 8 + (6 * kMaxExperts + 8) * 4;
}

int router_max_stages() { return kMaxStages; }
int router_stage_multiple() { return kComputeWarps; }

cudaError_t launch_router(const RouterParams& p, const CUtensorMap* tx, const CUtensorMap* tw,
                          size_t smem, cudaStream_t s, bool pdl) {
    if (p.stages < 1 || p.stages > kMaxStages) return cudaErrorInvalidValue;
    if (p.ksplit < 1 || p.ksplit > kMaxRouterSlices) return cudaErrorInvalidValue;
    cudaError_t err = cudaFuncSetAttribute(router_topk_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.nblocks, p.egroups, p.ksplit);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (p.ksplit > 1) {
        // the K slices of one (token block, expert group) form a cluster
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = 1;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = static_cast<unsigned>(p.ksplit);
        ++na;
    }
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, router_topk_kernel, p, *tx, *tw);
}

}  // namespace moe
