// Expert permutation on the device, with no host synchronisation (xserv
// docs/19-gpt-oss-moe.md, "Phase 19: gpt-oss-20b", §2 "MoE 前向": topk_ids
// stay on the GPU and the host never waits for them).
//
// The T*k assignments a = t*k + j are placed in rows sorted by
// (expert, a) ascending -- a stable counting sort.  The router kernel left,
// per expert e and 32-token block b, the block's count of e (blk_cnt[e][b])
// and the expert offsets.  CTA (b, y):
//   1. sums the counts of the earlier blocks, base(e) = sum over b' < b of
//      blk_cnt[e][b'] (a warp per expert, loads in flight together), and ranks
//      block b's assignments per expert in order of a (warp match), so
//      row(a) = offsets[e] + base(e) + rank; the y == 0 CTA writes
//      sorted_assign / assign_row;
//   2. copies its share (1/gather_split) of those assignments' activation
//      rows into x_perm[row] -- the contiguous per-expert operand of the
//      gate_up GEMM -- one warp per row, 16-byte loads kept in flight.
//      With MXFP4 weights x_perm takes the layout that GEMM reads: chunk-
//      major [H/64][T*k][64] (one TMA box then spans several 64-wide K
//      chunks), each group of 8 columns in the order 0,4,1,5,2,6,3,7 (the
//      order in which the GEMM expands E2M1 codes).  With FP8 W8A8 weights
//      the row is quantised on the way: E4M3 codes of x * (448 / max|x|)
//      with the token's own max|x|, and the row's scale max|x| / 448.
//      With MXFP8 activations every block of 32 elements is quantised by the
//      OCP MX rule (scale 2^(floor(log2 max|x|) - 8) as a UE8M0 byte, codes
//      E4M3 of x / scale) into the padded layout of mx_pos.
#include <cuda_fp16.h>

#include "moe_internal.cuh"
#include "ptx.cuh"
#include "trace.cuh"
#include "../../include/moe.h"

namespace moe {
namespace {

MOE_TRACE_ARRAY(g_trace_permute, 1);

constexpr int kThreads = 256;
constexpr int kRowVecUnroll = 12;   // 16-byte vectors per lane in flight (H <= 6144)

// Eight bf16 (k = 0..7) to the order 0,4,1,5,2,6,3,7.
__device__ __forceinline__ uint4 kperm8(const uint4 v) {
    uint4 r;
    r.x = __byte_perm(v.x, v.z, 0x5410);
    r.y = __byte_perm(v.x, v.z, 0x7632);
    r.z = __byte_perm(v.y, v.w, 0x5410);
    r.w = __byte_perm(v.y, v.w, 0x7632);
    return r;
}

// Eight bf16 values to eight f16 values in the same order (round to
// nearest even; exact for magnitudes in [2^-14, 65504]); magnitudes beyond
// the f16 range saturate to +-65504 and set *range.
__device__ __forceinline__ uint4 f16x8(const uint4 v, bool& range) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float lo = __uint_as_float(w[i] << 16), hi = __uint_as_float(w[i] & 0xFFFF0000u);
        range |= fabsf(lo) > 65504.f || fabsf(hi) > 65504.f;
        lo = fminf(fmaxf(lo, -65504.f), 65504.f);
        hi = fminf(fmaxf(hi, -65504.f), 65504.f);
        const __half2 h = __floats2half2_rn(lo, hi);
        o[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// Largest magnitude of eight bf16 values (exact, in fp32).
__device__ __forceinline__ float absmax8(const uint4 v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        m = fmaxf(m, fabsf(__uint_as_float(w[i] << 16)));
        m = fmaxf(m, fabsf(__uint_as_float(w[i] & 0xFFFF0000u)));
    }
    return m;
}

// Eight bf16 values times `inv` to eight E4M3 codes, in element order.
__device__ __forceinline__ uint2 e4m3x8(const uint4 v, float inv) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t c[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        c[i] = cvt_e4m3x2(__uint_as_float(w[i] << 16) * inv,
                          __uint_as_float(w[i] & 0xFFFF0000u) * inv);
    return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

__global__ void __launch_bounds__(kThreads) permute_kernel(const PermuteParams p) {
    __shared__ int base[kMaxExperts];
    __shared__ int running[kMaxExperts];
    __shared__ int rows_s[kRouterTokens * kMaxTopK];

    const int trace_cta = blockIdx.y * gridDim.x + blockIdx.x;
    if (threadIdx.x == 0) MOE_TRACE_POINT(g_trace_permute, 0, trace_cta, 0);
    pdl_wait();                 // routing tables of the previous kernel
    pdl_launch_dependents();    // the GEMM may start its prologue
    if (threadIdx.x == 0) MOE_TRACE_POINT(g_trace_permute, 0, trace_cta, 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int E = p.E, k = p.top_k, b = blockIdx.x;

    // base(e) = offsets[e] + rows of e that earlier token blocks own.  Warp
    // w sums experts w, w + 8, ... (its lanes stride the blocks b' < b of
    // the expert's row of blk_cnt), eight experts and two blocks per lane in
    // flight, then a warp reduction: no atomics, and with few blocks every
    // load (offsets included) is in flight at once.
    constexpr int kWarps = kThreads / 32;
    constexpr int kExpertBatch = 8;
    for (int e0 = warp; e0 < E; e0 += kWarps * kExpertBatch) {
        int sum[kExpertBatch], off[kExpertBatch];
#pragma unroll
        for (int m = 0; m < kExpertBatch; ++m) {
            const int e = e0 + m * kWarps;
            off[m] = e < E ? __ldcg(p.offsets + e) : 0;
            sum[m] = 0;
        }
#pragma unroll 2
        for (int j = lane; j < b; j += 32) {
#pragma unroll
            for (int m = 0; m < kExpertBatch; ++m) {
                const int e = e0 + m * kWarps;
                if (e < E) sum[m] += __ldcg(p.blk_cnt + static_cast<size_t>(e) * p.nblocks + j);
            }
        }
#pragma unroll
        for (int m = 0; m < kExpertBatch; ++m) {
            int v = sum[m];
#pragma unroll
            for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
            const int e = e0 + m * kWarps;
            if (lane == 0 && e < E) base[e] = off[m] + v;
        }
    }
    if (tid < E) running[tid] = 0;
    __syncthreads();

    // Stable ranks of this block's assignments (warp 0, 32 at a time).
    const int a0 = b * kRouterTokens * k;
    const int a1 = min(p.T, (b + 1) * kRouterTokens) * k;
    const int rows_total = p.T * k;
    if (warp == 0) {
        for (int ab = a0; ab < a1; ab += 32) {
            const int a = ab + lane;
            const bool valid = a < a1;
            int e = valid ? __ldcg(p.topk_ids + a) : -1;
            const bool good = valid && e >= 0 && e < E;
            if (valid && !good && blockIdx.y == 0)
                atomicOr(p.status + kStatusWord, MOE_DEV_BAD_EXPERT_ID);
            if (!good) e = -1 - lane;   // unique per lane: never matches a real expert
            const unsigned peers = __match_any_sync(0xffffffffu, e);
            const int rank = __popc(peers & ((1u << lane) - 1u));
            const int r0 = good ? running[e] : 0;
            __syncwarp();
            if (good && rank == 0) running[e] = r0 + __popc(peers);
            __syncwarp();
            int row = good ? base[e] + r0 + rank : -1;
            // counts that do not add up (a corrupted counter region) must not
            // place a row outside [0, T*k): report it and drop the row
            if (good && (row < 0 || row >= rows_total)) {
                if (blockIdx.y == 0) atomicOr(p.status + kStatusWord, MOE_DEV_BAD_TILE);
                row = -1;
            }
            if (valid) {
                if (blockIdx.y == 0) {
                    if (row >= 0) p.sorted_assign[row] = a;
                    p.assign_row[a] = row;
                }
                // the gather copies only the rows of this device's experts
                rows_s[a - a0] = row >= 0 && e >= p.ex_lo && e < p.ex_hi ? row : -1;
            }
        }
    }
    __syncthreads();

    if (threadIdx.x == 0) MOE_TRACE_POINT(g_trace_permute, 0, trace_cta, 2);
    // Clear this CTA's share of the block's fp32 output rows (the down
    // projection's epilogue accumulates into them).
    if (p.zero_out) {
        const int rows = min(kRouterTokens, p.T - b * kRouterTokens);
        const size_t n4 = static_cast<size_t>(rows) * p.H / 4;
        const size_t per4 = (n4 + p.gather_split - 1) / p.gather_split;
        const size_t lo = blockIdx.y * per4, hi = min(n4, lo + per4);
        float4* dst = reinterpret_cast<float4*>(p.zero_out +
                                                static_cast<size_t>(b) * kRouterTokens * p.H);
        for (size_t i = lo + tid; i < hi; i += kThreads) dst[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }

    // Gather: x_perm[row(a)] = x[a / k], this CTA's slice of the block.
    if (p.x_perm) {
        const int n = a1 - a0;
        const int per = (n + p.gather_split - 1) / p.gather_split;
        const int l0 = blockIdx.y * per;
        const int l1 = min(n, l0 + per);
        const int vec_per_row = p.H / 8;
        for (int la = l0 + warp; la < l1; la += kThreads / 32) {
            const int row = rows_s[la];
            if (row < 0) continue;
            if (!MOE_BOUNDS(row < rows_total && (a0 + la) / k < p.T, p.status + kStatusWord))
                continue;
            const uint4* src = reinterpret_cast<const uint4*>(p.x + static_cast<size_t>((a0 + la) / k) * p.H);
            if (p.mx8) {
                // MXFP8: a block of 32 elements is the 4 vectors of 4
                // adjacent lanes; kRowVecUnroll vectors per lane are loaded
                // before any is used (loads in flight), and the shuffles run
                // in every lane (the batch's bounds are warp-uniform)
                const int kp = mx_padded_k(p.H), tail0 = mx_tail0(p.H);
                uint8_t* dst8 = reinterpret_cast<uint8_t*>(p.x_perm) + static_cast<size_t>(row) * kp;
                uint8_t* dsts = reinterpret_cast<uint8_t*>(p.x_scale) +
                                static_cast<size_t>(row) * mx_scale_row_bytes(p.H);
                for (int v0 = 0; v0 < vec_per_row; v0 += 32 * kRowVecUnroll) {
                    uint4 buf[kRowVecUnroll];
#pragma unroll
                    for (int u = 0; u < kRowVecUnroll; ++u) {
                        const int v = v0 + u * 32 + lane;
                        buf[u] = v < vec_per_row ? src[v] : make_uint4(0u, 0u, 0u, 0u);
                    }
#pragma unroll
                    for (int u = 0; u < kRowVecUnroll; ++u) {
                        if (v0 + u * 32 >= vec_per_row) break;        // warp-uniform
                        const int v = v0 + u * 32 + lane;
                        float m = absmax8(buf[u]);
                        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
                        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
                        if (v >= vec_per_row) continue;
                        // floor(log2 m) = biased exponent - 127 (0 for zero and
                        // subnormal m: the scale then clamps at 2^-127, byte 0)
                        const int ex = static_cast<int>(__float_as_uint(m) >> 23);
                        const int sbyte = ex > 8 ? ex - 8 : 0;
                        const float inv = __uint_as_float(static_cast<uint32_t>(254 - sbyte) << 23);
                        const int k0 = 8 * v;
                        *reinterpret_cast<uint2*>(dst8 + mx_pos(k0, tail0)) = e4m3x8(buf[u], inv);
                        if (k0 >= tail0) *reinterpret_cast<uint2*>(dst8 + k0) = make_uint2(0u, 0u);
                        if ((lane & 3) == 0) {
                            dsts[mx_pos(k0, tail0) / 32] = static_cast<uint8_t>(sbyte);
                            if (k0 >= tail0) dsts[k0 / 32] = 127;   // the gap's blocks: scale 1
                        }
                    }
                }
                continue;
            }
            if (p.fp8) {
                // FP8 W8A8: the token's own scale, max|x| / 448, then the row
                // as E4M3 codes of x * (448 / max|x|) (1 for an all-zero row).
                // Rows of up to 32 x kRowVecUnroll vectors stay in registers
                // (one pass over memory, loads in flight); longer rows are
                // read twice.
                uint2* dst8 = reinterpret_cast<uint2*>(reinterpret_cast<uint8_t*>(p.x_perm) +
                                                       static_cast<size_t>(row) * p.H);
                if (vec_per_row <= 32 * kRowVecUnroll) {
                    uint4 buf[kRowVecUnroll];
                    float m = 0.f;
#pragma unroll
                    for (int u = 0; u < kRowVecUnroll; ++u) {
                        const int v = u * 32 + lane;
                        buf[u] = v < vec_per_row ? src[v] : make_uint4(0u, 0u, 0u, 0u);
                    }
#pragma unroll
                    for (int u = 0; u < kRowVecUnroll; ++u) m = fmaxf(m, absmax8(buf[u]));
#pragma unroll
                    for (int d = 16; d > 0; d >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, d));
                    const float inv = m > 0.f ? 448.0f / m : 1.0f;
                    if (lane == 0) p.x_scale[row] = m > 0.f ? m / 448.0f : 1.0f;
#pragma unroll
                    for (int u = 0; u < kRowVecUnroll; ++u) {
                        const int v = u * 32 + lane;
                        if (v < vec_per_row) dst8[v] = e4m3x8(buf[u], inv);
                    }
                    continue;
                }
                float m = 0.f;
                for (int v = lane; v < vec_per_row; v += 32) m = fmaxf(m, absmax8(src[v]));
#pragma unroll
                for (int d = 16; d > 0; d >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, d));
                const float inv = m > 0.f ? 448.0f / m : 1.0f;
                if (lane == 0) p.x_scale[row] = m > 0.f ? m / 448.0f : 1.0f;
                for (int v = lane; v < vec_per_row; v += 32) dst8[v] = e4m3x8(src[v], inv);
                continue;
            }
            uint4* dst = reinterpret_cast<uint4*>(p.x_perm + static_cast<size_t>(row) * p.H);
            // chunk-major: vector v (8 columns) of the row goes to chunk v/8
            uint4* dst_mx = reinterpret_cast<uint4*>(p.x_perm) + static_cast<size_t>(row) * 8;
            const size_t chunk_vecs = static_cast<size_t>(p.T) * p.top_k * 8;
            for (int v0 = 0; v0 < vec_per_row; v0 += 32 * kRowVecUnroll) {
                uint4 buf[kRowVecUnroll];
#pragma unroll
                for (int u = 0; u < kRowVecUnroll; ++u) {
                    const int v = v0 + u * 32 + lane;
                    if (v < vec_per_row) buf[u] = src[v];
                }
#pragma unroll
                bool range = false;
#pragma unroll
                for (int u = 0; u < kRowVecUnroll; ++u) {
                    const int v = v0 + u * 32 + lane;
                    if (v < vec_per_row) {
                        if (p.mx_layout)
                            dst_mx[static_cast<size_t>(v >> 3) * chunk_vecs + (v & 7)] =
                                p.mx_f16 ? f16x8(buf[u], range) : kperm8(buf[u]);
                        else
                            dst[v] = buf[u];
                    }
                }
                if (range) atomicOr(p.status + kStatusWord, MOE_DEV_RANGE);
            }
        }
    }
#ifdef MOE_TRACE
    __syncthreads();
    if (threadIdx.x == 0) MOE_TRACE_POINT(g_trace_permute, 0, trace_cta, 3);
#endif
}

}  // namespace

size_t trace_copy_permute(unsigned long long* dst, size_t cap) {
    MOE_TRACE_COPY(g_trace_permute, dst, cap);
}

cudaError_t launch_permute(const PermuteParams& p, cudaStream_t s, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.nblocks, p.gather_split);
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
