// Router Linear + bias, top-k selection and softmax over the selected logits,
// fused in one kernel (xserv docs/19-gpt-oss-moe.md, "Phase 19: gpt-oss-20b":
// §1 table "MoE" row -- the router is a plain Linear [2880 -> 32] with bias;
// §2 "MoE 前向" -- router GEMV then topk_softmax on the GPU, ids stay there).
//
// One CTA of 128 threads handles 32 tokens against all E experts.  The
// logits are an fp32-accumulated bf16 contraction on the tensor cores
// (mma.sync m16n8k16; the router is ~0.1% of the layer's flops, far too
// small for a TMEM pipeline).  Operands are staged through shared memory in
// 64-wide K chunks with cp.async double buffering.  Each warp then takes
// 8 tokens and selects the top k with a warp argmax (higher logit first,
// equal logits -> lower expert index), computes the softmax over the k
// selected logits (max-subtracted, expf), and counts the assignments per
// expert for the permutation kernel.  Optionally clears the fp32 output rows
// of its tokens, which the down-projection epilogue accumulates into.
//
// Tails: rows past T and experts past E are zero-filled by cp.async (source
// size 0) and masked out of the selection; every thread reaches every
// barrier (no early exit before a __syncthreads, the failure mode of §4).
#include <cfloat>
#include <climits>

#include "moe_internal.cuh"
#include "ptx.cuh"
#include "../../include/moe.h"

namespace moe {
namespace {

constexpr int kThreads = 128;
constexpr int kRowStride = kBlockK + 8;  // padded smem row (bf16): 144 B, conflict-free ldmatrix

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;"
                 ::"r"(dst), "l"(src), "r"(valid ? 16 : 0) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                            uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];"
                 : "=r"(r0), "=r"(r1) : "r"(addr));
}
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4],
                                               uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// NTW: n-tiles of 8 experts per warp; the CTA covers E_pad = 32 * NTW experts.
template <int NTW>
__global__ void __launch_bounds__(kThreads) router_topk_kernel(const RouterParams p) {
    constexpr int kEPad = 32 * NTW;
    extern __shared__ __align__(16) uint8_t smem[];
    __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(smem);            // [2][32][72]
    __nv_bfloat16* ws = xs + 2 * kRouterTokens * kRowStride;                // [2][E_pad][72]
    int* hist = reinterpret_cast<int*>(ws + 2 * kEPad * kRowStride);        // [256]
    float* logits = reinterpret_cast<float*>(ws);                           // [32][E_pad+1], reuses ws

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int t0 = blockIdx.x * kRouterTokens;
    const int H = p.H, E = p.E;
    const int nchunks = H / kBlockK;

    for (int e = tid; e < kMaxExperts; e += kThreads) hist[e] = 0;

    auto load_chunk = [&](int c, int buf) {
        const int k0 = c * kBlockK;
        // activations: 32 rows x 8 segments of 16 B
        for (int i = tid; i < kRouterTokens * 8; i += kThreads) {
            const int r = i >> 3, seg = i & 7;
            const int t = t0 + r;
            const bool ok = t < p.T;
            const __nv_bfloat16* src = p.x + static_cast<size_t>(ok ? t : 0) * H + k0 + seg * 8;
            cp_async16(smem_u32(xs + (buf * kRouterTokens + r) * kRowStride + seg * 8), src, ok);
        }
        // router weights: E_pad rows x 8 segments
        for (int i = tid; i < kEPad * 8; i += kThreads) {
            const int r = i >> 3, seg = i & 7;
            const bool ok = r < E;
            const __nv_bfloat16* src = p.wr + static_cast<size_t>(ok ? r : 0) * H + k0 + seg * 8;
            cp_async16(smem_u32(ws + (buf * kEPad + r) * kRowStride + seg * 8), src, ok);
        }
    };

    float acc[2][NTW][4];
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int j = 0; j < NTW; ++j)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[m][j][q] = 0.f;

    load_chunk(0, 0);
    cp_async_commit();
    for (int c = 0; c < nchunks; ++c) {
        if (c + 1 < nchunks) {
            load_chunk(c + 1, (c + 1) & 1);
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const int buf = c & 1;
#pragma unroll
        for (int ks = 0; ks < kBlockK / 16; ++ks) {
            uint32_t a[2][4];
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                const int mi = lane >> 3, r = lane & 7;
                const int row = m * 16 + (mi & 1) * 8 + r;
                const int col = ks * 16 + (mi >> 1) * 8;
                ldmatrix_x4(smem_u32(xs + (buf * kRouterTokens + row) * kRowStride + col),
                            a[m][0], a[m][1], a[m][2], a[m][3]);
            }
#pragma unroll
            for (int j = 0; j < NTW; ++j) {
                const int nt = warp + 4 * j;
                const int l16 = lane & 15;
                const int row = nt * 8 + (l16 & 7);
                const int col = ks * 16 + (l16 >> 3) * 8;
                uint32_t b0, b1;
                ldmatrix_x2(smem_u32(ws + (buf * kEPad + row) * kRowStride + col), b0, b1);
#pragma unroll
                for (int m = 0; m < 2; ++m) mma_bf16_16816(acc[m][j], a[m], b0, b1);
            }
        }
        __syncthreads();
    }

    // Scatter the fragments to smem (ws is free now): logits[token][expert].
    {
        const int g = lane >> 2, cq = lane & 3;
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
            for (int j = 0; j < NTW; ++j) {
                const int col = (warp + 4 * j) * 8 + 2 * cq;
                const int row = m * 16 + g;
                logits[row * (kEPad + 1) + col] = acc[m][j][0];
                logits[row * (kEPad + 1) + col + 1] = acc[m][j][1];
                logits[(row + 8) * (kEPad + 1) + col] = acc[m][j][2];
                logits[(row + 8) * (kEPad + 1) + col + 1] = acc[m][j][3];
            }
    }
    __syncthreads();

    // Top-k + softmax: warp w handles tokens 8w .. 8w+7.
    const int k = p.top_k;
    float bias[NTW];
#pragma unroll
    for (int i = 0; i < NTW; ++i) {
        const int e = lane + 32 * i;
        bias[i] = e < E ? __bfloat162float(p.br[e]) : 0.f;
    }
    for (int r = warp * 8; r < warp * 8 + 8; ++r) {
        const int t = t0 + r;
        if (t >= p.T) break;  // warp-uniform; no block barrier follows inside
        float v[NTW];
        uint32_t taken = 0;
#pragma unroll
        for (int i = 0; i < NTW; ++i) {
            const int e = lane + 32 * i;
            float l = logits[r * (kEPad + 1) + e] + bias[i];
            if (!(l == l)) l = -FLT_MAX;            // NaN never wins
            v[i] = e < E ? l : -INFINITY;
            if (e >= E) taken |= 1u << i;
        }
        int sel_e[kMaxTopK];
        float sel_v[kMaxTopK];
        for (int j = 0; j < k; ++j) {
            float bv = -INFINITY;
            int be = INT_MAX;
#pragma unroll
            for (int i = 0; i < NTW; ++i) {
                const int e = lane + 32 * i;
                if (!(taken & (1u << i)) && (v[i] > bv || (v[i] == bv && e < be))) {
                    bv = v[i];
                    be = e;
                }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
                const int oe = __shfl_xor_sync(0xffffffffu, be, off);
                if (ov > bv || (ov == bv && oe < be)) {
                    bv = ov;
                    be = oe;
                }
            }
            if ((be & 31) == lane) taken |= 1u << (be >> 5);
            sel_e[j] = be;
            sel_v[j] = bv;
        }
        float ex[kMaxTopK];
        float denom = 0.f;
        for (int j = 0; j < k; ++j) {
            ex[j] = expf(sel_v[j] - sel_v[0]);
            denom += ex[j];
        }
        for (int j = 0; j < k; ++j) {
            if (lane == j) {
                p.topk_ids[static_cast<size_t>(t) * k + j] = sel_e[j];
                p.topk_w[static_cast<size_t>(t) * k + j] = ex[j] / denom;
                atomicAdd(&hist[sel_e[j]], 1);
            }
        }
    }
    __syncthreads();
    for (int e = tid; e < E; e += kThreads)
        p.blk_cnt[static_cast<size_t>(blockIdx.x) * E + e] = hist[e];

    if (p.zero_out) {
        const int rows = min(kRouterTokens, p.T - t0);
        float4* dst = reinterpret_cast<float4*>(p.zero_out + static_cast<size_t>(t0) * H);
        const int n4 = rows * H / 4;
        for (int i = tid; i < n4; i += kThreads) dst[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

template <int NTW>
cudaError_t launch_router_t(const RouterParams& p, cudaStream_t s) {
    constexpr int kEPad = 32 * NTW;
    const size_t smem = (2 * kRouterTokens * kRowStride + 2 * kEPad * kRowStride) * 2 +
                        kMaxExperts * 4;
    auto kern = router_topk_kernel<NTW>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    const int grid = (p.T + kRouterTokens - 1) / kRouterTokens;
    kern<<<grid, kThreads, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_router(const RouterParams& p, cudaStream_t s) {
    switch ((p.E + 31) / 32) {
        case 1: return launch_router_t<1>(p, s);
        case 2: return launch_router_t<2>(p, s);
        case 3: return launch_router_t<3>(p, s);
        case 4: return launch_router_t<4>(p, s);
        case 5: return launch_router_t<5>(p, s);
        case 6: return launch_router_t<6>(p, s);
        case 7: return launch_router_t<7>(p, s);
        case 8: return launch_router_t<8>(p, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace moe
