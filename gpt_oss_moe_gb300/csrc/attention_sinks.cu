// Attention with sinks and an optional sliding window, the other half of a
// gpt-oss block (xserv docs/19-gpt-oss-moe.md, "Phase 19: gpt-oss-20b": §1
// model-architecture table, "attention" row -- sliding (128) / full layers
// alternate, one learnable sink logit per head, 64 query / 8 KV heads of
// dim 64; §3 on the fully masked tile of a sliding window).
//
// One CTA per (64 query rows, query head, key split), four warps of 16
// rows.  Small grids (decode: one query block per head) split each block's
// key tiles over several CTAs (flash-decoding); each writes its unnormalised
// output with its running max and sum, and a second kernel merges the splits
// and adds the sink's share once.  Per KV
// tile of 64 keys: S = Q K^T on the tensor cores (mma.sync m16n8k16, bf16 in,
// fp32 out), scale and mask, online softmax in the exp2 domain, O += P V
// (P rounded to bf16).  The sink enters as the running max's starting value
// with one unit in the denominator (exp2(sink - m) after rescaling), so it
// weighs in the softmax and carries no value.  A row whose tile is fully
// masked (its tile max is -inf: all keys in the future or slid out of the
// window) leaves the row's state untouched -- the guard whose absence, with
// a running max of -inf, turns exp(-inf - -inf) into NaN.
#include <atomic>

#include "moe_internal.cuh"
#include "ptx.cuh"
#include "../../include/moe.h"

namespace moe {
namespace {

constexpr int kD = 64;          // head dim
constexpr int kBq = 64;         // query rows per CTA
constexpr int kBk = 64;         // keys per tile
constexpr int kLd = kD + 8;     // shared-memory row stride (bf16): 144 B
constexpr int kThreadsAttn = 128;

struct AttnParams {
    const __nv_bfloat16* q;     // [Tq, Hq, D]
    const __nv_bfloat16* k;     // [Tkv, Hkv, D]
    const __nv_bfloat16* v;     // [Tkv, Hkv, D]
    const float* sinks;         // [Hq]
    float* out;                 // [Tq, Hq, D]
    int Tq, Tkv, Hq, Hkv, window, q_start;
    float scale_log2;           // log2(e) / sqrt(D)
    int group;                  // 1: a CTA's 64 rows are (query, head) pairs of one
                                // KV head (64 / rep queries x its rep query heads),
                                // so its K/V tiles serve every head that reads
                                // them; 0: 64 queries of one query head
    int nsplit;                 // key splits per query block (grid.z)
    float* part_o;              // [nsplit, Tq, Hq, D] unnormalised (nsplit > 1)
    float2* part_ml;            // [nsplit, Tq, Hq] (running max log2, sum)
};

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4],
                                               uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// Rows [r0, r0 + 64) of a [T, H, D] tensor's head h into shared memory,
// copied asynchronously (cp.async, 16 B per thread and step; rows past T are
// zero-filled: source size 0).
__device__ __forceinline__ void load_tile_async(__nv_bfloat16* dst, const __nv_bfloat16* src,
                                                int r0, int T, int H, int h) {
    for (int i = threadIdx.x; i < 64 * (kD / 8); i += kThreadsAttn) {
        const int r = i / (kD / 8), c = (i % (kD / 8)) * 8;
        const bool in = r0 + r < T;
        const __nv_bfloat16* g = in ? src + (static_cast<size_t>(r0 + r) * H + h) * kD + c : src;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;"
                     ::"r"(smem_u32(dst + r * kLd + c)), "l"(g), "r"(in ? 16 : 0) : "memory");
    }
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Four 8x8 bf16 matrices, transposed: lane L gives the address of row L % 8
// of matrix L / 8; each register receives, for its matrix, the elements
// (2t, g) and (2t + 1, g) -- a B fragment of m16n8k16 from a [k][n] tile.
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                              uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

__global__ void __launch_bounds__(kThreadsAttn) attention_sinks_kernel(const AttnParams p) {
    __shared__ __align__(16) __nv_bfloat16 qs[kBq * kLd];
    __shared__ __align__(16) __nv_bfloat16 ks[2][kBk * kLd];   // double-buffered
    __shared__ __align__(16) __nv_bfloat16 vs[2][kBk * kLd];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    // later query blocks see the most keys (causal): they start first
    const int qb = gridDim.x - 1 - blockIdx.x;
    const int rep = p.Hq / p.Hkv;
    const int qpb = p.group ? kBq / rep : kBq;          // queries per CTA
    const int q_first = qb * qpb;
    const int q_last = min(q_first + qpb, p.Tq) - 1;
    const int hk = p.group ? static_cast<int>(blockIdx.y) : static_cast<int>(blockIdx.y) / rep;
    // row rho of the CTA: query q_first + rho / rep and head hk * rep + rho % rep
    // (grouped), or query q_first + rho of head blockIdx.y
    const auto query_of = [&](int rho) { return q_first + (p.group ? rho / rep : rho); };
    const auto head_of = [&](int rho) {
        return p.group ? hk * rep + rho % rep : static_cast<int>(blockIdx.y);
    };

    for (int idx = threadIdx.x; idx < kBq * (kD / 8); idx += kThreadsAttn) {
        const int rho = idx / (kD / 8), c = (idx % (kD / 8)) * 8;
        const int i = query_of(rho);
        uint4 val = make_uint4(0u, 0u, 0u, 0u);
        if (i <= q_last)
            val = *reinterpret_cast<const uint4*>(
                p.q + (static_cast<size_t>(i) * p.Hq + head_of(rho)) * kD + c);
        *reinterpret_cast<uint4*>(qs + rho * kLd + c) = val;
    }
    __syncthreads();

    // this warp's Q fragments (16 rows x 64), kept in registers
    uint32_t qa[4][4];
    {
        const __nv_bfloat16* base = qs + (warp * 16) * kLd;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const int c = kk * 16 + 2 * t;
            qa[kk][0] = *reinterpret_cast<const uint32_t*>(base + g * kLd + c);
            qa[kk][1] = *reinterpret_cast<const uint32_t*>(base + (g + 8) * kLd + c);
            qa[kk][2] = *reinterpret_cast<const uint32_t*>(base + g * kLd + c + 8);
            qa[kk][3] = *reinterpret_cast<const uint32_t*>(base + (g + 8) * kLd + c + 8);
        }
    }

    // rows g and g + 8 of this warp: positions, running max (log2 domain),
    // denominator, output accumulators
    const int row_a = query_of(warp * 16 + g), row_b = query_of(warp * 16 + g + 8);
    const int h_a = head_of(warp * 16 + g), h_b = head_of(warp * 16 + g + 8);
    const bool ok_a = row_a <= q_last, ok_b = row_b <= q_last;
    const int pos_a = p.q_start + row_a, pos_b = p.q_start + row_b;
    const float sink2_a = p.sinks[h_a] * 1.4426950408889634f;
    const float sink2_b = p.sinks[h_b] * 1.4426950408889634f;
    // split runs start without the sink (the merge adds it once)
    const bool whole = p.nsplit == 1;
    float m_a = whole ? sink2_a : -INFINITY, m_b = whole ? sink2_b : -INFINITY;
    float l_a = !whole || (isinf(sink2_a) && sink2_a < 0.f) ? 0.f : 1.f;
    float l_b = !whole || (isinf(sink2_b) && sink2_b < 0.f) ? 0.f : 1.f;
    float o[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;

    // key tiles that any row of this CTA can see
    const int kv_hi = min(p.Tkv, p.q_start + q_last + 1);
    int kv_lo = p.window > 0 ? max(0, p.q_start + q_first - p.window + 1) : 0;
    kv_lo = kv_lo / kBk * kBk;
    // this split's share of the block's key tiles
    const int ntile = kv_hi > kv_lo ? (kv_hi - kv_lo + kBk - 1) / kBk : 0;
    const int per = (ntile + p.nsplit - 1) / p.nsplit;
    const int t_lo = blockIdx.z * per, t_hi = min(ntile, t_lo + per);

    // tile it + 1 loads while tile it computes
    if (t_lo < t_hi) {
        load_tile_async(ks[0], p.k, kv_lo + t_lo * kBk, p.Tkv, p.Hkv, hk);
        load_tile_async(vs[0], p.v, kv_lo + t_lo * kBk, p.Tkv, p.Hkv, hk);
        cp_async_commit();
    }
    for (int it = t_lo; it < t_hi; ++it) {
        const int kv0 = kv_lo + it * kBk;
        const int buf = (it - t_lo) & 1;
        if (it + 1 < t_hi) {
            // buffer buf ^ 1 was last read in the previous iteration, which
            // ended with a barrier
            load_tile_async(ks[buf ^ 1], p.k, kv0 + kBk, p.Tkv, p.Hkv, hk);
            load_tile_async(vs[buf ^ 1], p.v, kv0 + kBk, p.Tkv, p.Hkv, hk);
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();

        // S = Q K^T: 16 x 64 per warp, 8 n-tiles of 8 keys
        float s[8][4];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
            const __nv_bfloat16* kr = ks[buf] + (j * 8 + g) * kLd;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const int c = kk * 16 + 2 * t;
                mma_bf16_16816(s[j], qa[kk], *reinterpret_cast<const uint32_t*>(kr + c),
                               *reinterpret_cast<const uint32_t*>(kr + c + 8));
            }
        }
        // scale, mask (future keys, keys that slid out of the window, keys
        // past Tkv), tile row maxima
        float tm_a = -INFINITY, tm_b = -INFINITY;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int kv = kv0 + j * 8 + 2 * t + (e & 1);
                const int pos = e < 2 ? pos_a : pos_b;
                const bool ok = kv <= pos && kv < p.Tkv && (p.window <= 0 || kv > pos - p.window);
                const float v = ok ? s[j][e] * p.scale_log2 : -INFINITY;
                s[j][e] = v;
                if (e < 2) tm_a = fmaxf(tm_a, v); else tm_b = fmaxf(tm_b, v);
            }
        }
        tm_a = fmaxf(tm_a, __shfl_xor_sync(0xffffffffu, tm_a, 1));
        tm_a = fmaxf(tm_a, __shfl_xor_sync(0xffffffffu, tm_a, 2));
        tm_b = fmaxf(tm_b, __shfl_xor_sync(0xffffffffu, tm_b, 1));
        tm_b = fmaxf(tm_b, __shfl_xor_sync(0xffffffffu, tm_b, 2));
        // empty-tile guard: a fully masked row keeps its state (its p = 0)
        const bool live_a = tm_a != -INFINITY, live_b = tm_b != -INFINITY;
        const float mn_a = live_a ? fmaxf(m_a, tm_a) : m_a;
        const float mn_b = live_b ? fmaxf(m_b, tm_b) : m_b;
        const float al_a = live_a && m_a != -INFINITY ? exp2f(m_a - mn_a) : (live_a ? 0.f : 1.f);
        const float al_b = live_b && m_b != -INFINITY ? exp2f(m_b - mn_b) : (live_b ? 0.f : 1.f);
        m_a = mn_a;
        m_b = mn_b;
        float ps_a = 0.f, ps_b = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            s[j][0] = live_a ? exp2f(s[j][0] - m_a) : 0.f;
            s[j][1] = live_a ? exp2f(s[j][1] - m_a) : 0.f;
            s[j][2] = live_b ? exp2f(s[j][2] - m_b) : 0.f;
            s[j][3] = live_b ? exp2f(s[j][3] - m_b) : 0.f;
            ps_a += s[j][0] + s[j][1];
            ps_b += s[j][2] + s[j][3];
            o[j][0] *= al_a;
            o[j][1] *= al_a;
            o[j][2] *= al_b;
            o[j][3] *= al_b;
        }
        ps_a += __shfl_xor_sync(0xffffffffu, ps_a, 1);
        ps_a += __shfl_xor_sync(0xffffffffu, ps_a, 2);
        ps_b += __shfl_xor_sync(0xffffffffu, ps_b, 1);
        ps_b += __shfl_xor_sync(0xffffffffu, ps_b, 2);
        l_a = l_a * al_a + ps_a;
        l_b = l_b * al_b + ps_b;

        // O += P V: P from the S accumulators (bf16), V columns as B
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            uint32_t pa[4];
            pa[0] = pack_bf16(s[2 * kk][0], s[2 * kk][1]);
            pa[1] = pack_bf16(s[2 * kk][2], s[2 * kk][3]);
            pa[2] = pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]);
            pa[3] = pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3]);
            // V rows kk*16 .. +15 (k) x columns 8j .. 8j+15 (two n-tiles)
            const int mat = lane >> 3;
            const uint32_t vrow = smem_u32(vs[buf] + (kk * 16 + (mat & 1) * 8 + (lane & 7)) * kLd +
                                           (mat >> 1) * 8);
#pragma unroll
            for (int j = 0; j < 8; j += 2) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4_trans(vrow + j * 16, b0, b1, b2, b3);
                mma_bf16_16816(o[j], pa, b0, b1);
                mma_bf16_16816(o[j + 1], pa, b2, b3);
            }
        }
        __syncthreads();                      // both buffers' readers are done
    }

    if (!whole) {
        // this split's unnormalised output, running max and sum
        const size_t plane = static_cast<size_t>(blockIdx.z) * p.Tq * p.Hq;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int c = j * 8 + 2 * t;
            if (ok_a)
                *reinterpret_cast<float2*>(p.part_o + ((plane + static_cast<size_t>(row_a) * p.Hq + h_a) * kD + c)) =
                    make_float2(o[j][0], o[j][1]);
            if (ok_b)
                *reinterpret_cast<float2*>(p.part_o + ((plane + static_cast<size_t>(row_b) * p.Hq + h_b) * kD + c)) =
                    make_float2(o[j][2], o[j][3]);
        }
        if (t == 0) {
            if (ok_a) p.part_ml[plane + static_cast<size_t>(row_a) * p.Hq + h_a] = make_float2(m_a, l_a);
            if (ok_b) p.part_ml[plane + static_cast<size_t>(row_b) * p.Hq + h_b] = make_float2(m_b, l_b);
        }
        return;
    }
    // out = O / l (l includes the sink's share)
    const float inv_a = l_a > 0.f ? 1.f / l_a : 0.f, inv_b = l_b > 0.f ? 1.f / l_b : 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int c = j * 8 + 2 * t;
        if (ok_a) {
            float* dst = p.out + (static_cast<size_t>(row_a) * p.Hq + h_a) * kD + c;
            *reinterpret_cast<float2*>(dst) = make_float2(o[j][0] * inv_a, o[j][1] * inv_a);
        }
        if (ok_b) {
            float* dst = p.out + (static_cast<size_t>(row_b) * p.Hq + h_b) * kD + c;
            *reinterpret_cast<float2*>(dst) = make_float2(o[j][2] * inv_b, o[j][3] * inv_b);
        }
    }
}

// Merge of the key splits: one CTA of 64 threads (one per output column) per
// (query row, head).  M = max(sink, m_s), L = exp2(sink - M) + sum l_s
// exp2(m_s - M), out = sum o_s exp2(m_s - M) / L; splits without live keys
// (m_s = -inf) add nothing.
__global__ void __launch_bounds__(kD) attention_merge_kernel(const AttnParams p) {
    const int r = blockIdx.x, h = blockIdx.y, d = threadIdx.x;
    const size_t rh = static_cast<size_t>(r) * p.Hq + h;
    const size_t plane = static_cast<size_t>(p.Tq) * p.Hq;
    const float sink2 = p.sinks[h] * 1.4426950408889634f;
    float M = sink2;
    for (int z = 0; z < p.nsplit; ++z) M = fmaxf(M, p.part_ml[z * plane + rh].x);
    float L = M == -INFINITY || sink2 == -INFINITY ? 0.f : exp2f(sink2 - M);
    float acc = 0.f;
    for (int z = 0; z < p.nsplit; ++z) {
        const float2 ml = p.part_ml[z * plane + rh];
        if (ml.x == -INFINITY) continue;
        const float f = exp2f(ml.x - M);
        L += ml.y * f;
        acc += p.part_o[(z * plane + rh) * kD + d] * f;
    }
    p.out[rh * kD + d] = L > 0.f ? acc / L : 0.f;
}

// Key splits: enough CTAs for about four waves, at least two key tiles per
// split (counted for the last query block, the widest under causality), at
// most kMaxSplit.  Grids of four waves or more need none.
constexpr int kMaxSplit = 32;
// Grouped rows when all queries fit in one CTA's 64 / rep (decode steps):
// measured, grouping took a 4096-key decode step from 37.4 to 19.9 us but
// slowed prefill (T = 4096: 862.6 -> 909.7 us full, 96.7 -> 117.0 us with a
// 128-key window; 64 queries: 43.4 -> 49.7 us).
bool attn_grouped(const moe_attn_shape& s) {
    const int rep = s.Hq / s.Hkv;
    return rep <= kBq && kBq % rep == 0 && s.Tq <= kBq / rep;
}

int attn_qpb(const moe_attn_shape& s) { return attn_grouped(s) ? kBq / (s.Hq / s.Hkv) : kBq; }

int attn_splits(const moe_attn_shape& s, int sms) {
    const int qpb = attn_qpb(s);
    const int qb = (s.Tq + qpb - 1) / qpb;
    const long long ctas = static_cast<long long>(qb) * (attn_grouped(s) ? s.Hkv : s.Hq);
    if (ctas == 0) return 1;                               // Tq == 0: nothing to split
    const int kv_hi = min(s.Tkv, s.q_start + s.Tq);
    int kv_lo = s.window > 0 ? max(0, s.q_start + (qb - 1) * qpb - s.window + 1) : 0;
    kv_lo = kv_lo / kBk * kBk;
    const int tiles = kv_hi > kv_lo ? (kv_hi - kv_lo + kBk - 1) / kBk : 0;
    long long n = (4LL * sms + ctas - 1) / ctas;
    if (n > tiles / 2) n = tiles / 2;
    if (n > kMaxSplit) n = kMaxSplit;
    return n < 1 ? 1 : static_cast<int>(n);
}

int sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return 152;
    }
    return sms;
}

bool attn_shape_ok(const moe_attn_shape& s) {
    return s.D == kD && s.Hkv >= 1 && s.Hq >= s.Hkv && s.Hq % s.Hkv == 0 && s.Hq <= 65535 &&
           s.Tq >= 0 && s.Tkv >= 1 && s.q_start >= 0 && s.q_start + s.Tq <= s.Tkv &&
           s.window >= 0;
}

size_t attn_ws_bytes(const moe_attn_shape& s, int nsplit) {
    if (nsplit <= 1) return 0;
    const size_t rows = static_cast<size_t>(nsplit) * s.Tq * s.Hq;
    return rows * kD * sizeof(float) + 256 + rows * sizeof(float2);
}

// Prefill-sized calls run on the tcgen05 kernel (attention_tc.cu): at least
// kTcMinTq queries (one 128-row block per query head keeps few SMs busy
// below that, where the 64-row kernel with key splits does better).
// "attn_tc" tuning: 0 = automatic, 1 = never, 2 = always.
constexpr int kTcMinTq = 512;
std::atomic<int> g_attn_tc{0};
// softmax hand-off waits of the tcgen05 kernel: 1 polling
// (mbarrier.test_wait), 0 suspending (mbarrier.try_wait; measured faster:
// a polling warp takes issue slots from the other softmax group)
std::atomic<int> g_attn_poll{0};

bool attn_use_tc(const moe_attn_shape& s) {
    const int mode = g_attn_tc.load();
    return mode == 2 || (mode == 0 && s.Tq >= kTcMinTq);
}

}  // namespace

size_t attention_tc_smem_bytes();
cudaError_t launch_attention_tc(const moe_attn_shape& s, const void* q, const void* k,
                                const void* v, const float* sinks, float* out, int32_t* status,
                                PFN_cuTensorMapEncodeTiled_v12000 enc, int poll,
                                cudaStream_t stream);

int set_attn_tc_mode(int mode) {
    if (mode < 0 || mode > 2) return MOE_ERR_ARG;
    g_attn_tc.store(mode);
    return MOE_OK;
}

int set_attn_poll(int mode) {
    if (mode != 0 && mode != 1) return MOE_ERR_ARG;
    g_attn_poll.store(mode);
    return MOE_OK;
}

}  // namespace moe

using namespace moe;

extern "C" size_t moe_attention_workspace_bytes(const moe_attn_shape* shape) {
    if (!shape || !attn_shape_ok(*shape)) return 0;
    // the tcgen05 kernel: a status word
    if (attn_use_tc(*shape)) return 256;
    return attn_ws_bytes(*shape, attn_splits(*shape, sm_count()));
}

extern "C" moe_status moe_attention_sinks(const moe_attn_shape* shape, const void* q,
                                          const void* k, const void* v, const float* sinks,
                                          float* out, void* workspace, size_t workspace_bytes,
                                          cudaStream_t stream) {
    if (!shape) return MOE_ERR_ARG;
    const moe_attn_shape s = *shape;
    if (!attn_shape_ok(s)) return MOE_ERR_SHAPE;
    if (s.Tq == 0) return MOE_OK;            // nothing to do (pointers may be null)
    if (!q || !k || !v || !sinks || !out) return MOE_ERR_ARG;
    for (const void* ptr : {q, k, v, static_cast<const void*>(out)})
        if (reinterpret_cast<uintptr_t>(ptr) & 15) return MOE_ERR_ALIGN;
    if (reinterpret_cast<uintptr_t>(sinks) & 3) return MOE_ERR_ALIGN;
    if (attn_use_tc(s)) {
        // status word at the workspace's start, cleared for this call
        if (!workspace || workspace_bytes < 256) return MOE_ERR_WORKSPACE;
        if (reinterpret_cast<uintptr_t>(workspace) & 15) return MOE_ERR_ALIGN;
        PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
        if (!enc) return MOE_ERR_CUDA;
        int32_t* status = static_cast<int32_t*>(workspace);
        if (cudaMemsetAsync(status, 0, sizeof(int32_t), stream) != cudaSuccess) return MOE_ERR_CUDA;
        return launch_attention_tc(s, q, k, v, sinks, out, status, enc, g_attn_poll.load(),
                                   stream) == cudaSuccess
                   ? MOE_OK : MOE_ERR_CUDA;
    }
    const int nsplit = attn_splits(s, sm_count());
    const size_t need = attn_ws_bytes(s, nsplit);
    if (need > 0 && (!workspace || workspace_bytes < need)) return MOE_ERR_WORKSPACE;
    if (need > 0 && (reinterpret_cast<uintptr_t>(workspace) & 15)) return MOE_ERR_ALIGN;
    AttnParams p;
    p.q = static_cast<const __nv_bfloat16*>(q);
    p.k = static_cast<const __nv_bfloat16*>(k);
    p.v = static_cast<const __nv_bfloat16*>(v);
    p.sinks = sinks;
    p.out = out;
    p.Tq = s.Tq;
    p.Tkv = s.Tkv;
    p.Hq = s.Hq;
    p.Hkv = s.Hkv;
    p.window = s.window;
    p.q_start = s.q_start;
    p.scale_log2 = 1.4426950408889634f / 8.0f;     // log2(e) / sqrt(64)
    p.nsplit = nsplit;
    p.group = attn_grouped(s) ? 1 : 0;
    const size_t rows = static_cast<size_t>(nsplit) * s.Tq * s.Hq;
    p.part_o = static_cast<float*>(workspace);
    p.part_ml = need > 0 ? reinterpret_cast<float2*>(static_cast<uint8_t*>(workspace) +
                                                     (rows * kD * sizeof(float) + 255) / 256 * 256)
                         : nullptr;
    const int qpb = attn_qpb(s);
    const dim3 grid((s.Tq + qpb - 1) / qpb, p.group ? s.Hkv : s.Hq, nsplit);
    attention_sinks_kernel<<<grid, kThreadsAttn, 0, stream>>>(p);
    if (nsplit > 1)
        attention_merge_kernel<<<dim3(s.Tq, s.Hq), kD, 0, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
