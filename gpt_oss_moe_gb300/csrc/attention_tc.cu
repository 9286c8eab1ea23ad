// Attention with sinks on the 5th-generation tensor cores, for prefill-sized
// query blocks (xserv docs/19-gpt-oss-moe.md, "Phase 19: gpt-oss-20b": §1
// model-architecture table, "attention" row -- sliding (128) / full layers,
// one sink logit per head, GQA 64 / 8 heads of dim 64; §3 on the fully
// masked tile of a sliding window).
//
// One CTA per (128 query rows, query head); the blocks start with every head
// of the query block that sees the most keys (the last, under causality),
// then the next, so that the longest blocks do not end the launch.  The
// key tiles of 128 keys are
// dealt alternately to two softmax groups, each with its own running max,
// sum and output accumulator, merged once at the end (the same online-
// softmax merge as a split over keys): while one group works on its scores
// the other's are being computed, and no exchange between threads is needed
// inside a tile.  Roles:
//   warp 0      TMA producer: the Q tile once, then K and V tiles of 128
//               keys (128-byte swizzle) into a three-slot ring.
//   warp 1      TMEM owner and MMA issuer: S_g = Q K_j^T (M = 128 queries,
//               N = 128 keys, K = 64) into group g's score buffer, and
//               O_g += P_g V_j (M = 128, N = 64, K = 128 keys) with P_g read
//               from TMEM and V as an MN-major operand (the head dimension,
//               64 bf16 = one 128-byte swizzle row, is contiguous in shared
//               memory).  Order S_0, S_1, S_2, O_0, S_3, O_1, ...: the
//               scores of a group's next tile are computed while it works
//               on the current one.
//   warps 2..5  softmax group 0 (tiles 0, 2, 4, ...), warps 6..9 group 1
//               (tiles 1, 3, 5, ...): one query row per thread (its TMEM
//               lane), all 128 scores of a tile: the row maximum, P =
//               exp2(scaled, masked score - m) as bf16 pairs into TMEM.
//               When a tile raises the row's running max m, the thread that
//               owns the row rescales its row of O_g (held in TMEM) before
//               the next product adds to it (kRescaleLog2 = 0: m stays the
//               exact running max, so the row's largest weight is exactly 1
//               in bf16).
// The sink is the starting reference max with one unit in group 0's sum, so
// it weighs in the softmax and carries no value.  A row with no visible key
// yet keeps a reference of -inf and weights of zero: the guard whose absence
// turns exp(-inf - -inf) into NaN.
//
// TMEM: S_g at columns [128 g, 128 g + 128), P_g (bf16 pairs) at
// [256 + 64 g, +64), O_g at [384 + 64 g, +64); one CTA per SM.  K and V
// tiles sit in a three-slot ring, K released after its S product, V after
// its O product.  Every mbarrier wait is bounded; a wait that gives up sets
// MOE_DEV_WAIT_TIMEOUT in the caller's status word, makes every role leave
// and frees TMEM.
#include <cudaTypedefs.h>

#include "moe_internal.cuh"
#include "ptx.cuh"
#include "trace.cuh"
#include "../../include/moe.h"

namespace moe {
namespace {

// trace build: per CTA 0 entry, 1 set-up done, 2 Q landed (MMA warp), 3 last
// S issued, 4 softmax done, 7 exit; per tile j of the CTA with blockIdx
// (0, 0) (kernel slot 1, "CTA" j): 0 S_j issued, 1 O_j issued, 2 the
// tile's group has S_j, 3 row maximum done, 4 P_j computed, 5 P_j written
MOE_TRACE_ARRAY(g_trace_attn, 2);

constexpr int kTcBq = 128;              // query rows per CTA (MMA M)
constexpr int kTcBk = 128;              // keys per tile
constexpr int kTcD = 64;                // head dim
constexpr int kTcStages = 3;            // K / V ring slots
constexpr int kTcGroups = 2;            // softmax groups (alternate key tiles)
constexpr int kTcThreads = 64 + kTcGroups * 128;   // producer, MMA issuer, softmax
constexpr uint32_t kTileBytes = kTcBk * kTcD * 2;   // 16 KB (Q, K or V tile)
// TMEM columns of group g: scores, P (bf16 pairs), O
constexpr uint32_t kColS = 0, kColP = 256, kColO = 384, kTcTmemCols = 512;
// the reference max is raised when a tile's maximum exceeds it by more than
// this (log2 domain).  0 keeps it the exact running max, so that the row's
// largest weight is exactly 1 in bf16: a larger threshold saves rescales of
// O but rounds that weight (measured: ~2 % faster, 8x the error)
constexpr float kRescaleLog2 = 0.0f;
// merge of the groups: per row and group, m, l and 32 output columns
constexpr int kXchFloats = 2 + 32;

struct AttnTcParams {
    const float* sinks;         // [Hq]
    float* out;                 // [Tq, Hq, D]
    int32_t* status;            // word 0: MOE_DEV_* bits
    int Tq, Tkv, Hq, Hkv, window, q_start;
    float scale_log2;           // log2(e) / sqrt(D)
    int poll;                   // hand-off waits: 1 = polling test_wait, 0 = try_wait
};

// 2^x by the hardware approximation (relative error ~2^-22); -inf gives 0.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Packed fp32 pairs (one instruction for two lanes of arithmetic): a pair
// of floats travels as one 64-bit register.
__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
// {y0, y1} = {x0, x1} * s2 + b2
__device__ __forceinline__ void fma_f32x2(float& y0, float& y1, float x0, float x1, uint64_t s2,
                                          uint64_t b2) {
    asm("{\n\t.reg .b64 a, d;\n\t"
        "mov.b64 a, {%2, %3};\n\t"
        "fma.rn.f32x2 d, a, %4, %5;\n\t"
        "mov.b64 {%0, %1}, d;\n\t}"
        : "=f"(y0), "=f"(y1)
        : "f"(x0), "f"(x1), "l"(s2), "l"(b2));
}
// acc2 += {x0, x1}
__device__ __forceinline__ void add_f32x2(uint64_t& acc2, float x0, float x1) {
    asm("{\n\t.reg .b64 a;\n\t"
        "mov.b64 a, {%1, %2};\n\t"
        "add.f32x2 %0, %0, a;\n\t}"
        : "+l"(acc2)
        : "f"(x0), "f"(x1));
}
__device__ __forceinline__ float f32x2_sum(uint64_t v) {
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
    return lo + hi;
}
// max(a, b, c) in one instruction
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float y;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(y) : "f"(a), "f"(b), "f"(c));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// Shared-memory descriptor of a 128-byte-swizzled tile whose 128-byte rows
// are 1024 bytes apart per group of eight, with both byte-offset fields set
// to that 1024: for a K-major operand the leading offset is unused, for an
// MN-major operand of one swizzle row's width (64 bf16) the strides between
// groups of eight rows along K are 1024 bytes whichever field holds them.
__device__ __forceinline__ uint64_t smem_desc_sw128_both(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>(1024u >> 4) << 16;
    d |= static_cast<uint64_t>(1024u >> 4) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(2u) << 61;
    return d;
}

__global__ void __launch_bounds__(kTcThreads, 1)
    attention_tc_kernel(const AttnTcParams p, const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t* q_s = smem;                                         // [128][64] bf16
    uint8_t* k_s = q_s + kTileBytes;                             // [3][128][64]
    uint8_t* v_s = k_s + kTcStages * kTileBytes;                 // [3][128][64]
    uint64_t* bars = reinterpret_cast<uint64_t*>(v_s + kTcStages * kTileBytes);
    uint64_t* q_full = bars;
    uint64_t* k_full = bars + 1;                                 // [3]
    uint64_t* v_full = k_full + kTcStages;                       // [3]
    uint64_t* k_empty = v_full + kTcStages;                      // [3]
    uint64_t* v_empty = k_empty + kTcStages;                     // [3]
    uint64_t* s_full = v_empty + kTcStages;                      // [group]
    uint64_t* s_free = s_full + kTcGroups;                       // [group]
    uint64_t* p_full = s_free + kTcGroups;                       // [group]
    uint64_t* o_full = p_full + kTcGroups;                       // [group]
    uint64_t* drain = o_full + kTcGroups;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* flags = reinterpret_cast<volatile int*>(tmem_slot + 1);
    // the groups' merge: [group][kXchFloats][128 rows]
    float* xch = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(bars) + 256);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tcta = static_cast<int>(blockIdx.y * gridDim.x + blockIdx.x);
    const bool ttile = blockIdx.x == 0 && blockIdx.y == 0;
    (void)tcta;
    (void)ttile;
    if (threadIdx.x == 0) MOE_TRACE_POINT(g_trace_attn, 0, tcta, 0);
    // blocks start in linear order (x fastest): all heads of the query block
    // with the most keys (the last, under causality) first, then the next
    const int qb = static_cast<int>(gridDim.y - 1 - blockIdx.y), h = blockIdx.x;
    const int kvh = h / (p.Hq / p.Hkv);
    const int q0 = qb * kTcBq;                                   // first query row
    const int pos0 = p.q_start + q0;                             // its position
    // key tiles: from the first key any row of the block sees to the last
    const int kv_hi = min(p.Tkv, pos0 + kTcBq);
    int kv_lo = p.window > 0 ? max(0, pos0 - p.window + 1) : 0;
    kv_lo = kv_lo / kTcBk * kTcBk;
    const int n_tiles = kv_hi > kv_lo ? (kv_hi - kv_lo + kTcBk - 1) / kTcBk : 0;
    // a hand-off wait (bounded either way)
    const auto await = [&](uint64_t* bar, uint32_t parity) {
        return p.poll ? mbar_wait_poll(smem_u32(bar), parity, flags)
                      : mbar_wait(smem_u32(bar), parity, flags);
    };

    if (threadIdx.x == 0) {
        mbar_init(smem_u32(q_full), 1);
        for (int s = 0; s < kTcStages; ++s) {
            mbar_init(smem_u32(k_full + s), 1);
            mbar_init(smem_u32(v_full + s), 1);
            mbar_init(smem_u32(k_empty + s), 1);
            mbar_init(smem_u32(v_empty + s), 1);
        }
        for (int g = 0; g < kTcGroups; ++g) {
            mbar_init(smem_u32(s_full + g), 1);
            mbar_init(smem_u32(s_free + g), 4);     // one arrival per warp of the group
            mbar_init(smem_u32(p_full + g), 4);
            mbar_init(smem_u32(o_full + g), 1);
        }
        mbar_init(smem_u32(drain), 1);
        flags[0] = 0;
        mbar_fence_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
    }
    if (warp == 1) {
        tmem_alloc<1>(smem_u32(tmem_slot), kTcTmemCols);
        tmem_relinquish<1>();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (threadIdx.x == 0) MOE_TRACE_POINT(g_trace_attn, 0, tcta, 1);

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t pol = policy_evict_last();
            mbar_arrive_expect_tx(smem_u32(q_full), kTileBytes);
            tma_load_3d(smem_u32(q_s), &tm_q, smem_u32(q_full), 0, h, q0, pol);
            bool ok = true;
            int nk = 0, nv = 0;                      // tiles whose K / V loads were issued
            for (int j = 0; j < n_tiles && ok; ++j) {
                const int s = j % kTcStages;
                const uint32_t ph = static_cast<uint32_t>(j / kTcStages) & 1u;
                const int key0 = kv_lo + j * kTcBk;
                // K_j once S_{j-3} is done with the slot, V_j once O_{j-3} is
                if (!mbar_wait(smem_u32(k_empty + s), ph ^ 1u, flags)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(smem_u32(k_full + s), kTileBytes);
                tma_load_3d(smem_u32(k_s + s * kTileBytes), &tm_k, smem_u32(k_full + s), 0, kvh,
                            key0, pol);
                ++nk;
                if (!mbar_wait(smem_u32(v_empty + s), ph ^ 1u, flags)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(smem_u32(v_full + s), kTileBytes);
                tma_load_3d(smem_u32(v_s + s * kTileBytes), &tm_v, smem_u32(v_full + s), 0, kvh,
                            key0, pol);
                ++nv;
            }
            if (!ok) {
                flags[0] = 1;
                atomicOr(p.status, MOE_DEV_WAIT_TIMEOUT);
            }
            // every load issued must land before the CTA may leave (bounded)
            mbar_wait(smem_u32(q_full), 0, nullptr);
            for (int i = nk - kTcStages > 0 ? nk - kTcStages : 0; i < nk; ++i)
                mbar_wait(smem_u32(k_full + i % kTcStages),
                          static_cast<uint32_t>(i / kTcStages) & 1u, nullptr);
            for (int i = nv - kTcStages > 0 ? nv - kTcStages : 0; i < nv; ++i)
                mbar_wait(smem_u32(v_full + i % kTcStages),
                          static_cast<uint32_t>(i / kTcStages) & 1u, nullptr);
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        const bool leader = elect_one();
        const uint32_t idesc_s = idesc_bf16_f32(kTcBq, kTcBk);
        const uint32_t idesc_o = idesc_bf16_f32(kTcBq, kTcD) | (1u << 16);   // B MN-major
        const uint64_t qd = smem_desc_sw128(smem_u32(q_s));
        // (the issuer's waits always suspend: a polling warp takes issue
        // slots from the softmax warps that share its scheduler)
        const auto wwait = [&](uint64_t* bar, uint32_t parity) {
            return __all_sync(0xffffffffu, mbar_wait(smem_u32(bar), parity, flags));
        };
        bool ok = wwait(q_full, 0);
        if (lane == 0) MOE_TRACE_POINT(g_trace_attn, 0, tcta, 2);
        // S_g = Q K_j^T (g = j % 2, the group's t-th tile, t = j / 2) once K_j
        // landed and the group has read its previous scores
        const auto issue_s = [&](int j) {
            const int s = j % kTcStages, g = j & 1, t = j >> 1;
            if (!wwait(k_full + s, static_cast<uint32_t>(j / kTcStages) & 1u) ||
                (t >= 1 && !wwait(s_free + g, static_cast<uint32_t>(t - 1) & 1u)))
                return false;
            tc_fence_after();
            if (leader) {
                const uint64_t kd = smem_desc_sw128(smem_u32(k_s + s * kTileBytes));
#pragma unroll
                for (int kk = 0; kk < kTcD / 16; ++kk)
                    tc_mma_bf16(tmem + kColS + 128u * g, qd + 2 * kk, kd + 2 * kk, idesc_s,
                                kk > 0 ? 1u : 0u);
                tc_commit(smem_u32(s_full + g));
                tc_commit(smem_u32(k_empty + s));
                if (ttile) MOE_TRACE_POINT(g_trace_attn, 1, j, 0);
                if (j == n_tiles - 1) MOE_TRACE_POINT(g_trace_attn, 0, tcta, 3);
            }
            __syncwarp();
            return true;
        };
        // O_g += P_g V_j once the group wrote P_g (the first product of a
        // group overwrites its accumulator)
        const auto issue_o = [&](int j) {
            const int s = j % kTcStages, g = j & 1, t = j >> 1;
            if (!wwait(p_full + g, static_cast<uint32_t>(t) & 1u) ||
                !wwait(v_full + s, static_cast<uint32_t>(j / kTcStages) & 1u))
                return false;
            tc_fence_after();
            if (leader) {
                const uint64_t vd = smem_desc_sw128_both(smem_u32(v_s + s * kTileBytes));
#pragma unroll
                for (int kk = 0; kk < kTcBk / 16; ++kk)      // 16 keys: 8 P columns, 2 KB of V
                    tc_mma_bf16_ts(tmem + kColO + 64u * g, tmem + kColP + 64u * g + 8u * kk,
                                   vd + 128u * kk, idesc_o, (t > 0 || kk > 0) ? 1u : 0u);
                tc_commit(smem_u32(o_full + g));
                tc_commit(smem_u32(v_empty + s));
                if (ttile) MOE_TRACE_POINT(g_trace_attn, 1, j, 1);
            }
            __syncwarp();
            return true;
        };
        for (int j = 0; j < n_tiles && ok; ++j) {
            ok = issue_s(j);
            if (ok && j >= 2) ok = issue_o(j - 2);
        }
        for (int j = n_tiles - 2 > 0 ? n_tiles - 2 : 0; j < n_tiles && ok; ++j) ok = issue_o(j);
        if (!ok && leader) {
            flags[0] = 1;
            atomicOr(p.status, MOE_DEV_WAIT_TIMEOUT);
        }
        if (leader) {
            tc_commit(smem_u32(drain));                 // every MMA issued has finished
            mbar_wait(smem_u32(drain), 0, nullptr);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ softmax groups
        const int g = (warp - 2) >> 2;                  // group: tiles g, g + 2, ...
        const int quad = warp & 3;
        const int r = quad * 32 + lane;                 // query row of this thread
        const int qrow = q0 + r;
        const int pos = p.q_start + qrow;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        const uint32_t col_s = lane_base + kColS + 128u * g;
        const uint32_t col_p = lane_base + kColP + 64u * g;
        const uint32_t col_o = lane_base + kColO + 64u * g;
        const bool tr = ttile && lane == 0 && quad == 2;   // the group's first warp
        const float sink2 = p.sinks[h] * 1.4426950408889634f;
        float m = sink2;                                // reference max (log2 domain)
        float l = (g == 0 && sink2 != -INFINITY) ? 1.f : 0.f;   // (the sink's unit, once)
        const int n_g = (n_tiles - g + 1) / 2;          // this group's tiles
        bool ok = true;
        // (the TMEM loads are warp-collective: every wait's outcome is made
        // warp-uniform first)
        for (int t = 0; t < n_g; ++t) {
            const int j = 2 * t + g;
            if (!__all_sync(0xffffffffu, await(s_full + g, static_cast<uint32_t>(t) & 1u))) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (tr) MOE_TRACE_POINT(g_trace_attn, 1, j, 2);
            // all 128 scores of the row: eight loads in flight, one wait
            uint32_t sr[8][16];
#pragma unroll
            for (int c = 0; c < 8; ++c) tmem_ld16_nowait(col_s + 16u * c, sr[c]);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 8; ++c) tmem_regs_ready(sr[c]);
            // the scores are in registers: the buffer may take the next ones
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(s_free + g));
            const int key0 = kv_lo + j * kTcBk;
            // keys [key0, key0 + 128) all visible to this row?
            const bool full = key0 + kTcBk - 1 <= pos && key0 + kTcBk <= p.Tkv &&
                              (p.window == 0 || key0 > pos - p.window);
            // raw scores, masked to -inf (the scale is positive: the maximum
            // is taken before scaling and the scale folds into the exponent)
            float mx[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) mx[i] = -INFINITY;
            if (!full) {
                // visible: tile columns [lo, hi) (not in the future, inside
                // the window, before Tkv)
                const int hi = min(pos + 1, p.Tkv) - key0;
                const int lo = p.window > 0 ? pos - p.window + 1 - key0 : 0;
                if (p.window == 0) {           // (one compare per key)
#pragma unroll
                    for (int i = 0; i < kTcBk; ++i)
                        if (i >= hi) sr[i >> 4][i & 15] = __float_as_uint(-INFINITY);
                } else {
#pragma unroll
                    for (int i = 0; i < kTcBk; ++i)
                        if (i < lo || i >= hi) sr[i >> 4][i & 15] = __float_as_uint(-INFINITY);
                }
            }
#pragma unroll
            for (int i = 0; i < kTcBk; i += 2)
                mx[(i >> 1) & 3] = fmax3(mx[(i >> 1) & 3], __uint_as_float(sr[i >> 4][i & 15]),
                                         __uint_as_float(sr[(i + 1) >> 4][(i + 1) & 15]));
            const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * p.scale_log2;
            if (tr) MOE_TRACE_POINT(g_trace_attn, 1, j, 3);
            // raise the reference only when the tile's maximum is well above it
            // (a row with no visible key so far has m = -inf: any visible key
            // raises it, and the zero sum and output rescale to zero)
            const bool raise = mt > m + kRescaleLog2;
            const float alpha = raise ? (m == -INFINITY ? 0.f : ex2(m - mt)) : 1.f;
            if (raise) m = mt;
            const float mneg = m == -INFINITY ? 0.f : -m;
            // P_g is free and O_g final for the previous tile once that
            // tile's product completed; a raised reference rescales O_g
            // (16 columns at a time: it is rare, and the scores hold most
            // registers)
            if (t > 0) {
                if (!__all_sync(0xffffffffu,
                                await(o_full + g, static_cast<uint32_t>(t - 1) & 1u))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (__any_sync(0xffffffffu, raise)) {
#pragma unroll 1
                    for (int c = 0; c < 4; ++c) {
                        uint32_t ov[16];
                        tmem_ld16_nowait(col_o + 16u * c, ov);
                        tmem_wait_ld();
                        tmem_regs_ready(ov);
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
                        tmem_st16(col_o + 16u * c, ov);
                    }
                }
            }
            // P_g = exp2(scaled score - m) as bf16 pairs, 32 keys per store
            // (scale and shift, and the row sum, on packed fp32 pairs)
            const uint64_t sc2 = f32x2(p.scale_log2, p.scale_log2);
            const uint64_t mn2 = f32x2(mneg, mneg);
            uint64_t ls2[2] = {0ull, 0ull};
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t pc[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int k0 = 32 * c + 2 * i;
                    float xa, xb;
                    fma_f32x2(xa, xb, __uint_as_float(sr[k0 >> 4][k0 & 15]),
                              __uint_as_float(sr[(k0 + 1) >> 4][(k0 + 1) & 15]), sc2, mn2);
                    const float pa = ex2(xa), pb = ex2(xb);
                    add_f32x2(ls2[i & 1], pa, pb);
                    pc[i] = pack_bf16x2(pa, pb);
                }
                tmem_st16(col_p + 16u * c, pc);
            }
            l = l * alpha + (f32x2_sum(ls2[0]) + f32x2_sum(ls2[1]));
            if (tr) MOE_TRACE_POINT(g_trace_attn, 1, j, 4);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(p_full + g));
            if (tr) MOE_TRACE_POINT(g_trace_attn, 1, j, 5);
        }
        if (threadIdx.x == 64) MOE_TRACE_POINT(g_trace_attn, 0, tcta, 4);
        // this group's output accumulator, once its last product completed
        float o[kTcD];
#pragma unroll
        for (int i = 0; i < kTcD; ++i) o[i] = 0.f;
        if (ok && n_g > 0) {
            if (__all_sync(0xffffffffu, await(o_full + g, static_cast<uint32_t>(n_g - 1) & 1u))) {
                tc_fence_after();
                uint32_t ov[4][16];
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_ld16_nowait(col_o + 16u * c, ov[c]);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    tmem_regs_ready(ov[c]);
#pragma unroll
                    for (int i = 0; i < 16; ++i) o[16 * c + i] = __uint_as_float(ov[c][i]);
                }
            } else {
                ok = false;
            }
        }
        if (!ok) {
            flags[0] = 1;
            atomicOr(p.status, MOE_DEV_WAIT_TIMEOUT);
        }
        // merge: group g finishes output columns [32 g, 32 g + 32) from its
        // own accumulator and the other group's m, l and those columns (every
        // softmax thread reaches the barrier, also after an abort)
        float* mine = xch + g * kXchFloats * kTcBq;
        mine[r] = m;
        mine[kTcBq + r] = l;
#pragma unroll
        for (int i = 0; i < 32; ++i) mine[(2 + i) * kTcBq + r] = g == 0 ? o[32 + i] : o[i];
        named_bar_sync(1, kTcGroups * 128);
        const float* other = xch + (1 - g) * kXchFloats * kTcBq;
        const float m_o = other[r], l_o = other[kTcBq + r];
        const float mm = fmaxf(m, m_o);
        const float f_me = m == -INFINITY ? 0.f : ex2(m - mm);
        const float f_o = m_o == -INFINITY ? 0.f : ex2(m_o - mm);
        const float lt = l * f_me + l_o * f_o;
        if (ok && qrow < p.Tq) {
            // out = O / l (l includes the sink's share; 0 only for a row that
            // sees no key and has no sink -- then O is 0 as well)
            const float inv = lt > 0.f ? 1.f / lt : 0.f;
            float4* dst = reinterpret_cast<float4*>(
                p.out + (static_cast<size_t>(qrow) * p.Hq + h) * kTcD + 32 * g);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float v4[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int c = 4 * i + e;
                    const float mine_c = g == 0 ? o[c] : o[32 + c];
                    v4[e] = (mine_c * f_me + other[(2 + c) * kTcBq + r] * f_o) * inv;
                }
                dst[i] = make_float4(v4[0], v4[1], v4[2], v4[3]);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<1>(tmem, kTcTmemCols);
    }
    if (threadIdx.x == 0) MOE_TRACE_POINT(g_trace_attn, 0, tcta, 7);
}

}  // namespace

size_t trace_copy_attn(unsigned long long* dst, size_t cap) {
    MOE_TRACE_COPY(g_trace_attn, dst, cap);
}

size_t attention_tc_smem_bytes() {
    return 1024 + (1 + 2 * kTcStages) * static_cast<size_t>(kTileBytes) + 256 +
           static_cast<size_t>(kTcGroups) * kXchFloats * kTcBq * 4;
}

// q [Tq, Hq, 64], k / v [Tkv, Hkv, 64] bf16 through 3-D tensor maps (dim,
// head, row), box 64 x 1 x 128 rows.
cudaError_t launch_attention_tc(const moe_attn_shape& s, const void* q, const void* k,
                                const void* v, const float* sinks, float* out, int32_t* status,
                                PFN_cuTensorMapEncodeTiled_v12000 enc, int poll,
                                cudaStream_t stream) {
    CUtensorMap tq, tk, tv;
    const auto make = [&](CUtensorMap* m, const void* base, int heads, int rows) {
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kTcD), static_cast<cuuint64_t>(heads),
                                    static_cast<cuuint64_t>(rows)};
        const cuuint64_t str[2] = {static_cast<cuuint64_t>(kTcD) * 2,
                                   static_cast<cuuint64_t>(heads) * kTcD * 2};
        const cuuint32_t box[3] = {static_cast<cuuint32_t>(kTcD), 1u, static_cast<cuuint32_t>(kTcBq)};
        const cuuint32_t estr[3] = {1, 1, 1};
        return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, str, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    };
    if (make(&tq, q, s.Hq, s.Tq) != CUDA_SUCCESS || make(&tk, k, s.Hkv, s.Tkv) != CUDA_SUCCESS ||
        make(&tv, v, s.Hkv, s.Tkv) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    AttnTcParams p;
    p.sinks = sinks;
    p.out = out;
    p.status = status;
    p.Tq = s.Tq;
    p.Tkv = s.Tkv;
    p.Hq = s.Hq;
    p.Hkv = s.Hkv;
    p.window = s.window;
    p.q_start = s.q_start;
    p.scale_log2 = 1.4426950408889634f / 8.0f;     // log2(e) / sqrt(64)
    p.poll = poll;
    const size_t smem = attention_tc_smem_bytes();
    cudaError_t err = cudaFuncSetAttribute(attention_tc_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    const int n_qb = (s.Tq + kTcBq - 1) / kTcBq;
    if (n_qb > 65535) return cudaErrorInvalidConfiguration;   // grid y limit
    const dim3 grid(s.Hq, n_qb);
    attention_tc_kernel<<<grid, kTcThreads, smem, stream>>>(p, tq, tk, tv);
    return cudaGetLastError();
}

}  // namespace moe
