// Attention with sinks on the 5th-generation tensor cores, for prefill-sized
// query blocks (xserv docs/19-gpt-oss-moe.md, "Phase 19: gpt-oss-20b": §1
// model-architecture table, "attention" row -- sliding (128) / full layers,
// one sink logit per head, GQA 64 / 8 heads of dim 64; §3 on the fully
// masked tile of a sliding window).
//
// One CTA per (128 query rows, query head); roles:
//   warp 0      TMA producer: the Q tile once, then K and V tiles of 128
//               keys (128-byte swizzle) into a three-slot ring.
//   warp 1      TMEM owner and MMA issuer: S = Q K^T (M = 128 queries,
//               N = 128 keys, K = 64, into TMEM), then O_j = P_j V_j
//               (M = 128, N = 64, K = 128 keys) with P read from TMEM and V
//               as an MN-major operand (the head dimension, 64 bf16 = one
//               128-byte swizzle row, is contiguous in shared memory).  The
//               warp issues S_{j+1} before O_j, so the tensor cores compute
//               the next scores while the softmax warps work.
//   warps 2..17 softmax, four warps per TMEM lane quadrant, a query row per
//               thread and a quarter of the keys (and of the output columns)
//               per warp: load the part's 32 scores (one wait for two
//               loads), take the row maximum with the other parts through
//               shared memory, write P_j = exp2(scaled, masked score - max)
//               (bf16) to TMEM, and accumulate O_{j-1} into registers with
//               the running-max rescale O <- O * exp2(m_{j-2} - m_{j-1}) + O_{j-1}.
// The sink is the running max's starting value with one unit in the
// denominator, so it weighs in the softmax and carries no value.  A row with
// no visible key yet keeps a running max of -inf and weights of zero: the
// guard whose absence turns exp(-inf - -inf) into NaN.
//
// TMEM: two score buffers at columns [0, 256) (S_{j+1} is computed while
// the softmax reads S_j), P at [256, 320) (bf16 pairs), O_j at [320, 384);
// one CTA per SM.  K and V tiles
// sit in a three-slot ring, K released after its S product, V after its O
// product.  Every mbarrier wait is bounded; a wait that gives up sets
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
// (0, 0) (kernel slot 1, "CTA" j): 0 S_j issued, 1 O_{j-1} issued, 2 softmax
// has S_j, 3 pass 1 done, 4 O_{j-1} accumulated, 5 P_j written
MOE_TRACE_ARRAY(g_trace_attn, 2);

constexpr int kTcBq = 128;              // query rows per CTA (MMA M)
constexpr int kTcBk = 128;              // keys per tile
constexpr int kTcD = 64;                // head dim
constexpr int kTcStages = 3;            // K / V ring slots
constexpr int kSmxWarps = 16;                  // softmax warps: 4 per TMEM lane quadrant
constexpr int kSmxParts = kSmxWarps / 4;       // column parts of a row
constexpr int kSmxKeys = kTcBk / kSmxParts;    // keys per thread and tile (32)
constexpr int kSmxCols = 64 / kSmxParts;       // output columns per thread (16)
constexpr int kSmxThreads = kSmxWarps * 32;
constexpr int kTcThreads = 64 + kSmxThreads;   // producer, MMA issuer, softmax
constexpr uint32_t kTileBytes = kTcBk * kTcD * 2;   // 16 KB (Q, K or V tile)
// TMEM: two score buffers, P (bf16 pairs), O_j
constexpr uint32_t kColS = 0, kColP = 256, kColO = 320, kTcTmemCols = 512;

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
    uint64_t* s_full = v_empty + kTcStages;                      // [2]
    uint64_t* s_free = s_full + 2;                               // [2]
    uint64_t* p_full = s_free + 2;
    uint64_t* o_full = p_full + 1;
    uint64_t* drain = o_full + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* flags = reinterpret_cast<volatile int*>(tmem_slot + 1);
    // softmax exchange: [2 tile parities][parts][128 rows] maxima, then
    // [parts][128 rows] sums
    float* red_s = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(bars) + 256);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tcta = static_cast<int>(blockIdx.y * gridDim.x + blockIdx.x);
    const bool ttile = blockIdx.x == 0 && blockIdx.y == 0;
    if (threadIdx.x == 0) MOE_TRACE_POINT(g_trace_attn, 0, tcta, 0);
    // query blocks with the most keys (the last, under causality) first
    const int qb = static_cast<int>(gridDim.x - 1 - blockIdx.x), h = blockIdx.y;
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
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(s_full + b), 1);
            mbar_init(smem_u32(s_free + b), kSmxWarps);   // one arrival per softmax warp
        }
        mbar_init(smem_u32(p_full), kSmxWarps);
        mbar_init(smem_u32(o_full), 1);
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
        // Order: S_0, S_1, O_0, S_2, O_1, ...: the scores of the next tile
        // (second TMEM buffer) are computed while the softmax works on the
        // current one, and O_j waits only for P_j.
        const bool leader = elect_one();
        const uint32_t idesc_s = idesc_bf16_f32(kTcBq, kTcBk);
        const uint32_t idesc_o = idesc_bf16_f32(kTcBq, kTcD) | (1u << 16);   // B MN-major
        const uint64_t qd = smem_desc_sw128(smem_u32(q_s));
        const auto wwait = [&](uint64_t* bar, uint32_t parity) {
            return __all_sync(0xffffffffu, await(bar, parity));
        };
        bool ok = wwait(q_full, 0);
        if (lane == 0) MOE_TRACE_POINT(g_trace_attn, 0, tcta, 2);
        // O_j = P_j V_j (after the softmax wrote P_j)
        const auto issue_o = [&](int j) {
            const int s = j % kTcStages;
            if (!wwait(p_full, static_cast<uint32_t>(j) & 1u) ||
                !wwait(v_full + s, static_cast<uint32_t>(j / kTcStages) & 1u))
                return false;
            tc_fence_after();
            if (leader) {
                const uint64_t vd = smem_desc_sw128_both(smem_u32(v_s + s * kTileBytes));
#pragma unroll
                for (int kk = 0; kk < kTcBk / 16; ++kk)      // 16 keys: 8 P columns, 2 KB of V
                    tc_mma_bf16_ts(tmem + kColO, tmem + kColP + 8u * kk, vd + 128u * kk, idesc_o,
                                   kk > 0 ? 1u : 0u);
                tc_commit(smem_u32(o_full));
                tc_commit(smem_u32(v_empty + s));
                if (ttile) MOE_TRACE_POINT(g_trace_attn, 1, j + 1, 1);
            }
            __syncwarp();
            return true;
        };
        for (int j = 0; j < n_tiles && ok; ++j) {
            const int s = j % kTcStages, sb = j & 1;
            // S_j = Q K_j^T into buffer j % 2 once K_j landed and the softmax
            // read S_{j-2} from that buffer
            if (!wwait(k_full + s, static_cast<uint32_t>(j / kTcStages) & 1u) ||
                (j >= 2 && !wwait(s_free + sb, static_cast<uint32_t>((j - 2) >> 1) & 1u))) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (leader) {
                const uint64_t kd = smem_desc_sw128(smem_u32(k_s + s * kTileBytes));
#pragma unroll
                for (int kk = 0; kk < kTcD / 16; ++kk)
                    tc_mma_bf16(tmem + kColS + 128u * sb, qd + 2 * kk, kd + 2 * kk, idesc_s,
                                kk > 0 ? 1u : 0u);
                tc_commit(smem_u32(s_full + sb));
                tc_commit(smem_u32(k_empty + s));
                if (ttile) MOE_TRACE_POINT(g_trace_attn, 1, j, 0);
                if (j == n_tiles - 1) MOE_TRACE_POINT(g_trace_attn, 0, tcta, 3);
            }
            __syncwarp();
            if (j > 0 && !issue_o(j - 1)) {
                ok = false;
                break;
            }
        }
        if (ok && n_tiles > 0 && !issue_o(n_tiles - 1)) ok = false;
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
        // ------------------------------------------------ softmax (warps 2..17)
        // kSmxParts warps per TMEM lane quadrant: the thread of row r in part
        // hf takes key columns [32 hf, 32 hf + 32) of each score tile and
        // output columns [16 hf, 16 hf + 16).  The parts of a row agree on
        // the running max through shared memory once per tile; each keeps
        // its own part of the running sum (the same rescales apply to all),
        // added once at the end.
        const int quad = warp & 3;
        const int hf = (warp - 2) >> 2;
        const int r = quad * 32 + lane;                 // query row of this thread
        const int qrow = q0 + r;
        const int pos = p.q_start + qrow;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        const float sink2 = p.sinks[h] * 1.4426950408889634f;
        float m = sink2;                                // running max (log2 domain)
        float l = (hf == 0 && sink2 != -INFINITY) ? 1.f : 0.f;   // (the sink's unit, once)
        float o[kSmxCols];
#pragma unroll
        for (int i = 0; i < kSmxCols; ++i) o[i] = 0.f;
        float alpha_prev = 1.f;                         // rescale for O_{j-1}
        bool ok = true;
        // (the TMEM loads are warp-collective: the wait's outcome is made
        // warp-uniform first)
        const auto accumulate_o = [&](int j, float alpha) {
            if (!__all_sync(0xffffffffu, await(o_full, static_cast<uint32_t>(j) & 1u)))
                return false;
            tc_fence_after();
            uint32_t v[16];
            tmem_ld16_nowait(lane_base + kColO + kSmxCols * hf, v);
            tmem_wait_ld();
            tmem_regs_ready(v);
#pragma unroll
            for (int i = 0; i < kSmxCols; ++i) o[i] = fmaf(o[i], alpha, __uint_as_float(v[i]));
            return true;
        };
        // Every decision to stop is taken by all softmax threads at once (the
        // per-tile barrier reduces their outcomes), so that none of them
        // waits at a barrier the others have left.
        for (int j = 0; j < n_tiles; ++j) {
            const int sb = j & 1;
            const bool got =
                __all_sync(0xffffffffu, ok && await(s_full + sb, static_cast<uint32_t>(j >> 1) & 1u));
            tc_fence_after();
            if (ttile && threadIdx.x == 64) MOE_TRACE_POINT(g_trace_attn, 1, j, 2);
            // this part's 32 scores, two loads in flight, one wait
            uint32_t sr[2][16];
            const uint32_t sbase = lane_base + kColS + 128u * sb + kSmxKeys * hf;
            if (got) {
                tmem_ld16_nowait(sbase, sr[0]);
                tmem_ld16_nowait(sbase + 16u, sr[1]);
                tmem_wait_ld();
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) sr[0][i] = sr[1][i] = 0u;
            }
            tmem_regs_ready(sr[0]);
            tmem_regs_ready(sr[1]);
            // the scores are in registers: the buffer may take S_{j+2}
            tc_fence_before();
            __syncwarp();
            if (lane == 0 && got) mbar_arrive(smem_u32(s_free + sb));
            const int key0 = kv_lo + j * kTcBk + kSmxKeys * hf;
            // keys [key0, key0 + 32) all visible to this row?
            const bool full = key0 + kSmxKeys - 1 <= pos && key0 + kSmxKeys <= p.Tkv &&
                              (p.window == 0 || key0 > pos - p.window);
            float x[kSmxKeys];
            float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
            if (full) {
#pragma unroll
                for (int i = 0; i < kSmxKeys; ++i) {
                    x[i] = __uint_as_float(sr[i >> 4][i & 15]) * p.scale_log2;
                    mx[i & 3] = fmaxf(mx[i & 3], x[i]);
                }
            } else {
#pragma unroll
                for (int i = 0; i < kSmxKeys; ++i) {
                    const int key = key0 + i;
                    const bool vis =
                        key <= pos && key < p.Tkv && (p.window == 0 || key > pos - p.window);
                    x[i] = vis ? __uint_as_float(sr[i >> 4][i & 15]) * p.scale_log2 : -INFINITY;
                    mx[i & 3] = fmaxf(mx[i & 3], x[i]);
                }
            }
            // the row's tile maximum: all parts
            float* red = red_s + (j & 1) * kSmxParts * kTcBq;
            red[hf * kTcBq + r] = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
            if (!named_bar_and(1, kSmxThreads, got)) {
                ok = false;                             // every softmax thread
                break;
            }
            float mt = red[r];
#pragma unroll
            for (int q4 = 1; q4 < kSmxParts; ++q4) mt = fmaxf(mt, red[q4 * kTcBq + r]);
            if (ttile && threadIdx.x == 64) MOE_TRACE_POINT(g_trace_attn, 1, j, 3);
            const float m_new = fmaxf(m, mt);
            // rescale of everything so far; a row with no visible key yet
            // keeps m = -inf and weighs nothing
            const float alpha = m_new == -INFINITY ? 1.f : ex2(m - m_new);
            const float mneg = m_new == -INFINITY ? 0.f : -m_new;
            float ls[4] = {0.f, 0.f, 0.f, 0.f};
            uint32_t pk[kSmxKeys / 2];
#pragma unroll
            for (int i = 0; i < kSmxKeys / 2; ++i) {
                const float pa = ex2(x[2 * i] + mneg), pb = ex2(x[2 * i + 1] + mneg);
                ls[i & 3] += pa + pb;
                pk[i] = pack_bf16x2(pa, pb);
            }
            // before P_j overwrites P_{j-1}: the product reading P_{j-1} has
            // completed once O_{j-1} is ready; accumulate O_{j-1} (a failed
            // wait stops this thread's work; all stop at the next barrier)
            if (j > 0 && !accumulate_o(j - 1, alpha_prev)) {
                ok = false;
                continue;
            }
            if (ttile && threadIdx.x == 64) MOE_TRACE_POINT(g_trace_attn, 1, j, 4);
            tmem_st16(lane_base + kColP + (kSmxKeys / 2) * hf, pk);
            l = l * alpha + ((ls[0] + ls[1]) + (ls[2] + ls[3]));
            m = m_new;
            alpha_prev = alpha;
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(p_full));
            if (ttile && threadIdx.x == 64) MOE_TRACE_POINT(g_trace_attn, 1, j, 5);
        }
        if (threadIdx.x == 64) MOE_TRACE_POINT(g_trace_attn, 0, tcta, 4);
        if (ok && n_tiles > 0 && !accumulate_o(n_tiles - 1, alpha_prev)) ok = false;
        if (!ok) {
            flags[0] = 1;
            atomicOr(p.status, MOE_DEV_WAIT_TIMEOUT);
        }
        // the row's whole sum: all parts (every softmax thread takes part,
        // also after an abort, so that the barrier is reached by all)
        float* red = red_s + 2 * kSmxParts * kTcBq;
        red[hf * kTcBq + r] = l;
        named_bar_sync(1, kSmxThreads);
        float lt = red[r];
#pragma unroll
        for (int q4 = 1; q4 < kSmxParts; ++q4) lt += red[q4 * kTcBq + r];
        if (ok && qrow < p.Tq) {
            // out = O / l (l includes the sink's share; 0 only for a row that
            // sees no key and has no sink -- then O is 0 as well)
            const float inv = lt > 0.f ? 1.f / lt : 0.f;
            float4* dst = reinterpret_cast<float4*>(
                p.out + (static_cast<size_t>(qrow) * p.Hq + h) * kTcD + kSmxCols * hf);
#pragma unroll
            for (int i = 0; i < kSmxCols / 4; ++i)
                dst[i] = make_float4(o[4 * i] * inv, o[4 * i + 1] * inv, o[4 * i + 2] * inv,
                                     o[4 * i + 3] * inv);
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
           3 * kSmxParts * kTcBq * 4;
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
    const dim3 grid((s.Tq + kTcBq - 1) / kTcBq, s.Hq);
    attention_tc_kernel<<<grid, kTcThreads, smem, stream>>>(p, tq, tk, tv);
    return cudaGetLastError();
}

}  // namespace moe
