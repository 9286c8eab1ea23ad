// Grouped expert GEMMs on the 5th-generation tensor cores (tcgen05 + TMEM),
// fed by TMA, with the bias + clamped GLU fused into the gate_up epilogue and
// the bias + top-k weighted combine fused into the down epilogue
// (xserv docs/19-gpt-oss-moe.md, "Phase 19: gpt-oss-20b": §2 "MoE 前向"
// step list gate_up -> bias -> GLU -> down -> bias -> weighted_sum; §1 table
// "激活" row for the GLU; §5 "量化" for MXFP4 weights).
//
// Orientation.  The weight matrix is the MMA's A operand (M = 128 weight
// rows per tile) and the tokens routed to one expert are the B operand
// (N = 16..256 token rows).  Putting the tokens on N lets every tile use
// exactly round_up(rows, 16) columns, so an expert with few tokens (decode)
// costs a 16-wide MMA instead of a 128-row one, and the weights -- the bytes
// that dominate at small T -- stream through TMA once per token tile.
//
// Work unit = (token tile, 128-row weight block).  A persistent grid walks
// the units in order; units of one token tile are consecutive, so the
// token tile stays hot in L2 while its 128-row weight blocks stream past.
//
// CTA roles:
//   warp 0      TMA producer (one lane): W tile [128 x 64] via a 3-D map
//               (k, row, expert) and token tile [box x 64] via a 2-D map,
//               both 128-byte swizzled, into a ring of `stages` slots.
//               MXFP4: the W tile arrives as packed E2M1 codes [128 x 32 B]
//               (unswizzled), and once per unit one bulk copy brings the
//               unit's E8M0 scales [128 x K/32 B] (double-buffered).
//   warp 1      TMEM owner + MMA issuer (one lane): 4 x (128 x N x 16)
//               tcgen05.mma per slot into one of two TMEM accumulators.
//   warps 2..5  epilogue (128 threads): tcgen05.ld of the accumulator, one
//               TMEM lane (= weight row) per thread, 16 token columns at a
//               time, then
//                 kEpiGlu:     + bias, pair gate/up rows (adjacent lanes,
//                              shfl.xor 1), clamp, GLU, bf16 store of h;
//                 kEpiCombine: + bias, x routing weight, red.global.add.f32
//                              into out[token, row].
//   warps 6..9  (MXFP4 only) converters: thread r expands row r of the code
//               tile to bf16 (E2M1 via byte-permute lookups -- every E2M1
//               value is a normal bf16 -- times 2^(s-127), an exact bf16x2
//               multiply), writes the 128-byte-swizzled A tile, fences the
//               async proxy and arrives on the slot's "converted" barrier,
//               which the MMA issuer waits for.
// The two accumulators let the epilogue of one unit overlap the main loop
// of the next.  Tails: weight rows past the matrix are zero-filled by TMA
// and masked at the store; token rows past the tile are computed on
// whatever TMA loaded (zeros past the end) and never stored; K = 64 * k.
//
// Every mbarrier wait is bounded (ptx.cuh).  A wait that gives up sets
// MOE_DEV_WAIT_TIMEOUT in the status word and makes all roles leave their
// loops; the producer then waits (bounded) for the loads it still has in
// flight, the MMA issuer for its last MMAs, and TMEM is freed before exit.
#include "moe_internal.cuh"
#include "ptx.cuh"
#include "../../include/moe.h"

namespace moe {
namespace {

constexpr int kEpiThreads = 128;
constexpr int kConvThreads = 256;   // two threads per weight row (half a row each)
constexpr uint32_t kATileBytes = kWeightTileRows * kBlockK * 2;      // 16 KB bf16
constexpr uint32_t kCodeTileBytes = kWeightTileRows * kBlockK / 2;   // 4 KB E2M1
constexpr int kMaxStages = 12;

template <int WF>
constexpr int kThreadsOf = WF == 1 ? 192 + kConvThreads : 192;

struct SmemPlan {
    uint8_t* a;          // stages x 16 KB bf16 W tiles (1024-aligned)
    uint8_t* b;          // stages x box*128 B token tiles (1024-aligned)
    uint8_t* codes;      // stages x 4 KB E2M1 tiles (MXFP4)
    uint8_t* scales;     // 2 x 128*kscale B (MXFP4)
    int* meta_tok;       // [box] token of each tile row (combine)
    float* meta_w;       // [box] routing weight of each tile row (combine)
    uint64_t* full;      // [stages] TMA landed
    uint64_t* conv;      // [stages] A tile converted (MXFP4)
    uint64_t* empty;     // [stages] MMAs done with the slot
    uint64_t* tfull;     // [2]
    uint64_t* tempty;    // [2]
    uint64_t* sfull;     // [2] scales landed (MXFP4)
    uint64_t* sempty;    // [2] scales consumed (MXFP4)
    uint64_t* drain;     // [1]
    uint32_t* tmem_base;
    int* flags;          // [0] abort, [1..2] epilogue broadcast (alternating)
};

__device__ __forceinline__ SmemPlan plan_smem(uint8_t* raw, int stages, int box, int wf,
                                              int kscale) {
    SmemPlan s;
    const uint32_t base = smem_u32(raw);
    uint8_t* p = raw + ((1024u - (base & 1023u)) & 1023u);
    s.a = p;
    p += static_cast<size_t>(stages) * kATileBytes;
    s.b = p;
    p += static_cast<size_t>(stages) * box * 128;
    s.codes = p;
    s.scales = p;
    if (wf == 1) {
        p += static_cast<size_t>(stages) * kCodeTileBytes;
        s.scales = p;
        p += 2 * ((kWeightTileRows * kscale + 15) / 16 * 16);
    }
    s.meta_tok = reinterpret_cast<int*>(p);
    p += box * 4;
    s.meta_w = reinterpret_cast<float*>(p);
    p += box * 4;
    uint64_t* bars = reinterpret_cast<uint64_t*>(p);
    s.full = bars;
    s.conv = bars + stages;
    s.empty = bars + 2 * stages;
    s.tfull = bars + 3 * stages;
    s.tempty = s.tfull + 2;
    s.sfull = s.tempty + 2;
    s.sempty = s.sfull + 2;
    s.drain = s.sempty + 2;
    s.tmem_base = reinterpret_cast<uint32_t*>(s.drain + 1);
    s.flags = reinterpret_cast<int*>(s.tmem_base + 1);
    return s;
}

__device__ __forceinline__ void raise_abort(volatile int* flags, int32_t* status, int bit) {
    flags[0] = 1;
    atomicOr(status + kStatusWord, bit);
}

__device__ __forceinline__ bool tile_ok(const int4& t, const GemmParams& p) {
    return t.x >= 0 && t.x < p.num_experts && t.z >= 1 && t.z <= p.token_box && t.y >= 0 &&
           t.y + t.z <= p.rows_total;
}

__device__ __forceinline__ float clamped_glu(float gate, float up) {
    gate = fminf(gate, 7.0f);
    up = fminf(fmaxf(up, -7.0f), 7.0f);
    const float g = gate / (1.0f + __expf(-1.702f * gate));
    return (up + 1.0f) * g;
}

// Eight E2M1 codes (one 32-bit word, element 2i in the low nibble of byte i)
// to eight bf16 values times 2^(s-127).
//
// For the byte b of elements (2i, 2i+1), two integer multiplies place the
// nibbles at the bf16 bit positions: b * (2^6 + 2^18) puts the magnitude bits
// (exponent e, mantissa m) of the low nibble at bits 6..8 and of the high
// nibble at 22..24; b * (2^12 + 2^24) puts their sign bits at 15 and 31.
// Read as bf16, each half is then exactly e2m1(code) * 2^-126 -- a normal
// number for e >= 1 and the subnormal 2^-127 for the code 0.5 (e = 0,
// m = 1) -- so one exact bf16x2 multiply by 2^(s-1) yields
// e2m1(code) * 2^(s-127).  The multiplies run on the FMA pipe, leaving the
// integer pipe two masks and one byte extraction per pair.
__device__ __forceinline__ uint4 e2m1x8_to_bf16(uint32_t w, uint32_t scale2, uint32_t scale2b) {
    uint4 r;
    uint32_t* rr = reinterpret_cast<uint32_t*>(&r);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t b = __byte_perm(w, 0u, 0x4440u | static_cast<uint32_t>(i));
        const uint32_t mag = (b * 0x00040040u) & 0x01C001C0u;
        const uint32_t emb = mag | ((b * 0x01001000u) & 0x80008000u);
        __nv_bfloat162 v = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&emb),
                                   *reinterpret_cast<const __nv_bfloat162*>(&scale2));
        if (scale2b != 0x3F803F80u)   // only for scales above 2^1 (s > 128)
            v = __hmul2(v, *reinterpret_cast<const __nv_bfloat162*>(&scale2b));
        rr[i] = *reinterpret_cast<uint32_t*>(&v);
    }
    return r;
}

// The factor(s) that turn an embedded code into e2m1(code) * 2^(s-127),
// as bf16x2: 2^(s-1) when s <= 128 (bf16 exponent field s + 126), else
// 2^127 then 2^(s-128).  Scale bytes 0 and 255 (zero, NaN) are not produced
// by MX quantisers for weights and are not supported.
__device__ __forceinline__ void e8m0_factors(uint32_t s, uint32_t& f1, uint32_t& f2) {
    s &= 0xFFu;
    if (s <= 128u) {
        const uint32_t h = (s + 126u) << 7;
        f1 = h | (h << 16);
        f2 = 0x3F803F80u;                       // 1.0
    } else {
        const uint32_t h1 = 254u << 7;          // 2^127
        const uint32_t h2 = (s - 1u) << 7;      // 2^(s-128)
        f1 = h1 | (h1 << 16);
        f2 = h2 | (h2 << 16);
    }
}

template <int EPI, int WF>
__global__ void __launch_bounds__(kThreadsOf<WF>, 1)
    grouped_gemm_kernel(const GemmParams p, const __grid_constant__ CUtensorMap tmap_w,
                        const __grid_constant__ CUtensorMap tmap_x) {
    extern __shared__ uint8_t smem_raw[];
    const int stages = p.stages, box = p.token_box;
    const uint32_t b_bytes = static_cast<uint32_t>(box) * 128u;
    SmemPlan sm = plan_smem(smem_raw, stages, box, WF, p.kscale);
    volatile int* flags = sm.flags;
    const uint32_t scale_buf_bytes =
        static_cast<uint32_t>((kWeightTileRows * p.kscale + 15) / 16 * 16);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(smem_u32(sm.full + s), 1);
            mbar_init(smem_u32(sm.conv + s), kConvThreads);
            mbar_init(smem_u32(sm.empty + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(sm.tfull + b), 1);
            mbar_init(smem_u32(sm.tempty + b), kEpiThreads);
            mbar_init(smem_u32(sm.sfull + b), 1);
            mbar_init(smem_u32(sm.sempty + b), kConvThreads);
        }
        mbar_init(smem_u32(sm.drain), 1);
        flags[0] = 0;
        flags[1] = 0;
        flags[2] = 0;
        mbar_fence_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmap_w);
        tma_prefetch_desc(&tmap_x);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(sm.tmem_base), static_cast<uint32_t>(p.tmem_cols));
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *sm.tmem_base;
    const uint32_t acc_stride = static_cast<uint32_t>(p.tmem_cols) / 2u;

    pdl_wait();                 // tiles, activations and outputs of earlier kernels
    pdl_launch_dependents();

    const int num_units = p.num_tiles[0] * p.n_wblocks;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();
            const uint64_t pol_x = policy_evict_last();
            const uint32_t w_bytes = WF == 1 ? kCodeTileBytes : kATileBytes;
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            int local = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
                const int4 t = p.tiles[u / p.n_wblocks];
                if (!tile_ok(t, p)) continue;
                const int mb = u % p.n_wblocks;
                if (WF == 1) {
                    // this unit's scale rows, one bulk copy, double-buffered
                    const int sb = local & 1;
                    const uint32_t sph = static_cast<uint32_t>(local >> 1) & 1u;
                    if (!mbar_wait(smem_u32(sm.sempty + sb), sph ^ 1u, flags)) {
                        raise_abort(flags, p.status, MOE_DEV_WAIT_TIMEOUT);
                        ok = false;
                        break;
                    }
                    const int rows = min(kWeightTileRows, p.w_rows - mb * kWeightTileRows);
                    const uint32_t bytes = static_cast<uint32_t>(rows * p.kscale);
                    const uint32_t sf = smem_u32(sm.sfull + sb);
                    mbar_arrive_expect_tx(sf, bytes);
                    bulk_load(smem_u32(sm.scales + sb * scale_buf_bytes),
                              p.scales + (static_cast<size_t>(t.x) * p.w_rows +
                                          static_cast<size_t>(mb) * kWeightTileRows) * p.kscale,
                              bytes, sf);
                }
                ++local;
                for (int kb = 0; kb < p.k_blocks; ++kb) {
                    if (!mbar_wait(smem_u32(sm.empty + stage), phase ^ 1u, flags)) {
                        raise_abort(flags, p.status, MOE_DEV_WAIT_TIMEOUT);
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_u32(sm.full + stage);
                    mbar_arrive_expect_tx(fb, w_bytes + b_bytes);
                    if (WF == 1)
                        tma_load_3d(smem_u32(sm.codes + static_cast<size_t>(stage) * kCodeTileBytes),
                                    &tmap_w, fb, kb * (kBlockK / 2), mb * kWeightTileRows, t.x, pol_w);
                    else
                        tma_load_3d(smem_u32(sm.a + static_cast<size_t>(stage) * kATileBytes),
                                    &tmap_w, fb, kb * kBlockK, mb * kWeightTileRows, t.x, pol_w);
                    tma_load_2d(smem_u32(sm.b + static_cast<size_t>(stage) * b_bytes), &tmap_x, fb,
                                kb * kBlockK, t.y, pol_x);
                    ++issued;
                    if (++stage == stages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                // Wait (bounded) for the loads still in flight before the CTA
                // may release its shared memory.
                const long long pending = issued < stages ? issued : stages;
                int s = stage;
                uint32_t ph = phase;
                for (long long i = 0; i < pending; ++i) {
                    if (--s < 0) {
                        s = stages - 1;
                        ph ^= 1u;
                    }
                    mbar_wait(smem_u32(sm.full + s), ph, nullptr);
                }
                if (WF == 1 && local > 0) {
                    const int sb = (local - 1) & 1;
                    mbar_wait(smem_u32(sm.sfull + sb), static_cast<uint32_t>((local - 1) >> 1) & 1u,
                              nullptr);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int local = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
                const int4 t = p.tiles[u / p.n_wblocks];
                if (!tile_ok(t, p)) continue;
                const uint32_t n_mma = static_cast<uint32_t>((t.z + 15) & ~15);
                const uint32_t idesc = idesc_bf16_f32(kWeightTileRows, n_mma);
                const int buf = local & 1;
                const uint32_t tph = static_cast<uint32_t>(local >> 1) & 1u;
                ++local;
                if (!mbar_wait(smem_u32(sm.tempty + buf), tph ^ 1u, flags)) {
                    raise_abort(flags, p.status, MOE_DEV_WAIT_TIMEOUT);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf) * acc_stride;
                for (int kb = 0; kb < p.k_blocks; ++kb) {
                    const uint32_t ready = smem_u32((WF == 1 ? sm.conv : sm.full) + stage);
                    if (!mbar_wait(ready, phase, flags)) {
                        raise_abort(flags, p.status, MOE_DEV_WAIT_TIMEOUT);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(sm.a + static_cast<size_t>(stage) * kATileBytes);
                    const uint32_t b_addr = smem_u32(sm.b + static_cast<size_t>(stage) * b_bytes);
#pragma unroll
                    for (int kk = 0; kk < kBlockK / 16; ++kk) {
                        tc_mma_bf16(d_tmem, smem_desc_sw128(a_addr + kk * 32),
                                    smem_desc_sw128(b_addr + kk * 32), idesc,
                                    (kb | kk) != 0 ? 1u : 0u);
                    }
                    tc_commit(smem_u32(sm.empty + stage));
                    if (++stage == stages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                tc_commit(smem_u32(sm.tfull + buf));
            }
            // Every MMA issued so far has finished once this arrives.
            tc_commit(smem_u32(sm.drain));
            mbar_wait(smem_u32(sm.drain), 0, nullptr);
        }
    } else if (warp < 6) {
        // ------------------------------------------------ epilogue
        const int ep = threadIdx.x - 64;          // 0..127
        const int quad = warp & 3;                // TMEM lane quadrant of this warp
        const int row_in_tile = quad * 32 + lane;
        int local = 0;
        for (int u = blockIdx.x; u < num_units; u += gridDim.x) {
            const int4 t = p.tiles[u / p.n_wblocks];
            if (!tile_ok(t, p)) {
                if (ep == 0) atomicOr(p.status + kStatusWord, MOE_DEV_BAD_TILE);
                continue;
            }
            const int mb = u % p.n_wblocks;
            const int buf = local & 1;
            const uint32_t tph = static_cast<uint32_t>(local >> 1) & 1u;
            ++local;

            if (EPI == kEpiCombine) {
                named_bar_sync(1, kEpiThreads);   // previous unit done with meta
                for (int c = ep; c < t.z; c += kEpiThreads) {
                    const int a = p.sorted_assign[t.y + c];
                    sm.meta_tok[c] = a / p.top_k;
                    sm.meta_w[c] = p.topk_w[a];
                }
            }
            // One thread waits; the decision is broadcast so all 128 agree.
            // The slot alternates so it is never rewritten before every
            // thread has read it (a barrier of the next unit lies between).
            if (ep == 0) {
                const bool got = mbar_wait(smem_u32(sm.tfull + buf), tph, flags);
                if (!got) raise_abort(flags, p.status, MOE_DEV_WAIT_TIMEOUT);
                flags[1 + buf] = got ? 0 : 1;
            }
            named_bar_sync(1, kEpiThreads);
            if (flags[1 + buf]) break;
            tc_fence_after();

            const int wrow = mb * kWeightTileRows + row_in_tile;
            const bool row_ok = wrow < p.w_rows;
            const float bias =
                row_ok ? __bfloat162float(p.bias[static_cast<size_t>(t.x) * p.w_rows + wrow]) : 0.f;
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                                   static_cast<uint32_t>(buf) * acc_stride;
            const int n_mma = (t.z + 15) & ~15;
            for (int c0 = 0; c0 < n_mma; c0 += 16) {
                float v[16];
                tmem_ld16(taddr + static_cast<uint32_t>(c0), v);
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] += bias;
                if (EPI == kEpiGlu) {
                    // even lane: gate row 2j, odd lane: up row 2j+1 (same j)
                    const bool odd = lane & 1;
                    const int hcols = p.w_rows >> 1;
                    __nv_bfloat16* hrow0 =
                        p.h + static_cast<size_t>(t.y) * hcols + (wrow >> 1);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float send = odd ? v[i] : v[8 + i];
                        const float recv = __shfl_xor_sync(0xffffffffu, send, 1);
                        const float gate = odd ? recv : v[i];
                        const float up = odd ? v[8 + i] : recv;
                        const int c = c0 + i + (odd ? 8 : 0);
                        if (c < t.z)
                            hrow0[static_cast<size_t>(c) * hcols] =
                                __float2bfloat16_rn(clamped_glu(gate, up));
                    }
                } else {
                    if (row_ok) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const int c = c0 + i;
                            if (c < t.z) {
                                atomicAdd(p.out + static_cast<size_t>(sm.meta_tok[c]) * p.w_rows + wrow,
                                          sm.meta_w[c] * v[i]);
                            }
                        }
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(smem_u32(sm.tempty + buf));
        }
    } else if (WF == 1) {
        // ------------------------------------------------ MXFP4 converters
        const int ct = threadIdx.x - 192;         // 0..255
        const int r = ct & 127;                   // weight row within the tile
        const int half = ct >> 7;                 // chunks 4*half .. 4*half+3 of the row
        const uint32_t a_row_off = static_cast<uint32_t>(r) * 128u;
        const uint32_t swz = static_cast<uint32_t>(r & 7);
        int stage = 0;
        uint32_t phase = 0;
        int local = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
            const int4 t = p.tiles[u / p.n_wblocks];
            if (!tile_ok(t, p)) continue;
            const int sb = local & 1;
            const uint32_t sph = static_cast<uint32_t>(local >> 1) & 1u;
            ++local;
            if (!mbar_wait(smem_u32(sm.sfull + sb), sph, flags)) {
                raise_abort(flags, p.status, MOE_DEV_WAIT_TIMEOUT);
                break;
            }
            const uint8_t* srow = sm.scales + sb * scale_buf_bytes + r * p.kscale;
            // rows past the matrix: codes are TMA zero-fill and no scale bytes
            // were copied for them; use scale 1 so they stay exactly zero
            const bool row_ok = (u % p.n_wblocks) * kWeightTileRows + r < p.w_rows;
            for (int kb = 0; kb < p.k_blocks; ++kb) {
                if (!mbar_wait(smem_u32(sm.full + stage), phase, flags)) {
                    raise_abort(flags, p.status, MOE_DEV_WAIT_TIMEOUT);
                    ok = false;
                    break;
                }
                uint32_t f1, f2;
                e8m0_factors(row_ok ? srow[2 * kb + half] : 127u, f1, f2);
                const uint4 cw = *reinterpret_cast<const uint4*>(
                    sm.codes + static_cast<size_t>(stage) * kCodeTileBytes + r * 32 + half * 16);
                const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
                uint8_t* arow = sm.a + static_cast<size_t>(stage) * kATileBytes + a_row_off;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint32_t chunk = static_cast<uint32_t>(4 * half + c);
                    const uint4 v = e2m1x8_to_bf16(words[c], f1, f2);
                    *reinterpret_cast<uint4*>(arow + ((chunk ^ swz) << 4)) = v;
                }
                fence_proxy_async_smem();
                mbar_arrive(smem_u32(sm.conv + stage));
                if (++stage == stages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
            mbar_arrive(smem_u32(sm.sempty + sb));
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, static_cast<uint32_t>(p.tmem_cols));
    }
}

template <int EPI, int WF>
cudaError_t launch_gemm_t(const GemmParams& p, const CUtensorMap* tmap_w, const CUtensorMap* tmap_x,
                          int grid, size_t smem, cudaStream_t s, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreadsOf<WF>);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    cudaError_t err = cudaFuncSetAttribute(grouped_gemm_kernel<EPI, WF>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    return cudaLaunchKernelEx(&cfg, grouped_gemm_kernel<EPI, WF>, p, *tmap_w, *tmap_x);
}

}  // namespace

cudaError_t launch_gemm(int epi, int wf, const GemmParams& p, const CUtensorMap* tmap_w,
                        const CUtensorMap* tmap_x, int grid, size_t smem, cudaStream_t s,
                        bool pdl) {
    if (p.stages < 2 || p.stages > kMaxStages) return cudaErrorInvalidValue;
    if (epi == kEpiGlu)
        return wf == 1 ? launch_gemm_t<kEpiGlu, 1>(p, tmap_w, tmap_x, grid, smem, s, pdl)
                       : launch_gemm_t<kEpiGlu, 0>(p, tmap_w, tmap_x, grid, smem, s, pdl);
    return wf == 1 ? launch_gemm_t<kEpiCombine, 1>(p, tmap_w, tmap_x, grid, smem, s, pdl)
                   : launch_gemm_t<kEpiCombine, 0>(p, tmap_w, tmap_x, grid, smem, s, pdl);
}

// fp32 -> bf16 (round to nearest even) of the combined output.
namespace {
__global__ void to_bf16_kernel(const float* __restrict__ in, __nv_bfloat16* __restrict__ out,
                               size_t n) {
    pdl_wait();
    const size_t n4 = n / 4;
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n4;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const float4 v = reinterpret_cast<const float4*>(in)[i];
        __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
        __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
        uint2 pk;
        pk.x = *reinterpret_cast<uint32_t*>(&lo);
        pk.y = *reinterpret_cast<uint32_t*>(&hi);
        reinterpret_cast<uint2*>(out)[i] = pk;
    }
}
}  // namespace

cudaError_t launch_to_bf16(const float* in, __nv_bfloat16* out, size_t n, cudaStream_t s,
                           bool pdl) {
    cudaLaunchConfig_t cfg = {};
    const size_t n4 = n / 4;
    size_t blocks = (n4 + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    if (blocks == 0) blocks = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, to_bf16_kernel, in, out, n);
}

}  // namespace moe
