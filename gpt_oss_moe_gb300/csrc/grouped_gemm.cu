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
//   warp 1      TMEM owner + MMA issuer: the warp walks the ring, one
//               elected lane issues 4 x (128 x N x 16) tcgen05.mma per slot
//               into one of two TMEM accumulators (CTA pairs: 256 x N x 16
//               from the even CTA).
//   warps 2..5  epilogue (128 threads): tcgen05.ld of the accumulator, one
//               TMEM lane (= weight row) per thread, 16 token columns at a
//               time, then
//                 kEpiGlu:     + bias, pair gate/up rows (adjacent lanes,
//                              shfl.xor 1), clamp, GLU, bf16 store of h;
//                 kEpiCombine: + bias, x routing weight, red.global.add.f32
//                              into out[token, row].
//   warps 6..21 (MXFP4 only) converters, two teams of 8 warps taking
//               alternate k-blocks: two threads per weight row, each
//               expanding half a row of the code tile to bf16 (E2M1 by
//               integer multiplies into bf16 bit positions, times
//               2^(s-127) by an exact bf16x2 multiply) and storing it to
//               TMEM (tcgen05.st: the row's lane, 32 columns per A tile);
//               one lane per warp then arrives on the A slot's "converted"
//               barrier, which the MMA issuer waits for.  The MMAs read A
//               from TMEM and the token tile from shared memory, so the
//               converted tile costs no shared-memory bandwidth.  MXFP4 uses
//               two rings: `stages` slots of code + token tiles (deep, to
//               keep HBM busy) and `astages` A tiles in TMEM.
// The two accumulators let the epilogue of one unit overlap the main loop
// of the next.  Tails: weight rows past the matrix are zero-filled by TMA
// and masked at the store; token rows past the tile are computed on
// whatever TMA loaded (zeros past the end) and never stored; K = 64 * k.
//
// Every mbarrier wait is bounded (ptx.cuh).  A wait that gives up sets
// MOE_DEV_WAIT_TIMEOUT in the status word and makes all roles leave their
// loops; the producer then waits (bounded) for the loads it still has in
// flight, the MMA issuer for its last MMAs, and TMEM is freed before exit.
#include <type_traits>

#include <cuda_fp16.h>

#include "moe_internal.cuh"
#include "ptx.cuh"
#include "trace.cuh"
#include "../../include/moe.h"

namespace moe {
namespace {

// gate_up (kernel 0) and down (kernel 1): 0 entry, 1 set-up done, 2 weight
// loads issued before the wait, 3 producer past the wait, 4 first MMA slot
// full, 5 last MMA commit, 6 epilogue done, 7 exit
MOE_TRACE_ARRAY(g_trace_gemm, 2);

constexpr int kConvThreads = 256;   // per team: two threads per weight row (half a row each)
constexpr int kConvTeams = 2;
constexpr uint32_t kATileBytes = kWeightTileRows * kBlockK * 2;      // 16 KB bf16
// k-blocks (of 64) per ring slot: MXFP4 slots carry 4, so that each slot is
// two TMA operations of 16 KB codes + 4 token chunks (an SM keeps only about
// ten TMA operations in flight, so bytes per operation set the bandwidth).
template <int WF>
constexpr int kKbPerStage = WF == 1 ? kMxfp4KbPerStage : WF == 3 ? kMxKbPerStage : 1;
constexpr uint32_t kCodeStageBytes = kWeightTileRows * kMxfp4KbPerStage * kBlockK / 2;  // 16 KB
constexpr uint32_t kASlotCols = 32u * kMxfp4KbPerStage;    // TMEM columns of one MXFP4 A slot
constexpr int kMaxStages = 24;
constexpr int kBarBytes = 768;

// MXFP4 x MXFP8: bytes one weight slot moves from global memory (128 rows
// x 64 B of codes; shared memory receives them padded to 128 B per row)
constexpr uint32_t kMxCodeTxBytes = kWeightTileRows * 64;
constexpr int kMxScaleWarps = 4;        // MXFP4 x MXFP8: warps 6..9 write the scales

// Epilogue warps (from warp 2): bf16 and FP8 kernels run two warps per TMEM
// lane quadrant, each taking alternate 16-column chunks of the accumulator,
// so that a prefill unit's epilogue (GLU, or the output reductions) ends
// within the next unit's main loop; the MXFP4 kernels keep one per quadrant
// (their other warps convert or write scales).
template <int WF>
constexpr int kEpiWarps = (WF == 0 || WF == 2) ? 8 : 4;
// bf16 kernels: one more warp, the last of the CTA, gathers token rows from
// the layer input for small batches (GemmParams::gather_x); in gate_up
// without gathering it clears the output rows the down projection
// accumulates into (GemmParams::zero_out), alongside the pipeline.
template <int WF>
constexpr int kGatherWarpOf = WF == 0 ? 2 + kEpiWarps<WF> : -1;
template <int WF>
constexpr int kThreadsOf = WF == 1 ? 192 + kConvTeams * kConvThreads + 32
                         : WF == 3 ? 192 + kMxScaleWarps * 32
                         : 64 + kEpiWarps<WF> * 32 + (kGatherWarpOf<WF> >= 0 ? 32 : 0);
// token-row copies of the gather warp in flight, in ring slots
constexpr int kGatherLag = 3;
constexpr int kSecondIssuerWarp = 6 + kConvTeams * kConvThreads / 32;    // MXFP4: warp 22

struct SmemPlan {
    uint8_t* a;          // stages x 16 KB bf16 W tiles (1024-aligned)
    uint8_t* b;          // stages x kb_per_stage x box*128 B token tiles (1024-aligned)
    uint8_t* codes;      // stages x 16 KB E2M1 tiles [128 rows x 128 B], 128-byte swizzled (MXFP4)
    uint8_t* scales;     // 2 x 128*kscale B (MXFP4, MXFP4 x MXFP8)
    uint8_t* tscales;    // 2 x box*xs_row_bytes B: token tile scale rows (MXFP4 x MXFP8)
    int* meta_tok;       // [box] token of each tile row (combine)
    float* meta_w;       // [box] routing weight of each tile row (combine)
    uint64_t* full;      // [stages] TMA landed
    uint64_t* empty;     // [stages] MMAs done with the slot
    uint64_t* afull;     // [astages] A tile converted (MXFP4)
    uint64_t* aempty;    // [astages] MMAs done with the A tile (MXFP4)
    uint64_t* tfull;     // [2]
    uint64_t* tempty;    // [2]
    uint64_t* sfull;     // [2] scales landed (MXFP4)
    uint64_t* sempty;    // [2] scales consumed (MXFP4)
    uint64_t* drain;     // [2] one per MMA issuer
    uint64_t* gfull;     // [stages] gathered token rows landed (bf16 small batches)
    uint32_t* tmem_base;
    int* flags;          // [0] abort, [1..2] epilogue broadcast (alternating),
                         // [3] K-split: this epilogue holds the last part
};

// bf16: one ring of `stages` slots, each a W tile + a token tile.
// MXFP4: one ring of `stages` slots, each a code tile + a token tile; the
// converted bf16 W tiles live in TMEM, not here.
__device__ __forceinline__ SmemPlan plan_smem(uint8_t* raw, int stages, int astages, int box,
                                              int bbox, int wf, int kscale, int xs_row_bytes) {
    SmemPlan s;
    const uint32_t base = smem_u32(raw);
    uint8_t* p = raw + ((1024u - (base & 1023u)) & 1023u);
    s.a = p;
    p += static_cast<size_t>(wf == 1 ? 0 : stages) * (wf == 3 ? kMxKbPerStage : 1) * kATileBytes;
    s.b = p;
    p += static_cast<size_t>(stages) * (wf == 1 ? kMxfp4KbPerStage : wf == 3 ? kMxKbPerStage : 1) *
         bbox * 128;
    s.codes = p;
    s.scales = p;
    s.tscales = p;
    if (wf == 1) {
        p += static_cast<size_t>(stages) * kCodeStageBytes;
        s.scales = p;
        p += 2 * ((kWeightTileRows * kscale + 15) / 16 * 16);
    } else if (wf == 3) {
        s.scales = p;
        p += 2 * ((kWeightTileRows * kscale + 15) / 16 * 16);
        s.tscales = p;
        p += 2 * static_cast<size_t>(box) * xs_row_bytes;
    }
    s.meta_tok = reinterpret_cast<int*>(p);
    p += box * 4;
    s.meta_w = reinterpret_cast<float*>(p);
    p += box * 4;
    uint64_t* bars = reinterpret_cast<uint64_t*>(p);
    s.full = bars;
    s.empty = bars + stages;
    s.afull = bars + 2 * stages;
    s.aempty = s.afull + astages;
    s.tfull = s.aempty + astages;
    s.tempty = s.tfull + 2;
    s.sfull = s.tempty + 2;
    s.sempty = s.sfull + 2;
    s.drain = s.sempty + 2;
    s.gfull = s.drain + 2;
    s.tmem_base = reinterpret_cast<uint32_t*>(s.gfull + stages);
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

// Work unit u of a call: K-split part `split` of (token tile, 128-row weight
// block) pair `pair` = tile * n_wblocks + mb; it covers ring slots
// [st_lo, st_hi) of the n_st slots of the weights' K range.
struct Unit {
    int pair, tile, mb, split, st_lo, st_hi;
};
__device__ __forceinline__ Unit unit_of(int u, const GemmParams& p, int n_st) {
    Unit x;
    x.split = u % p.ksplit;
    x.pair = u / p.ksplit;
    x.tile = x.pair / p.n_wblocks;
    x.mb = x.pair % p.n_wblocks;
    const int per = (n_st + p.ksplit - 1) / p.ksplit;
    x.st_lo = x.split * per;
    x.st_hi = min(n_st, x.st_lo + per);
    return x;
}

__device__ __forceinline__ float clamped_glu(float gate, float up) {
    gate = fminf(gate, 7.0f);
    up = fminf(fmaxf(up, -7.0f), 7.0f);
    const float g = gate / (1.0f + __expf(-1.702f * gate));
    return (up + 1.0f) * g;
}

// Eight E2M1 codes (one 32-bit word, code q in nibble q) to eight bf16
// values times 2^(s-127), as four bf16x2 words holding the codes in the
// order (0,4), (1,5), (2,6), (3,7).  The tile's K positions are permuted the
// same way within every group of 8, and so are the token operand's (the
// gather and the GLU epilogue store them in that order), so the products
// and their sum over K are unchanged.
//
// Codes q and q+4 sit 16 bits apart, one per bf16 half.  Masking the pair
// and multiplying by 2^a + 2^(a+6) leaves two non-overlapping copies of each
// nibble (no carries): the first puts the magnitude bits (exponent e,
// mantissa m) at bits 6..8 of its half, the second the sign at bit 15.  Read
// as bf16, each half is then exactly e2m1(code) * 2^-126 -- a normal number
// for e >= 1 and the subnormal 2^-127 for the code 0.5 (e = 0, m = 1) -- so
// one exact bf16x2 multiply by 2^(s-1) yields e2m1(code) * 2^(s-127).  Per
// pair of values: AND, IMAD, AND on the integer pipes, one multiply on the
// FMA pipe.
template <bool kTwoFactors>
__device__ __forceinline__ uint4 e2m1x8_to_bf16(uint32_t w, uint32_t scale2, uint32_t scale2b) {
    const uint32_t w2 = w >> 8;
    const uint32_t emb[4] = {((w & 0x000F000Fu) * 0x1040u) & 0x81C081C0u,
                             ((w & 0x00F000F0u) * 0x0104u) & 0x81C081C0u,
                             ((w2 & 0x000F000Fu) * 0x1040u) & 0x81C081C0u,
                             ((w2 & 0x00F000F0u) * 0x0104u) & 0x81C081C0u};
    uint4 r;
    uint32_t* rr = reinterpret_cast<uint32_t*>(&r);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 v = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&emb[i]),
                                   *reinterpret_cast<const __nv_bfloat162*>(&scale2));
        if (kTwoFactors)   // only for scales above 2^1 (s > 128)
            v = __hmul2(v, *reinterpret_cast<const __nv_bfloat162*>(&scale2b));
        rr[i] = *reinterpret_cast<uint32_t*>(&v);
    }
    return r;
}

// Column c of a row stored in the order above: position of natural column c.
__device__ __forceinline__ int kperm8_pos(int c) {
    return (c & ~7) | ((c & 3) << 1) | ((c >> 2) & 1);
}

// f16 mode of the MXFP4 kernels: scale bytes whose every E2M1 multiple is
// an f16 (0.5 * 2^(s-127) >= 2^-24, 6 * 2^(s-127) <= 65504).
constexpr uint32_t kF16ScaleLo = 104;
constexpr uint32_t kF16ScaleHi = 140;

// 2^e as f16x2, -24 <= e <= 15 (subnormal below 2^-14).
__device__ __forceinline__ __half2 f16_pow2_x2(int e) {
    const uint32_t h = e >= -14 ? static_cast<uint32_t>(e + 15) << 10
                                : 1u << static_cast<uint32_t>(e + 24);
    const uint32_t hh = h | (h << 16);
    return *reinterpret_cast<const __half2*>(&hh);
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

template <int EPI, int WF, int CG>
__global__ void __launch_bounds__(kThreadsOf<WF>, 1)
    grouped_gemm_kernel(const GemmParams p, const __grid_constant__ CUtensorMap tmap_w,
                        const __grid_constant__ CUtensorMap tmap_x) {
    extern __shared__ uint8_t smem_raw[];
    constexpr int KPS = kKbPerStage<WF>;
    // K elements per k-block (one 128-byte swizzled row of an operand tile):
    // 64 bf16, or 128 E4M3 codes (WF = 2; WF = 3: 128 E4M3 token codes and
    // 128 E2M1 weight codes, padded to a byte each in shared memory)
    constexpr int kKB = WF >= 2 ? kBlockKFp8 : kBlockK;
    const int stages = p.stages, astages = p.astages, box = p.token_box;
    // CTA pair (CG = 2, bf16 weights): the cluster's two CTAs share each unit
    // of 256 weight rows; CTA r loads rows 128r.. of the block and half of
    // the token tile, the even CTA issues M = 256 MMAs over both.
    constexpr bool kPair = CG == 2;
    constexpr int kUnitRows = kPair ? 2 * kWeightTileRows : kWeightTileRows;
    const uint32_t rank = kPair ? cluster_ctarank() : 0u;
    const int cta0 = kPair ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
    const int ncta = kPair ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
    const int bbox = kPair ? box / 2 : box;   // token rows of this CTA's B tile
    // TMEM columns: per MMA issuer two accumulators of acc_stride columns
    // (issuer i, buffer b at (2i + b) * acc_stride), then (MXFP4) astages A
    // slots of 128 columns, each the converted weights of one ring slot
    // (4 k-blocks x 32 columns: 128 rows x 64 bf16 per k-block).  MXFP4 runs
    // n_iss = 2 issuers on alternate ring slots of a unit, each into its own
    // accumulators (a thread issues an N <= 64 MMA only every ~23 ns, the
    // tensor core takes them faster); the epilogue adds the two.
    const int n_iss = p.n_iss;
    const uint32_t acc_stride = (WF == 1 || WF == 3) ? static_cast<uint32_t>((box + 31) & ~31)
                                                     : static_cast<uint32_t>(p.tmem_cols) / 2u;
    const uint32_t a_col0 = 2u * static_cast<uint32_t>(n_iss) * acc_stride;
    // MXFP4 x MXFP8: after the two accumulators, 8 scale columns per
    // k-block of a ring slot: A (weight rows, column sf + row / 32) at
    // +0..3, B (token rows, column sf + 4 + row / 32, lanes row % 32) at +4..7
    const uint32_t sf_col0 = 2u * acc_stride;
    // ring sizes the converter teams rely on and the TMEM plan (uniform
    // exit, nothing started)
    if (stages < 2 || stages > kMaxStages || n_iss < 1 || n_iss > (WF == 1 ? 2 : 1) ||
        p.ksplit < 1 || p.ksplit > kMaxKSplit ||
        (EPI == kEpiGlu && p.ksplit > 1 && (p.partial == nullptr || p.tickets == nullptr)) ||
        (kPair && (WF == 1 || WF == 3 || p.ksplit != 1 || (gridDim.x & 1u) || (box & 15))) ||
        (p.gather_x != nullptr && (WF != 0 || kPair || stages <= kGatherLag || box > 64 ||
                                   p.sorted_assign == nullptr || p.top_k < 1)) ||
        (WF == 3 && (box > 128 || p.mx_cmax < 0 ||
                     sf_col0 + 8u * KPS * static_cast<uint32_t>(stages) >
                         static_cast<uint32_t>(p.tmem_cols))) ||
        (WF == 1 && (astages < 2 || astages > kMxfp4AStages || 2 * stages < astages + 2 ||
                     (n_iss == 2 && (astages & 1)) ||
                     a_col0 + kASlotCols * static_cast<uint32_t>(astages) >
                         static_cast<uint32_t>(p.tmem_cols)))) {
        if (threadIdx.x == 0) atomicOr(p.status + kStatusWord, MOE_DEV_BAD_TILE);
        return;
    }
    const uint32_t b_bytes = static_cast<uint32_t>(bbox) * 128u;      // one 64-wide K chunk
    const uint32_t b_stage_bytes = b_bytes * KPS;
    const int n_st = (p.k_blocks + KPS - 1) / KPS;                     // ring slots per unit
    SmemPlan sm = plan_smem(smem_raw, stages, astages, box, bbox, WF, p.kscale, p.xs_row_bytes);
    const uint32_t tscale_buf_bytes = static_cast<uint32_t>(box * p.xs_row_bytes);
    volatile int* flags = sm.flags;
    const uint32_t scale_buf_bytes =
        static_cast<uint32_t>((kWeightTileRows * p.kscale + 15) / 16 * 16);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) MOE_TRACE_POINT(g_trace_gemm, EPI, blockIdx.x, 0);

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            // MXFP4 x MXFP8: the producer's arrival + one per scale warp
            mbar_init(smem_u32(sm.full + s), WF == 3 ? 1 + kMxScaleWarps : 1);
            mbar_init(smem_u32(sm.gfull + s), 1);
            mbar_init(smem_u32(sm.empty + s), 1);
        }
        for (int s = 0; s < astages; ++s) {
            mbar_init(smem_u32(sm.afull + s), kConvThreads / 32);
            mbar_init(smem_u32(sm.aempty + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(sm.tfull + b), static_cast<uint32_t>(n_iss));
            // pair: one arrival from each CTA's epilogue, on the even CTA's
            mbar_init(smem_u32(sm.tempty + b),
                      kPair ? 2u : static_cast<uint32_t>(kEpiWarps<WF> * 32));
            mbar_init(smem_u32(sm.sfull + b), 1);
            mbar_init(smem_u32(sm.sempty + b), WF == 3 ? kMxScaleWarps : kConvTeams * kConvThreads);
        }
        mbar_init(smem_u32(sm.drain), 1);
        mbar_init(smem_u32(sm.drain + 1), 1);
        flags[0] = 0;
        flags[1] = 0;
        flags[2] = 0;
        flags[3] = 0;
        mbar_fence_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmap_w);
        tma_prefetch_desc(&tmap_x);
    }
    if (warp == 1) {
        tmem_alloc<CG>(smem_u32(sm.tmem_base), static_cast<uint32_t>(p.tmem_cols));
        tmem_relinquish<CG>();
    }
    tc_fence_before();
    __syncthreads();
    // pair: both CTAs' barriers are initialised before either CTA's TMA
    // loads, MMAs or arrivals reach them
    if (kPair) cluster_sync();
    tc_fence_after();
    const uint32_t tmem_base = *sm.tmem_base;
    if (threadIdx.x == 0) MOE_TRACE_POINT(g_trace_gemm, EPI, blockIdx.x, 1);

    // The GEMM token tiles were written by the router.  With p.prewait set
    // the router has completed before this kernel starts: the launch order
    // is router -> permutation -> gate_up -> down, and each of the later
    // kernels lets its successor start only after its own
    // griddepcontrol.wait has returned, i.e. after its predecessor
    // completed.  The token operand (gathered activations, or h) is written
    // by the kernel launched just before this one and is read only after
    // griddepcontrol.wait.  The producer therefore streams the first ring
    // slots' weight tiles (and weight scales) before that wait, overlapping
    // the previous kernel; every other role waits first.  Without p.prewait
    // (small batches: the router launched just before gate_up) the producer
    // too waits before reading the tile list.
    if (warp != 0) {
        pdl_wait();
        pdl_launch_dependents();
    }

    // (read at L2: the producer reads it before griddepcontrol.wait)
    const int num_units = __ldcg(p.num_tiles) * p.n_wblocks * p.ksplit;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();
            const uint64_t pol_x = policy_evict_last();
            const uint32_t w_bytes = WF == 1 ? kCodeStageBytes : WF == 3 ? kMxCodeTxBytes : kATileBytes;
            // Loads of one ring slot: the weight part (`wpart`) and/or the
            // token part; the slot's full barrier expects both.
            const auto slot_loads = [&](const Unit& un, const int4& t, int st, int stage,
                                        bool wpart, bool tpart, bool expect) {
                (void)tpart;
                const uint32_t fb = smem_u32(sm.full + stage);
                const int mb = un.mb;
                // full boxes are counted, zero-filled past K included;
                // pair: the even CTA's barrier counts both CTAs' bytes
                // MXFP4 x MXFP8: nk k-blocks (the K range's last slot may
                // hold one), 8 KB of codes + the token tile each
                const int nk = min(KPS, p.k_blocks - st * KPS);
                // (gathered token rows arrive through the gather warp)
                const bool gathered = WF == 0 && p.gather_x != nullptr;
                if (gathered) tpart = false;
                if (expect && rank == 0)
                    mbar_arrive_expect_tx(
                        fb, WF == 3 ? static_cast<uint32_t>(nk) * (kMxCodeTxBytes + b_bytes)
                                    : (kPair ? 2u : 1u) *
                                          (w_bytes + (gathered ? 0u : b_stage_bytes)));
                const uint32_t b_dst = smem_u32(sm.b + static_cast<size_t>(stage) * b_stage_bytes);
                if (WF == 1) {
                    // codes of k-blocks 4st..4st+3 (128 B per row), and the
                    // token rows' K chunks 4st..4st+3 (chunk-major operand)
                    if (wpart)
                        tma_load_3d(smem_u32(sm.codes + static_cast<size_t>(stage) * kCodeStageBytes),
                                    &tmap_w, fb, st * KPS * (kBlockK / 2), mb * kWeightTileRows, t.x,
                                    pol_w);
                    if (tpart) tma_load_3d(b_dst, &tmap_x, fb, 0, t.y, st * KPS, pol_x);
                } else if (WF == 3) {
                    // E2M1 codes of K 64c..64c+127 (c = 2 st, or the last
                    // chunk starting 64 early), padded by TMA to 128 B rows
                    for (int jj = 0; jj < nk; ++jj) {
                        const int kb = st * KPS + jj;
                        if (wpart)
                            tma_load_4d(smem_u32(sm.a + (static_cast<size_t>(stage) * KPS + jj) *
                                                            kATileBytes),
                                        &tmap_w, fb, 0, min(2 * kb, p.mx_cmax),
                                        mb * kWeightTileRows, t.x, pol_w);
                        if (tpart)
                            tma_load_2d(b_dst + static_cast<uint32_t>(jj) * b_bytes, &tmap_x, fb,
                                        kb * kKB, t.y, pol_x);
                    }
                } else if (kPair) {
                    // rows 128 * rank.. of the 256-row block; token rows
                    // n/2 * rank.. of the tile (each CTA holds N/2 of B)
                    const uint32_t fb0 = mapa_shared(fb, 0);
                    const int half_n = ((t.z + 15) & ~15) / 2;
                    if (wpart)
                        tma_load_3d_pair(smem_u32(sm.a + static_cast<size_t>(stage) * kATileBytes),
                                         &tmap_w, fb0, st * kKB,
                                         mb * kUnitRows + static_cast<int>(rank) * kWeightTileRows,
                                         t.x, pol_w);
                    if (tpart)
                        tma_load_2d_pair(b_dst, &tmap_x, fb0, st * kKB,
                                         t.y + static_cast<int>(rank) * half_n, pol_x);
                } else {
                    if (wpart)
                        tma_load_3d(smem_u32(sm.a + static_cast<size_t>(stage) * kATileBytes),
                                    &tmap_w, fb, st * kKB, mb * kWeightTileRows, t.x, pol_w);
                    if (tpart) tma_load_2d(b_dst, &tmap_x, fb, st * kKB, t.y, pol_x);
                }
            };
            // A unit's scale rows (MXFP4 and MXFP4 x MXFP8), one bulk copy
            // into buffer sb: the weight scales and/or (MXFP4 x MXFP8) the
            // token tile's scales, written by the previous kernel.
            const auto scale_loads = [&](const Unit& un, const int4& t, int sb, bool wpart,
                                         bool tpart, bool expect) {
                const int rows = min(kWeightTileRows, p.w_rows - un.mb * kWeightTileRows);
                const uint32_t bytes = static_cast<uint32_t>(rows * p.kscale);
                const bool tok = WF == 3 && p.xs_mx != nullptr;
                const uint32_t tbytes = tok ? static_cast<uint32_t>(t.z * p.xs_row_bytes) : 0u;
                const uint32_t sf = smem_u32(sm.sfull + sb);
                if (expect) mbar_arrive_expect_tx(sf, bytes + tbytes);
                if (wpart)
                    bulk_load(smem_u32(sm.scales + sb * scale_buf_bytes),
                              p.scales + (static_cast<size_t>(t.x) * p.w_rows +
                                          static_cast<size_t>(un.mb) * kWeightTileRows) * p.kscale,
                              bytes, sf);
                if (tok && tpart)
                    bulk_load(smem_u32(sm.tscales + sb * tscale_buf_bytes),
                              p.xs_mx + static_cast<size_t>(t.y) * p.xs_row_bytes, tbytes, sf);
            };

            // Before the wait: the weight parts of the first ring slots (at
            // most one ring), and the first two units' weight scales.
            int npre = 0, npre_units = 0;
            if (p.prewait) {
                int stage = 0, local = 0;
                for (int u = cta0; u < num_units && npre < stages; u += ncta) {
                    const Unit un = unit_of(u, p, n_st);
                    const int4 t = __ldcg(p.tiles + un.tile);
                    if (!tile_ok(t, p)) continue;
                    if (WF == 1 || WF == 3) {
                        if (local == 2) break;              // both scale buffers taken
                        scale_loads(un, t, local & 1, true, false, true);
                        npre_units = ++local;
                    }
                    for (int st = un.st_lo; st < un.st_hi && npre < stages; ++st) {
                        slot_loads(un, t, st, stage, true, false, true);
                        ++npre;
                        ++stage;
                    }
                }
            }
            MOE_TRACE_POINT(g_trace_gemm, EPI, blockIdx.x, 2);
            pdl_wait();
            pdl_launch_dependents();
            MOE_TRACE_POINT(g_trace_gemm, EPI, blockIdx.x, 3);
            // without the early pass the tile list may come from the kernel
            // just before this one: count the units only now
            const int num_units_p =
                p.prewait ? num_units : __ldcg(p.num_tiles) * p.n_wblocks * p.ksplit;

            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            int local = 0;
            bool ok = true;
            for (int u = cta0; u < num_units_p && ok; u += ncta) {
                const Unit un = unit_of(u, p, n_st);
                const int4 t = p.tiles[un.tile];
                if (!tile_ok(t, p)) continue;
                if (WF == 1 || WF == 3) {
                    // this unit's scale rows, one bulk copy, double-buffered
                    // (MXFP4 x MXFP8: and the token tile's scale rows)
                    const int sb = local & 1;
                    const uint32_t sph = static_cast<uint32_t>(local >> 1) & 1u;
                    if (local < npre_units) {
                        scale_loads(un, t, sb, false, true, false);
                    } else {
                        if (!mbar_wait(smem_u32(sm.sempty + sb), sph ^ 1u, flags)) {
                            raise_abort(flags, p.status, MOE_DEV_WAIT_TIMEOUT);
                            ok = false;
                            break;
                        }
                        scale_loads(un, t, sb, true, true, true);
                    }
                }
                ++local;
                for (int st = un.st_lo; st < un.st_hi; ++st) {
                    if (issued < npre) {
                        // weight part already in flight: the token part only
                        slot_loads(un, t, st, stage, false, true, false);
                    } else {
                        if (!mbar_wait(smem_u32(sm.empty + stage), phase ^ 1u, flags)) {
                            raise_abort(flags, p.status, MOE_DEV_WAIT_TIMEOUT);
                            ok = false;
                            break;
                        }
                        slot_loads(un, t, st, stage, true, true, true);
                    }
                    ++issued;
                    if (++stage == stages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok && rank == 0) {
                // Wait (bounded) for the loads still in flight before the CTA
                // may release its shared memory (pair: the even CTA's
                // barriers count the odd CTA's loads too).
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
                if ((WF == 1 || WF == 3) && local > 0) {
                    const int sb = (local - 1) & 1;
                    mbar_wait(smem_u32(sm.sfull + sb), static_cast<uint32_t>((local - 1) >> 1) & 1u,
                              nullptr);
                }
            }
        } else {
            pdl_wait();
            pdl_launch_dependents();
        }
    } else if (WF != 1 && warp == 1) {
        // ------------------------------------------------ MMA issuer (bf16)
        // The whole warp walks the loop, so the barrier waits and the
        // descriptors are warp-uniform, and one elected lane issues the MMAs
        // and commits: 4 MMAs + commit then take ~170 SM cycles, against
        // ~450 when a lone lane walks the loop.  Pair: the even CTA issues
        // for both; the odd CTA's warp 1 only allocates and frees its TMEM.
        if (rank == 0) {
            const bool leader = elect_one();
            int stage = 0;
            uint32_t phase = 0;
            int local = 0;
            bool ok = true;
            // test fault: a wait on a barrier that nothing arrives on (the
            // second drain barrier, unused by this issuer) runs out
            if (!kPair && p.inject_stall && !warp_wait(smem_u32(sm.drain + 1), 0, flags)) {
                if (leader) raise_abort(flags, p.status, MOE_DEV_WAIT_TIMEOUT);
                ok = false;
            }
            for (int u = cta0; u < num_units && ok; u += ncta) {
                const Unit un = unit_of(u, p, n_st);
                const int4 t = p.tiles[un.tile];
                if (!tile_ok(t, p)) continue;
                const uint32_t n_mma = static_cast<uint32_t>((t.z + 15) & ~15);
                const uint32_t idesc = WF == 3   ? idesc_mx_e2m1_e4m3(kUnitRows, n_mma, 0)
                                       : WF == 2 ? idesc_e4m3_f32(kUnitRows, n_mma)
                                                 : idesc_bf16_f32(kUnitRows, n_mma);
                const int buf = local & 1;
                const uint32_t tph = static_cast<uint32_t>(local >> 1) & 1u;
                ++local;
                if (!warp_wait(smem_u32(sm.tempty + buf), tph ^ 1u, flags)) {
                    if (leader) raise_abort(flags, p.status, MOE_DEV_WAIT_TIMEOUT);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf) * acc_stride;
                for (int st = un.st_lo; st < un.st_hi; ++st) {
                    // (gathered token rows: their own barrier)
                    if (!warp_wait(smem_u32(sm.full + stage), phase, flags) ||
                        (p.gather_x != nullptr &&
                         !warp_wait(smem_u32(sm.gfull + stage), phase, flags))) {
                        if (leader) raise_abort(flags, p.status, MOE_DEV_WAIT_TIMEOUT);
                        ok = false;
                        break;
                    }
                    if (local == 1 && st == un.st_lo && lane == 0)
                        MOE_TRACE_POINT(g_trace_gemm, EPI, blockIdx.x, 4);
                    tc_fence_after();
                    // K steps of 16: +32 bytes along the swizzled rows, +2 in
                    // the descriptors' start-address field (address >> 4)
                    const uint64_t ad =
                        smem_desc_sw128(smem_u32(sm.a + static_cast<size_t>(stage) * kATileBytes));
                    const uint64_t bd =
                        smem_desc_sw128(smem_u32(sm.b + static_cast<size_t>(stage) * b_stage_bytes));
                    const uint32_t acc0 = st != un.st_lo ? 1u : 0u;   // the part's first k-block
                    if (WF == 3 && leader) {
                        // nk k-blocks, each 4 MMAs with scale byte kk of the
                        // k-block's 8 scale columns
                        const int nk = min(KPS, p.k_blocks - st * KPS);
                        for (int jj = 0; jj < nk; ++jj) {
                            const uint64_t adj = smem_desc_sw128(smem_u32(
                                sm.a + (static_cast<size_t>(stage) * KPS + jj) * kATileBytes));
                            const uint64_t bdj = smem_desc_sw128(smem_u32(
                                sm.b + static_cast<size_t>(stage) * b_stage_bytes +
                                static_cast<size_t>(jj) * b_bytes));
                            const uint32_t sfa = tmem_base + sf_col0 +
                                                 8u * static_cast<uint32_t>(stage * KPS + jj);
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                tc_mma_mx(d_tmem, adj + 2 * kk, bdj + 2 * kk,
                                          idesc | (static_cast<uint32_t>(kk) << 4) |
                                              (static_cast<uint32_t>(kk) << 29),
                                          sfa, sfa + 4u, (jj == 0 && kk == 0) ? acc0 : 1u);
                        }
                        tc_commit(smem_u32(sm.empty + stage));
                    } else if (leader) {
#pragma unroll
                        for (int kk = 0; kk < kBlockK / 16; ++kk) {
                            const uint32_t acc = kk == 0 ? acc0 : 1u;
                            // one MMA per 32 bytes of K (16 bf16, 32 E4M3)
                            if constexpr (kPair && WF == 2)
                                tc_mma_e4m3_pair(d_tmem, ad + 2 * kk, bd + 2 * kk, idesc, acc);
                            else if constexpr (kPair)
                                tc_mma_bf16_pair(d_tmem, ad + 2 * kk, bd + 2 * kk, idesc, acc);
                            else if constexpr (WF == 2)
                                tc_mma_e4m3(d_tmem, ad + 2 * kk, bd + 2 * kk, idesc, acc);
                            else
                                tc_mma_bf16(d_tmem, ad + 2 * kk, bd + 2 * kk, idesc, acc);
                        }
                        // pair: the slot is free in both CTAs
                        if constexpr (kPair)
                            tc_commit_pair_mc(smem_u32(sm.empty + stage), 3);
                        else
                            tc_commit(smem_u32(sm.empty + stage));
                    }
                    __syncwarp();
                    if (++stage == stages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                if (leader) {
                    if constexpr (kPair)
                        tc_commit_pair_mc(smem_u32(sm.tfull + buf), 3);
                    else
                        tc_commit(smem_u32(sm.tfull + buf));
                }
                __syncwarp();
            }
            // Every MMA issued so far has finished once this arrives.
            if (leader) {
                MOE_TRACE_POINT(g_trace_gemm, EPI, blockIdx.x, 5);
                if constexpr (kPair)
                    tc_commit_pair(smem_u32(sm.drain));
                else
                    tc_commit(smem_u32(sm.drain));
                mbar_wait(smem_u32(sm.drain), 0, nullptr);
            }
            __syncwarp();
        }
    } else if (WF == 1 && (warp == 1 || warp == kSecondIssuerWarp)) {
        // ------------------------------------------------ MMA issuers (MXFP4)
        // Issuer `is` takes the ring slots whose use (the ring position counted
        // over the CTA's units) has parity `is`, so that an A slot and a
        // converter team always meet the same issuer -- their barrier phases
        // then advance in order even when a unit has an odd slot count; as
        // for bf16, its whole warp walks the loop and one elected lane issues.
        const int is = warp == 1 ? 0 : 1;
        if constexpr (WF == 1) if (is < n_iss) {
            const bool leader = elect_one();
            int local = 0;
            int sbase = 0;                        // ring use of the unit's first slot
            // ring positions of use `cur`, advanced (not divided) to each use
            int cur = 0, stage = 0, astage = 0;
            uint32_t phase = 0, aphase = 0;
            bool ok = true;
            for (int u = cta0; u < num_units && ok; u += ncta) {
                const Unit un = unit_of(u, p, n_st);
                const int4 t = p.tiles[un.tile];
                if (!tile_ok(t, p)) continue;
                const uint32_t n_mma = static_cast<uint32_t>((t.z + 15) & ~15);
                const uint32_t idesc = p.mx_f16 ? idesc_f16_f32(kWeightTileRows, n_mma)
                                                : idesc_bf16_f32(kWeightTileRows, n_mma);
                const int buf = local & 1;
                const uint32_t tph = static_cast<uint32_t>(local >> 1) & 1u;
                ++local;
                if (!warp_wait(smem_u32(sm.tempty + buf), tph ^ 1u, flags)) {
                    if (leader) raise_abort(flags, p.status, MOE_DEV_WAIT_TIMEOUT);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem =
                    tmem_base + static_cast<uint32_t>(2 * is + buf) * acc_stride;
                // issuer `is` takes the unit's slots of use parity `is` (the
                // parity of its A slot and converter team in every unit)
                const int off = n_iss == 2 ? ((is ^ sbase) & 1) : 0;
                for (int st = un.st_lo + off; st < un.st_hi && ok; st += n_iss) {
                    for (const int use = sbase + (st - un.st_lo); cur < use; ++cur) {
                        if (++stage == stages) {
                            stage = 0;
                            phase ^= 1u;
                        }
                        if (++astage == astages) {
                            astage = 0;
                            aphase ^= 1u;
                        }
                    }
                    const int nk = min(KPS, p.k_blocks - st * KPS);
                    // The slot's A slot is converted (which implies its codes
                    // and token chunks landed).  One wait per slot: a wait
                    // issued behind in-flight MMAs costs about as much as four
                    // N = 16 MMAs.
                    if (!warp_wait(smem_u32(sm.afull + astage), aphase, flags)) {
                        if (leader) raise_abort(flags, p.status, MOE_DEV_WAIT_TIMEOUT);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t b_stage =
                        smem_u32(sm.b + static_cast<size_t>(stage) * b_stage_bytes);
                    const uint32_t a_tm = tmem_base + a_col0 + kASlotCols * static_cast<uint32_t>(astage);
                    if (leader) {
                        for (int jj = 0; jj < nk; ++jj) {
                            // the issuer's first MMA of the unit starts its sum
                            const bool first = st == un.st_lo + off && jj == 0;
                            const uint64_t bd =
                                smem_desc_sw128(b_stage + static_cast<uint32_t>(jj) * b_bytes);
#pragma unroll
                            for (int kk = 0; kk < kBlockK / 16; ++kk)
                                tc_mma_bf16_ts(d_tmem, a_tm + 32u * jj + 8u * kk, bd + 2 * kk, idesc,
                                               (first && kk == 0) ? 0u : 1u);
                        }
                        tc_commit(smem_u32(sm.aempty + astage));
                        tc_commit(smem_u32(sm.empty + stage));
                    }
                    __syncwarp();
                }
                if (!ok) break;
                sbase += un.st_hi - un.st_lo;
                if (leader) tc_commit(smem_u32(sm.tfull + buf));
                __syncwarp();
            }
            // Every MMA this issuer issued has finished once this arrives.
            if (leader) {
                tc_commit(smem_u32(sm.drain + is));
                mbar_wait(smem_u32(sm.drain + is), 0, nullptr);
            }
            __syncwarp();
        }
    } else if (warp < 2 + kEpiWarps<WF>) {
        // ------------------------------------------------ epilogue
        constexpr int kEpiThreads = kEpiWarps<WF> * 32;
        constexpr int kHalves = kEpiWarps<WF> / 4;     // warps per lane quadrant
        const int ep = threadIdx.x - 64;          // 0 .. kEpiThreads-1
        const int quad = warp & 3;                // TMEM lane quadrant of this warp
        const int half = (warp - 2) >> 2;         // this warp's share of the columns
        const int row_in_tile = quad * 32 + lane;
        // the output rows the down projection will accumulate into (with
        // bf16 weights and no gathering to do, the gather warp clears them
        // in the background instead)
        if (p.zero_out != nullptr && !(kGatherWarpOf<WF> >= 0 && p.gather_x == nullptr)) {
            float4* z = reinterpret_cast<float4*>(p.zero_out);
            for (size_t i = static_cast<size_t>(blockIdx.x) * kEpiThreads + ep; i < p.n_zero / 4;
                 i += static_cast<size_t>(gridDim.x) * kEpiThreads)
                z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        int local = 0;
        int sbase = 0;                            // ring use of the unit's first slot
        for (int u = cta0; u < num_units; u += ncta) {
            const Unit un = unit_of(u, p, n_st);
            const int4 t = p.tiles[un.tile];
            if (!tile_ok(t, p)) {
                if (ep == 0) atomicOr(p.status + kStatusWord, MOE_DEV_BAD_TILE);
                continue;
            }
            const int mb = un.mb;
            const int buf = local & 1;
            const uint32_t tph = static_cast<uint32_t>(local >> 1) & 1u;
            ++local;

            if (EPI == kEpiCombine) {
                named_bar_sync(1, kEpiThreads);   // previous unit done with meta
                for (int c = ep; c < t.z; c += kEpiThreads) {
                    // a row the permutation could not fill (a bad expert id,
                    // inconsistent counts) holds a stale entry: never let it
                    // address memory outside this call's buffers
                    const int a = p.sorted_assign[t.y + c];
                    const bool a_ok = a >= 0 && a < p.rows_total;
                    if (!a_ok) atomicOr(p.status + kStatusWord, MOE_DEV_BAD_TILE);
                    sm.meta_tok[c] = a_ok ? a / p.top_k : -1;
                    sm.meta_w[c] = a_ok ? p.topk_w[a] : 0.f;
                }
            } else if (WF == 2) {
                // FP8 gate_up: the activation scale of each routed row
                named_bar_sync(1, kEpiThreads);   // previous unit done with meta
                for (int c = ep; c < t.z; c += kEpiThreads) sm.meta_w[c] = p.xscale[t.y + c];
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

            const int wrow = mb * kUnitRows + static_cast<int>(rank) * kWeightTileRows + row_in_tile;
            const bool row_ok = wrow < p.w_rows;
            // the bias enters once: down adds it with part 0, gate_up after the sum
            const float bias =
                row_ok && (EPI == kEpiGlu || un.split == 0)
                    ? __bfloat162float(p.bias[static_cast<size_t>(t.x) * p.w_rows + wrow])
                    : 0.f;
            // FP8: the expert's weight scale (applied to the finished sum)
            const float wsc = WF == 2 ? p.wscale[t.x] : 1.f;
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                                   static_cast<uint32_t>(buf) * acc_stride;
            const int n_mma = (t.z + 15) & ~15;
            // issuers that had ring slots in this unit (MXFP4 issuer i takes
            // the slots of use parity i)
            const int nsl = un.st_hi - un.st_lo;
            const bool has0 = n_iss == 1 || nsl > (sbase & 1);
            const bool has1 = n_iss == 2 && nsl > ((1 ^ sbase) & 1);
            sbase += nsl;
            // This part's accumulator, 16 token columns from c0 (both issuers added).
            auto load_acc = [&](int c0, float (&v)[16]) {
                if (has0) {
                    tmem_ld16(taddr + static_cast<uint32_t>(c0), v);
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] = 0.f;
                }
                if (has1) {
                    float v2[16];
                    tmem_ld16(taddr + 2u * acc_stride + static_cast<uint32_t>(c0), v2);
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] += v2[i];
                }
            };
            // bias + clamped GLU of 16 token columns, bf16 store of h
            auto glu_store = [&](int c0, float (&v)[16]) {
                // even lane: gate row 2j, odd lane: up row 2j+1 (same j)
                const bool odd = lane & 1;
                const int hcols = p.w_rows >> 1;
                // MXFP4: h is the down projection's token operand in its
                // layout -- chunk-major [I/64][T*k][64], each group of 8
                // columns in the order 0,4,1,5,2,6,3,7
                // (f16 mode: natural order, f16 values)
                const int hcol = WF == 1 && !p.mx_f16 ? kperm8_pos(wrow >> 1) : (wrow >> 1);
                __nv_bfloat16* hrow0 =
                    WF == 1 ? p.h + (static_cast<size_t>(hcol >> 6) * p.rows_total + t.y) * 64 +
                                  (hcol & 63)
                            : p.h + static_cast<size_t>(t.y) * hcols + hcol;
                const size_t hstride = WF == 1 ? 64 : static_cast<size_t>(hcols);
                // FP8: h as E4M3 codes of h / kFp8HScale, [T*k, I] bytes;
                // MXFP4 x MXFP8: the same codes in the padded layout
                // [T*k, h_pad], column hcol at mx_pos (the gap zeroed by the
                // threads of the last 64 columns)
                const size_t h8stride = WF == 3 ? static_cast<size_t>(p.h_pad)
                                                : static_cast<size_t>(hcols);
                uint8_t* h8row0 = p.h8 + static_cast<size_t>(t.y) * h8stride +
                                  (WF == 3 ? mx_pos(hcol, p.h_tail0) : hcol);
                const bool h8gap = WF == 3 && hcol >= p.h_tail0;
                if (WF == 2) {
                    // the sum of code products times weight scale x row scale
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] = v[i] * (wsc * sm.meta_w[c0 + i]) + bias;
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] += bias;
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float send = odd ? v[i] : v[8 + i];
                    const float recv = __shfl_xor_sync(0xffffffffu, send, 1);
                    const float gate = odd ? recv : v[i];
                    const float up = odd ? v[8 + i] : recv;
                    const int c = c0 + i + (odd ? 8 : 0);
                    // rows past 2I exist only in the last 256-row block of
                    // CTA pairs (gate and up rows share their validity)
                    if (c < t.z && row_ok &&
                        MOE_BOUNDS(t.y + c < p.rows_total && hcol < hcols, p.status)) {
                        if (WF >= 2) {
                            uint8_t* dst = h8row0 + static_cast<size_t>(c) * h8stride;
                            *dst = static_cast<uint8_t>(
                                cvt_e4m3x2(clamped_glu(gate, up) * (1.f / kFp8HScale), 0.f));
                            if (h8gap) dst[-64] = 0;
                        } else if (WF == 1 && p.mx_f16) {
                            reinterpret_cast<__half*>(hrow0)[static_cast<size_t>(c) * hstride] =
                                __float2half_rn(clamped_glu(gate, up));
                        } else {
                            hrow0[static_cast<size_t>(c) * hstride] =
                                __float2bfloat16_rn(clamped_glu(gate, up));
                        }
                    }
                }
            };

            if (EPI == kEpiGlu && p.ksplit > 1) {
                // K split: store this part's fp32 tile [col][row], release the
                // accumulator, take a ticket; the last part adds all parts in
                // part order (the same sum whichever part arrives last).
                // part q of this unit: rows t.y.. of block mb in part q's plane
                const size_t part_floats =
                    static_cast<size_t>(p.n_wblocks) * p.rows_total * kWeightTileRows;
                const size_t unit_off =
                    (static_cast<size_t>(mb) * p.rows_total + t.y) * kWeightTileRows + row_in_tile;
                float* mine = p.partial + un.split * part_floats + unit_off;
                for (int c0 = 16 * half; c0 < n_mma; c0 += 16 * kHalves) {
                    float v[16];
                    load_acc(c0, v);
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        if (c0 + i < t.z &&
                            MOE_BOUNDS(un.split < p.ksplit && mb < p.n_wblocks &&
                                           t.y + c0 + i < p.rows_total, p.status))
                            mine[static_cast<size_t>(c0 + i) * kWeightTileRows] = v[i];
                }
                tc_fence_before();
                mbar_arrive(smem_u32(sm.tempty + buf));
                __threadfence();
                named_bar_sync(1, kEpiThreads);
                if (ep == 0) {
                    const int ticket = atomicAdd(p.tickets + un.pair, 1);
                    const int last = ticket == p.ksplit - 1;
                    if (last) p.tickets[un.pair] = 0;   // zero for the next call
                    flags[3] = last;
                }
                named_bar_sync(1, kEpiThreads);
                if (!flags[3]) continue;
                __threadfence();
                const float* parts = p.partial + unit_off;
                for (int c0 = 16 * half; c0 < n_mma; c0 += 16 * kHalves) {
                    float v[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] = 0.f;
                    for (int q = 0; q < p.ksplit; ++q) {
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            if (c0 + i < t.z)
                                v[i] += __ldcg(parts + q * part_floats +
                                               static_cast<size_t>(c0 + i) * kWeightTileRows);
                    }
                    glu_store(c0, v);
                }
                continue;
            }

            for (int c0 = 16 * half; c0 < n_mma; c0 += 16 * kHalves) {
                float v[16];
                load_acc(c0, v);
                if (EPI == kEpiGlu) {
                    glu_store(c0, v);
                } else {
                    if (WF == 2) {
                        // FP8 down: weight scale x the h codes' scale
                        const float dsc = wsc * p.hscale;
#pragma unroll
                        for (int i = 0; i < 16; ++i) v[i] = v[i] * dsc + bias;
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i) v[i] += bias;
                    }
                    if (row_ok && p.y_rows) {
                        // deterministic combine: this slot's weighted row,
                        // summed in slot order by a later kernel
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const int c = c0 + i;
                            if (c < t.z && MOE_BOUNDS(t.y + c < p.rows_total, p.status))
                                p.y_rows[static_cast<size_t>(t.y + c) * p.w_rows + wrow] =
                                    sm.meta_w[c] * v[i];
                        }
                    } else if (row_ok) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const int c = c0 + i;
                            const int tok = c < t.z ? sm.meta_tok[c] : -1;
                            if (tok >= 0 &&
                                MOE_BOUNDS(tok < p.rows_total / p.top_k && wrow < p.w_rows,
                                           p.status))
                                atomicAdd(p.out + static_cast<size_t>(tok) * p.w_rows + wrow,
                                          sm.meta_w[c] * v[i]);
                        }
                    }
                }
            }
            tc_fence_before();
            if (kPair) {
                // one arrival per CTA, on the even CTA's barrier, once all
                // 128 threads' TMEM loads are done
                named_bar_sync(1, kEpiThreads);
                if (ep == 0) mbar_arrive_cluster(mapa_shared(smem_u32(sm.tempty + buf), 0));
            } else {
                mbar_arrive(smem_u32(sm.tempty + buf));
            }
        }
        if (ep == 0) MOE_TRACE_POINT(g_trace_gemm, EPI, blockIdx.x, 6);
    } else if (kGatherWarpOf<WF> >= 0 && warp == kGatherWarpOf<WF>) {
        // ------------------------------------------------ token-row gather
        // Small batches (bf16 gate_up): each ring slot's token tile is copied
        // here from the layer input, row r of tile t being input row
        // sorted_assign[t.y + r] / top_k, 16 bytes per lane with cp.async into
        // the 128-byte-swizzled layout TMA would have written (chunk c of row
        // r at chunk c ^ (r % 8)).  Copies of kGatherLag slots stay in
        // flight; a slot's copies are awaited, made visible to the tensor
        // cores (proxy fence) and announced with one arrival.  Rows past the
        // tile keep whatever they held: their products are never stored.
        // (The slot's own "gfull" barrier, not "full", takes the arrival, so
        // that "full" still tracks the TMA bytes alone for the producer's
        // bounded drain after an abort.)
        if (p.gather_x == nullptr && p.zero_out != nullptr) {
            // nothing to gather: this warp clears the output rows the down
            // projection will accumulate into, alongside the pipeline
            float4* z = reinterpret_cast<float4*>(p.zero_out);
            for (size_t i = static_cast<size_t>(blockIdx.x) * 32 + lane; i < p.n_zero / 4;
                 i += static_cast<size_t>(gridDim.x) * 32)
                z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        if (p.gather_x != nullptr) {
            int stage = 0;
            uint32_t phase = 0;
            int inflight = 0;
            bool ok = true;
            const auto announce_oldest = [&](int pending) {
                int s0 = stage - (pending - 1);
                if (s0 < 0) s0 += stages;
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(sm.gfull + s0));
            };
            for (int u = cta0; u < num_units && ok; u += ncta) {
                const Unit un = unit_of(u, p, n_st);
                const int4 t = p.tiles[un.tile];
                if (!tile_ok(t, p)) continue;
                // input rows of tile rows lane and lane + 32 (t.z <= 64 here)
                int tok0 = -1, tok1 = -1;
                if (lane < t.z) {
                    const int a = p.sorted_assign[t.y + lane];
                    if (a >= 0 && a < p.rows_total) tok0 = a / p.top_k;
                }
                if (lane + 32 < t.z) {
                    const int a = p.sorted_assign[t.y + lane + 32];
                    if (a >= 0 && a < p.rows_total) tok1 = a / p.top_k;
                }
                const int nchunk = t.z * 8;
                for (int st = un.st_lo; st < un.st_hi; ++st) {
                    if (!warp_wait(smem_u32(sm.empty + stage), phase ^ 1u, flags)) {
                        if (lane == 0) raise_abort(flags, p.status, MOE_DEV_WAIT_TIMEOUT);
                        ok = false;
                        break;
                    }
                    const uint32_t b_dst = smem_u32(sm.b + static_cast<size_t>(stage) * b_stage_bytes);
                    for (int base = 0; base < nchunk; base += 32) {
                        const int i = base + lane, r = i >> 3, c = i & 7;
                        const int ta = __shfl_sync(0xffffffffu, tok0, r & 31);
                        const int tb = __shfl_sync(0xffffffffu, tok1, r & 31);
                        const int tk = r < 32 ? ta : tb;
                        if (i < nchunk && tk >= 0)
                            cp_async_16(b_dst + static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4)),
                                        p.gather_x + static_cast<size_t>(tk) * p.gather_K +
                                            st * kBlockK + c * 8);
                    }
                    cp_async_commit();
                    if (++inflight > kGatherLag) {
                        cp_async_wait<kGatherLag>();
                        announce_oldest(inflight);
                        --inflight;
                    }
                    if (++stage == stages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // the last slots: every copy landed (also on an abort, before the
            // CTA's shared memory is released)
            cp_async_wait<0>();
            if (ok) {
                for (; inflight > 0; --inflight) {
                    int s0 = stage - inflight;
                    if (s0 < 0) s0 += stages;
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(sm.gfull + s0));
                }
            }
        }
    } else if (WF == 3) {
        // ------------------------------------------------ MX scale writers
        // Warps 6..9 (one per TMEM lane quadrant) copy each ring slot's
        // UE8M0 scales into the slot's 8 TMEM columns once the MMAs are done
        // with the slot's previous use (the same barrier the producer waits
        // for), then arrive on the slot's "full" barrier beside the TMA
        // bytes.  A: weight row r (this quadrant's lanes) at column r / 32 =
        // quad, the 4 bytes of K blocks 2c..2c+3 (c the slot's code chunk).
        // B: token row n at lane n % 32 of every quadrant (each quadrant of
        // the MMA reads the token scales from its own lanes), column
        // 4 + n / 32, the 4 bytes of the slot's K blocks 4 st..4 st+3 of the
        // padded operand, or 2^-3 for every block of the h operand.
        const int quad = warp & 3;
        const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(quad * 32) << 16);
        int stage = 0;
        uint32_t phase = 0;
        int local = 0;
        bool ok = true;
        for (int u = cta0; u < num_units && ok; u += ncta) {
            const Unit un = unit_of(u, p, n_st);
            const int4 t = p.tiles[un.tile];
            if (!tile_ok(t, p)) continue;
            const int wrow = un.mb * kWeightTileRows + quad * 32 + lane;
            const bool row_ok = wrow < p.w_rows;
            // this unit's scale rows, staged in shared memory by the producer
            // (one bulk copy per unit, double-buffered): a per-slot load from
            // L2 kept the slot's MMAs waiting ~0.5 us for these warps
            const int sb = local & 1;
            const uint32_t sph = static_cast<uint32_t>(local >> 1) & 1u;
            ++local;
            if (!warp_wait(smem_u32(sm.sfull + sb), sph, flags)) {
                if (lane == 0) raise_abort(flags, p.status, MOE_DEV_WAIT_TIMEOUT);
                ok = false;
                break;
            }
            // rows past the matrix are TMA zero-fill: scale 1 keeps them zero
            const uint8_t* srow = sm.scales + sb * scale_buf_bytes + (quad * 32 + lane) * p.kscale;
            const uint8_t* trow = sm.tscales + sb * tscale_buf_bytes;
            // the scale values of k-block kb (weight rows: two aligned halves,
            // as kscale = K / 32 and 2c are even; token rows, or 2^-3 for h)
            const auto load_vals = [&](int kb, uint32_t& va, uint32_t (&vb)[4]) {
                va = 0x7F7F7F7Fu;
                if (row_ok) {
                    const uint16_t* s16 =
                        reinterpret_cast<const uint16_t*>(srow + 2 * min(2 * kb, p.mx_cmax));
                    va = static_cast<uint32_t>(s16[0]) | (static_cast<uint32_t>(s16[1]) << 16);
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int n = 32 * j + lane;
                    vb[j] = 0x7C7C7C7Cu;
                    if (p.xs_mx != nullptr)
                        vb[j] = n < t.z ? *reinterpret_cast<const uint32_t*>(
                                              trow + n * p.xs_row_bytes + 4 * kb)
                                        : 0x7F7F7F7Fu;
                }
            };
            for (int st = un.st_lo; st < un.st_hi; ++st) {
                // the slot's values first: their loads overlap the wait (loading
                // one slot further ahead measured slower)
                const int nk = min(KPS, p.k_blocks - st * KPS);
                uint32_t va[KPS], vb[KPS][4];
#pragma unroll
                for (int jj = 0; jj < KPS; ++jj)
                    if (jj < nk) load_vals(st * KPS + jj, va[jj], vb[jj]);
                if (!warp_wait(smem_u32(sm.empty + stage), phase ^ 1u, flags)) {
                    if (lane == 0) raise_abort(flags, p.status, MOE_DEV_WAIT_TIMEOUT);
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int jj = 0; jj < KPS; ++jj) {
                    if (jj >= nk) break;
                    const uint32_t col = sf_col0 + 8u * static_cast<uint32_t>(stage * KPS + jj);
                    tmem_st1(lane_base + col + static_cast<uint32_t>(quad), va[jj]);
                    tmem_st4(lane_base + col + 4u, vb[jj][0], vb[jj][1], vb[jj][2], vb[jj][3]);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(sm.full + stage));
                if (++stage == stages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
            // this unit's staged scales are consumed (their values are in
            // TMEM): the producer may refill the buffer
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(sm.sempty + sb));
        }
    } else if (WF == 1) {
        // ------------------------------------------------ MXFP4 converters
        // Two teams of 8 warps take alternate ring slots (team = parity of
        // the slot use g): a team converts the slot's (up to) 4 k-blocks into
        // A slot g % astages in TMEM, then each warp arrives once on its
        // barrier.  Barrier waits cost tens of nanoseconds even when ready,
        // so they are taken once per slot, not per k-block.  No wait runs
        // two phases early (a parity wait would then pass at once):
        //  - code slot of use g: the team has converted g-2, so the producer,
        //    which loads in use order, has loaded every use up to g-2, which
        //    includes g - stages (stages >= 2);
        //  - A slot of use g: the team has waited for the MMAs of g-2-astages.
        //    MMAs complete in order only per issuer, so with two issuers
        //    astages is even: all uses of one A slot then belong to one team
        //    and one issuer, and g - 2 x astages <= g-2-astages is complete.
        //    The issuer at use g has consumed g-2 (two issuers; g-1 with
        //    one), so this team (or the other one, converting in order) has
        //    converted g - astages.
        // Arrivals for use g come only after the MMAs of use g-astages, i.e.
        // after that phase was consumed.
        // A warp may touch only its own TMEM lane quadrant (warp % 4), so
        // the warp's rows are that quadrant's 32 rows.
        const int cw_idx = warp - 6;              // 0..15
        const int team = cw_idx >> 3;
        const int half = (cw_idx >> 2) & 1;       // K 32*half .. 32*half+31 of each k-block
        const int quad = warp & 3;
        const int r = quad * 32 + lane;           // weight row within the tile
        const uint32_t a_tm_row = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + a_col0 +
                                  16u * static_cast<uint32_t>(half);
        const uint32_t swz = static_cast<uint32_t>(r & 7);
        int sbase = 0;                            // ring use of the unit's first slot
        int local = 0;
        // ring positions of use `cur`, advanced (not divided: a division by
        // the runtime ring sizes costs dozens of instructions) to each use
        int cur = 0, stage = 0, aslot = 0;
        uint32_t phase = 0, aphase = 0;
        bool ok = true;
        for (int u = cta0; u < num_units && ok; u += ncta) {
            const Unit un = unit_of(u, p, n_st);
            const int4 t = p.tiles[un.tile];
            if (!tile_ok(t, p)) continue;
            const int sb = local & 1;
            const uint32_t sph = static_cast<uint32_t>(local >> 1) & 1u;
            ++local;
            if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(sm.sfull + sb), sph, flags))) {
                raise_abort(flags, p.status, MOE_DEV_WAIT_TIMEOUT);
                break;
            }
            const uint8_t* srow = sm.scales + sb * scale_buf_bytes + r * p.kscale;
            // rows past the matrix: codes are TMA zero-fill and no scale bytes
            // were copied for them; use scale 1 so they stay exactly zero
            const bool row_ok = un.mb * kWeightTileRows + r < p.w_rows;
            const int nsl = un.st_hi - un.st_lo;      // ring slots of this unit
            for (int i = (team ^ sbase) & 1; i < nsl; i += 2) {
                const int st = un.st_lo + i;
                for (const int use = sbase + i; cur < use; ++cur) {
                    if (++stage == stages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                    if (++aslot == astages) {
                        aslot = 0;
                        aphase ^= 1u;
                    }
                }
                // the outcome is made warp-uniform: the lanes must not split
                // before the warp's single arrival below
                const bool got = mbar_wait(smem_u32(sm.full + stage), phase, flags) &&
                                 mbar_wait(smem_u32(sm.aempty + aslot), aphase ^ 1u, flags);
                if (!__all_sync(0xffffffffu, got)) {
                    raise_abort(flags, p.status, MOE_DEV_WAIT_TIMEOUT);
                    ok = false;
                    break;
                }
                const int nk = min(KPS, p.k_blocks - st * KPS);
                const uint8_t* crow = sm.codes + static_cast<size_t>(stage) * kCodeStageBytes + r * 128;
                const uint32_t a_tm = a_tm_row + kASlotCols * static_cast<uint32_t>(aslot);
                // k-block jj of the slot: codes = 16-byte unit jj * 2 + half of the
                // row (128-byte swizzled), its E8M0 byte; the bf16 values go to
                // row r, columns 32*jj + 16*half .. +15 of the A slot (word c of
                // the 16 bytes = K 8c..8c+7 = columns 4c..4c+3)
                // k-block jj: E2M1 codes to bf16 times 2^(s-127), stored to TMEM.
                // kTwo: the bf16 scale factor needs two multiplies (s > 128).
                const auto convert_store = [&](auto two_tag, int jj, const uint4 cw, uint32_t sbyte) {
                    constexpr bool kTwo = decltype(two_tag)::value;
                    uint32_t f1, f2;
                    if (kTwo) {
                        e8m0_factors(sbyte, f1, f2);
                    } else {
                        const uint32_t h = (sbyte + 126u) << 7;     // 2^(s-1), s <= 128
                        f1 = h | (h << 16);
                        f2 = 0x3F803F80u;
                    }
                    const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
                    uint32_t v[16];
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const uint4 q = e2m1x8_to_bf16<kTwo>(words[c], f1, f2);
                        v[4 * c] = q.x; v[4 * c + 1] = q.y; v[4 * c + 2] = q.z; v[4 * c + 3] = q.w;
                    }
                    tmem_st16(a_tm + 32u * static_cast<uint32_t>(jj), v);
                };
                const auto code_of = [&](int jj) {
                    return *reinterpret_cast<const uint4*>(
                        crow + ((static_cast<uint32_t>(jj * 2 + half) ^ swz) << 4));
                };
                const auto scale_of = [&](int jj) {
                    return row_ok ? static_cast<uint32_t>(srow[2 * (st * KPS + jj) + half]) : 127u;
                };
                // every load first, then the expansions; whether any lane of
                // the warp needs the second scale factor is decided once per
                // slot (a per-lane, per-k-block choice cost ~17 instructions
                // per k-block)
                uint4 cw[KPS];
                uint32_t sb[KPS];
                bool big = false;
#pragma unroll
                for (int jj = 0; jj < KPS; ++jj) {
                    if (jj < nk) {
                        cw[jj] = code_of(jj);
                        sb[jj] = scale_of(jj);
                        big |= p.mx_f16 ? (sb[jj] < kF16ScaleLo || sb[jj] > kF16ScaleHi)
                                        : sb[jj] > 128u;
                    }
                }
                if (p.mx_f16) {
                    // f16 operands: each byte of codes is two f16 values by
                    // the hardware conversion, times 2^(s-127) in f16 (one
                    // multiply per pair, exact for scale bytes in
                    // [kF16ScaleLo, kF16ScaleHi]); a scale outside that
                    // range is clamped into it and reported
                    if (__any_sync(0xffffffffu, big) && lane == 0)
                        atomicOr(p.status + kStatusWord, MOE_DEV_RANGE);
#pragma unroll
                    for (int jj = 0; jj < KPS; ++jj) {
                        if (jj >= nk) break;
                        const uint32_t sc = min(max(sb[jj], kF16ScaleLo), kF16ScaleHi);
                        const __half2 f = f16_pow2_x2(static_cast<int>(sc) - 127);
                        const uint32_t words[4] = {cw[jj].x, cw[jj].y, cw[jj].z, cw[jj].w};
                        uint32_t v[16];
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            const uint4 q = e2m1x8_to_f16x8(words[c]);
                            const uint32_t qq[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const __half2 m =
                                    __hmul2(*reinterpret_cast<const __half2*>(&qq[e]), f);
                                v[4 * c + e] = *reinterpret_cast<const uint32_t*>(&m);
                            }
                        }
                        tmem_st16(a_tm + 32u * static_cast<uint32_t>(jj), v);
                    }
                } else if (__any_sync(0xffffffffu, big)) {
#pragma unroll
                    for (int jj = 0; jj < KPS; ++jj)
                        if (jj < nk) convert_store(std::true_type{}, jj, cw[jj], sb[jj]);
                } else {
#pragma unroll
                    for (int jj = 0; jj < KPS; ++jj)
                        if (jj < nk) convert_store(std::false_type{}, jj, cw[jj], sb[jj]);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(sm.afull + aslot));
            }
            if (!ok) break;
            sbase += nsl;
            mbar_arrive(smem_u32(sm.sempty + sb));
        }
    }

    tc_fence_before();
    __syncthreads();
    // pair: the even CTA's MMAs have drained (into both CTAs' TMEM) and the
    // odd CTA's arrivals on its barriers have landed before either CTA frees
    // TMEM or exits
    if (kPair) cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<CG>(tmem_base, static_cast<uint32_t>(p.tmem_cols));
    }
    if (threadIdx.x == 0) MOE_TRACE_POINT(g_trace_gemm, EPI, blockIdx.x, 7);
}

template <int EPI, int WF, int CG>
cudaError_t launch_gemm_t(const GemmParams& p, const CUtensorMap* tmap_w, const CUtensorMap* tmap_x,
                          int grid, size_t smem, cudaStream_t s, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreadsOf<WF>);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (CG == 2) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = 2;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attr;
    cudaError_t err = cudaFuncSetAttribute(grouped_gemm_kernel<EPI, WF, CG>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    if (CG == 2) {
        // A persistent grid of pairs: no more pairs than fit at once (the
        // SMs of a GPU partition may not all pair up), and an even count.
        cfg.numAttrs = na;
        cfg.gridDim = dim3(2);
        int clusters = 0;
        err = cudaOccupancyMaxActiveClusters(&clusters, grouped_gemm_kernel<EPI, WF, CG>, &cfg);
        if (err != cudaSuccess) return err;
        if (clusters < 1) return cudaErrorInvalidConfiguration;
        grid &= ~1;
        if (grid > 2 * clusters) grid = 2 * clusters;
        if (grid < 2) grid = 2;
    }
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.numAttrs = na;
    cfg.gridDim = dim3(grid);
    return cudaLaunchKernelEx(&cfg, grouped_gemm_kernel<EPI, WF, CG>, p, *tmap_w, *tmap_x);
}

}  // namespace

size_t trace_copy_gemm(unsigned long long* dst, size_t cap) {
    MOE_TRACE_COPY(g_trace_gemm, dst, cap);
}

cudaError_t launch_gemm(int epi, int wf, int cg, const GemmParams& p, const CUtensorMap* tmap_w,
                        const CUtensorMap* tmap_x, int grid, size_t smem, cudaStream_t s,
                        bool pdl) {
    if (p.stages < 2 || p.stages > kMaxStages) return cudaErrorInvalidValue;
    if (cg == 2) {
        if (wf == 1 || wf == 3) return cudaErrorInvalidValue;
        if (wf == 2)
            return epi == kEpiGlu
                       ? launch_gemm_t<kEpiGlu, 2, 2>(p, tmap_w, tmap_x, grid, smem, s, pdl)
                       : launch_gemm_t<kEpiCombine, 2, 2>(p, tmap_w, tmap_x, grid, smem, s, pdl);
        return epi == kEpiGlu
                   ? launch_gemm_t<kEpiGlu, 0, 2>(p, tmap_w, tmap_x, grid, smem, s, pdl)
                   : launch_gemm_t<kEpiCombine, 0, 2>(p, tmap_w, tmap_x, grid, smem, s, pdl);
    }
    if (wf == 2)
        return epi == kEpiGlu
                   ? launch_gemm_t<kEpiGlu, 2, 1>(p, tmap_w, tmap_x, grid, smem, s, pdl)
                   : launch_gemm_t<kEpiCombine, 2, 1>(p, tmap_w, tmap_x, grid, smem, s, pdl);
    if (wf == 3)
        return epi == kEpiGlu
                   ? launch_gemm_t<kEpiGlu, 3, 1>(p, tmap_w, tmap_x, grid, smem, s, pdl)
                   : launch_gemm_t<kEpiCombine, 3, 1>(p, tmap_w, tmap_x, grid, smem, s, pdl);
    if (epi == kEpiGlu)
        return wf == 1 ? launch_gemm_t<kEpiGlu, 1, 1>(p, tmap_w, tmap_x, grid, smem, s, pdl)
                       : launch_gemm_t<kEpiGlu, 0, 1>(p, tmap_w, tmap_x, grid, smem, s, pdl);
    return wf == 1 ? launch_gemm_t<kEpiCombine, 1, 1>(p, tmap_w, tmap_x, grid, smem, s, pdl)
                   : launch_gemm_t<kEpiCombine, 0, 1>(p, tmap_w, tmap_x, grid, smem, s, pdl);
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
// Ordered combine: one thread per 4 output columns of a token; the token's
// slots are added in slot order (j = 0, 1, ...), starting from zero.
__global__ void combine_rows_kernel(const float* __restrict__ y_rows,
                                    const int32_t* __restrict__ assign_row,
                                    const int32_t* __restrict__ topk_ids, int T, int H, int k,
                                    int ex_lo, int ex_hi, float* __restrict__ out32,
                                    __nv_bfloat16* __restrict__ out16) {
    pdl_wait();
    const int h4 = H / 4;
    const size_t n = static_cast<size_t>(T) * h4;
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const int t = static_cast<int>(i / h4), c4 = static_cast<int>(i % h4);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < k; ++j) {
            const int a = t * k + j;
            const int e = __ldg(topk_ids + a), row = __ldg(assign_row + a);
            if (row < 0 || e < ex_lo || e >= ex_hi) continue;
#ifdef MOE_DEBUG_BOUNDS
            if (row >= T * k) continue;    // (no status word here: skip only)
#endif
            const float4 y = __ldcg(reinterpret_cast<const float4*>(
                                        y_rows + static_cast<size_t>(row) * H) + c4);
            acc.x += y.x;
            acc.y += y.y;
            acc.z += y.z;
            acc.w += y.w;
        }
        if (out16) {
            __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
            __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
            uint2 pk;
            pk.x = *reinterpret_cast<uint32_t*>(&lo);
            pk.y = *reinterpret_cast<uint32_t*>(&hi);
            reinterpret_cast<uint2*>(out16)[i] = pk;
        } else {
            reinterpret_cast<float4*>(out32)[i] = acc;
        }
    }
}
}  // namespace

cudaError_t launch_combine_rows(const float* y_rows, const int32_t* assign_row,
                                const int32_t* topk_ids, int T, int H, int k, int ex_lo,
                                int ex_hi, float* out32, __nv_bfloat16* out16, cudaStream_t s,
                                bool pdl) {
    cudaLaunchConfig_t cfg = {};
    const size_t n = static_cast<size_t>(T) * (H / 4);
    size_t blocks = (n + 255) / 256;
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
    return cudaLaunchKernelEx(&cfg, combine_rows_kernel, y_rows, assign_row, topk_ids, T, H, k,
                              ex_lo, ex_hi, out32, out16);
}

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
