// Internal declarations shared by the kernels and the C-ABI host code:
// workspace layout, kernel parameter blocks and launch helpers.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace moe {

constexpr int kRouterTokens = 32;      // tokens per router / permutation block
constexpr int kMaxExperts = 256;
constexpr int kMaxTopK = 8;
constexpr int kBlockK = 64;            // K elements per pipeline stage (128 B of bf16)
constexpr int kBlockKFp8 = 128;        // E4M3: K elements per stage (128 B)
constexpr float kFp8HScale = 0.125f;   // FP8 h codes = e4m3(h / kFp8HScale)
constexpr int kWeightTileRows = 128;   // MMA M: weight rows per tile
constexpr int kMaxTokenTile = 256;     // MMA N upper bound

// Status region: word 0 is the device status word (MOE_DEV_* bits),
// word 1 the number of GEMM token tiles written by the router kernel,
// word 2 the router's grid-completion counter (zero between calls).
constexpr int kStatusWord = 0;
constexpr int kNumTilesWord = 1;
constexpr int kGridCounterWord = 2;
// Stage checks (MOE_CHECK_STAGES=1): per stage s, the non-finite count at
// word kStageStatsWord + 2 s and the largest finite magnitude (fp32 bits,
// ordered as integers) at word kStageStatsWord + 2 s + 1.
constexpr int kStageStatsWord = 16;
constexpr int kNumStages = 3;

// MOE_DEBUG_BOUNDS builds check the index of every store of the layer's
// kernels against its buffer and skip a store that fails, reporting
// MOE_DEV_BOUNDS; other builds compile the checks away.
#ifdef MOE_DEBUG_BOUNDS
__device__ __forceinline__ bool bounds_ok(bool ok, int32_t* status) {
    if (!ok) atomicOr(status, 0x10);
    return ok;
}
#define MOE_BOUNDS(cond, status) ::moe::bounds_ok((cond), (status))
#else
#define MOE_BOUNDS(cond, status) true
#endif

// Router ticket counters live at a fixed offset, right after the status
// region, with one slot for every (token block, expert group) pair that can
// use a K split (fewer than 304 pairs) and one per token block (T <= 2^20):
// the same slots for every shape, so a workspace reused for another shape
// still finds them at zero (every call leaves them at zero).
constexpr int kPairSlots = 304;
constexpr int kMaxTokenBlocks = (1 << 20) / 32;

// GEMM K split for small batches.  When the work units (token tiles x
// 128-row weight blocks) cannot fill two waves of GB300's 152 SMs, each
// unit's ring slots are cut into up to kMaxKSplit contiguous parts handled
// by different CTAs (each part at least 2 slots, none empty); the part count
// minimises the persistent grid's makespan, ceil(units * parts / SMs) waves
// of ceil(slots / parts) slots.  The down
// projection adds the parts through its fp32 atomics; gate_up parts store
// fp32 partial tiles and the last part to arrive (a ticket per unit) adds
// them in part order before the bias and the GLU.  The split depends on the
// shape only, and at most kSplitTargetUnits tickets exist, so they too live
// in the fixed counter region.
constexpr int kSplitTargetUnits = 304;
constexpr int kMaxKSplit = 8;
constexpr int kSplitPartsAlloc = 4;    // partial-tile region: parts at R* rows
inline bool gemm_may_split(long long max_units, int n_slots) {
    return max_units > 0 && max_units < kSplitTargetUnits && n_slots >= 4;
}
inline int gemm_ksplit(long long max_units, int n_slots, int sms) {
    if (!gemm_may_split(max_units, n_slots) || sms < 1) return 1;
    int best = 1;
    long long best_cost = ((max_units + sms - 1) / sms) * n_slots;
    for (int ks = 2; ks <= kMaxKSplit && ks <= n_slots / 2; ++ks) {
        const int per = (n_slots + ks - 1) / ks;
        const int parts = (n_slots + per - 1) / per;      // no empty part
        const long long cost = ((max_units * parts + sms - 1) / sms) * per;
        if (cost < best_cost) {
            best_cost = cost;
            best = parts;
        }
    }
    return best;
}
// Upper bound of the token tiles of a call (every tile holds >= 1 row).
inline long long max_token_tiles(long long R, int max_tiles) {
    return R < max_tiles ? R : max_tiles;
}

constexpr size_t kCounterBytes =
    static_cast<size_t>(kPairSlots + kMaxTokenBlocks + kSplitTargetUnits + kMaxExperts) * 4;
// GEMM split tickets: counters + kSplitTicketOffset (ints)
constexpr int kSplitTicketOffset = kPairSlots + kMaxTokenBlocks;
// Per-expert assignment totals, summed by the router's token blocks and
// read (then zeroed) by the last one: counters + kExpertTotalsOffset (ints)
constexpr int kExpertTotalsOffset = kPairSlots + kMaxTokenBlocks + kSplitTargetUnits;

// K slices of the router: the hidden dimension is cut into `ksplit` slices
// handled by separate CTAs when there are few (token block, expert group)
// pairs, so that a small batch still spreads its loads over ~2 CTAs per SM,
// but never so many that the grid needs a second wave (two router CTAs fit
// on an SM; sized for GB300's 152 SMs; each slice keeps at least 4 chunks of
// 64).  Measured at T = 4096: 3 slices (384 CTAs) left the last CTAs
// starting 8 us after the first.
// The slices of one pair form a thread-block cluster (at most the portable
// 8 CTAs), which adds their partial logits through distributed shared memory.
constexpr int kMaxRouterSlices = 8;
inline int router_ksplit(int pairs, int nchunks) {
    if (pairs < 1 || nchunks < 1) return 1;
    int ks = 304 / pairs;                            // one wave of 2 CTAs per SM
    if (ks > kMaxRouterSlices) ks = kMaxRouterSlices;
    const int cap = nchunks / 4 > 1 ? nchunks / 4 : 1;
    if (ks > cap) ks = cap;
    if (ks < 1) ks = 1;
    const int per = (nchunks + ks - 1) / ks;       // chunks per slice
    return (nchunks + per - 1) / per;              // no empty slice
}

// MXFP4 weights x MXFP8 activations: token operands hold K padded to a
// multiple of 128.  When K = 128 m + 64, the last 128-wide k-block holds 64
// zero codes, then the last 64 elements: the weights' last k-block is read
// through an overlapping chunk view that starts 64 elements early, so its
// first half (already counted) meets the zeros.
__host__ __device__ inline int mx_padded_k(int K) { return (K + 127) / 128 * 128; }
// position of element k of a row in that padded layout (tail0 = K rounded
// down to 128 when K % 128 == 64, else K)
__host__ __device__ inline int mx_tail0(int K) { return K % 128 ? K / 128 * 128 : K; }
__host__ __device__ inline int mx_pos(int k, int tail0) { return k < tail0 ? k : k + 64; }
// bytes of one token row's UE8M0 scales (mx_padded_k(K) / 32, padded to 16
// so that a tile's rows are one 16-byte-aligned bulk copy)
__host__ __device__ inline int mx_scale_row_bytes(int K) {
    return (mx_padded_k(K) / 32 + 15) / 16 * 16;
}

struct WsLayout {
    size_t status, topk_ids, topk_w, blk_cnt, logits, partials, counters, offsets, gemm_partial;
    size_t sorted_assign, assign_row, tiles, x_perm, x_scale, h, out_acc, y_rows, total;
    size_t gemm_partial_bytes;
    int max_tiles;
};

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// deterministic: room for the per-slot output rows of the ordered combine
// (fp32 [T*k, H], after every other region so that the others keep their
// offsets whatever the mode).
inline WsLayout ws_layout(long long T, int H, int I, int E, int k, bool deterministic = false) {
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
    L.counters = take(kCounterBytes);
    L.topk_ids = take(R * 4);
    L.topk_w = take(R * 4);
    L.blk_cnt = take(nb * E * 4);
    const size_t eg = (static_cast<size_t>(E) + 31) / 32;
    const int ks = router_ksplit(static_cast<int>(nb * eg), H / kBlockK);
    L.logits = take(eg > 1 ? nb * kRouterTokens * E * 4 : 0);
    (void)ks;                              // (slices merge in shared memory)
    L.partials = take(0);
    L.offsets = take((E + 1) * 4);
    L.sorted_assign = take(R * 4);
    L.assign_row = take(R * 4);
    L.tiles = take(static_cast<size_t>(L.max_tiles) * 16);
    L.x_perm = take(R * H * 2);            // bf16, or E4M3 codes (FP8)
    // FP8: fp32 scale of each routed row; MXFP4 x MXFP8: UE8M0 block scales
    // [T*k][mx_padded_k(H) / 32]
    L.x_scale = take(R * (mx_scale_row_bytes(H) > 4 ? mx_scale_row_bytes(H) : 4));
    L.h = take(R * I * 2);
    L.out_acc = take(static_cast<size_t>(T) * H * 4);
    // gate_up K-split partial tiles, fp32 [part][weight block][routed row][128].
    // A call splits only while its unit bound
    // (token tiles x weight blocks) is below kSplitTargetUnits, which holds
    // for R up to some R* (the tile bound grows with R); the region holds
    // kSplitPartsAlloc parts of R* rows whatever T is (a call with R rows may
    // use as many parts as fit), so a workspace sized for one call of a layer
    // shape serves every other T of that shape.
    {
        const int nwb = (2 * I + kWeightTileRows - 1) / kWeightTileRows;
        const int slots_bf16 = H / kBlockK, slots_mx = (H / kBlockK + 3) / 4;
        long long rstar = 0;
        // (units grow by >= nwb per 16 rows, so the loop ends before 16 x 304 rows)
        for (long long r = 1;; ++r) {
            const long long mt = r / 16 + (r < E ? r : E) + 1;
            const long long units = max_token_tiles(r, static_cast<int>(mt)) * nwb;
            if (!gemm_may_split(units, slots_bf16) && !gemm_may_split(units, slots_mx)) break;
            rstar = r;
        }
        L.gemm_partial_bytes = static_cast<size_t>(kSplitPartsAlloc) * nwb * rstar * kWeightTileRows * 4;
        L.gemm_partial = take(L.gemm_partial_bytes);
    }
    L.y_rows = take(deterministic ? R * H * 4 : 0);
    L.total = o;
    return L;
}

// ------------------------------------------------------------ router (K1)

struct RouterParams {
    const __nv_bfloat16* br;     // [E]
    int T, H, E, top_k;
    int nblocks;                 // grid = (token blocks of 32, expert groups of 32,
    int egroups;                 //         K slices)
    int ksplit;
    int stages;                  // TMA ring depth
    float* logits;               // [nblocks, 32, E] when egroups > 1
    int32_t* counters;           // fixed counter region, zero between calls
    int32_t* topk_ids;           // [T, k]
    float* topk_w;               // [T, k]
    int32_t* blk_cnt;            // [E, nblocks]: assignments per expert and token block
    int32_t* offsets;            // [E+1]
    int4* tiles;                 // GEMM token tiles (expert, first row, rows, 0)
    int max_tiles;
    int token_tile;              // rows of tokens per GEMM tile
    // expert-parallel form: GEMM tiles only for experts [ex_lo, ex_lo + ex_n),
    // numbered from 0 (the local weight banks); 0, E for the whole layer
    int ex_lo, ex_n;
    int inject;                  // test faults: 1 = token 0's first id set to E
                                 // after counting, 2 = tile 0 names expert ex_n
    // small batches (T * top_k <= kSmallPermRows): the last CTA also writes
    // the stable permutation (no permutation kernel)
    int small_perm;
    int32_t* sorted_assign;      // [T*k] (small_perm)
    int32_t* assign_row;         // [T*k] (small_perm)
    int32_t* status;             // status region (status word, tile count, counter)
};
// Largest T * top_k whose permutation the router's last CTA makes itself,
// and the largest T of that path (measured on gpt-oss-20b: 5-10 us faster
// at T = 16 and 32, 6.4 us faster at T = 48, 4 us slower at T = 64, where
// gate_up cannot load weights before the router, its immediate
// predecessor, has finished).
constexpr int kSmallPermRows = 256;
constexpr int kSmallPathMaxT = 48;

// ------------------------------------------------------------ permutation (K2)

struct PermuteParams {
    const int32_t* topk_ids;     // [T, k]
    const int32_t* blk_cnt;      // [E, nblocks] assignments per expert and token block
    const int32_t* offsets;      // [E+1]
    const __nv_bfloat16* x;      // [T, H]
    int T, H, E, top_k, nblocks;
    int gather_split;            // CTAs per 32-token block (grid.y)
    float* zero_out;             // [T, H] fp32 rows to clear, or null
    int32_t* sorted_assign;      // [T*k]
    int32_t* assign_row;         // [T*k]
    __nv_bfloat16* x_perm;       // [T*k, H] or null (no gather)
    int mx_layout;               // MXFP4 operand layout: chunk-major
                                 // [H/64][T*k][64], each group of 8 columns
                                 // in the order 0,4,1,5,2,6,3,7
    int fp8;                     // FP8 W8A8: x_perm holds E4M3 codes [T*k, H]
    float* x_scale;              // FP8: [T*k] scale of each routed row's codes
    int ex_lo, ex_hi;            // gather only the rows of experts [ex_lo, ex_hi)
    int mx_f16;                  // with mx_layout: f16 values in natural order
                                 // (values beyond +-65504 reported, saturated)
    int mx8;                     // MXFP8 activations: x_perm holds E4M3 codes
                                 // [T*k, mx_padded_k(H)] and x_scale UE8M0
                                 // bytes [T*k, mx_padded_k(H) / 32]
    int32_t* status;
};

// ------------------------------------------------------------ grouped GEMM

enum EpilogueKind { kEpiGlu = 0, kEpiCombine = 1 };

struct GemmParams {
    const int4* tiles;           // token tiles from the permutation kernel
    const int32_t* num_tiles;    // device count of tiles
    int n_wblocks;               // weight-row blocks per expert (128 rows; CTA pairs: 256)
    int k_blocks;                // K / 64
    int w_rows;                  // weight rows per expert (2I or H)
    int token_box;               // token rows per TMA box (= MMA N bound)
    int stages;                  // ring of W (bf16) or code (MXFP4) + token tiles
    int astages;                 // MXFP4: ring of converted bf16 W tiles
    int n_iss;                   // MMA issuers (1; MXFP4 tiles up to 64 rows: 2)
    int tmem_cols;               // allocated TMEM columns (2 accumulators)
    int num_experts;             // E (tile bounds check)
    int rows_total;              // T * k (tile bounds check)
    const uint8_t* scales;       // MXFP4: E8M0 [E, w_rows, kscale]
    int kscale;                  // MXFP4: scale bytes per weight row (K / 32)
    const __nv_bfloat16* bias;   // [E, w_rows]
    // kEpiGlu: h[row, w_rows/2] bf16
    __nv_bfloat16* h;
    // FP8 W8A8 (WF = 2): per-expert weight scales [E]; gate_up: the scale of
    // each routed row's activation codes [T*k] and h written as E4M3 codes
    // [T*k, w_rows/2] (scale kFp8HScale); down: the scale of the h codes
    const float* wscale;
    const float* xscale;
    uint8_t* h8;
    float hscale;
    // MXFP4 x MXFP8 (WF = 3): weights through the chunk view (the last
    // chunk index is mx_cmax = K/64 - 2); token operand scales UE8M0
    // [rows_total, xs_row_bytes] (null: every block scale 2^-3, the h
    // operand); gate_up stores h codes [T*k, h_pad] (positions mx_pos)
    int mx_cmax;
    const uint8_t* xs_mx;
    int xs_row_bytes;
    int h_pad;
    int h_tail0;
    // kEpiCombine: out[t, w_rows] += w * y (fp32 atomics), or, when y_rows
    // is set (deterministic combine), y_rows[routed row, w_rows] = w * y
    float* out;
    float* y_rows;
    const int32_t* sorted_assign;
    const float* topk_w;
    int top_k;
    int32_t* status;
    // K split (small batches): parts per unit; gate_up partial tiles
    // [part][weight block][routed row][128] fp32 and per-unit tickets
    // (ksplit > 1 only)
    int ksplit;
    float* partial;
    int32_t* tickets;
    // test fault: the MMA issuer first waits on a barrier that nothing
    // arrives on (the wait gives up after its bound and the kernel aborts)
    int inject_stall;
    // small batches, bf16 gate_up: token rows come straight from the layer
    // input (row = sorted_assign[tile row] / top_k), gathered by the kernel
    // (null: the token operand is read through tmap_x); zero_out[0, n_zero)
    // fp32 is cleared first (the output the down projection accumulates
    // into); prewait = 0: the tile list comes from the immediately preceding
    // kernel, so no load may start before the dependency wait
    // MXFP4 (WF = 1) f16 mode: the token operands hold f16 in natural K
    // order and the converters expand E2M1 to f16 (else bf16, with the
    // 0,4,1,5,2,6,3,7 order within groups of 8)
    int mx_f16;
    const __nv_bfloat16* gather_x;
    int gather_K;                // elements per row of gather_x
    float* zero_out;
    size_t n_zero;
    int prewait;
};

// Shared memory of one GEMM pipeline stage and of the fixed part (bytes,
// excluding the 1 KB alignment slack).  wf: 0 = bf16, 1 = MXFP4.  An MXFP4
// stage holds kMxfp4KbPerStage k-blocks (codes [128 x 128 B] + that many
// 64-wide token chunks); its converted weights take an A slot of 128 TMEM
// columns after the two accumulators -- up to kMxfp4AStages slots, as many
// as fit in 512 columns and, with two MMA issuers, an even count (2 for every
// token tile up to 128 rows) -- and token tiles are at most
// kMxfp4MaxTokenTile rows.
constexpr int kMxfp4AStages = 3;
constexpr int kMxfp4MaxTokenTile = 128;
constexpr int kMxfp4KbPerStage = 4;     // k-blocks of 64 per MXFP4 ring slot
constexpr int kMxKbPerStage = 2;        // k-blocks of 128 per MXFP4 x MXFP8 ring slot
inline size_t gemm_stage_bytes(int token_box, int wf) {
    size_t a = static_cast<size_t>(kWeightTileRows) * kBlockK * 2;
    size_t b = static_cast<size_t>(token_box) * kBlockK * 2;
    size_t codes = static_cast<size_t>(kWeightTileRows) * kBlockK / 2;
    // FP8: one 128-wide k-block of byte codes, the same bytes; MXFP4 x
    // MXFP8: kMxKbPerStage of them (the codes padded to a byte each)
    return wf == 1 ? kMxfp4KbPerStage * (codes + b) : wf == 3 ? kMxKbPerStage * (a + b) : a + b;
}
inline size_t gemm_fixed_bytes(int token_box, int wf, int kscale, int xs_row_bytes = 0) {
    // MXFP4 and MXFP4 x MXFP8: each unit's weight scale rows, double-buffered;
    // MXFP4 x MXFP8 also the token tile's scale rows
    size_t scales = (wf == 1 || wf == 3)
                        ? 2 * align_up(static_cast<size_t>(kWeightTileRows) * kscale, 16) : 0;
    if (wf == 3) scales += 2 * static_cast<size_t>(token_box) * xs_row_bytes;
    size_t meta = static_cast<size_t>(token_box) * 8;
    size_t bars = 768;
    return scales + meta + bars;
}

// Kernel launchers (defined next to each kernel).
// Router: x [T, H] and Wr [E, H] through 2-D tensor maps (box 64 x 32,
// 128-byte swizzle); each CTA covers 32 tokens x 32 experts.
size_t router_stage_bytes();
size_t router_smem_bytes(int stages);
int router_max_stages();
int router_stage_multiple();
cudaError_t launch_router(const RouterParams& p, const CUtensorMap* tmap_x,
                          const CUtensorMap* tmap_wr, size_t smem, cudaStream_t s, bool pdl);
// Tiny batches (T <= 8, the small-batch path): one CTA routes everything.
bool router_tiny_fits(int T, int H, int E);
int router_tiny_tokens_per_cta(int T, int H, int E);
cudaError_t launch_router_tiny(const RouterParams& p, const void* x, const void* wr,
                               cudaStream_t s, bool pdl);
cudaError_t launch_permute(const PermuteParams& p, cudaStream_t s, bool pdl);
// cg = 2 (bf16 only): CTA pairs (clusters of 2) on 256-row weight blocks,
// each CTA holding token_box / 2 rows of every token tile; `grid` counts CTAs.
cudaError_t launch_gemm(int epi, int wf, int cg, const GemmParams& p, const CUtensorMap* tmap_w,
                        const CUtensorMap* tmap_x, int grid, size_t smem,
                        cudaStream_t s, bool pdl);
// "attn_tc" tuning switch of the attention step (0 automatic, 1 never, 2
// always the tcgen05 kernel); returns a moe_status value.
int set_attn_tc_mode(int mode);
int set_attn_poll(int mode);
// cuTensorMapEncodeTiled from the driver (looked up once); null if absent.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// Stage check: counts the non-finite elements of buf (n elements of type
// dtype: 0 = bf16, 1 = fp32, 2 = E4M3 codes, 3 = f16) and their largest finite
// magnitude into the stage's status words.
cudaError_t launch_stage_check(const void* buf, size_t n, int dtype, int stage, int32_t* status,
                               cudaStream_t s);
// moe_forward_noalloc's test switch (moe_set_tuning "noalloc_poison").
void set_noalloc_poison(int on);
// Deterministic combine: out[t] = sum over j in order of y_rows[assign_row[t*k + j]]
// for the slots whose expert lies in [ex_lo, ex_hi); fp32 out32 or bf16 out16.
cudaError_t launch_combine_rows(const float* y_rows, const int32_t* assign_row,
                                const int32_t* topk_ids, int T, int H, int k, int ex_lo,
                                int ex_hi, float* out32, __nv_bfloat16* out16, cudaStream_t s,
                                bool pdl);
cudaError_t launch_to_bf16(const float* in, __nv_bfloat16* out, size_t n, cudaStream_t s,
                           bool pdl);

}  // namespace moe
