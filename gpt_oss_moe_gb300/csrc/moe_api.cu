// C ABI of the library (include/moe.h): argument validation on the host,
// workspace layout, TMA tensor maps and the launch sequence
//   router+top-k -> permutation -> gate_up GEMM (+GLU) -> down GEMM (+combine)
//   [-> fp32->bf16 when a bf16 output is asked for]
// all on the caller's stream, with no host synchronisation (xserv
// docs/19-gpt-oss-moe.md, "Phase 19: gpt-oss-20b", §2 "MoE 前向").
#include <cudaTypedefs.h>
#include <nvtx3/nvToolsExt.h>

#include <atomic>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "moe_internal.cuh"
#include "trace.cuh"
#include "../../include/moe.h"

namespace moe {
namespace {

// ------------------------------------------------------------ device cache

struct DevInfo {
    int sms = 0;
    int max_smem = 0;
    bool ok = false;
};
constexpr int kMaxDevices = 64;
DevInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

moe_status device_info(DevInfo* out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_dev_mu);
    DevInfo& d = g_dev[dev];
    if (!d.ok) {
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
                cudaSuccess)
            return MOE_ERR_CUDA;
        int major = 0, minor = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (major != 10) return MOE_ERR_UNSUPPORTED;   // built for sm_103a only
        d.ok = true;
    }
    *out = d;
    return MOE_OK;
}

// ------------------------------------------------------------ tensor maps

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

moe_status encode_fn(PFN_cuTensorMapEncodeTiled_v12000* fn) {
    std::call_once(g_encode_once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    if (!g_encode) return MOE_ERR_CUDA;
    *fn = g_encode;
    return MOE_OK;
}

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    return encode_fn(&fn) == MOE_OK ? fn : nullptr;
}

namespace {

// Every map uses the 128-byte swizzle: box inner extent 128 B (64 bf16
// elements, or 128 MXFP4 code bytes = 4 k-blocks of one row).
moe_status make_tmap_dt(CUtensorMap* m, CUtensorMapDataType dt, const void* base, int rank,
                        const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box) {
    PFN_cuTensorMapEncodeTiled_v12000 enc;
    moe_status st = encode_fn(&enc);
    if (st != MOE_OK) return st;
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(m, dt, static_cast<cuuint32_t>(rank), const_cast<void*>(base), dims, strides, box,
                     estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_CUDA;
}

moe_status make_tmap(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
                     const cuuint64_t* strides, const cuuint32_t* box, bool bytes = false) {
    return make_tmap_dt(m, bytes ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                        base, rank, dims, strides, box);
}

// MXFP4 codes [E, rows, K/2] for the block-scaled MMA: a 4-D view (element
// in chunk, chunk, row, expert) whose chunks of 128 E2M1 codes start every
// 64 elements (stride 32 B, overlapping), so that the K range's last 128
// codes form a chunk even when K = 128 m + 64.  The 4-bit type with 16-byte
// alignment makes TMA spread every 8 bytes of codes over 16 bytes of shared
// memory, the form the MMA reads; box 128 codes x 1 chunk x 128 rows.
moe_status mx_weight_tmap(CUtensorMap* m, const void* w, int E, int rows, int K) {
    const cuuint64_t row_bytes = static_cast<cuuint64_t>(K) / 2;
    const cuuint64_t dims[4] = {128, static_cast<cuuint64_t>(K / 64 - 1),
                                static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(E)};
    const cuuint64_t str[3] = {32, row_bytes, row_bytes * static_cast<cuuint64_t>(rows)};
    const cuuint32_t boxd[4] = {128u, 1u, 128u, 1u};
    return make_tmap_dt(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, w, 4, dims, str, boxd);
}

// 3-D map over one expert weight bank [E, rows, K]: bf16 values (box 64 K
// elements x 128 rows x 1 expert) or MXFP4 codes (K/2 bytes per row; box
// 128 bytes = kMxfp4KbPerStage k-blocks x 128 rows x 1 expert).
moe_status weight_tmap(CUtensorMap* m, const void* w, int E, int rows, int K, bool mxfp4,
                       bool fp8 = false) {
    if (fp8) {
        // E4M3 codes [E, rows, K], one byte each: box 128 K x 128 rows
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows),
                                    static_cast<cuuint64_t>(E)};
        const cuuint64_t str[2] = {static_cast<cuuint64_t>(K),
                                   static_cast<cuuint64_t>(K) * static_cast<cuuint64_t>(rows)};
        const cuuint32_t boxd[3] = {static_cast<cuuint32_t>(kBlockKFp8), 128u, 1u};
        return make_tmap(m, w, 3, dims, str, boxd, true);
    }
    const cuuint64_t row_bytes = mxfp4 ? static_cast<cuuint64_t>(K) / 2
                                       : static_cast<cuuint64_t>(K) * 2;
    const cuuint64_t dims[3] = {mxfp4 ? static_cast<cuuint64_t>(K) / 2 : static_cast<cuuint64_t>(K),
                                static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(E)};
    const cuuint64_t str[2] = {row_bytes, row_bytes * static_cast<cuuint64_t>(rows)};
    const cuuint32_t boxd[3] = {mxfp4 ? kMxfp4KbPerStage * 32u : 64u, 128u, 1u};
    return make_tmap(m, w, 3, dims, str, boxd, mxfp4);
}

// ------------------------------------------------------------ tuning

std::atomic<int> g_token_tile{0};
std::atomic<int> g_ksplit_mode{0};  // 0: automatic, 1: never split, n >= 2: n parts
std::atomic<int> g_pdl{1};
std::atomic<int> g_pair_mode{0};   // 0: automatic, 1: never, 2: always (bf16 and FP8 weights)
// 1: the combine adds each token's k expert outputs in slot order (bitwise
// reproducible); 0: fp32 atomics in the down projection's epilogue
std::atomic<int> g_deterministic{0};
// test faults (moe_set_tuning "inject"): 1 = a routed id out of range, 2 = a
// GEMM tile naming an expert out of range, 4 = a gate_up wait that runs out
std::atomic<int> g_inject{0};
// 1: small bf16 batches skip the permutation kernel (the router permutes,
// gate_up gathers token rows itself); 0: always the permutation kernel
std::atomic<int> g_small_path{1};
// 1: small-batch calls of at most 8 tokens route in one CTA (router_tiny)
std::atomic<int> g_tiny_router{1};
// 1: MXFP4 weights with bf16 activations run on f16 operands (hardware E2M1
// conversion; exact for scale bytes in [104, 140] and activations within
// +-65504, others reported as MOE_DEV_RANGE); 0: bf16 operands, exact for
// every scale
std::atomic<int> g_mxfp4_f16{1};
// bf16 token boxes from which the GEMMs run on CTA pairs (automatic mode):
// measured on gpt-oss-20b, pairs are 3 % slower at a 128-row box (T = 128),
// even at 256 (T = 256) and 2-5 % faster at T >= 512
constexpr int kPairMinBox = 256;
// FP8 layers (box 256) on gpt-oss-20b: pairs are 10-12 % faster while the
// mean routed rows per expert stay below 128 (T = 256, 512), even at 128
// (T = 1024) and 4 % slower at 512 (T = 4096).
constexpr long long kFp8PairMaxMeanRows = 128;

// ------------------------------------------------------------ profiling
//
// When enabled for C calls, each of the next C calls records one CUDA event
// before its first kernel and one after each kernel, on the call's stream.
// Reading waits for the last event and averages each kernel over the calls.

constexpr int kMaxProf = 8;          // kernels per call
constexpr int kMaxProfCalls = 8192;
struct Prof {
    int capacity = 0;                // calls to record (0 = off)
    int calls = 0;                   // calls recorded so far
    int created = 0;                 // events created (capacity * (kMaxProf + 1))
    cudaEvent_t* ev = nullptr;
    const char* names[kMaxProf];
    int n = 0;                       // kernels in the current call
    int n_first = 0;                 // kernels per call (from the first call)
};
Prof g_prof;
std::mutex g_prof_mu;

cudaEvent_t* prof_slot() {
    return g_prof.ev + static_cast<size_t>(g_prof.calls) * (kMaxProf + 1);
}
void prof_reset(cudaStream_t s) {
    g_prof.n = -1;
    if (g_prof.calls >= g_prof.capacity) return;
    g_prof.n = 0;
    cudaEventRecord(prof_slot()[0], s);
}
void prof_mark(const char* name, cudaStream_t s) {
    if (g_prof.n < 0 || g_prof.n >= kMaxProf) return;
    if (g_prof.calls == 0) g_prof.names[g_prof.n] = name;
    cudaEventRecord(prof_slot()[g_prof.n + 1], s);
    ++g_prof.n;
}
void prof_finish() {
    if (g_prof.n < 0) return;
    if (g_prof.calls == 0) g_prof.n_first = g_prof.n;
    if (g_prof.n == g_prof.n_first) ++g_prof.calls;   // calls of another shape are dropped
    g_prof.n = -1;
}

// ------------------------------------------------------------ NVTX
//
// With MOE_NVTX=1 in the environment (read once per process), every call
// opens an NVTX range ("moe_forward", ...) and every kernel launch a nested
// range named after the kernel, for timeline tools.  Off, the ranges cost a
// branch.

bool nvtx_on() {
    static const bool on = [] {
        const char* v = std::getenv("MOE_NVTX");
        return v != nullptr && v[0] == '1';
    }();
    return on;
}
struct NvtxRange {
    bool on;
    explicit NvtxRange(const char* name) : on(nvtx_on()) {
        if (on) nvtxRangePushA(name);
    }
    ~NvtxRange() {
        if (on) nvtxRangePop();
    }
};

// With MOE_CHECK_STAGES=1 (read once per process) every forward call
// checks each stage's output for NaN / infinity and its largest magnitude
// (stage_check.cu; read with moe_stage_stats).
bool stage_checks_on() {
    static const bool on = [] {
        const char* v = std::getenv("MOE_CHECK_STAGES");
        return v != nullptr && v[0] == '1';
    }();
    return on;
}

// ------------------------------------------------------------ validation

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

moe_status check_shape(const moe_shape* s) {
    if (!s) return MOE_ERR_ARG;
    if (s->wfmt != MOE_W_BF16 && s->wfmt != MOE_W_MXFP4 && s->wfmt != MOE_W_FP8 &&
        s->wfmt != MOE_W_MXFP4_MXFP8)
        return MOE_ERR_ARG;
    if (s->T < 0 || s->T > (1 << 20)) return MOE_ERR_SHAPE;
    if (s->H <= 0 || s->H % 64 || s->H > 32768) return MOE_ERR_SHAPE;
    if (s->I <= 0 || s->I % 64 || s->I > 32768) return MOE_ERR_SHAPE;
    if (s->E < 1 || s->E > kMaxExperts) return MOE_ERR_SHAPE;
    if (s->top_k < 1 || s->top_k > kMaxTopK || s->top_k > s->E) return MOE_ERR_SHAPE;
    // MXFP8 activations: the weights' chunk view needs K >= 128
    if (s->wfmt == MOE_W_MXFP4_MXFP8 && (s->H < 128 || s->I < 128)) return MOE_ERR_SHAPE;
    return MOE_OK;
}

moe_status check_ptr(const void* p) {
    if (!p) return MOE_ERR_ARG;
    if (!aligned16(p)) return MOE_ERR_ALIGN;
    return MOE_OK;
}

#define MOE_TRY(expr)                         \
    do {                                      \
        moe_status _st = (expr);              \
        if (_st != MOE_OK) return _st;        \
    } while (0)

#define MOE_CUDA(expr)                                \
    do {                                              \
        if ((expr) != cudaSuccess) return MOE_ERR_CUDA; \
    } while (0)

// Rows of tokens per GEMM tile.  bf16: round_up(T, 16), in [16, 256] -- a
// box that fits every expert's rows when T is small (one tile per touched
// expert), the widest MMA N otherwise; measured at T = 64 (k = 4, E = 32),
// boxes of 16 or 32 rows are 4-6 % slower than 64 (hot experts then take
// several tiles, re-streaming their weights).  MXFP4: about twice the mean
// rows per expert, round_up(2 * ceil(T * k / E), 16) in [16, 128] -- its
// ring slots carry 4 token chunks, so a smaller box buys a deeper ring (at
// T = 64: 113 us for gate_up with 16 rows against 133 us with 64), and its
// converted weights need TMEM beside the accumulators (at most 128 rows).
int auto_token_tile(const moe_shape& s) {
    const int tuned = g_token_tile.load();
    long long t;
    if (tuned > 0) {
        t = tuned;
    } else if (s.wfmt == MOE_W_MXFP4 || s.wfmt == MOE_W_MXFP4_MXFP8) {
        const long long mean = (static_cast<long long>(s.T) * s.top_k + s.E - 1) / s.E;
        t = (2 * mean + 15) / 16 * 16;
        // MXFP4 x MXFP8: at most 96 rows, so that the ring keeps three slots
        // beside the staged scales; measured on gpt-oss-20b (layer, us):
        // T=64 box 16/64: 104.2/117.4, T=512 box 96/128: 134.2/164.0,
        // T=4096 box 96/128: 605.3/633.0
        if (s.wfmt == MOE_W_MXFP4_MXFP8 && t > 96) t = 96;
    } else {
        t = (static_cast<long long>(s.T) + 15) / 16 * 16;
    }
    if (t < 16) t = 16;
    if (t > kMaxTokenTile) t = kMaxTokenTile;
    // MXFP4 (TMEM A slots) and MXFP4 x MXFP8 (TMEM scale slots) share 512
    // TMEM columns with the two accumulators
    if ((s.wfmt == MOE_W_MXFP4 || s.wfmt == MOE_W_MXFP4_MXFP8) && t > kMxfp4MaxTokenTile)
        t = kMxfp4MaxTokenTile;
    return static_cast<int>(t);
}

int next_pow2(int v) {
    int p = 1;
    while (p < v) p <<= 1;
    return p;
}

struct Routing {
    int32_t* ids;
    float* w;
    int32_t* offsets;
    int32_t* sorted_assign;
};

// K1 + K2.  x_perm null = no gather (routing only).
// small_perm: the router's last CTA writes the permutation (T * top_k <=
// kSmallPermRows) and the permutation kernel is not launched (the GEMM
// then gathers the token rows and clears the output itself).
moe_status launch_routing(const moe_shape& s, const WsLayout& L, uint8_t* ws, const void* hidden,
                          const void* router_w, const void* router_b, const Routing& r,
                          float* zero_out, __nv_bfloat16* x_perm, int token_tile,
                          const DevInfo& dev, cudaStream_t stream, int ex_lo, int ex_n,
                          bool small_perm = false) {
    int32_t* status = reinterpret_cast<int32_t*>(ws + L.status);
    const int nb = (s.T + kRouterTokens - 1) / kRouterTokens;

    // Router operands through TMA: x [T, H] box 64 x 32, Wr [E, H] box 64 x E_pad.
    CUtensorMap tm_x, tm_wr;
    {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(s.H), static_cast<cuuint64_t>(s.T)};
        const cuuint64_t str[1] = {static_cast<cuuint64_t>(s.H) * 2};
        const cuuint32_t boxd[2] = {64, static_cast<cuuint32_t>(kRouterTokens)};
        MOE_TRY(make_tmap(&tm_x, hidden, 2, dims, str, boxd));
    }
    {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(s.H), static_cast<cuuint64_t>(s.E)};
        const cuuint64_t str[1] = {static_cast<cuuint64_t>(s.H) * 2};
        const cuuint32_t boxd[2] = {64, static_cast<cuuint32_t>(kRouterTokens)};
        MOE_TRY(make_tmap(&tm_wr, router_w, 2, dims, str, boxd));
    }
    const int nchunks = s.H / kBlockK;
    const size_t fixed = router_smem_bytes(0);
    int stages = static_cast<int>((static_cast<size_t>(dev.max_smem) - fixed) /
                                  router_stage_bytes());
    if (stages > router_max_stages()) stages = router_max_stages();
    const int per_slice = (nchunks + router_ksplit(nb * ((s.E + 31) / 32), nchunks) - 1) /
                          router_ksplit(nb * ((s.E + 31) / 32), nchunks);
    if (stages >= per_slice) {
        stages = per_slice;                        // the ring never wraps
    } else {
        stages -= stages % router_stage_multiple();   // one consumer warp per slot
    }
    if (stages < 1) return MOE_ERR_UNSUPPORTED;

    RouterParams rp{};
    rp.br = static_cast<const __nv_bfloat16*>(router_b);
    rp.T = s.T;
    rp.H = s.H;
    rp.E = s.E;
    rp.top_k = s.top_k;
    rp.nblocks = nb;
    rp.egroups = (s.E + 31) / 32;
    rp.ksplit = router_ksplit(nb * rp.egroups, nchunks);
    rp.stages = stages;
    rp.logits = reinterpret_cast<float*>(ws + L.logits);
    rp.counters = reinterpret_cast<int32_t*>(ws + L.counters);
    rp.topk_ids = r.ids;
    rp.topk_w = r.w;
    rp.blk_cnt = reinterpret_cast<int32_t*>(ws + L.blk_cnt);
    rp.offsets = r.offsets;
    rp.tiles = reinterpret_cast<int4*>(ws + L.tiles);
    rp.max_tiles = L.max_tiles;
    rp.token_tile = token_tile;
    rp.ex_lo = ex_lo;
    rp.ex_n = ex_n;
    rp.inject = g_inject.load() & 3;
    rp.small_perm = small_perm ? 1 : 0;
    rp.sorted_assign = r.sorted_assign;
    rp.assign_row = reinterpret_cast<int32_t*>(ws + L.assign_row);
    rp.status = status;
    // few tokens: the single-block router (a grid of 4-token blocks up to 64
    // tokens when the router matrix can be staged in shared memory)
    const int tiny_tb = g_tiny_router.load() != 0 ? router_tiny_tokens_per_cta(s.T, s.H, s.E) : 0;
    if (tiny_tb > 0) {
        NvtxRange nv("moe.router_tiny");
        rp.nblocks = (s.T + tiny_tb - 1) / tiny_tb;
        MOE_CUDA(launch_router_tiny(rp, hidden, router_w, stream, g_pdl.load() != 0));
    } else {
        NvtxRange nv("moe.router_topk");
        MOE_CUDA(launch_router(rp, &tm_x, &tm_wr, router_smem_bytes(stages), stream,
                               g_pdl.load() != 0));
    }
    prof_mark("router_topk", stream);

    if (small_perm) return MOE_OK;

    PermuteParams pp{};
    pp.topk_ids = r.ids;
    pp.blk_cnt = rp.blk_cnt;
    pp.offsets = r.offsets;
    pp.x = static_cast<const __nv_bfloat16*>(hidden);
    pp.T = s.T;
    pp.H = s.H;
    pp.E = s.E;
    pp.top_k = s.top_k;
    pp.nblocks = nb;
    const int rows_per_block = (s.T < kRouterTokens ? s.T : kRouterTokens) * s.top_k;
    // CTAs per token block: as many as keep the grid within one wave (two
    // permutation CTAs fit on an SM); rounding up left a second wave that
    // started 18 us late at T = 4096
    int g = (x_perm || zero_out) ? (2 * dev.sms) / nb : 1;
    if (g > 32) g = 32;
    if (g > rows_per_block) g = rows_per_block;
    pp.gather_split = g < 1 ? 1 : g;
    pp.zero_out = zero_out;
    pp.sorted_assign = r.sorted_assign;
    pp.assign_row = reinterpret_cast<int32_t*>(ws + L.assign_row);
    pp.x_perm = x_perm;
    pp.mx_layout = s.wfmt == MOE_W_MXFP4 ? 1 : 0;
    pp.mx_f16 = s.wfmt == MOE_W_MXFP4 && g_mxfp4_f16.load() != 0 ? 1 : 0;
    pp.fp8 = s.wfmt == MOE_W_FP8 ? 1 : 0;
    pp.mx8 = s.wfmt == MOE_W_MXFP4_MXFP8 ? 1 : 0;
    pp.x_scale = reinterpret_cast<float*>(ws + L.x_scale);
    pp.ex_lo = ex_lo;
    pp.ex_hi = ex_lo + ex_n;
    pp.status = status;
    {
        NvtxRange nv(x_perm ? "moe.permute_gather" : "moe.permute");
        MOE_CUDA(launch_permute(pp, stream, g_pdl.load() != 0));
    }
    prof_mark(x_perm ? "permute_gather" : "permute", stream);
    return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

size_t moe_workspace_bytes(const moe_shape* shape) {
    if (check_shape(shape) != MOE_OK) return 0;
    return ws_layout(shape->T, shape->H, shape->I, shape->E, shape->top_k,
                     g_deterministic.load() != 0).total;
}

moe_status moe_route(const moe_shape* shape, const void* hidden, const void* router_w,
                     const void* router_b, int32_t* topk_ids, float* topk_w,
                     int32_t* expert_offsets, int32_t* sorted_assign, void* workspace,
                     size_t workspace_bytes, cudaStream_t stream) {
    MOE_TRY(check_shape(shape));
    const moe_shape s = *shape;
    if (s.T == 0) return MOE_OK;
    MOE_TRY(check_ptr(hidden));
    MOE_TRY(check_ptr(router_w));
    MOE_TRY(check_ptr(router_b));
    MOE_TRY(check_ptr(workspace));
    for (const void* p : {static_cast<const void*>(topk_ids), static_cast<const void*>(topk_w),
                          static_cast<const void*>(expert_offsets),
                          static_cast<const void*>(sorted_assign)})
        if (p && !aligned16(p)) return MOE_ERR_ALIGN;
    const WsLayout L = ws_layout(s.T, s.H, s.I, s.E, s.top_k);
    if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE;
    DevInfo dev;
    MOE_TRY(device_info(&dev));
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    Routing r;
    r.ids = topk_ids ? topk_ids : reinterpret_cast<int32_t*>(ws + L.topk_ids);
    r.w = topk_w ? topk_w : reinterpret_cast<float*>(ws + L.topk_w);
    r.offsets = expert_offsets ? expert_offsets : reinterpret_cast<int32_t*>(ws + L.offsets);
    r.sorted_assign =
        sorted_assign ? sorted_assign : reinterpret_cast<int32_t*>(ws + L.sorted_assign);
    NvtxRange nv("moe_route");
    std::lock_guard<std::mutex> lock(g_prof_mu);
    prof_reset(stream);
    const moe_status st = launch_routing(s, L, ws, hidden, router_w, router_b, r, nullptr,
                                         nullptr, auto_token_tile(s), dev, stream, 0, s.E);
    prof_finish();
    return st;
}

namespace moe {
namespace {

// moe_forward for the local experts [ex_lo, ex_lo + ex_n) of the layer's E
// (all of them for moe_forward); the weight banks hold those ex_n experts.
moe_status forward_impl(const moe_shape* shape, int ex_lo, int ex_n, const void* hidden,
                        const void* router_w, const void* router_b, moe_weight gate_up,
                        moe_weight down, void* out, int out_is_fp32, int32_t* topk_ids_out,
                        float* topk_w_out, void* workspace, size_t workspace_bytes,
                        cudaStream_t stream) {
    MOE_TRY(check_shape(shape));
    if (ex_lo < 0 || ex_n < 1 || ex_lo + ex_n > shape->E) return MOE_ERR_ARG;
    const moe_shape s = *shape;
    if (s.T == 0) return MOE_OK;
    MOE_TRY(check_ptr(hidden));
    MOE_TRY(check_ptr(router_w));
    MOE_TRY(check_ptr(router_b));
    MOE_TRY(check_ptr(gate_up.w));
    MOE_TRY(check_ptr(gate_up.bias));
    MOE_TRY(check_ptr(down.w));
    MOE_TRY(check_ptr(down.bias));
    MOE_TRY(check_ptr(out));
    MOE_TRY(check_ptr(workspace));
    const bool mxfp4 = s.wfmt == MOE_W_MXFP4;
    const bool fp8 = s.wfmt == MOE_W_FP8;
    const bool mx = s.wfmt == MOE_W_MXFP4_MXFP8;
    if (mxfp4 || mx) {
        MOE_TRY(check_ptr(gate_up.scale));
        MOE_TRY(check_ptr(down.scale));
    } else if (fp8) {
        // per-expert fp32 scales, read one float at a time: 4-byte alignment
        // (a slice of an expert-parallel rank is 4-byte aligned)
        if (!gate_up.scale || !down.scale) return MOE_ERR_ARG;
        if ((reinterpret_cast<uintptr_t>(gate_up.scale) | reinterpret_cast<uintptr_t>(down.scale)) & 3)
            return MOE_ERR_ALIGN;
    }
    // the 4-bit tensor maps of the block-scaled path want 32-byte alignment
    if (mx && ((reinterpret_cast<uintptr_t>(gate_up.w) | reinterpret_cast<uintptr_t>(down.w)) & 31))
        return MOE_ERR_ALIGN;
    if ((topk_ids_out && !aligned16(topk_ids_out)) || (topk_w_out && !aligned16(topk_w_out)))
        return MOE_ERR_ALIGN;
    const bool det = g_deterministic.load() != 0;
    const WsLayout L = ws_layout(s.T, s.H, s.I, s.E, s.top_k, det);
    if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE;
    DevInfo dev;
    MOE_TRY(device_info(&dev));

    uint8_t* ws = static_cast<uint8_t*>(workspace);
    int32_t* status = reinterpret_cast<int32_t*>(ws + L.status);
    const int R = s.T * s.top_k;
    const int box = auto_token_tile(s);
    const bool pdl = g_pdl.load() != 0;

    // CTA pairs (bf16 or FP8, wide token boxes): M = 256 MMAs over two SMs, each SM
    // loading 128 weight rows and half of the token tile, so a ring slot
    // holds 32 KB instead of 48 KB (box 256) for the same tensor work.
    const int pair_mode = g_pair_mode.load();
    const bool pair_auto =
        box >= kPairMinBox &&
        (!fp8 || static_cast<long long>(R) < kFp8PairMaxMeanRows * s.E);
    const bool pair = !mxfp4 && !mx && (pair_mode == 2 || (pair_mode == 0 && pair_auto));
    const int bbox = pair ? box / 2 : box;     // token rows of one CTA's B tile
    // Pipeline depth: as many stages as the shared memory allows (2..12).
    const int wf = mxfp4 ? 1 : fp8 ? 2 : mx ? 3 : 0;
    const int kscale_max = (s.H > s.I ? s.H : s.I) / 32;
    const size_t stage_bytes = gemm_stage_bytes(bbox, wf);
    const size_t budget = static_cast<size_t>(dev.max_smem) - 1024;
    // MXFP4: per MMA issuer two accumulators of round_up(box, 32) TMEM
    // columns, then A slots of 128 columns, all in 512.  Two issuers (one N
    // <= 64 MMA per ~23 ns each) while their accumulators leave room for two
    // A slots, else one.
    int astages = 0, n_iss = 1;
    if (mxfp4) {
        const int acc = (box + 31) & ~31;
        n_iss = 2 * 2 * acc + 2 * 128 <= 512 ? 2 : 1;
        astages = (512 - 2 * n_iss * acc) / 128;
        if (astages > kMxfp4AStages) astages = kMxfp4AStages;
        // two issuers: an even count, so that every A slot is always used by
        // the same issuer and converter team (their barrier phases then
        // advance in order)
        if (n_iss == 2) astages &= ~1;
        if (astages < 2) return MOE_ERR_UNSUPPORTED;
    }
    const size_t fixed = gemm_fixed_bytes(box, wf, kscale_max, mx ? mx_scale_row_bytes(s.H) : 0);
    int stages = budget < fixed ? 0 : static_cast<int>((budget - fixed) / stage_bytes);
    // MXFP4 converter teams need 2 x stages >= astages + 2
    if (stages < 2 || (mxfp4 && 2 * stages < astages + 2)) return MOE_ERR_UNSUPPORTED;
    const int max_stages = mxfp4 ? 24 : 12;   // MXFP4 slots carry 4 KB of HBM bytes
    if (stages > max_stages) stages = max_stages;
    // MXFP4 x MXFP8: 8 TMEM scale columns per k-block of a ring slot after the two
    // accumulators of round_up(box, 32) columns
    const int mx_acc = (box + 31) & ~31;
    if (mx && stages > (512 - 2 * mx_acc) / (8 * kMxKbPerStage))
        stages = (512 - 2 * mx_acc) / (8 * kMxKbPerStage);
    if (stages < 2) return MOE_ERR_UNSUPPORTED;
    const size_t smem = fixed + stages * stage_bytes + 1024;
    // two accumulators (+ MXFP4: A tiles of 32 columns after them)
    const int tmem_cols =
        mxfp4 ? 512 : mx ? next_pow2(2 * mx_acc + 8 * kMxKbPerStage * stages) : next_pow2(2 * box < 32 ? 32 : 2 * box);
    if (tmem_cols > 512) return MOE_ERR_UNSUPPORTED;

    __nv_bfloat16* x_perm = reinterpret_cast<__nv_bfloat16*>(ws + L.x_perm);
    __nv_bfloat16* h = reinterpret_cast<__nv_bfloat16*>(ws + L.h);
    float* out32 = out_is_fp32 ? static_cast<float*>(out) : reinterpret_cast<float*>(ws + L.out_acc);

    // Tensor maps (host-side descriptors; cheap to build per call).
    CUtensorMap tm_wgu, tm_x, tm_wd, tm_h;
    if (mx) {
        MOE_TRY(mx_weight_tmap(&tm_wgu, gate_up.w, ex_n, 2 * s.I, s.H));
        MOE_TRY(mx_weight_tmap(&tm_wd, down.w, ex_n, s.H, s.I));
    } else {
        MOE_TRY(weight_tmap(&tm_wgu, gate_up.w, ex_n, 2 * s.I, s.H, mxfp4, fp8));
        MOE_TRY(weight_tmap(&tm_wd, down.w, ex_n, s.H, s.I, mxfp4, fp8));
    }
    // Token operands: bf16 layers read [R, K] row-major, one 64-wide K chunk
    // per box; MXFP4 layers read the chunk-major [K/64, R, 64] layout the
    // gather and the GLU epilogue write, kMxfp4KbPerStage chunks per box.
    const auto token_tmap = [&](CUtensorMap* m, const void* base, int K) {
        if (mxfp4) {
            const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(R),
                                        static_cast<cuuint64_t>(K) / 64};
            const cuuint64_t str[2] = {128, static_cast<cuuint64_t>(R) * 128};
            const cuuint32_t boxd[3] = {64, static_cast<cuuint32_t>(box), kMxfp4KbPerStage};
            return make_tmap(m, base, 3, dims, str, boxd);
        }
        if (mx) {
            // E4M3 codes [R, mx_padded_k(K)], one byte each: box 128 K x box rows
            const cuuint64_t kp = static_cast<cuuint64_t>(mx_padded_k(K));
            const cuuint64_t dims[2] = {kp, static_cast<cuuint64_t>(R)};
            const cuuint64_t str[1] = {kp};
            const cuuint32_t boxd[2] = {static_cast<cuuint32_t>(kBlockKFp8),
                                        static_cast<cuuint32_t>(bbox)};
            return make_tmap(m, base, 2, dims, str, boxd, true);
        }
        if (fp8) {
            // E4M3 codes [R, K], one byte each: box 128 K x box rows
            const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(R)};
            const cuuint64_t str[1] = {static_cast<cuuint64_t>(K)};
            const cuuint32_t boxd[2] = {static_cast<cuuint32_t>(kBlockKFp8),
                                        static_cast<cuuint32_t>(bbox)};
            return make_tmap(m, base, 2, dims, str, boxd, true);
        }
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(R)};
        const cuuint64_t str[1] = {static_cast<cuuint64_t>(K) * 2};
        const cuuint32_t boxd[2] = {64, static_cast<cuuint32_t>(bbox)};
        return make_tmap(m, base, 2, dims, str, boxd);
    };
    MOE_TRY(token_tmap(&tm_x, x_perm, s.H));
    MOE_TRY(token_tmap(&tm_h, h, s.I));

    std::lock_guard<std::mutex> lock(g_prof_mu);
    prof_reset(stream);

    Routing r;
    r.ids = topk_ids_out ? topk_ids_out : reinterpret_cast<int32_t*>(ws + L.topk_ids);
    r.w = topk_w_out ? topk_w_out : reinterpret_cast<float*>(ws + L.topk_w);
    r.offsets = reinterpret_cast<int32_t*>(ws + L.offsets);
    r.sorted_assign = reinterpret_cast<int32_t*>(ws + L.sorted_assign);
    const bool checks = stage_checks_on();
    if (checks)
        MOE_CUDA(cudaMemsetAsync(status + kStageStatsWord, 0, 2 * kNumStages * sizeof(int32_t),
                                 stream));
    // Small bf16 batches: the router makes the permutation and gate_up
    // gathers its token rows from `hidden` (no permutation kernel, no x_perm
    // round trip; gate_up clears the output rows)
    const bool small = g_small_path.load() != 0 && !mxfp4 && !fp8 && !mx && !pair &&
                       R <= kSmallPermRows && s.T <= kSmallPathMaxT && box <= 64 && stages > 4;
    // The output rows the down projection accumulates into are cleared by
    // gate_up's epilogue warps, not by the permutation: at prefill the
    // permutation is bound by its writes (the gathered rows), while gate_up
    // is bound by the tensor cores (20b T=4096: 47 MB of zeros off the
    // permutation's path).  The deterministic combine writes every output
    // element, so its output needs no clearing.
    MOE_TRY(launch_routing(s, L, ws, hidden, router_w, router_b, r, nullptr,
                           small ? nullptr : x_perm, box, dev, stream, ex_lo, ex_n, small));
    // element type of the GEMM token operands: E4M3 codes (FP8, MXFP8) or bf16
    const int tok_dtype = (fp8 || mx) ? 2 : (mxfp4 && g_mxfp4_f16.load() != 0) ? 3 : 0;
    if (checks)
        MOE_CUDA(launch_stage_check(small ? hidden : static_cast<const void*>(x_perm),
                                    small ? static_cast<size_t>(s.T) * s.H
                                          : static_cast<size_t>(R) * (mx ? mx_padded_k(s.H) : s.H),
                                    tok_dtype, 0, status, stream));

    GemmParams g{};
    g.tiles = reinterpret_cast<const int4*>(ws + L.tiles);
    g.num_tiles = status + kNumTilesWord;
    g.token_box = box;
    g.stages = stages;
    g.astages = astages;
    g.n_iss = n_iss;
    g.tmem_cols = tmem_cols;
    g.num_experts = ex_n;            // tiles number the local experts from 0
    g.rows_total = R;
    g.status = status;
    g.mx_f16 = mxfp4 && g_mxfp4_f16.load() != 0 ? 1 : 0;

    const int unit_rows = pair ? 2 * kWeightTileRows : kWeightTileRows;
    const int cg = pair ? 2 : 1;

    // gate_up + bias + GLU -> h
    g.n_wblocks = (2 * s.I + unit_rows - 1) / unit_rows;
    // k-blocks of 64 bf16 / E4M3: 128 (a K tail past the last full block is
    // zero-filled by TMA)
    g.k_blocks = (fp8 || mx) ? (s.H + kBlockKFp8 - 1) / kBlockKFp8 : s.H / kBlockK;
    g.w_rows = 2 * s.I;
    g.bias = static_cast<const __nv_bfloat16*>(gate_up.bias);
    g.h = h;
    g.scales = static_cast<const uint8_t*>(gate_up.scale);
    g.wscale = fp8 ? static_cast<const float*>(gate_up.scale) : nullptr;
    g.xscale = reinterpret_cast<const float*>(ws + L.x_scale);
    g.h8 = reinterpret_cast<uint8_t*>(h);
    g.hscale = kFp8HScale;
    g.kscale = s.H / 32;
    g.mx_cmax = s.H / 64 - 2;
    g.xs_mx = mx ? reinterpret_cast<const uint8_t*>(ws + L.x_scale) : nullptr;
    g.xs_row_bytes = mx_scale_row_bytes(s.H);
    g.h_pad = mx_padded_k(s.I);
    g.h_tail0 = mx_tail0(s.I);
    // K split when the units cannot fill two waves (small batches)
    const int kb_per_slot = mxfp4 ? kMxfp4KbPerStage : mx ? kMxKbPerStage : 1;
    const long long tiles_max = max_token_tiles(R, L.max_tiles);
    const int split_mode = g_ksplit_mode.load();
    // parts for `slots` ring slots: the model's choice (at most auto_max), or
    // the forced count (no empty part, at least 2 slots each)
    const auto parts_of = [](int want, int slots) {
        if (want > slots / 2) want = slots / 2;
        if (want < 2) return 1;
        const int per = (slots + want - 1) / want;
        return (slots + per - 1) / per;
    };
    const auto parts_for = [&](long long units, int slots, int auto_max) {
        if (split_mode == 1) return 1;
        if (split_mode >= 2) return parts_of(split_mode, slots);
        const int m = gemm_ksplit(units, slots, dev.sms);
        return m > auto_max ? parts_of(auto_max, slots) : m;
    };
    // gate_up: at most 2 parts -- each part's epilogue stores, fences and
    // tickets its partial tile and the last one reloads all of them; at
    // 20b T=1 (180 units) 2 parts gave 33 us, 3 gave 39, 5 gave 46 (1: 37)
    g.ksplit = pair ? 1 : parts_for(tiles_max * g.n_wblocks, (g.k_blocks + kb_per_slot - 1) / kb_per_slot, 2);
    {
        // no more parts than the partial-tile region holds at R rows
        const size_t part_bytes = static_cast<size_t>(g.n_wblocks) * R * kWeightTileRows * 4;
        const size_t cap = part_bytes ? L.gemm_partial_bytes / part_bytes : 0;
        if (static_cast<size_t>(g.ksplit) > cap) {
            const int slots = (g.k_blocks + kb_per_slot - 1) / kb_per_slot;
            const int want = cap < 2 ? 1 : static_cast<int>(cap);
            const int per = (slots + want - 1) / want;
            g.ksplit = want < 2 ? 1 : (slots + per - 1) / per;
        }
    }
    g.partial = reinterpret_cast<float*>(ws + L.gemm_partial);
    g.tickets = reinterpret_cast<int32_t*>(ws + L.counters) + kSplitTicketOffset;
    long long units = tiles_max * g.n_wblocks * g.ksplit;
    long long ctas = units * cg;
    int grid = static_cast<int>(ctas < dev.sms ? ctas : dev.sms);
    g.inject_stall = (g_inject.load() & 4) && !mxfp4 ? 1 : 0;
    // small batches: token rows gathered from the input; the tile list comes
    // from the router, the kernel just before, so nothing starts before the
    // dependency wait.  Every batch: the output rows are cleared here
    g.gather_x = small ? static_cast<const __nv_bfloat16*>(hidden) : nullptr;
    g.gather_K = s.H;
    // (the gather reads the permutation: row r of a tile is assignment
    // sorted_assign[r] of token sorted_assign[r] / top_k)
    g.sorted_assign = r.sorted_assign;
    g.top_k = s.top_k;
    g.zero_out = det ? nullptr : out32;
    g.n_zero = static_cast<size_t>(s.T) * s.H;
    g.prewait = small ? 0 : 1;
    {
        NvtxRange nv("moe.gate_up_glu");
        MOE_CUDA(launch_gemm(kEpiGlu, wf, cg, g, &tm_wgu, &tm_x, grid, smem, stream, pdl));
    }
    if (checks)
        MOE_CUDA(launch_stage_check(h, static_cast<size_t>(R) * (mx ? mx_padded_k(s.I) : s.I),
                                    tok_dtype, 1, status, stream));
    g.inject_stall = 0;
    g.gather_x = nullptr;
    g.zero_out = nullptr;
    g.prewait = 1;           // tiles from the router, two kernels back
    prof_mark("gate_up_glu", stream);

    // down + bias + weighted combine -> out (fp32 accumulation)
    g.n_wblocks = (s.H + unit_rows - 1) / unit_rows;
    g.k_blocks = (fp8 || mx) ? (s.I + kBlockKFp8 - 1) / kBlockKFp8 : s.I / kBlockK;
    g.w_rows = s.H;
    g.bias = static_cast<const __nv_bfloat16*>(down.bias);
    g.h = nullptr;
    g.out = out32;
    g.sorted_assign = r.sorted_assign;
    g.topk_w = r.w;
    g.top_k = s.top_k;
    g.scales = static_cast<const uint8_t*>(down.scale);
    g.wscale = fp8 ? static_cast<const float*>(down.scale) : nullptr;
    g.kscale = s.I / 32;
    g.mx_cmax = s.I / 64 - 2;
    g.xs_mx = nullptr;                      // h codes: every block scale 2^-3
    // the down projection adds its K parts through the output's atomics
    // (deterministic combine: whole K ranges, one stored row per slot)
    g.ksplit = pair || det ? 1 : parts_for(tiles_max * g.n_wblocks, (g.k_blocks + kb_per_slot - 1) / kb_per_slot, kMaxKSplit);
    g.partial = nullptr;
    g.tickets = nullptr;
    g.y_rows = det ? reinterpret_cast<float*>(ws + L.y_rows) : nullptr;
    units = tiles_max * g.n_wblocks * g.ksplit;
    ctas = units * cg;
    grid = static_cast<int>(ctas < dev.sms ? ctas : dev.sms);
    {
        NvtxRange nv("moe.down_combine");
        MOE_CUDA(launch_gemm(kEpiCombine, wf, cg, g, &tm_wd, &tm_h, grid, smem, stream, pdl));
    }
    prof_mark("down_combine", stream);

    if (det) {
        NvtxRange nv("moe.combine_ordered");
        MOE_CUDA(launch_combine_rows(
            g.y_rows, reinterpret_cast<const int32_t*>(ws + L.assign_row), r.ids, s.T, s.H,
            s.top_k, ex_lo, ex_lo + ex_n, out_is_fp32 ? static_cast<float*>(out) : nullptr,
            out_is_fp32 ? nullptr : static_cast<__nv_bfloat16*>(out), stream, pdl));
        prof_mark("combine_ordered", stream);
    } else if (!out_is_fp32) {
        NvtxRange nv("moe.to_bf16");
        MOE_CUDA(launch_to_bf16(out32, static_cast<__nv_bfloat16*>(out),
                                static_cast<size_t>(s.T) * s.H, stream, pdl));
        prof_mark("to_bf16", stream);
    }
    if (checks)
        MOE_CUDA(launch_stage_check(out, static_cast<size_t>(s.T) * s.H, out_is_fp32 ? 1 : 0, 2,
                                    status, stream));
    prof_finish();
    return MOE_OK;
}

}  // namespace
}  // namespace moe

moe_status moe_forward(const moe_shape* shape, const void* hidden, const void* router_w,
                       const void* router_b, moe_weight gate_up, moe_weight down, void* out,
                       int out_is_fp32, int32_t* topk_ids_out, float* topk_w_out,
                       void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (!shape) return MOE_ERR_ARG;
    NvtxRange nv("moe_forward");
    return forward_impl(shape, 0, shape->E, hidden, router_w, router_b, gate_up, down, out,
                        out_is_fp32, topk_ids_out, topk_w_out, workspace, workspace_bytes,
                        stream);
}

moe_status moe_forward_ep(const moe_shape* shape, int expert_start, int local_experts,
                          const void* hidden, const void* router_w, const void* router_b,
                          moe_weight gate_up, moe_weight down, void* out, int out_is_fp32,
                          int32_t* topk_ids_out, float* topk_w_out, void* workspace,
                          size_t workspace_bytes, cudaStream_t stream) {
    if (!shape) return MOE_ERR_ARG;
    NvtxRange nv("moe_forward_ep");
    return forward_impl(shape, expert_start, local_experts, hidden, router_w, router_b,
                        gate_up, down, out, out_is_fp32, topk_ids_out, topk_w_out, workspace,
                        workspace_bytes, stream);
}

moe_status moe_get_device_status(const void* workspace, int32_t* host_status) {
    if (!workspace || !host_status) return MOE_ERR_ARG;
    int32_t v = 0;
    if (cudaMemcpy(&v, workspace, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess)
        return MOE_ERR_CUDA;
    *host_status = v;
    return v ? MOE_ERR_DEVICE : MOE_OK;
}

moe_status moe_stage_stats(const void* workspace, int32_t nonfinite[3], float maxabs[3]) {
    if (!workspace || !nonfinite || !maxabs) return MOE_ERR_ARG;
    int32_t w[2 * kNumStages];
    if (cudaMemcpy(w, static_cast<const int32_t*>(workspace) + kStageStatsWord, sizeof w,
                   cudaMemcpyDeviceToHost) != cudaSuccess)
        return MOE_ERR_CUDA;
    for (int i = 0; i < kNumStages; ++i) {
        nonfinite[i] = w[2 * i];
        std::memcpy(&maxabs[i], &w[2 * i + 1], sizeof(float));
    }
    return MOE_OK;
}

moe_status moe_trace_read(uint64_t* out, size_t cap, size_t* count) {
    if (!count) return MOE_ERR_ARG;
    *count = 0;
    if (!out) return MOE_ERR_ARG;
    unsigned long long* o = reinterpret_cast<unsigned long long*>(out);
    size_t n = trace_copy_router(o, cap);
    if (n == 0) return MOE_ERR_UNSUPPORTED;
    const size_t n2 = trace_copy_permute(o + n, cap - n);
    if (n2 == 0) return MOE_ERR_UNSUPPORTED;
    n += n2;
    const size_t n3 = trace_copy_gemm(o + n, cap - n);
    if (n3 == 0) return MOE_ERR_UNSUPPORTED;
    n += n3;
    const size_t n4 = trace_copy_attn(o + n, cap - n);
    if (n4 == 0) return MOE_ERR_UNSUPPORTED;
    *count = n + n4;
    return MOE_OK;
}

moe_status moe_clear_device_status(void* workspace, cudaStream_t stream) {
    if (!workspace) return MOE_ERR_ARG;
    // the status word and the router's ticket counters (fixed offsets)
    return cudaMemsetAsync(workspace, 0, 256 + kCounterBytes, stream) == cudaSuccess
               ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_set_tuning(const char* key, int value) {
    if (!key) return MOE_ERR_ARG;
    if (std::strcmp(key, "token_tile") == 0) {
        if (value != 0 && (value < 16 || value > kMaxTokenTile || value % 16)) return MOE_ERR_ARG;
        g_token_tile.store(value);
        return MOE_OK;
    }
    if (std::strcmp(key, "ksplit") == 0) {
        if (value < 0 || value > kMaxKSplit) return MOE_ERR_ARG;
        g_ksplit_mode.store(value);
        return MOE_OK;
    }
    if (std::strcmp(key, "pair") == 0) {
        if (value < 0 || value > 2) return MOE_ERR_ARG;
        g_pair_mode.store(value);
        return MOE_OK;
    }
    if (std::strcmp(key, "mxfp4_f16") == 0) {
        if (value != 0 && value != 1) return MOE_ERR_ARG;
        g_mxfp4_f16.store(value);
        return MOE_OK;
    }
    if (std::strcmp(key, "attn_tc") == 0) return static_cast<moe_status>(set_attn_tc_mode(value));
    if (std::strcmp(key, "attn_poll") == 0) return static_cast<moe_status>(set_attn_poll(value));
    if (std::strcmp(key, "tiny_router") == 0) {
        if (value != 0 && value != 1) return MOE_ERR_ARG;
        g_tiny_router.store(value);
        return MOE_OK;
    }
    if (std::strcmp(key, "small_path") == 0) {
        if (value != 0 && value != 1) return MOE_ERR_ARG;
        g_small_path.store(value);
        return MOE_OK;
    }
    if (std::strcmp(key, "inject") == 0) {
        if (value < 0 || value > 7) return MOE_ERR_ARG;
        g_inject.store(value);
        return MOE_OK;
    }
    if (std::strcmp(key, "deterministic") == 0) {
        if (value != 0 && value != 1) return MOE_ERR_ARG;
        g_deterministic.store(value);
        return MOE_OK;
    }
    if (std::strcmp(key, "noalloc_poison") == 0) {
        if (value != 0 && value != 1) return MOE_ERR_ARG;
        set_noalloc_poison(value);
        return MOE_OK;
    }
    if (std::strcmp(key, "pdl") == 0) {
        if (value != 0 && value != 1) return MOE_ERR_ARG;
        g_pdl.store(value);
        return MOE_OK;
    }
    return MOE_ERR_ARG;
}

moe_status moe_profile_enable(int calls) {
    std::lock_guard<std::mutex> lock(g_prof_mu);
    if (calls < 0 || calls > kMaxProfCalls) return MOE_ERR_ARG;
    const int need = calls * (kMaxProf + 1);
    if (need > g_prof.created) {
        cudaEvent_t* ev = static_cast<cudaEvent_t*>(
            std::realloc(g_prof.ev, sizeof(cudaEvent_t) * static_cast<size_t>(need)));
        if (!ev) return MOE_ERR_ARG;
        g_prof.ev = ev;
        for (int i = g_prof.created; i < need; ++i) {
            if (cudaEventCreate(&g_prof.ev[i]) != cudaSuccess) {
                g_prof.created = i;
                g_prof.capacity = 0;
                return MOE_ERR_CUDA;
            }
        }
        g_prof.created = need;
    }
    g_prof.capacity = calls;
    g_prof.calls = 0;
    g_prof.n = -1;
    g_prof.n_first = 0;
    return MOE_OK;
}

moe_status moe_profile_read(const char** names, float* ms, int cap, int* count) {
    std::lock_guard<std::mutex> lock(g_prof_mu);
    if (!count) return MOE_ERR_ARG;
    *count = 0;
    const int calls = g_prof.calls, nk = g_prof.n_first;
    if (calls == 0 || nk == 0) return MOE_OK;
    cudaEvent_t* last = g_prof.ev + static_cast<size_t>(calls - 1) * (kMaxProf + 1);
    if (cudaEventSynchronize(last[nk]) != cudaSuccess) return MOE_ERR_CUDA;
    const int n = nk < cap ? nk : cap;
    for (int i = 0; i < n; ++i) {
        double sum = 0.0;
        for (int c = 0; c < calls; ++c) {
            cudaEvent_t* e = g_prof.ev + static_cast<size_t>(c) * (kMaxProf + 1);
            float t = 0.f;
            if (cudaEventElapsedTime(&t, e[i], e[i + 1]) != cudaSuccess) return MOE_ERR_CUDA;
            sum += t;
        }
        if (names) names[i] = g_prof.names[i];
        if (ms) ms[i] = static_cast<float>(sum / calls);
    }
    *count = n;
    return MOE_OK;
}

const char* moe_status_str(moe_status st) {
    switch (st) {
        case MOE_OK: return "ok";
        case MOE_ERR_ARG: return "invalid argument (null pointer or bad enum)";
        case MOE_ERR_SHAPE: return "unsupported shape";
        case MOE_ERR_ALIGN: return "pointer not 16-byte aligned";
        case MOE_ERR_WORKSPACE: return "workspace missing or too small";
        case MOE_ERR_UNSUPPORTED: return "unsupported by this build or device";
        case MOE_ERR_CUDA: return "CUDA runtime/driver call failed";
        case MOE_ERR_DEVICE: return "device status word reports an error";
    }
    return "unknown status";
}

}  // extern "C"
