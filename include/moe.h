/*
 * gpt-oss mixture-of-experts layer forward on one GB300 (sm_103a).
 *
 * The operation (xserv docs/19-gpt-oss-moe.md, "Phase 19: gpt-oss-20b",
 * §1 model-architecture table "MoE" and "激活" rows, §2 "MoE 前向"):
 *
 *   logits[t,e] = sum_h x[t,h] * Wr[e,h] + br[e]                 (router)
 *   ids[t,:]    = the top_k experts by logit, descending, ties to the lower
 *                 expert index; w[t,:] = softmax over those k logits
 *   gu          = W_gu[e] x[t] + b_gu[e]           (2I features, interleaved)
 *   gate_j      = min(gu[2j], 7),  up_j = clamp(gu[2j+1], -7, 7)
 *   h_j         = (up_j + 1) * gate_j * sigmoid(1.702 * gate_j)
 *   y           = W_d[e] h + b_d[e]
 *   out[t,:]    = sum_{j<top_k} w[t,j] * y(expert ids[t,j], token t)
 *
 * Unselected experts are skipped (never multiplied by zero).  Expert ids stay
 * on the device: no call below synchronises the host with the GPU, except
 * moe_get_device_status, which says so.
 *
 * Conventions for every call:
 *   - All tensor pointers are DEVICE pointers, row-major, densely packed,
 *     16-byte aligned (FP8 per-expert scale arrays: 4-byte aligned).  The caller owns every buffer; the library allocates
 *     no device memory and keeps no state beyond a per-device cache of device
 *     attributes and the optional profiling events below.
 *   - bf16 is IEEE-754 binary16-brain (uint16 storage).
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default).
 *   - Argument errors are detected on the host before anything is enqueued
 *     and returned as a negative moe_status; nothing is launched then.
 *   - Errors that only the device can see (an expert id out of range, a
 *     pipeline wait that timed out) set bits in the device status word held
 *     in the workspace; read it with moe_get_device_status.
 *   - T == 0 is valid and enqueues nothing.
 *
 * Supported shapes: H % 64 == 0, I % 64 == 0, 1 <= E <= 256,
 * 1 <= top_k <= min(E, 8), 0 <= T <= 1048576.
 */
#ifndef GPT_OSS_MOE_H
#define GPT_OSS_MOE_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_ARG = -1,          /* null pointer or bad enum value */
    MOE_ERR_SHAPE = -2,        /* a dimension outside the supported set */
    MOE_ERR_ALIGN = -3,        /* a pointer not 16-byte aligned */
    MOE_ERR_WORKSPACE = -4,    /* workspace missing or smaller than needed */
    MOE_ERR_UNSUPPORTED = -5,  /* valid request this build cannot serve */
    MOE_ERR_CUDA = -6,         /* a CUDA runtime/driver call failed */
    MOE_ERR_DEVICE = -7        /* the device status word reported an error */
} moe_status;

/* Expert weight storage format. */
typedef enum {
    MOE_W_BF16 = 0,   /* bf16 values */
    MOE_W_MXFP4 = 1,  /* OCP MX FP4: E2M1 codes, two per byte (element 2i in
                         the low nibble of byte i), plus one E8M0 scale byte
                         (value 2^(s-127)) per 32 consecutive input elements
                         of each output row (§5 "量化") */
    MOE_W_FP8 = 2,    /* FP8 W8A8 (§5 "量化"): E4M3 codes ("fn": max 448),
                         one byte per weight, [E, N, K] like bf16, and
                         moe_weight.scale = fp32 [E], one scale per expert,
                         applied to the finished products.  The layer
                         quantises the activations itself: each token with
                         its own scale max|x| / 448 (round to nearest even,
                         saturating), h with the fixed scale 1/8 (the GLU
                         clamps keep |h| * 8 <= 448) */
    MOE_W_MXFP4_MXFP8 = 3 /* MXFP4 weights exactly as MOE_W_MXFP4 (codes
                         32-byte aligned), with the activations quantised
                         by the layer to MXFP8 (OCP MX): every block of 32
                         consecutive elements of a token gets the scale
                         2^(floor(log2 max|x|) - 8) (a UE8M0 byte, at least
                         2^-127) and E4M3 codes of x / scale (round to
                         nearest even, saturating); h likewise with every
                         block scale 1/8.  The GEMMs run on the tensor cores'
                         block-scaled MMA, with no software dequantisation.
                         Needs H, I >= 128 */
} moe_wfmt;

/* Layer shape.  T tokens, hidden size H, expert intermediate size I,
 * E experts, top_k experts per token. */
typedef struct {
    int T, H, I, E, top_k;
    int wfmt;                  /* a moe_wfmt */
} moe_shape;

/* One expert weight bank.
 *   gate_up: w bf16 [E, 2I, H] (row 2j = gate_j, row 2j+1 = up_j) or MXFP4
 *            codes u8 [E, 2I, H/2] with scale u8 [E, 2I, H/32] or FP8 codes
 *            u8 [E, 2I, H] with scale fp32 [E];
 *            bias bf16 [E, 2I].
 *   down:    w bf16 [E, H, I] or codes u8 [E, H, I/2], scale u8 [E, H, I/32],
 *            or FP8 codes u8 [E, H, I] with scale fp32 [E];
 *            bias bf16 [E, H].
 * MOE_W_MXFP4_MXFP8 takes the MXFP4 bank.  scale is NULL for bf16 weights. */
typedef struct {
    const void* w;
    const void* scale;
    const void* bias;
} moe_weight;

/* Device status word bits (moe_get_device_status). */
#define MOE_DEV_BAD_EXPERT_ID  0x1   /* a routed id fell outside [0, E) */
#define MOE_DEV_WAIT_TIMEOUT   0x2   /* a pipeline wait gave up (~1 s) */
#define MOE_DEV_BAD_TILE       0x4   /* a work tile or a permutation row
                                        failed its bounds check */
#define MOE_DEV_NONFINITE      0x8   /* a stage check (MOE_CHECK_STAGES=1) met
                                        a NaN or an infinity */
#define MOE_DEV_BOUNDS         0x10  /* an index check of a MOE_DEBUG_BOUNDS
                                        build failed (the access was skipped) */
#define MOE_DEV_RANGE          0x20  /* MXFP4 weights, f16 mode: a scale byte
                                        outside [104, 140] or an activation
                                        beyond +-65504 was clamped; the
                                        result is inexact (rerun with the
                                        "mxfp4_f16" switch off) */

/* Bytes of device workspace moe_route / moe_forward need for this shape
 * (0 for an invalid shape).  The workspace is scratch owned by the caller.
 * A new workspace must be zero-filled once before its first use (e.g.
 * cudaMemsetAsync(ws, 0, bytes), or moe_clear_device_status): it starts
 * with the status word and a fixed block of completion counters that every
 * call leaves at zero again, so one workspace (large enough) may serve any
 * shape.  After a device error is reported, clear it again.  Apart from
 * those, its contents between calls are unspecified.  Calls that share a
 * workspace must not overlap on the GPU. */
size_t moe_workspace_bytes(const moe_shape* shape);

/* Router + top-k softmax + expert permutation (§2: "router GEMV ->
 * topk_softmax", ids kept on the GPU).
 *   hidden   bf16 [T, H];  router_w bf16 [E, H];  router_b bf16 [E]
 *   topk_ids int32 [T, top_k]   out: expert of slot j of token t
 *   topk_w   fp32  [T, top_k]   out: its softmax weight
 *   expert_offsets int32 [E+1]  out: exclusive scan of per-expert counts
 *   sorted_assign  int32 [T*top_k] out: assignment a = t*top_k + j placed at
 *                  row r, rows sorted by (expert, a) ascending
 * Any of the four outputs may be NULL (that result is then kept in the
 * workspace only).  Returns MOE_OK once the work is enqueued. */
moe_status moe_route(const moe_shape* shape, const void* hidden,
                     const void* router_w, const void* router_b,
                     int32_t* topk_ids, float* topk_w,
                     int32_t* expert_offsets, int32_t* sorted_assign,
                     void* workspace, size_t workspace_bytes,
                     cudaStream_t stream);

/* The whole layer forward (§2 step list, routed form).
 *   hidden, router_w, router_b as for moe_route;
 *   gate_up, down: expert weight banks (see moe_weight);
 *   out: [T, H], fp32 when out_is_fp32 != 0, else bf16 (rounded to nearest
 *        even from the fp32 sum);
 *   topk_ids_out int32 [T, top_k], topk_w_out fp32 [T, top_k]: optional
 *        copies of the routing (NULL to skip).
 * The fp32 combine adds the top_k expert outputs of a token in an order that
 * may vary from run to run (last-bit differences only), unless the
 * "deterministic" switch of moe_set_tuning is on. */
moe_status moe_forward(const moe_shape* shape, const void* hidden,
                       const void* router_w, const void* router_b,
                       moe_weight gate_up, moe_weight down,
                       void* out, int out_is_fp32,
                       int32_t* topk_ids_out, float* topk_w_out,
                       void* workspace, size_t workspace_bytes,
                       cudaStream_t stream);

/* Expert-parallel form of moe_forward (§2 "MoE 前向", the multi-device
 * path: a device holds a contiguous range of experts and skips tokens'
 * other experts, never multiplying them by zero).
 *   expert_start, local_experts: this device's experts [expert_start,
 *        expert_start + local_experts), 0 <= expert_start, local_experts >= 1,
 *        expert_start + local_experts <= shape->E;
 *   router_w, router_b: for all shape->E experts (routing is global);
 *   gate_up, down: banks holding only the local experts (local_experts
 *        experts in the layouts of moe_weight, local expert 0 first);
 *   out: this device's partial output, out[t] = sum over the slots j whose
 *        expert is local of w[t,j] * y (zero rows for tokens with none).
 * The partial outputs of devices whose ranges partition [0, E) add up to
 * moe_forward's output (in another order: last-bit differences); the caller
 * sums them (an all-reduce).  Other arguments and errors as for moe_forward;
 * MOE_ERR_ARG for a bad expert range. */
moe_status moe_forward_ep(const moe_shape* shape, int expert_start, int local_experts,
                          const void* hidden, const void* router_w, const void* router_b,
                          moe_weight gate_up, moe_weight down,
                          void* out, int out_is_fp32,
                          int32_t* topk_ids_out, float* topk_w_out,
                          void* workspace, size_t workspace_bytes,
                          cudaStream_t stream);

/* Size of the library-owned scratch array used by moe_forward_noalloc
 * (8 MiB per device that loads the library, held until the process exits).
 * A shape fits when moe_workspace_bytes(shape) <= this size; with
 * H = I = 2880 and top_k = 4 that is T <= 132 for E = 32 and T <= 131 for
 * E = 128. */
#define MOE_NOALLOC_SCRATCH_BYTES (8u << 20)

/* moe_forward for callers that cannot allocate device memory.  The source
 * page has no counterpart of this call: it exists for hosts that give a
 * plugin only its inputs and outputs and plan all other device memory
 * themselves (or cannot afford cudaMalloc's implicit synchronisation), so
 * they cannot provide moe_forward's workspace.
 *   Arguments as for moe_forward, minus the workspace; device_status_out
 *   (int32 [1], device memory, nullable) receives this call's device status
 *   word (MOE_DEV_* bits) when the call's work completes.
 * The scratch lives in one static device array of MOE_NOALLOC_SCRATCH_BYTES
 * inside the library; the call allocates and frees nothing.  Shapes whose
 * moe_workspace_bytes exceeds that size are rejected with MOE_ERR_WORKSPACE
 * (see MOE_NOALLOC_SCRATCH_BYTES for the token counts this admits).
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  Every call shares the one array and it keeps
 * the last call's contents; each call first clears (on its stream) the
 * status word and the completion counters that follow it, so a call that
 * gave up on the device does not leave the next one with stale counters.
 * Calls whose work overlaps on the GPU -- on different streams, or from
 * different threads -- race on the array and must be serialised by the
 * caller. */
moe_status moe_forward_noalloc(const moe_shape* shape, const void* hidden,
                               const void* router_w, const void* router_b,
                               moe_weight gate_up, moe_weight down,
                               void* out, int out_is_fp32,
                               int32_t* topk_ids_out, float* topk_w_out,
                               int32_t* device_status_out,
                               cudaStream_t stream);

/* Copies the device status word of `workspace` to *host_status.  This call
 * synchronises the calling thread with the device (cudaMemcpy).  Returns
 * MOE_ERR_DEVICE when the word is non-zero, MOE_OK otherwise. */
moe_status moe_get_device_status(const void* workspace, int32_t* host_status);

/* Zeroes the device status word and the workspace's completion counters
 * (enqueued on `stream`). */
moe_status moe_clear_device_status(void* workspace, cudaStream_t stream);

/* Stage checks, for finding the first stage of the layer that goes wrong
 * (§3 and §4 of the source page bisect their bugs this way: NaN and
 * magnitude checks after every stage behind an environment switch).  With
 * MOE_CHECK_STAGES=1 in the environment (read once per process), every
 * moe_forward / moe_forward_ep call also runs, after each stage, a check of
 * that stage's output: stage 0 the gathered activation rows (T * top_k rows
 * in the GEMM operand's format), stage 1 the GLU output h, stage 2 the
 * layer output.  Each check counts the elements that are NaN or infinite
 * and takes the largest finite magnitude; a count above zero also sets
 * MOE_DEV_NONFINITE.  This call copies the last checked call's figures to
 * the host (synchronising, like moe_get_device_status): nonfinite[3] and
 * maxabs[3], one entry per stage (0 and 0 when the checks are off). */
moe_status moe_stage_stats(const void* workspace, int32_t nonfinite[3], float maxabs[3]);

/* Phase timestamps of the last call's kernels, for timeline analysis.
 * Only the "trace" build of the library (compiled with MOE_TRACE) records
 * them; other builds return MOE_ERR_UNSUPPORTED.  Each kernel records the
 * GPU's global timer (ns) at fixed points of each of its first 512 CTAs
 * (CTA i: the linear block index).  *count receives the number of uint64
 * values written to out (cap at least 24576): the router's [512][8] (entry,
 * past the dependency wait, loads done, logits ready, routing tables
 * started, done), the permutation's [512][8] (entry, past the wait, ranks
 * done, exit), then the two GEMMs' [2][512][8] (gate_up, down: entry,
 * set-up done, weight loads issued before the wait, producer past the wait,
 * first MMA slot ready, last MMA commit, epilogue done, exit), then the
 * tensor-core attention kernel's [2][512][8] (per CTA: entry, set-up done, Q
 * landed, last scores issued, softmax done, exit; per key tile of the first
 * CTA: scores issued, previous P.V issued, softmax has the scores, row
 * maxima done, previous P.V accumulated, P written); unrecorded points hold
 * earlier values.  Synchronises with the device. */
moe_status moe_trace_read(uint64_t* out, size_t cap, size_t* count);

/* Process-wide tuning switches for tests and benchmarks:
 *   "token_tile": rows of tokens per GEMM tile, 0 = automatic, else a
 *                 multiple of 16 in [16, 256] (MXFP4 and MXFP4 x MXFP8
 *                 layers use at most 128);
 *   "pdl":        1 = launch dependent kernels with programmatic dependent
 *                 launch (default), 0 = plain stream order.  With 1 the
 *                 layer's kernels start reading weights (the router matrix,
 *                 expert weights and their scales) before the work that
 *                 precedes the call on the stream has finished: weights
 *                 written by that work need 0 here or a synchronisation
 *                 (an event the stream waits on) in between;
 *   "ksplit":     0 = split the GEMMs' K range when a small batch leaves
 *                 SMs idle (default), 1 = never split (every output then
 *                 sums its K range in one fixed order), 2..8 = split every
 *                 small-batch unit into that many parts (at most one per
 *                 two ring slots, and as many as the workspace holds);
 *   "deterministic": 1 = the down projection stores each slot's weighted
 *                 output row (fp32, T * top_k rows of H) and a last kernel
 *                 adds each token's top_k rows in slot order, so that the
 *                 output is bitwise reproducible run to run (the down
 *                 projection's K range is then never split);
 *                 moe_workspace_bytes includes those rows while the switch
 *                 is on, so query it after setting the switch (a workspace
 *                 sized without them is refused with MOE_ERR_WORKSPACE);
 *                 0 = fp32 atomics in the down projection (default);
 *   "mxfp4_f16":  MOE_W_MXFP4 layers: 1 = the GEMMs run on f16 operands
 *                 (the activations and h rounded to f16, the weights
 *                 expanded by the hardware E2M1 conversion), exact for scale
 *                 bytes in [104, 140] and activations within +-65504; a
 *                 value outside is clamped and MOE_DEV_RANGE reported
 *                 (default); 0 = bf16 operands, exact for every scale;
 *   "small_path": 1 = batches of bf16 weights with T * top_k <= 256 (and
 *                 T <= 48) skip the permutation kernel: the router's last
 *                 block computes the permutation and the gate_up GEMM copies
 *                 its token rows from `hidden` itself (default); 0 = always
 *                 the permutation kernel and the gathered activation rows;
 *   "attn_tc":    moe_attention_sinks: 0 = calls of at least 512 queries
 *                 run on the tensor-core (tcgen05) kernel, smaller ones on
 *                 the 64-row kernel with key splits (default); 1 = never the
 *                 tcgen05 kernel; 2 = always (query the workspace size
 *                 after setting this switch);
 *   "attn_poll":  softmax hand-off waits of the tcgen05 attention kernel:
 *                 0 = suspending try_wait (default), 1 = poll
 *                 (mbarrier.test_wait);
 *   "tiny_router": 1 = calls of at most 8 tokens and at most 64 experts
 *                 (at most 2 tokens: 128 experts) route in one thread block (with the permutation on the
 *                 small-batch path), and calls of 9 to 64 tokens whose
 *                 router matrix fits in shared memory beside four token
 *                 rows in a grid of 4-token blocks (default); 0 = the
 *                 multi-block router;
 *   "inject":     test faults that the device status word must report, as
 *                 a bit mask (0 = none, default): 1 = token 0's first
 *                 routed id is written as E (after it was counted), so the
 *                 permutation reports MOE_DEV_BAD_EXPERT_ID; 2 = the first
 *                 GEMM tile names an expert outside the banks, so the GEMMs
 *                 skip it and report MOE_DEV_BAD_TILE; 4 = the gate_up
 *                 GEMM's MMA issuer (bf16, FP8, MXFP4 x MXFP8 weights, no
 *                 CTA pairs) first waits on a barrier that nothing arrives
 *                 on, so the wait gives up after its ~1 s bound, the kernel
 *                 aborts and MOE_DEV_WAIT_TIMEOUT is reported.  The outputs
 *                 of such a call are not meaningful; clear the workspace
 *                 (moe_clear_device_status) before its next use;
 *   "noalloc_poison": 1 = the next moe_forward_noalloc call first fills the
 *                 status word and completion counters of its scratch with
 *                 non-zero bytes, as a failed call could leave them (a test
 *                 of the clear that follows); 0 = off (default);
 *   "pair":       0 = run the bf16 and FP8 GEMMs on CTA pairs (M = 256 MMAs
 *                 over two SMs, 256-row weight blocks) when the token box is
 *                 256 rows and, for FP8, T * top_k < 128 * E (default),
 *                 1 = never, 2 = always (bf16 and FP8 weights; the K range
 *                 is then never split).
 * Returns MOE_ERR_ARG for an unknown key or value. */
moe_status moe_set_tuning(const char* key, int value);

/* Optional per-kernel timing.  moe_profile_enable(n) with n > 0 makes the
 * next n calls of moe_route / moe_forward record a CUDA event before their
 * first kernel and after each kernel, on the call's stream (events break the
 * overlap of dependent launches, a few microseconds per kernel); n == 0
 * turns recording off.  moe_profile_read waits for the last recorded event
 * and returns, per kernel of those calls, its name (a static string) and its
 * mean duration in milliseconds; *count receives the number of kernels.
 * Not thread-safe against concurrent calls on other threads. */
moe_status moe_profile_enable(int calls);
moe_status moe_profile_read(const char** names, float* ms, int cap,
                            int* count);

/* Attention with sinks, the other half of a gpt-oss block (§1 model-
 * architecture table, "attention" row: sliding-window (128) and full layers
 * alternate; one learnable sink logit per head; GQA).
 *   Query i (position q_start + i) of head h attends to the keys j of KV
 *   head h / (Hq / Hkv) with j <= q_start + i and, when window > 0,
 *   j > q_start + i - window; scores s_j = q.k_j / sqrt(D); the sink is one
 *   more logit in the softmax's denominator that carries no value:
 *     out = sum_j exp(s_j) v_j / (exp(sink_h) + sum_j exp(s_j))
 *   (sink = -inf: plain causal / windowed softmax attention).
 * A prefill passes Tq = Tkv, q_start = 0; a decode step Tq new queries at
 * the end of a cache of Tkv keys, q_start = Tkv - Tq.
 *   q bf16 [Tq, Hq, D]; k, v bf16 [Tkv, Hkv, D] (post-rotary q and k);
 *   sinks fp32 [Hq] (4-byte aligned); out fp32 [Tq, Hq, D].
 * Supported: D == 64, Hq a multiple of Hkv, 0 <= q_start, q_start + Tq <=
 * Tkv, window >= 0 (0 = full).  Enqueued on `stream`; Tq == 0 is valid and
 * enqueues nothing (pointers may then be NULL). */
typedef struct {
    int Tq, Tkv, Hq, Hkv, D;
    int window;                /* keys per query's window, 0 = full */
    int q_start;               /* position of query 0 */
} moe_attn_shape;

/* Bytes of scratch moe_attention_sinks needs for this shape on the current
 * device (0: none; small grids -- decode -- split the keys over several
 * CTAs and merge their partial results through it; calls served by the
 * tensor-core kernel need 256 bytes, whose first word receives that call's
 * device status bits, readable with moe_get_device_status; 0 also for an
 * invalid shape). */
size_t moe_attention_workspace_bytes(const moe_attn_shape* shape);

/* workspace: device scratch of at least moe_attention_workspace_bytes
 * (NULL when that is 0), 16-byte aligned, owned by the caller; its contents
 * between calls are unspecified.  MOE_ERR_WORKSPACE when it is missing or
 * too small. */
moe_status moe_attention_sinks(const moe_attn_shape* shape, const void* q, const void* k,
                               const void* v, const float* sinks, float* out,
                               void* workspace, size_t workspace_bytes,
                               cudaStream_t stream);

/* Static description of a status code. */
const char* moe_status_str(moe_status status);

#ifdef __cplusplus
}
#endif

#endif /* GPT_OSS_MOE_H */
