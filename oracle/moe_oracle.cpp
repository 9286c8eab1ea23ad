// CPU oracle of the gpt-oss mixture-of-experts layer forward.
//
// TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
// cpu_baseline / reference legs of bench.py may load or call this library.
// It shares no code, header, table or helper with the CUDA library in
// gpt_oss_moe_gb300/; the two meet only in the seeded input buffers.
//
// It is plain and slow on purpose: every dot product is one sequential fp32
// sum in ascending index order, with no blocking, fusion or reordering, so a
// reader can check each step against the source by eye.  Build with
// -ffp-contract=off so that no multiply-add is contracted (the result is then
// the same on every host).  OpenMP only spreads independent output elements
// over threads; each element is summed by one thread in a fixed order, so the
// result does not depend on the thread count.
//
// Source: xserv docs/19-gpt-oss-moe.md, "Phase 19: gpt-oss-20b -- MoE 模型支持
// 与两次 CUDA 调试实战":
//   * §1 model-architecture table, "MoE" row: 32 experts, top-4, expert
//     intermediate 2880; the router is a plain Linear [2880 -> 32] with bias.
//   * §1 table, "激活" (activation) row: clamped GLU on interleaved columns,
//     gate = gu[::2], up = gu[1::2], gate <= 7, up in [-7, 7],
//     glu = gate * sigmoid(1.702 * gate), h = (up + 1) * glu.
//   * §2 "MoE 前向" (MoE forward): router GEMV -> topk_softmax -> replicate
//     -> batched GEMM gate_up -> bias -> GLU -> batched GEMM down -> bias ->
//     weighted_sum over the top-4 only; non-selected experts are skipped,
//     not multiplied by zero.
//   * §5 "量化" (quantization): MXFP4 = E2M1 values with one UE8M0 scale per
//     32 elements; FP8 W8A8 = E4M3 weights with one scalar scale per expert,
//     E4M3 activations, the scales applied after the product.
//
// Readings where the page leaves a step open (each is listed in the design
// notes of the repository):
//   * router logits stay fp32 (not rounded to bf16);
//   * top-k order is descending logit, equal logits -> lower expert index;
//   * the softmax runs over the k selected logits (max-subtracted), which is
//     the same as a full softmax renormalised over the selected ones;
//   * bias is added before the clamp (gate_up) and before the weighting
//     (down), following the step order of §2;
//   * gate has an upper clamp only; up is clamped on both sides; both clamps
//     come before the sigmoid and the product;
//   * h stays fp32 inside the oracle;
//   * MXFP4: element 2i of a row is the low nibble of byte i, element 2i+1
//     the high nibble; the 32-element scale blocks run along the input (K)
//     dimension of each output row; value = e2m1(code) * 2^(scale - 127).
//   * the permutation sorts assignments a = t*k + j by (expert, a) ascending.
//   * FP8 W8A8: weight = e4m3(code) * scale[e] (one fp32 scale per expert and
//     matrix); each token's activations are quantised with their own scale,
//     s = max|x| / 448 (1 when the row is all zero): code = e4m3 nearest to
//     x * (448 / max|x|), ties to the even code, magnitudes beyond 448
//     saturating to 448; h is quantised with the fixed scale 1/8 (the GLU
//     clamps keep h in [-42, 56), so h * 8 never exceeds 448).  A gate_up row
//     is (sum_k e4m3(w) * e4m3(xq)) * (scale[e] * s) + bias; a down row is
//     (sum_j e4m3(w) * e4m3(hq)) * (scale[e] * 1/8) + bias.
//   * MXFP4 weights with MXFP8 activations (the native block-scaled form of
//     §5's MXFP4): weights as MXFP4 above; each token's activations are cut
//     into blocks of 32 consecutive elements, each block quantised by the
//     OCP Microscaling (MX) v1.0 conversion rule: shared scale
//     X = 2^(floor(log2 max|x|) - 8) (8 = the largest exponent of E4M3),
//     clamped to [2^-127, 2^127] (2^-127 for an all-zero block), elements =
//     e4m3 nearest to x / X, ties to even, saturating at 448.  h is E4M3 with
//     every block scale 1/8, as in the FP8 reading.  A gate_up row is
//     sum_k w(k) * e4m3(xq_k) * X(k) + bias, a down row
//     sum_j w(j) * e4m3(hq_j) / 8 + bias, both in fp32.
//
// Parity pins (tests/test_oracle_pins.py): brute force over all k-subsets,
// closed-form special cases of top-k/softmax, permutation closed forms,
// GLU identities (odd part equals the input, logit of the gate equals
// 1.702*gate, clamp equivalences, range), an independent fp64 brute force of
// the whole layer on E=4/top-2/H=I=64, routed == dense bit-exactly, and the
// exact E2M1/E8M0 table.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

#ifdef _OPENMP
#include <omp.h>
#endif

#include "moe_oracle.h"

namespace {

// Exact widening of a bf16 bit pattern to fp32.
inline float bf16_value(uint16_t b) {
    uint32_t u = static_cast<uint32_t>(b) << 16;
    float f;
    std::memcpy(&f, &u, sizeof f);
    return f;
}

// E2M1: sign bit, 2 exponent bits, 1 mantissa bit.  Magnitude codes 0..7
// decode to 0, 0.5, 1, 1.5, 2, 3, 4, 6 (exponent bias 1; code 1 is the
// subnormal 0.5).  Computed from the bit fields, not from a table.
inline float e2m1_value(unsigned code) {
    unsigned s = (code >> 3) & 1u, ex = (code >> 1) & 3u, m = code & 1u;
    float mag = (ex == 0) ? 0.5f * static_cast<float>(m)
                          : std::ldexp(1.0f + 0.5f * static_cast<float>(m),
                                       static_cast<int>(ex) - 1);
    return s ? -mag : mag;
}

// E4M3 (OCP FP8, "fn" variant): sign, 4 exponent bits (bias 7), 3 mantissa
// bits; exponent field 0 holds the subnormals m * 2^-9; the all-ones code
// (exponent 15, mantissa 7) is NaN; the largest finite magnitude is 448.
inline float e4m3_value(uint8_t code) {
    const unsigned s = code >> 7, ex = (code >> 3) & 0xFu, m = code & 7u;
    if (ex == 15 && m == 7) return std::nanf("");
    const float mag = (ex == 0) ? std::ldexp(static_cast<float>(m), -9)
                                : std::ldexp(1.0f + static_cast<float>(m) / 8.0f,
                                             static_cast<int>(ex) - 7);
    return s ? -mag : mag;
}

// The e4m3 code nearest to v: a search over the 127 non-negative finite
// codes (their values increase with the code), ties to the even code; a
// magnitude beyond 448 gives 448 (saturation); the sign is kept.
inline uint8_t e4m3_round(float v) {
    if (std::isnan(v)) return 0x7F;
    const uint8_t sign = std::signbit(v) ? 0x80 : 0x00;
    const float a = std::fabs(v);
    int best = 0;
    float best_d = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {
        const float d = std::fabs(e4m3_value(static_cast<uint8_t>(c)) - a);
        if (d < best_d || (d == best_d && (c & 1) == 0)) {
            best = c;
            best_d = d;
        }
    }
    return static_cast<uint8_t>(sign | best);
}

// One token's activations to e4m3 with their own scale (FP8 W8A8 reading).
inline float fp8_quantize_row(const uint16_t* x, int n, uint8_t* codes) {
    float amax = 0.0f;
    for (int i = 0; i < n; ++i) amax = std::fmax(amax, std::fabs(bf16_value(x[i])));
    const float inv = amax > 0.0f ? 448.0f / amax : 1.0f;
    for (int i = 0; i < n; ++i) codes[i] = e4m3_round(bf16_value(x[i]) * inv);
    return amax > 0.0f ? amax / 448.0f : 1.0f;
}

// One block of 32 activations to MXFP8 (OCP MX v1.0 conversion: shared
// exponent floor(log2 max|x|) minus E4M3's largest exponent 8, clamped to
// the UE8M0 range; elements rounded to e4m3 after division by the scale).
// Returns the UE8M0 byte of the block's scale.
inline uint8_t mx_quantize_block(const uint16_t* x, uint8_t* codes) {
    float amax = 0.0f;
    for (int i = 0; i < 32; ++i) amax = std::fmax(amax, std::fabs(bf16_value(x[i])));
    int shared = -127;
    if (amax > 0.0f) {
        int ex = 0;
        std::frexp(amax, &ex);            // amax = m * 2^ex, m in [0.5, 1)
        shared = (ex - 1) - 8;            // floor(log2 amax) - 8
        if (shared < -127) shared = -127;
        if (shared > 127) shared = 127;
    }
    for (int i = 0; i < 32; ++i)
        codes[i] = e4m3_round(std::ldexp(bf16_value(x[i]), -shared));
    return static_cast<uint8_t>(shared + 127);
}

// UE8M0: an unsigned power-of-two exponent with bias 127.
inline float e8m0_value(uint8_t s) {
    return std::ldexp(1.0f, static_cast<int>(s) - 127);
}

// Element (row, col) of one expert's weight matrix with `cols` inputs.
inline float weight_at(int wfmt, const void* w, const uint8_t* s, size_t row,
                       size_t col, size_t cols) {
    if (wfmt == 0) {
        return bf16_value(static_cast<const uint16_t*>(w)[row * cols + col]);
    }
    if (wfmt == 2) {   // FP8: the code's value; the expert scale comes later
        return e4m3_value(static_cast<const uint8_t*>(w)[row * cols + col]);
    }
    const uint8_t* codes = static_cast<const uint8_t*>(w);
    uint8_t byte = codes[row * (cols / 2) + col / 2];
    unsigned code = (col & 1) ? (byte >> 4) : (byte & 0xFu);
    return e2m1_value(code) * e8m0_value(s[row * (cols / 32) + col / 32]);
}

inline float sigmoid(float v) { return 1.0f / (1.0f + std::exp(-v)); }

// Clamped interleaved GLU of one (gate, up) pair (§1 table, activation row).
inline float glu(float gate, float up) {
    if (gate > 7.0f) gate = 7.0f;
    if (up > 7.0f) up = 7.0f;
    if (up < -7.0f) up = -7.0f;
    float g = gate * sigmoid(1.702f * gate);
    return (up + 1.0f) * g;
}

// Router logit of token t for expert e: sequential fp32 dot product + bias.
float router_logit(const oracle_layer* L, int t, int e) {
    const uint16_t* xr = L->x + static_cast<size_t>(t) * L->H;
    const uint16_t* wr = L->wr + static_cast<size_t>(e) * L->H;
    float acc = 0.0f;
    for (int h = 0; h < L->H; ++h) acc += bf16_value(xr[h]) * bf16_value(wr[h]);
    return acc + bf16_value(L->br[e]);
}

// Top-k by (logit descending, index ascending), then softmax over the k.
void topk_softmax_row(const float* logit, int E, int k, int32_t* ids,
                      float* w) {
    std::vector<char> taken(E, 0);
    for (int j = 0; j < k; ++j) {
        int best = -1;
        for (int e = 0; e < E; ++e) {
            if (taken[e]) continue;
            if (best < 0 || logit[e] > logit[best]) best = e;  // strict: lower index wins ties
        }
        taken[best] = 1;
        ids[j] = best;
    }
    const float m = logit[ids[0]];
    float denom = 0.0f;
    std::vector<float> ex(k);
    for (int j = 0; j < k; ++j) {
        ex[j] = std::exp(logit[ids[j]] - m);
        denom += ex[j];
    }
    for (int j = 0; j < k; ++j) w[j] = ex[j] / denom;
}

// FP8 W8A8 form of expert_ffn (the readings above): quantised token row,
// code products summed in fp32, then the scales, then the bias.
void expert_ffn_fp8(const oracle_layer* L, int e, const uint16_t* xr, float* h_out,
                    float* y_out) {
    const int H = L->H, I = L->I;
    const size_t n_gu = static_cast<size_t>(2) * I;
    std::vector<uint8_t> xq(H);
    const float xs = fp8_quantize_row(xr, H, xq.data());
    std::vector<float> xv(H);
    for (int k = 0; k < H; ++k) xv[k] = e4m3_value(xq[k]);
    const float* sw_gu = static_cast<const float*>(L->s_gu);
    const float* sw_d = static_cast<const float*>(L->s_d);
    const float gu_scale = sw_gu[e] * xs;
    const size_t gu_row0 = static_cast<size_t>(e) * n_gu;
    std::vector<float> gu(n_gu);
    for (size_t n = 0; n < n_gu; ++n) {
        float acc = 0.0f;
        for (int k = 0; k < H; ++k)
            acc += weight_at(2, L->w_gu, nullptr, gu_row0 + n, k, H) * xv[k];
        gu[n] = acc * gu_scale + bf16_value(L->b_gu[gu_row0 + n]);
    }
    std::vector<float> h(I), hv(I);
    for (int j = 0; j < I; ++j) {
        const float gate = gu[2 * j], up = gu[2 * j + 1];
        h[j] = glu(gate, up);
        hv[j] = e4m3_value(e4m3_round(h[j] * 8.0f));
    }
    if (h_out) std::memcpy(h_out, h.data(), sizeof(float) * I);
    const float d_scale = sw_d[e] * 0.125f;
    const size_t d_row0 = static_cast<size_t>(e) * H;
    for (int n = 0; n < H; ++n) {
        float acc = 0.0f;
        for (int j = 0; j < I; ++j)
            acc += weight_at(2, L->w_d, nullptr, d_row0 + n, j, I) * hv[j];
        y_out[n] = acc * d_scale + bf16_value(L->b_d[d_row0 + n]);
    }
}

// MXFP4-weight / MXFP8-activation form of expert_ffn (the readings above).
void expert_ffn_mx(const oracle_layer* L, int e, const uint16_t* xr, float* h_out,
                   float* y_out) {
    const int H = L->H, I = L->I;
    const size_t n_gu = static_cast<size_t>(2) * I;
    std::vector<uint8_t> xq(H);
    std::vector<float> xv(H);
    for (int b = 0; b < H / 32; ++b) {
        const uint8_t sx = mx_quantize_block(xr + 32 * b, xq.data() + 32 * b);
        for (int i = 0; i < 32; ++i)
            xv[32 * b + i] = e4m3_value(xq[32 * b + i]) * e8m0_value(sx);
    }
    const uint8_t* s_gu = static_cast<const uint8_t*>(L->s_gu);
    const uint8_t* s_d = static_cast<const uint8_t*>(L->s_d);
    const size_t gu_row0 = static_cast<size_t>(e) * n_gu;
    const uint16_t* bias_gu = L->b_gu + gu_row0;
    std::vector<float> gu(n_gu);
    for (size_t n = 0; n < n_gu; ++n) {
        float acc = 0.0f;
        for (int k = 0; k < H; ++k)
            acc += weight_at(1, L->w_gu, s_gu, gu_row0 + n, k, H) * xv[k];
        gu[n] = acc + bf16_value(bias_gu[n]);
    }
    std::vector<float> h(I), hv(I);
    for (int j = 0; j < I; ++j) {
        const float gate = gu[2 * j], up = gu[2 * j + 1];
        h[j] = glu(gate, up);
        hv[j] = e4m3_value(e4m3_round(h[j] * 8.0f)) * 0.125f;
    }
    if (h_out) std::memcpy(h_out, h.data(), sizeof(float) * I);
    const size_t d_row0 = static_cast<size_t>(e) * H;
    const uint16_t* bias_d = L->b_d + d_row0;
    for (int n = 0; n < H; ++n) {
        float acc = 0.0f;
        for (int j = 0; j < I; ++j)
            acc += weight_at(1, L->w_d, s_d, d_row0 + n, j, I) * hv[j];
        y_out[n] = acc + bf16_value(bias_d[n]);
    }
}

// One expert applied to one token: gate_up + bias -> GLU -> down + bias.
// h_out may be null; y_out receives H values.
void expert_ffn(const oracle_layer* L, int e, int t, float* h_out,
                float* y_out) {
    const int H = L->H, I = L->I;
    const size_t n_gu = static_cast<size_t>(2) * I;
    const uint16_t* xr = L->x + static_cast<size_t>(t) * H;
    std::vector<float> xf(H);
    for (int k = 0; k < H; ++k) xf[k] = bf16_value(xr[k]);
    if (L->wfmt == 2) {
        expert_ffn_fp8(L, e, xr, h_out, y_out);
        return;
    }
    if (L->wfmt == 3) {
        expert_ffn_mx(L, e, xr, h_out, y_out);
        return;
    }

    // gate_up rows of expert e, then the per-pair GLU.
    const size_t gu_row0 = static_cast<size_t>(e) * n_gu;
    const uint8_t* s_gu = static_cast<const uint8_t*>(L->s_gu);
    std::vector<float> gu(n_gu);
    for (size_t n = 0; n < n_gu; ++n) {
        float acc = 0.0f;
        for (int k = 0; k < H; ++k)
            acc += weight_at(L->wfmt, L->w_gu, s_gu, gu_row0 + n, k, H) * xf[k];
        gu[n] = acc + bf16_value(L->b_gu[gu_row0 + n]);
    }
    std::vector<float> h(I);
    for (int j = 0; j < I; ++j) h[j] = glu(gu[2 * j], gu[2 * j + 1]);
    if (h_out) std::memcpy(h_out, h.data(), sizeof(float) * I);

    // down rows of expert e.
    const uint8_t* s_d = static_cast<const uint8_t*>(L->s_d);
    const size_t d_row0 = static_cast<size_t>(e) * H;
    for (int n = 0; n < H; ++n) {
        float acc = 0.0f;
        for (int j = 0; j < I; ++j)
            acc += weight_at(L->wfmt, L->w_d, s_d, d_row0 + n, j, I) * h[j];
        y_out[n] = acc + bf16_value(L->b_d[d_row0 + n]);
    }
}

void set_threads(int threads) {
#ifdef _OPENMP
    if (threads > 0) omp_set_num_threads(threads);
#else
    (void)threads;
#endif
}

}  // namespace

extern "C" {

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

float oracle_glu(float gate, float up) { return glu(gate, up); }

float oracle_e2m1(unsigned code) { return e2m1_value(code & 0xFu); }

float oracle_e8m0(uint8_t s) { return e8m0_value(s); }

float oracle_e4m3(uint8_t code) { return e4m3_value(code); }

uint8_t oracle_e4m3_round(float v) { return e4m3_round(v); }

// One token row of n bf16 activations to e4m3 codes; *scale receives its
// scale (max|x| / 448, or 1 for an all-zero row).
int oracle_fp8_quantize_row(const uint16_t* x, int n, uint8_t* codes, float* scale) {
    *scale = fp8_quantize_row(x, n, codes);
    return 0;
}

// One token row of n bf16 activations (n a multiple of 32) to MXFP8: codes
// [n] e4m3 and scales [n / 32] UE8M0 bytes.
int oracle_mx_quantize_row(const uint16_t* x, int n, uint8_t* codes, uint8_t* scales) {
    if (n % 32) return -1;
    for (int b = 0; b < n / 32; ++b) scales[b] = mx_quantize_block(x + 32 * b, codes + 32 * b);
    return 0;
}

// logits[T, E] (fp32).
int oracle_router_logits(const oracle_layer* L, float* logits, int threads) {
    set_threads(threads);
    const long long n = static_cast<long long>(L->T) * L->E;
#pragma omp parallel for schedule(static)
    for (long long i = 0; i < n; ++i)
        logits[i] = router_logit(L, static_cast<int>(i / L->E),
                                 static_cast<int>(i % L->E));
    return 0;
}

// ids[T, k] int32 and w[T, k] fp32 from logits[T, E].
int oracle_topk_softmax(const float* logits, int T, int E, int k, int32_t* ids,
                        float* w) {
    if (k < 1 || k > E) return -1;
    for (int t = 0; t < T; ++t)
        topk_softmax_row(logits + static_cast<size_t>(t) * E, E, k,
                         ids + static_cast<size_t>(t) * k,
                         w + static_cast<size_t>(t) * k);
    return 0;
}

// Stable counting sort of the T*k assignments a = t*k + j by expert id.
// offsets[E+1]: exclusive scan of the per-expert counts; sorted_assign[r] is
// the assignment placed at row r; assign_row[a] is the row of assignment a.
// Returns -1 if an id lies outside [0, E).
int oracle_permute(const int32_t* ids, int T, int k, int E, int32_t* offsets,
                   int32_t* sorted_assign, int32_t* assign_row) {
    const int n = T * k;
    std::vector<int32_t> count(E, 0);
    for (int a = 0; a < n; ++a) {
        if (ids[a] < 0 || ids[a] >= E) return -1;
        count[ids[a]] += 1;
    }
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + count[e];
    std::vector<int32_t> next(offsets, offsets + E);
    for (int a = 0; a < n; ++a) {
        const int r = next[ids[a]]++;
        sorted_assign[r] = a;
        assign_row[a] = r;
    }
    return 0;
}

// One expert on one token (for tests): h[I] (nullable) and y[H].
int oracle_expert_ffn(const oracle_layer* L, int e, int t, float* h, float* y) {
    expert_ffn(L, e, t, h, y);
    return 0;
}

// Routed forward of the tokens listed in `tokens` (n of them; all T tokens
// when tokens is null).  ids[n, k], w[n, k], logits[n, E] (nullable) and
// out[n, H] (fp32) are indexed by list position.
int oracle_forward_tokens(const oracle_layer* L, const int32_t* tokens, int n,
                          int32_t* ids, float* w, float* logits, float* out,
                          int threads) {
    set_threads(threads);
    const int H = L->H, E = L->E, k = L->top_k;
    if (k < 1 || k > E) return -1;
    if (!tokens) n = L->T;
    std::vector<float> lg(static_cast<size_t>(n) * E);
    const long long nl = static_cast<long long>(n) * E;
#pragma omp parallel for schedule(static)
    for (long long i = 0; i < nl; ++i) {
        const int p = static_cast<int>(i / E), e = static_cast<int>(i % E);
        const int t = tokens ? tokens[p] : p;
        lg[i] = router_logit(L, t, e);
    }
    for (int p = 0; p < n; ++p)
        topk_softmax_row(lg.data() + static_cast<size_t>(p) * E, E, k,
                         ids + static_cast<size_t>(p) * k,
                         w + static_cast<size_t>(p) * k);
    if (logits) std::memcpy(logits, lg.data(), sizeof(float) * lg.size());

    // Expert outputs of every (token, slot) pair, then the weighted sum in
    // slot order j = 0..k-1.
    std::vector<float> y(static_cast<size_t>(n) * k * H);
    const long long np = static_cast<long long>(n) * k;
#pragma omp parallel for schedule(dynamic, 1)
    for (long long q = 0; q < np; ++q) {
        const int p = static_cast<int>(q / k);
        const int t = tokens ? tokens[p] : p;
        expert_ffn(L, ids[q], t, nullptr, y.data() + static_cast<size_t>(q) * H);
    }
    for (int p = 0; p < n; ++p) {
        for (int c = 0; c < H; ++c) {
            float acc = 0.0f;
            for (int j = 0; j < k; ++j)
                acc += w[static_cast<size_t>(p) * k + j] *
                       y[(static_cast<size_t>(p) * k + j) * H + c];
            out[static_cast<size_t>(p) * H + c] = acc;
        }
    }
    return 0;
}

// Routed forward of all T tokens.
int oracle_moe_forward(const oracle_layer* L, int32_t* ids, float* w,
                       float* out, int threads) {
    return oracle_forward_tokens(L, nullptr, L->T, ids, w, nullptr, out,
                                 threads);
}

// Expert-parallel form of §2 (the page's multi-device path: a device holds
// the experts [ex_lo, ex_lo + ex_n) and skips tokens' other experts): the
// routing over all E experts as above, then out[p] = sum, in slot order, of
// w * y over the slots whose expert is local.  The devices' partial outputs
// of a partition of [0, E) add up to the full output.  L's weight banks hold
// all E experts (the expert index stays global here).  tokens may be null
// (all T tokens).
int oracle_moe_forward_ep(const oracle_layer* L, int ex_lo, int ex_n, const int32_t* tokens,
                          int n, float* out, int threads) {
    const int H = L->H, E = L->E, k = L->top_k;
    if (ex_lo < 0 || ex_n < 0 || ex_lo + ex_n > E) return -1;
    if (!tokens) n = L->T;
    std::vector<int32_t> ids(static_cast<size_t>(n) * k);
    std::vector<float> w(static_cast<size_t>(n) * k);
    set_threads(threads);
    std::vector<float> lg(static_cast<size_t>(n) * E);
    const long long nl = static_cast<long long>(n) * E;
#pragma omp parallel for schedule(static)
    for (long long i = 0; i < nl; ++i) {
        const int p = static_cast<int>(i / E), e = static_cast<int>(i % E);
        lg[i] = router_logit(L, tokens ? tokens[p] : p, e);
    }
    for (int p = 0; p < n; ++p)
        topk_softmax_row(lg.data() + static_cast<size_t>(p) * E, E, k,
                         ids.data() + static_cast<size_t>(p) * k,
                         w.data() + static_cast<size_t>(p) * k);
    std::vector<float> y(static_cast<size_t>(n) * k * H, 0.0f);
    const long long np = static_cast<long long>(n) * k;
#pragma omp parallel for schedule(dynamic, 1)
    for (long long q = 0; q < np; ++q) {
        const int e = ids[q];
        if (e < ex_lo || e >= ex_lo + ex_n) continue;      // not this device's expert
        const int p = static_cast<int>(q / k);
        expert_ffn(L, e, tokens ? tokens[p] : p, nullptr, y.data() + static_cast<size_t>(q) * H);
    }
    for (int p = 0; p < n; ++p) {
        for (int c = 0; c < H; ++c) {
            float acc = 0.0f;
            for (int j = 0; j < k; ++j) {    // other devices' slots hold y = 0
                const size_t q = static_cast<size_t>(p) * k + j;
                acc += w[q] * y[q * H + c];
            }
            out[static_cast<size_t>(p) * H + c] = acc;
        }
    }
    return 0;
}

// Dense form of §2: every token goes through every expert, then the weighted
// sum keeps the k selected ones only (a skip, never a multiply by zero).
int oracle_moe_forward_dense(const oracle_layer* L, int32_t* ids, float* w,
                             float* out, int threads) {
    set_threads(threads);
    const int T = L->T, H = L->H, E = L->E, k = L->top_k;
    if (k < 1 || k > E) return -1;
    std::vector<float> lg(static_cast<size_t>(T) * E);
    oracle_router_logits(L, lg.data(), threads);
    oracle_topk_softmax(lg.data(), T, E, k, ids, w);
    std::vector<float> y(static_cast<size_t>(T) * E * H);
    const long long np = static_cast<long long>(T) * E;
#pragma omp parallel for schedule(dynamic, 1)
    for (long long q = 0; q < np; ++q)
        expert_ffn(L, static_cast<int>(q % E), static_cast<int>(q / E), nullptr,
                   y.data() + static_cast<size_t>(q) * H);
    for (int t = 0; t < T; ++t) {
        for (int c = 0; c < H; ++c) {
            float acc = 0.0f;
            for (int j = 0; j < k; ++j) {
                const int e = ids[static_cast<size_t>(t) * k + j];
                acc += w[static_cast<size_t>(t) * k + j] *
                       y[(static_cast<size_t>(t) * E + e) * H + c];
            }
            out[static_cast<size_t>(t) * H + c] = acc;
        }
    }
    return 0;
}

// Attention with sinks (§1 model-architecture table, "attention" row:
// alternating sliding-window (128) / full layers, one learnable sink scalar
// per head; §3 on the empty-tile case).  Readings: GQA head h reads KV head
// h / (Hq / Hkv); scores are q.k / sqrt(D); query i sits at position
// q_start + i and sees key j when j <= q_start + i and, with a window W > 0,
// j > q_start + i - W (W keys including its own); the sink is one more logit
// in the softmax's denominator that carries no value:
//   out = sum_j exp(s_j - m) v_j / (exp(sink - m) + sum_j exp(s_j - m)),
// m = max(sink, s_j).  fp64 throughout (the page fixes no precision).
// q [Tq, Hq, D], k and v [Tkv, Hkv, D] bf16; sinks [Hq] fp32 (-inf: none);
// out [Tq, Hq, D] fp32.
int oracle_attention_sinks(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                           const float* sinks, int Tq, int Tkv, int Hq, int Hkv, int D,
                           int window, int q_start, float* out, int threads) {
    if (Hkv < 1 || Hq % Hkv || Tq < 0 || q_start < 0 || q_start + Tq > Tkv || window < 0)
        return -1;
    set_threads(threads);
    const int rep = Hq / Hkv;
    const double scale = 1.0 / std::sqrt(static_cast<double>(D));
    const long long n = static_cast<long long>(Tq) * Hq;
#pragma omp parallel for schedule(dynamic, 4)
    for (long long r = 0; r < n; ++r) {
        const int i = static_cast<int>(r / Hq), h = static_cast<int>(r % Hq);
        const int hk = h / rep;
        const int pos = q_start + i;
        const int j0 = window > 0 ? std::max(0, pos - window + 1) : 0;
        const uint16_t* qr = q + (static_cast<size_t>(i) * Hq + h) * D;
        std::vector<double> sc(static_cast<size_t>(pos - j0 + 1));
        double m = sinks[h];
        for (int j = j0; j <= pos; ++j) {
            const uint16_t* kr = k + (static_cast<size_t>(j) * Hkv + hk) * D;
            double acc = 0.0;
            for (int d = 0; d < D; ++d)
                acc += static_cast<double>(bf16_value(qr[d])) * bf16_value(kr[d]);
            sc[j - j0] = acc * scale;
            m = std::max(m, sc[j - j0]);
        }
        double denom = std::isinf(sinks[h]) && sinks[h] < 0 ? 0.0 : std::exp(sinks[h] - m);
        for (int j = j0; j <= pos; ++j) denom += std::exp(sc[j - j0] - m);
        float* o = out + (static_cast<size_t>(i) * Hq + h) * D;
        for (int d = 0; d < D; ++d) {
            double acc = 0.0;
            for (int j = j0; j <= pos; ++j)
                acc += std::exp(sc[j - j0] - m) *
                       bf16_value(v[(static_cast<size_t>(j) * Hkv + hk) * D + d]);
            o[d] = static_cast<float>(acc / denom);
        }
    }
    return 0;
}

// Dequantise MXFP4 rows: out[rows, K] fp32 from codes[rows, K/2] and
// scales[rows, K/32].
int oracle_dequant_mxfp4(const uint8_t* codes, const uint8_t* scales, int rows,
                         int K, float* out) {
    if (K % 32) return -1;
    for (long long r = 0; r < rows; ++r)
        for (int c = 0; c < K; ++c)
            out[r * K + c] = weight_at(1, codes, scales, static_cast<size_t>(r),
                                       static_cast<size_t>(c),
                                       static_cast<size_t>(K));
    return 0;
}

}  // extern "C"
