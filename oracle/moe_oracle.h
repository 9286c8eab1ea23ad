/* CPU oracle of the gpt-oss MoE layer forward -- TEST INFRASTRUCTURE ONLY.
 *
 * Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline/reference
 * legs may load or call it.  It shares no code with the CUDA library.
 * See moe_oracle.cpp for the definitions it follows and the readings taken.
 */
#ifndef GPT_OSS_MOE_ORACLE_H
#define GPT_OSS_MOE_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
    int T, H, I, E, top_k, wfmt;  /* 0 = bf16, 1 = MXFP4, 2 = FP8 W8A8,
                                     3 = MXFP4 weights, MXFP8 activations */
    const uint16_t* x;            /* [T, H] bf16 */
    const uint16_t* wr;           /* [E, H] bf16 */
    const uint16_t* br;           /* [E] bf16 */
    const void* w_gu;             /* bf16 [E, 2I, H] | u8 [E, 2I, H/2] | e4m3 [E, 2I, H] */
    const void* s_gu;             /* u8 [E, 2I, H/32] (MXFP4, 3) | fp32 [E] (FP8) */
    const uint16_t* b_gu;         /* [E, 2I] bf16 */
    const void* w_d;              /* bf16 [E, H, I] | u8 [E, H, I/2] | e4m3 [E, H, I] */
    const void* s_d;              /* u8 [E, H, I/32] (MXFP4, 3) | fp32 [E] (FP8) */
    const uint16_t* b_d;          /* [E, H] bf16 */
} oracle_layer;

int oracle_max_threads(void);
float oracle_glu(float gate, float up);
float oracle_e2m1(unsigned code);
float oracle_e8m0(uint8_t s);
float oracle_e4m3(uint8_t code);
uint8_t oracle_e4m3_round(float v);
int oracle_fp8_quantize_row(const uint16_t* x, int n, uint8_t* codes, float* scale);
int oracle_mx_quantize_row(const uint16_t* x, int n, uint8_t* codes, uint8_t* scales);
int oracle_router_logits(const oracle_layer* L, float* logits, int threads);
int oracle_topk_softmax(const float* logits, int T, int E, int k, int32_t* ids,
                        float* w);
int oracle_permute(const int32_t* ids, int T, int k, int E, int32_t* offsets,
                   int32_t* sorted_assign, int32_t* assign_row);
int oracle_expert_ffn(const oracle_layer* L, int e, int t, float* h, float* y);
int oracle_forward_tokens(const oracle_layer* L, const int32_t* tokens, int n,
                          int32_t* ids, float* w, float* logits, float* out,
                          int threads);
int oracle_moe_forward(const oracle_layer* L, int32_t* ids, float* w,
                       float* out, int threads);
int oracle_moe_forward_ep(const oracle_layer* L, int ex_lo, int ex_n, const int32_t* tokens,
                          int n, float* out, int threads);
int oracle_moe_forward_dense(const oracle_layer* L, int32_t* ids, float* w,
                             float* out, int threads);
int oracle_attention_sinks(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                           const float* sinks, int Tq, int Tkv, int Hq, int Hkv, int D,
                           int window, int q_start, float* out, int threads);
int oracle_dequant_mxfp4(const uint8_t* codes, const uint8_t* scales, int rows,
                         int K, float* out);

#ifdef __cplusplus
}
#endif

#endif
