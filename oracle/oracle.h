/*
 * CPU oracle for the routed-expert MoE FFN layer -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 restatement of what the layer computes.  Only the test
 * suite, the smoke check and the benchmark's CPU-baseline leg load it; the
 * product library never does.  It shares no code, header, table or constant
 * with the CUDA library.
 *
 * Sources (web pages; no code was published with them):
 *  [KT]   "KTransformers deep dive" (chenxutan.com/d/5425.html), section 1.2:
 *         256 routed experts plus 1 shared expert; a router sends each token
 *         to 8 of them.  Section 2.2: tokens hitting the same expert are
 *         batched (grouping GEMV into GEMM).
 *  [HYB]  "CPU-GPU hybrid inference (OSDI'26)" article (xingyun.xin):
 *         - SmallEP section / Fig. 5: standard expert parallelism = gating and
 *           sorting, dispatch, expert compute, combine, weighted reduction.
 *         - "Native FP8 GEMV" section / Fig. 9-10: E4M3FN weights, one
 *           inverse-scale per 128-element input block, partial dot products
 *           of a block accumulated first and the block scale applied once.
 *         - "CPU fine-grained parallelism" section: gate and up run side by
 *           side; their outputs go through the activation and an elementwise
 *           product before the down projection.
 *
 * Readings where the pages are silent:
 *  - scoring: softmax over the fp32 logits (+ optional per-expert bias),
 *    top-k with ties to the lower expert index, weights renormalised over
 *    the selected k; activation SiLU; shared expert weight 1; no residual.
 *  - activations are quantised to E4M3FN per token per 128 channels with
 *    s = amax/448 (s = 1 for an all-zero group), q = E4M3(fp32(v/s)); the
 *    intermediate h is rounded to fp32 first.
 *  - gate weights follow one fp32 operation sequence (see oracle_exp32 and
 *    oracle_route_from_logits) so that they are reproducible bit for bit.
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
    int32_t H, I, E, k;          /* hidden, expert inter, routed experts, top-k */
    int32_t n_shared, SI;        /* shared experts (0 or 1) and their inter     */
    const uint8_t *w_gate, *w_up;  /* [E][I][H] E4M3FN codes                   */
    const uint8_t *w_down;         /* [E][H][I]                                */
    const float *s_gate, *s_up;    /* [E][I/128][H/128] fp32 multipliers       */
    const float *s_down;           /* [E][H/128][I/128]                        */
    const uint8_t *sh_gate, *sh_up, *sh_down;      /* same with E = 1, I = SI  */
    const float *sh_s_gate, *sh_s_up, *sh_s_down;
} oracle_layer;

double  oracle_e4m3_decode(uint8_t code);
uint8_t oracle_e4m3_encode(float v);
float   oracle_exp32(float x);
void    oracle_quant_1x128(const float* v, int32_t n, uint8_t* q, float* s);
void    oracle_logits(const uint16_t* x_bf16, const float* router_w, const float* bias,
                      int32_t T, int32_t H, int32_t E, int32_t n_threads, float* logits);
void    oracle_route_from_logits(const float* logits, int32_t T, int32_t E, int32_t k,
                                 int32_t* ids, float* w, int32_t* offsets,
                                 int32_t* sorted_token, int32_t* inv_row);
int     oracle_forward(const oracle_layer* L, const uint16_t* x_bf16, int32_t T,
                       const int32_t* ids, const float* w,
                       const int32_t* rows, int32_t n_rows, int32_t exact_act,
                       int32_t n_threads, uint16_t* y_bf16, double* y64);
int     oracle_forward_ex(const oracle_layer* L, const uint16_t* x_bf16, int32_t T,
                          const int32_t* ids, const float* w,
                          const int32_t* rows, int32_t n_rows, int32_t exact_act,
                          const uint8_t* hq_in, const float* sh_in,
                          float* h32_out, uint8_t* hq_out, float* sh_out,
                          int32_t n_threads, uint16_t* y_bf16, double* y64);
int     oracle_threads(void);
void    oracle_e4m3_encode_n(const float* v, int64_t n, uint8_t* q);
void    oracle_e4m3_decode_n(const uint8_t* q, int64_t n, double* v);
void    oracle_exp32_n(const float* x, int64_t n, float* y);

#ifdef __cplusplus
}
#endif
#endif
