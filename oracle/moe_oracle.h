/*
 * moe_oracle.h -- the CPU oracle of the quantized MoE decode layer.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE. Only the tests, the smoke check and
 * the benchmark's CPU-baseline leg may load or call it. It shares no code,
 * header, table or helper with the CUDA library.
 *
 * Every routine is a plain restatement of what the layer computes, in f64
 * unless the page fixes the precision (the score's f32 chain, the selection's
 * f32 key arithmetic and the q8_1 quantisation decisions). Sources, by page:
 *   moe_v41.rs          -- module doc (three K-quant GEMVs on raw Q2_K / Q3_K
 *                          blocks, q8_1 activation, bf16 shared expert,
 *                          routing rule), MoeV41Cfg, MoeV41LayerWeights,
 *                          fn softplus, fn route_from_logits, fn bf16_bytes,
 *                          struct MoeV41 buffers (acc, out, shared side).
 *   moe_v41/device_route.rs -- module doc (header: miss flag, picks, weight
 *                          bits, plan slots), fn route_select_launch (pointer
 *                          = base + slot * slot_bytes + offset), fn
 *                          device_route_check (plan in ascending id).
 * Points the pages leave open take the readings listed in the design notes
 * (Q2_K / Q3_K byte layout = the public GGUF layout; q8_1 = 32 values with an
 * f16 scale; clamped SwiGLU; each f32 step of the score correctly rounded).
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H

#include <stdint.h>
#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
    int32_t dim, inter, n_routed, topk, norm_topk_prob;
    float gate_temp, route_scale, swiglu_limit;
} orc_cfg;

/* per-token flags written by orc_route */
#define ORC_FLAG_NONFINITE 2   /* a logit or key was NaN or infinite        */
#define ORC_FLAG_NEAR_MID  4   /* a step of a score's f32 chain lay within
                                  2^-56 (relative) of an f32 rounding
                                  midpoint: its rounding is not certain at
                                  long-double precision                     */

uint16_t orc_bf16_from_f32(float x);
double orc_bf16_to_f64(uint16_t h);
double orc_f16_to_f64(uint16_t h);
uint16_t orc_f16_from_f32(float x);

void orc_dequant_q2k(const uint8_t *blk, double w[256]);
void orc_dequant_q3k(const uint8_t *blk, double w[256]);
void orc_quant_q8_1(const float *x, int n, uint8_t *out);
void orc_dequant_q8_1(const uint8_t *blk, double v[32]);

void orc_quantize_q2k(const float *x, uint8_t *blk);
void orc_quantize_q3k(const float *x, uint8_t *blk);

void orc_router_logits(const uint16_t *x, const uint16_t *w, int dim, int n, int m,
                       float *logits);
float orc_score(float logit, float temp, int *near_mid);
int orc_route(const orc_cfg *c, const float *logits, const float *bias, int m,
              int32_t *picks, float *weights, float *scores, int32_t *flags);
double orc_swiglu(double g, double u, double limit);
int orc_plan(int m, int k, int n, const int32_t *picks, const float *weights,
             const int32_t *flags, const int32_t *slot_row, uint64_t base,
             uint64_t slot_bytes, uint64_t gate_off, uint64_t up_off, uint64_t down_off,
             int32_t *hdr, float *plan_w, int32_t *plan_rows, uint64_t *ptrs);

void orc_expert_token(const orc_cfg *c, const uint8_t *gate, const uint8_t *up,
                      const uint8_t *down, const uint8_t *x_q8, float *g, float *u,
                      float *h, uint8_t *h_q8, float *dn, int threads);
void orc_shared_token(const orc_cfg *c, const uint16_t *w1, const uint16_t *w3,
                      const uint16_t *w2, const uint16_t *x, float *gs, float *us,
                      uint16_t *hs, float *sd, int threads);

/* One layer step over m tokens. experts[e] = the host image of expert e's
 * slot (gate at gate_off, up at up_off, down at down_off), NULL when absent
 * (an absent pick is an error, return -1). sh_w* may be NULL (no shared
 * expert); bf16 matrices, or with sh_kquant Q2_K (w1, w3) and Q3_K (w2)
 * blocks run as a routed expert of weight 1. residual is updated in place;
 * x_next = bf16(residual). Optional
 * outputs (NULL to skip): logits [m,n], picks/weights [m,k], flags [m],
 * acc [m,dim], sd [m,dim]. */
int orc_layer(const orc_cfg *c, int m, const uint16_t *x, const uint16_t *router_w,
              const float *bias, const uint8_t *const *experts, uint64_t gate_off,
              uint64_t up_off, uint64_t down_off, const uint16_t *sh_w1,
              const uint16_t *sh_w3, const uint16_t *sh_w2, int sh_kquant, float *residual,
              uint16_t *x_next, float *logits, int32_t *picks, float *weights,
              int32_t *flags, float *acc, float *sd, int threads);

#ifdef __cplusplus
}
#endif
#endif
