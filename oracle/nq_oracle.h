/*
 * nq_oracle.h -- declarations of the CPU oracle (TEST INFRASTRUCTURE ONLY).
 * Only tests, the smoke check and the benchmark's CPU-baseline leg use it.
 * It shares nothing with the CUDA library's headers.
 */
#ifndef NQ_ORACLE_H
#define NQ_ORACLE_H
#include <stddef.h>
#include <stdint.h>

#define ORC_LEAF 16
#define ORC_SEG 1024

enum { ORC_FMT_NESTED44 = 0, ORC_FMT_INT4 = 1, ORC_FMT_FP8 = 2, ORC_FMT_FP16 = 3 };

typedef struct {
    int32_t n, k, group, format;
    const uint8_t *base;   /* nibbles [n][k/2] | e4m3 [n][k] | fp16 bits [n][k] */
    const uint8_t *resid;  /* nibbles [n][k/2] (NESTED44 only) */
    const void *scales;    /* fp16 bits [n][k/group] | fp32 [n] (FP8) | unused */
} nq_oracle_weights;

float orc_bf16_to_f32(uint16_t b);
float orc_f16_to_f32(uint16_t h);
uint16_t orc_f32_to_f16(float f);
float orc_e4m3_to_f32(uint8_t c);
uint8_t orc_f32_to_e4m3(float f);

int orc_nibble_value(unsigned nib);
int orc_get_code(const uint8_t *plane, size_t idx);
void orc_quantise_weight(float w, float s, int *q4, int *r);
int orc_pack_nested(const float *w, int n, int k, int g, uint8_t *base, uint8_t *resid, uint16_t *scales);
int orc_pack_fp8(const float *w, int n, int k, uint8_t *codes, float *row_scale);
int orc_pack_fp16(const float *w, int n, int k, uint16_t *w16);
int orc_linear(const nq_oracle_weights *W, int use_resid, const uint16_t *x, int M,
               const int32_t *rows, int nrows, double *y);

int orc_quantize_act_int8(const uint16_t *x, int M, int K, int8_t *xq, float *sx);
int orc_linear_a8(const nq_oracle_weights *W, int use_resid, const int8_t *xq, const float *sx, int M, double *y);

int orc_accept_greedy(const int32_t *draft, const float *tgt_logits, int B, int k, int V,
                      int32_t *out_tok, int32_t *out_cnt);

void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);
float orc_uniform(uint64_t seed, uint32_t j, uint32_t purpose, uint64_t round);
float orc_exp2c(float t);
float orc_exp2_coef(int i);
float orc_temper_coef(float T);
int orc_softmax_canonical(const float *l, int V, float T, float *p);
int orc_tree_sample(const float *w, int V, float u);
int orc_sample_p(const float *l, int V, float T, float u);
int orc_attn_decode(const float *q, int B, int M, int Hq, int Hkv, int d, int G, int L,
                    const uint8_t *kb, const uint8_t *kr, const uint16_t *ks,
                    const uint8_t *vb, const uint8_t *vr, const uint16_t *vs,
                    const int32_t *len, int planes, float scale, float *out);
int orc_draft_features(const int32_t *draft, const float *draft_logits, int B, int k, int V, float T, double *out);
int orc_draft_argmax(const float *logits, int M, int V, int32_t *tok);
int orc_round_commit(const int32_t *out_tok, const int32_t *out_cnt, int B, int k, int32_t *seq,
                     int32_t *seq_len, int max_len, int32_t *x0);
int orc_softmax_stats(const float *l, int V, float T, float *seg_mz, float *seg_s, float *M, float *S);
int orc_accept_sample(const int32_t *draft, const float *draft_logits, const float *tgt_logits,
                      int B, int k, int V, float T, const uint64_t *seeds, uint64_t round,
                      int32_t *out_tok, int32_t *out_cnt);
int orc_accept_sample_f64(const int32_t *draft, const float *draft_logits, const float *tgt_logits,
                          int B, int k, int V, float T, const uint64_t *seeds, uint64_t round,
                          int32_t *out_tok, int32_t *out_cnt, double *margin);
void orc_exp2c_n(const float *t, float *out, int n);
void orc_f32_to_f16_n(const float *f, uint16_t *out, int n);
void orc_f16_to_f32_n(const uint16_t *h, float *out, int n);
void orc_f32_to_e4m3_n(const float *f, uint8_t *out, int n);
void orc_e4m3_to_f32_n(const uint8_t *c, float *out, int n);
void orc_uniform_n(const uint64_t *seed, const uint32_t *j, const uint32_t *purpose, const uint64_t *round,
                   float *out, int n);
#endif
