/* CPU oracle for the 4-bit decode step — TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 restatement of the decoder that the aot-llm page
 * ("p10node/aot-llm", sequence diagram and "The static pipeline emitted for
 * every model") describes: embedding -> [RMSNorm -> GQA attention with RoPE
 * and a KV cache -> residual -> RMSNorm -> SwiGLU FFN -> residual] x N ->
 * RMSNorm -> logits. Only the tests, the smoke check and the bench's CPU
 * baseline may load this library; the product path never does. It shares no
 * code with the CUDA library.
 *
 * Parity pins: every function here is checked by tests/test_oracle_pins.py
 * against closed forms, brute force and the invariants the pages fix.
 */
#ifndef ORACLE_H
#define ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {            /* one group-64 4-bit linear, canonical layout */
  const uint8_t*  codes;    /* [rows][cols/2]: element 2j low nibble of byte j */
  const uint16_t* scales;   /* fp16 bits [rows][cols/64] */
  const uint16_t* mins;     /* fp16 bits [rows][cols/64] */
  int64_t rows, cols;
} orc_q4;

typedef struct {
  int32_t dim, n_layers, n_heads, n_kv_heads, head_dim, ffn_dim, vocab;
  int32_t rope_neox;        /* 0: pairs (2i,2i+1); 1: pairs (i, i+hd/2) */
  int32_t qk_norm;          /* per-head RMSNorm of q and k before RoPE */
  int32_t tied;             /* LM head = bf16 embedding table */
  int32_t embed_bf16;       /* embedding stored as bf16 (else fp32) */
  int32_t pad_;
  double  norm_eps, rope_theta;
} orc_config;

typedef struct {
  orc_q4 wq, wk, wv, wo, wg, wu, wd;
  const float *attn_norm, *ffn_norm, *q_norm, *k_norm;
} orc_layer;

typedef struct {
  orc_config cfg;
  const void* embed;        /* fp32 or bf16 bits, [vocab][dim] */
  const float* final_norm;
  orc_q4 lm_head;           /* unused when tied */
  const orc_layer* layers;
} orc_model;

typedef struct {            /* one sequence's cache, caller-owned storage */
  uint16_t* k;              /* bf16 bits [n_layers][n_kv_heads][cap][head_dim] */
  uint16_t* v;
  int32_t cap, len;
  int8_t* k8;               /* grouped int8 instead (k, v unused): codes [n_layers][n_kv_heads][cap][head_dim] */
  int8_t* v8;
  uint16_t* ks;             /* fp16 scales [n_layers][n_kv_heads][cap][head_dim / 32] */
  uint16_t* vs;
} orc_cache;

/* Grouped int8 storage of cached K/V (llmopt page, "grouped-Q8 attention
   state"; GGUF's q8_0 block): groups of 32 values, an fp16 scale d =
   fp16(amax / 127) from the fp32-rounded values, codes round(x / d) (half away
   from zero, clamped to +-127; all zero when d is), value = code * d. */
#define ORC_Q8_GROUP 32
uint16_t orc_half_from_float(float f);     /* RNE */
void     orc_q8_quantize(const double* x, int32_t n, int8_t* q, uint16_t* d);
double   orc_q8_value(int8_t q, uint16_t d);
/* orc_attend over grouped-int8 rows: codes [n_pos][hd], scales [n_pos][hd / 32]. */
void orc_attend_q8(const double* q, const int8_t* k, const uint16_t* ks, const int8_t* v,
                   const uint16_t* vs, int32_t n_pos, int32_t hd, double* out);
/* Full-prefix mode keeps K/V as grouped int8 (1) or bf16 (0, the default). */
void orc_set_kv_q8(int32_t on);

/* Planted mistakes for the mutation tests (0 = none). */
enum {
  ORC_MUT_NONE = 0, ORC_MUT_ROPE_PAIRING = 1, ORC_MUT_MASK_POLARITY = 2,
  ORC_MUT_CACHE_FRONTIER = 3, ORC_MUT_QK_ORIENTATION = 4, ORC_MUT_GQA_MAP = 5,
  ORC_MUT_NIBBLE_ORDER = 6, ORC_MUT_SCALE_MIN_SWAP = 7, ORC_MUT_NO_RESIDUAL = 8,
  ORC_MUT_ROPE_SIGN = 9
};
void    orc_set_mutation(int32_t m);
int32_t orc_num_threads(void);

double   orc_half_to_double(uint16_t h);
double   orc_bf16_to_double(uint16_t b);
uint16_t orc_bf16_from_double(double x);   /* via fp32: RNE to fp32, then RNE to bf16 */
float    orc_f32_from_double(double x);

void orc_dequant_row(const orc_q4* w, int64_t r, double* out);
void orc_matvec(const orc_q4* w, const double* x, double* y);
void orc_rmsnorm(const double* x, const float* w, int32_t n, double eps, double* out);
void orc_rope(double* v, int32_t hd, int32_t pos, double theta, int32_t neox);
void orc_silu_mul(const double* g, const double* u, int32_t n, double* out);
/* One query head over positions 0..n_pos-1 of one kv head's bf16 rows [n_pos][hd]. */
void orc_attend(const double* q, const uint16_t* k, const uint16_t* v, int32_t n_pos,
                int32_t hd, double* out);
int32_t orc_argmax_f32(const double* logits, int64_t n);

/* One cached decode step at position c->len for token tok: appends K/V, len += 1.
   logits [vocab] (may be NULL), hidden [(n_layers+1)][dim] (may be NULL). */
int32_t orc_step(const orc_model* m, orc_cache* c, int32_t tok, double* logits, double* hidden);

/* Full-prefix mode: positions 0..n-1 recomputed layer by layer with a causal
   mask and no cache object. logits [n][vocab] (every position), hidden
   [(n_layers+1)][n][dim] (may be NULL). */
int32_t orc_full_prefix(const orc_model* m, const int32_t* toks, int32_t n, double* logits,
                        double* hidden);

#ifdef __cplusplus
}
#endif
#endif
