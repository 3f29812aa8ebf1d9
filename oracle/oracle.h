/*
 * ORACLE — test infrastructure, not product code.  The interface of oracle.c: a plain
 * single-threaded f32 CPU decoder used only to check the GPU library.  See oracle.c for
 * the sources it follows and the readings it takes.
 */
#ifndef LLAMA_KV_ORACLE_H
#define LLAMA_KV_ORACLE_H
#include <stdint.h>

typedef struct {
  int32_t kv, g, half, ffn, layers, vocab; /* key/value heads, heads per group, half a head, MLP, layers, vocabulary */
  float eps, theta;                        /* RMSNorm epsilon, RoPE base */
  int32_t tied;                            /* 1: the LM head is the embedding */
  int32_t llama3;                          /* 1: llama3 three-band rescaling of inv_freq */
  float factor, low_freq, high_freq, orig_max;
  int32_t batch, cap;                      /* cache rows and positions */
  int32_t bf16;                            /* weights given as bf16 bits; cache rounded to bf16 */
  int32_t kv_f32;                          /* diagnostic: keep an f32 cache with bf16 weights */
} or_cfg;

typedef struct or_model or_model;

enum {
  OR_OK = 0,
  OR_ERR_CONFIG = -1,
  OR_ERR_WEIGHTS_SIZE = -2,
  OR_ERR_OOM = -3,
  OR_ERR_POS_RANGE = -4,
  OR_ERR_TOKEN_RANGE = -5,
  OR_ERR_ARG = -6,
};

uint64_t or_weight_count(const or_cfg* c);
or_model* or_create(const or_cfg* c, const void* weights, uint64_t nbytes, int32_t trace, int32_t* err);
void or_destroy(or_model* m);
void or_reset(or_model* m);
int32_t or_forward(or_model* m, int32_t b, int32_t tok, int32_t t, float* logits);
int32_t or_embed(or_model* m, int32_t tok);
int32_t or_layer(or_model* m, int32_t l, int32_t b, int32_t t);
void or_head(or_model* m, float* logits);
int32_t or_prefill(or_model* m, int32_t b, const int32_t* toks, int32_t S, int32_t pos, float* logits);
int32_t or_prefill_packed(or_model* m, const int32_t* toks, const int32_t* rows, const int32_t* positions,
                          const int32_t* segments, int32_t P, const int32_t* last, int32_t nlast, float* logits);
int32_t or_forward_full(const or_cfg* c, const void* weights, uint64_t nbytes, const int32_t* toks,
                        int32_t S, float* logits);
int32_t or_attend(or_model* m, int32_t layer, int32_t b, const float* q, int32_t t, float* out);
int32_t or_kv_write(or_model* m, int32_t layer, int32_t b, int32_t pos0, int32_t n, const void* k, const void* v);
int32_t or_kv_read(const or_model* m, int32_t layer, int32_t b, int32_t pos0, int32_t n, void* k, void* v);
int32_t or_trace(const or_model* m, int32_t layer, const char* name, float* dst);

float or_tree_sum(const float* xs, int32_t n);
void or_rmsnorm(const float* x, const float* g, int32_t n, float eps, float* out);
void or_split(const float* xs, int32_t n, int32_t half, float* lo, int32_t* nlo, float* hi, int32_t* nhi);
void or_join(const float* lo, int32_t nlo, const float* hi, int32_t nhi, float* out);
int32_t or_gqa_kv_head(int32_t h, int32_t g);
void or_rope_head(const float* x, int32_t half, const float* cs, const float* sn, float* out);
void or_inv_freq(const or_cfg* c, float* inv);
void or_rope_cs(const or_cfg* c, int32_t t, float* cs, float* sn);
float or_exp_s(float x);
uint16_t or_f32_to_bf16(float f);
int32_t or_argmax(const float* xs, int32_t n);
int32_t or_topk(const float* xs, int32_t n, int32_t k, int32_t* ids);
int32_t or_sample(const float* xs, int32_t n, float temp, int32_t k, float p, float u);
int32_t or_sample_detail(const float* xs, int32_t n, float temp, int32_t k, float p, float u,
                         int32_t* cand, int32_t* ncand, int32_t* nkept);
#endif
