/*
 * ORACLE — test infrastructure, not product code.
 *
 * A plain, slow, single-threaded f32 CPU decoder: the KV-cached forward step of a
 * Llama-architecture model followed by greedy or temperature/top-k/top-p sampling.
 * Only tests/, the smoke check and the CPU-baseline leg of bench.py load it.  It
 * shares no code, header or table with the GPU library.
 *
 * Sources (page title, section / definition):
 *   [P1] "bend-ml-llama 0.2.1.0, main.bend":
 *        "The numeric pieces" (list.*, squares, pair_sums, tree_sum, rmsnorm, inv_freq,
 *        angles, rot_at, rot_lo, rot_hi, silu, swiglu); "Heads" (split, join);
 *        "The key/value cache in flat arrays" (KV, KV.push); "Grouped-query attention
 *        over the arrays" (scores, weighted, head_att, group_att, seq_att, attention);
 *        "A layer" (LW, Act, block); "The model" (forward, forward_pre, head_of, argmax);
 *        "Sampling" (topk, weight, total, kept, stops, pick, sample).
 *   [P3] "Llama 3.1 8B Instruct" model card: README "Entries" and "Validation";
 *        rope.linnet (tables: llama3 rescaling); attention.linnet (forward, decode,
 *        prefill: the cache layout [Batch, KvHeads, MaxSeq, hd] and the seen-mask);
 *        lib.linnet (prefill_packed: prompts packed end to end, each seeing only itself).
 *
 * Build: gcc -std=c11 -O2 -ffp-contract=off -fno-fast-math -fPIC -shared oracle.c -lm
 * (-ffp-contract=off: no multiply-add contraction, every product and sum rounded on its
 * own, as the listed f32 operations are.)
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - matvec (P1 delegates it to an off-page package): y[r] = sum over c = 0..in-1 of
 *    W[r][c]*x[c], one f32 accumulator from 0, ascending c.  The dot products inside
 *    attention (q.K and w.V, also off-page gemms) are read the same way.
 *  - F32.pow, F32.cos, F32.sin (off-page): the f32 rounding of the exact value, computed as
 *    (float)pow/cos/sin of the f32 arguments widened to double.
 *  - inv_freq uses P1's 1 / theta^(2i/head) form; the llama3 band rescaling follows
 *    rope.linnet's select chain, in f32, with pi = 3.14159265f.
 *  - The cache of bf16-weight models stores keys and values rounded to bf16 (round to
 *    nearest even) on write, as P3's cache of element type T = bf16; the f32 model keeps
 *    an f32 cache (as P1 does).
 *  - prefill_packed's attention reads the pass's keys and values as the cache holds them
 *    (rounded to bf16 for bf16-weight models), as a decode step reads its own key and value.
 *  - F32.exp inside the sampler: exp_s below (Cody-Waite reduction by ln 2 split in two,
 *    degree-8 Taylor polynomial in Horner form with fused multiply-adds, scaling by 2^n),
 *    so that sampled ids can be reproduced bit for bit.  Softmax and silu use libm expf.
 *
 * parity pins: see tests/test_oracle_pins.py (laws, closed forms, brute force).  The whole
 * model beyond those pins is "parity unpinned": no page prints a worked input -> logits
 * example.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "oracle.h"

/* ------------------------------------------------------------------------------------ */
/* numbers                                                                               */
/* ------------------------------------------------------------------------------------ */

static inline float bf16_to_f32(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* round to nearest even; NaN stays NaN */
static inline uint16_t f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7f800000u) == 0x7f800000u) return (uint16_t)((u >> 16) | ((u & 0xffffu) ? 0x40u : 0u));
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* the bf16 cache rounding above, exported so that it can be checked on its own */
uint16_t or_f32_to_bf16(float f) { return f32_to_bf16(f); }

/* [P1] squares, pair_sums, tree_sum: adjacent pairs added, the odd tail carried, until one
 * value is left; 0 for an empty list. */
float or_tree_sum(const float* xs, int32_t n) {
  if (n <= 0) return 0.0f;
  float* t = (float*)malloc(sizeof(float) * (size_t)n);
  memcpy(t, xs, sizeof(float) * (size_t)n);
  while (n > 1) {
    int32_t m = n / 2;
    for (int32_t i = 0; i < m; ++i) t[i] = t[2 * i] + t[2 * i + 1];
    if (n & 1) t[m] = t[n - 1];
    n = m + (n & 1);
  }
  float r = t[0];
  free(t);
  return r;
}

/* [P1] rmsnorm: g * (x * (1 / sqrt(tree_sum(x^2) / dim + eps))), in this order. */
void or_rmsnorm(const float* x, const float* g, int32_t n, float eps, float* out) {
  float* sq = (float*)malloc(sizeof(float) * (size_t)(n > 0 ? n : 1));
  for (int32_t i = 0; i < n; ++i) sq[i] = x[i] * x[i];
  float ms = or_tree_sum(sq, n) / (float)n;
  float inv = 1.0f / sqrtf(ms + eps);
  for (int32_t i = 0; i < n; ++i) out[i] = g[i] * (inv * x[i]);
  free(sq);
}

/* [P1] Heads: split(half, xs) = (take half, drop half); join = append. */
void or_split(const float* xs, int32_t n, int32_t half, float* lo, int32_t* nlo, float* hi,
              int32_t* nhi) {
  int32_t a = half < n ? half : n;
  if (a < 0) a = 0;
  memcpy(lo, xs, sizeof(float) * (size_t)a);
  memcpy(hi, xs + a, sizeof(float) * (size_t)(n - a));
  *nlo = a;
  *nhi = n - a;
}

void or_join(const float* lo, int32_t nlo, const float* hi, int32_t nhi, float* out) {
  memcpy(out, lo, sizeof(float) * (size_t)nlo);
  memcpy(out + nlo, hi, sizeof(float) * (size_t)nhi);
}

/* [P1] query head h of group h / g (repeat_kv); the decode path walks groups (j, i) with
 * h = j * g + i, the full-sequence path uses this division. */
int32_t or_gqa_kv_head(int32_t h, int32_t g) { return h / g; }

/* [P1] inv_freq and [P3] rope.linnet tables (llama3 band rescaling). */
void or_inv_freq(const or_cfg* c, float* inv) {
  const int32_t hd = 2 * c->half;
  const float PI = 3.14159265f;
  for (int32_t i = 0; i < c->half; ++i) {
    float e = (float)(2 * i) / (float)hd;
    float pw = (float)pow((double)c->theta, (double)e);
    float base = 1.0f / pw;
    float f = base;
    if (c->llama3) {
      float wavelen = (2.0f * PI) / base;
      float low_wl = c->orig_max / c->low_freq;
      float high_wl = c->orig_max / c->high_freq;
      float smooth = (c->orig_max / wavelen - c->low_freq) / (c->high_freq - c->low_freq);
      float smoothed = (1.0f - smooth) * (base / c->factor) + smooth * base;
      if (wavelen > low_wl)
        f = base / c->factor;
      else if (wavelen < high_wl)
        f = base;
      else
        f = smoothed;
    }
    inv[i] = f;
  }
}

/* [P1] angles, cos.l, sin.l, rot_at: angle i = t * inv[i] in f32. */
void or_rope_cs(const or_cfg* c, int32_t t, float* cs, float* sn) {
  float inv[1024];
  or_inv_freq(c, inv);
  for (int32_t i = 0; i < c->half; ++i) {
    float a = (float)t * inv[i];
    cs[i] = (float)cos((double)a);
    sn[i] = (float)sin((double)a);
  }
}

/* [P1] rope on one head of 2*half numbers: split, rot_lo / rot_hi, join. */
void or_rope_head(const float* x, int32_t half, const float* cs, const float* sn, float* out) {
  float lo[512], hi[512], rl[512], rh[512];
  int32_t nlo, nhi;
  or_split(x, 2 * half, half, lo, &nlo, hi, &nhi);
  for (int32_t i = 0; i < half; ++i) {
    float a = lo[i], b = hi[i];
    rl[i] = (a * cs[i]) + ((-b) * sn[i]);
    rh[i] = (b * cs[i]) + (a * sn[i]);
  }
  or_join(rl, half, rh, half, out);
}

/* [P1] silu(x) = x / (1 + exp(-x)); swiglu = silu(g) * u. */
static inline float silu(float x) { return x / (1.0f + expf(-x)); }

/* ------------------------------------------------------------------------------------ */
/* the sampler's exp                                                                      */
/* ------------------------------------------------------------------------------------ */

/*
 * exp(x) for the sampler weights, built only from IEEE-exact operations (products, sums,
 * fused multiply-adds, integer bit assembly), so that any correctly rounding machine gives
 * the same bits.  Method: Cody-Waite range reduction x = n ln2 + r, |r| <= ln2 / 2, with ln 2
 * split as LN2_HI (ln 2 rounded to 16 significant bits, so n * LN2_HI is exact for |n| < 256)
 * plus LN2_LO (the f32 rounding of the remainder); exp(r) by its Taylor series to degree 8
 * (truncation < 6e-9 relative on |r| <= 0.347) in Horner form; then a multiplication by 2^n
 * (two steps below 2^-126 so that a subnormal result is rounded once).
 */
float or_exp_s(float x) {
  if (x != x) return x;
  if (x > 88.5f) return INFINITY;
  if (x < -104.0f) return 0.0f;
  const float LOG2E = 1.44269504088896340736f;
  const float LN2_HI = 0.693145751953125f;
  const float LN2_LO = (float)(0.69314718055994530942 - 0.693145751953125);
  float nf = rintf(x * LOG2E);
  int32_t n = (int32_t)nf;
  float r = fmaf(-nf, LN2_HI, x);
  r = fmaf(-nf, LN2_LO, r);
  const float c8 = (float)(1.0 / 40320.0), c7 = (float)(1.0 / 5040.0), c6 = (float)(1.0 / 720.0);
  const float c5 = (float)(1.0 / 120.0), c4 = (float)(1.0 / 24.0), c3 = (float)(1.0 / 6.0);
  float p = c8;
  p = fmaf(p, r, c7);
  p = fmaf(p, r, c6);
  p = fmaf(p, r, c5);
  p = fmaf(p, r, c4);
  p = fmaf(p, r, c3);
  p = fmaf(p, r, 0.5f);
  p = fmaf(p, r, 1.0f);
  p = fmaf(p, r, 1.0f);
  if (n >= -126) {
    uint32_t sb = (uint32_t)(n + 127) << 23;
    float s;
    memcpy(&s, &sb, 4);
    return p * s;
  }
  uint32_t s1b = (uint32_t)(n + 64 + 127) << 23, s2b = (uint32_t)(-64 + 127) << 23;
  float s1, s2;
  memcpy(&s1, &s1b, 4);
  memcpy(&s2, &s2b, 4);
  return (p * s1) * s2;
}

/* ------------------------------------------------------------------------------------ */
/* greedy and sampling                                                                    */
/* ------------------------------------------------------------------------------------ */

/* [P1] argmax: the first index of the largest value (strict >). */
int32_t or_argmax(const float* xs, int32_t n) {
  if (n <= 0) return 0;
  int32_t bi = 0;
  float bv = xs[0];
  for (int32_t i = 1; i < n; ++i)
    if (xs[i] > bv) {
      bv = xs[i];
      bi = i;
    }
  return bi;
}

/* order of two candidates: larger value first, equal values by lower id first */
static int before(const float* v, int32_t a, int32_t b) {
  if (v[a] > v[b]) return 1;
  if (v[a] < v[b]) return 0;
  return a < b;
}

static void merge_sort(const float* v, int32_t* ids, int32_t* tmp, int32_t n) {
  for (int32_t w = 1; w < n; w *= 2) {
    for (int32_t lo = 0; lo < n; lo += 2 * w) {
      int32_t mid = lo + w < n ? lo + w : n, hi = lo + 2 * w < n ? lo + 2 * w : n;
      int32_t i = lo, j = mid, k = lo;
      while (i < mid && j < hi) tmp[k++] = before(v, ids[j], ids[i]) ? ids[j++] : ids[i++];
      while (i < mid) tmp[k++] = ids[i++];
      while (j < hi) tmp[k++] = ids[j++];
    }
    memcpy(ids, tmp, sizeof(int32_t) * (size_t)n);
  }
}

/* [P1] topk: the k largest values (k > n clamps to n), largest first, equal values in
 * increasing id order (what the one-pass insertion computes).  Returns the count. */
int32_t or_topk(const float* xs, int32_t n, int32_t k, int32_t* ids) {
  if (k > n) k = n;
  if (k <= 0 || n <= 0) return 0;
  int32_t* all = (int32_t*)malloc(sizeof(int32_t) * (size_t)n);
  int32_t* tmp = (int32_t*)malloc(sizeof(int32_t) * (size_t)n);
  for (int32_t i = 0; i < n; ++i) all[i] = i;
  merge_sort(xs, all, tmp, n);
  memcpy(ids, all, sizeof(int32_t) * (size_t)k);
  free(all);
  free(tmp);
  return k;
}

/* [P1] weight(v) = exp(v/temp - top/temp) */
static inline float sweight(float v, float temp, float top) { return or_exp_s(v / temp - top / temp); }

/*
 * [P1] sample(xs, temp, k, p, u): top-k candidates; Z = their weights summed in order;
 * top-p keeps each candidate whose cumulative weight before it is below p*Z (the first is
 * always kept), Zp = the kept weights summed in order; the draw returns the first kept
 * candidate whose cumulative weight (itself included) is above u*Zp, else the last kept.
 * Outputs (optional): the candidate ids and their count, the number kept.
 */
int32_t or_sample_detail(const float* xs, int32_t n, float temp, int32_t k, float p, float u,
                         int32_t* cand, int32_t* ncand, int32_t* nkept) {
  int32_t kk = k > n ? n : k;
  int32_t* cs = (int32_t*)malloc(sizeof(int32_t) * (size_t)(kk > 0 ? kk : 1));
  int32_t m = or_topk(xs, n, kk, cs);
  int32_t id = 0;
  int32_t kept = 0;
  if (m > 0) {
    float top = xs[cs[0]];
    /* total */
    float Z = 0.0f;
    for (int32_t j = 0; j < m; ++j) Z = Z + sweight(xs[cs[j]], temp, top);
    float lim = p * Z;
    /* kept.go */
    float acc = 0.0f;
    int32_t take = 1;
    for (int32_t j = 0; j < m && take; ++j) {
      acc = acc + sweight(xs[cs[j]], temp, top);
      kept = j + 1;
      take = acc < lim;
    }
    float zp = acc;
    /* pick.go */
    float target = u * zp;
    float a = 0.0f;
    int32_t pick = kept - 1;
    for (int32_t j = 0; j < kept; ++j) {
      float a2 = a + sweight(xs[cs[j]], temp, top);
      if (j == kept - 1 || target < a2) {
        pick = j;
        break;
      }
      a = a2;
    }
    id = cs[pick];
  }
  if (cand) memcpy(cand, cs, sizeof(int32_t) * (size_t)m);
  if (ncand) *ncand = m;
  if (nkept) *nkept = kept;
  free(cs);
  return id;
}

int32_t or_sample(const float* xs, int32_t n, float temp, int32_t k, float p, float u) {
  return or_sample_detail(xs, n, temp, k, p, u, 0, 0, 0);
}

/* ------------------------------------------------------------------------------------ */
/* the model                                                                              */
/* ------------------------------------------------------------------------------------ */

enum { T_LN1, T_Q, T_K, T_V, T_O, T_LN2, T_GATE, T_UP, T_DOWN, T_PER_LAYER };
enum { A_X, A_N1, A_Q, A_K, A_V, A_QR, A_KR, A_ATTN, A_A, A_X1, A_N2, A_M, A_Y, A_COUNT };
static const char* ACT_NAMES[A_COUNT] = {"x", "n1", "q", "k", "v", "qr", "kr",
                                         "attn", "a", "x1", "n2", "m", "y"};

struct or_model {
  or_cfg c;
  int32_t hd, H, d, kvw, f, V, L;
  const void* w;
  uint64_t off_layer0, layer_size, off_lnf, off_head;
  int32_t cache_bf16;
  void* kc;
  void* vc;
  float* inv;
  float *x, *n1, *q, *k, *v, *qr, *kr, *att, *a, *x1, *n2, *gg, *uu, *m, *y, *nf;
  float *sc, *wt;
  float* act; /* trace: [L][A_COUNT][maxw] */
  int32_t act_w;
  int32_t trace;
};

uint64_t or_weight_count(const or_cfg* c) {
  uint64_t hd = 2 * (uint64_t)c->half, H = (uint64_t)c->kv * (uint64_t)c->g, d = H * hd;
  uint64_t kvw = (uint64_t)c->kv * hd, f = (uint64_t)c->ffn, V = (uint64_t)c->vocab;
  uint64_t layer = 2 * d + 2 * d * d + 2 * kvw * d + 3 * f * d;
  return V * d + (uint64_t)c->layers * layer + d + (c->tied ? 0 : V * d);
}

static inline float W(const or_model* M, uint64_t i) {
  return M->c.bf16 ? bf16_to_f32(((const uint16_t*)M->w)[i]) : ((const float*)M->w)[i];
}

static uint64_t toff(const or_model* M, int32_t l, int32_t t) {
  uint64_t d = (uint64_t)M->d, kvw = (uint64_t)M->kvw, f = (uint64_t)M->f;
  uint64_t sz[T_PER_LAYER] = {d, d * d, kvw * d, kvw * d, d * d, d, f * d, f * d, d * f};
  uint64_t o = M->off_layer0 + (uint64_t)l * M->layer_size;
  for (int32_t i = 0; i < t; ++i) o += sz[i];
  return o;
}

/* y = W x for W [rows][cols] at element offset off (see the matvec reading above): every y[r]
 * is one f32 accumulator summed over c = 0..cols-1 in order.  Eight rows are summed side by side
 * (eight independent accumulators, each in its own order: no result changes), so the processor
 * is not idle while one row's additions wait on each other. */
static void matvec(const or_model* M, uint64_t off, int32_t rows, int32_t cols, const float* x,
                   float* y) {
  int32_t r = 0;
  if (M->c.bf16) {
    const uint16_t* w = (const uint16_t*)M->w + off;
    for (; r + 8 <= rows; r += 8) {
      const uint16_t* w0 = w + (uint64_t)r * (uint64_t)cols;
      float a[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
      for (int32_t cc = 0; cc < cols; ++cc) {
        const float xv = x[cc];
        a[0] = a[0] + bf16_to_f32(w0[cc]) * xv;
        a[1] = a[1] + bf16_to_f32(w0[cols + cc]) * xv;
        a[2] = a[2] + bf16_to_f32(w0[2 * (uint64_t)cols + cc]) * xv;
        a[3] = a[3] + bf16_to_f32(w0[3 * (uint64_t)cols + cc]) * xv;
        a[4] = a[4] + bf16_to_f32(w0[4 * (uint64_t)cols + cc]) * xv;
        a[5] = a[5] + bf16_to_f32(w0[5 * (uint64_t)cols + cc]) * xv;
        a[6] = a[6] + bf16_to_f32(w0[6 * (uint64_t)cols + cc]) * xv;
        a[7] = a[7] + bf16_to_f32(w0[7 * (uint64_t)cols + cc]) * xv;
      }
      for (int32_t k = 0; k < 8; ++k) y[r + k] = a[k];
    }
  }
  for (; r < rows; ++r) {
    const uint64_t base = off + (uint64_t)r * (uint64_t)cols;
    float acc = 0.0f;
    for (int32_t cc = 0; cc < cols; ++cc) acc = acc + W(M, base + (uint64_t)cc) * x[cc];
    y[r] = acc;
  }
}

static void gains(const or_model* M, uint64_t off, int32_t n, float* out) {
  for (int32_t i = 0; i < n; ++i) out[i] = W(M, off + (uint64_t)i);
}

static inline uint64_t cidx(const or_model* M, int32_t l, int32_t b, int32_t j, int32_t p) {
  return ((((uint64_t)l * (uint64_t)M->c.batch + (uint64_t)b) * (uint64_t)M->c.kv + (uint64_t)j) *
              (uint64_t)M->c.cap +
          (uint64_t)p) *
         (uint64_t)M->hd;
}

static inline float cget(const or_model* M, const void* cache, uint64_t i) {
  return M->cache_bf16 ? bf16_to_f32(((const uint16_t*)cache)[i]) : ((const float*)cache)[i];
}

static inline void cput(const or_model* M, void* cache, uint64_t i, float v) {
  if (M->cache_bf16)
    ((uint16_t*)cache)[i] = f32_to_bf16(v);
  else
    ((float*)cache)[i] = v;
}

static int32_t valid_cfg(const or_cfg* c) {
  if (c->kv <= 0 || c->g <= 0 || c->half <= 0 || c->half > 256 || c->ffn <= 0 || c->layers <= 0 ||
      c->vocab <= 0 || c->batch <= 0 || c->cap <= 0)
    return 0;
  if (!(c->eps >= 0.0f) || !(c->theta > 0.0f)) return 0;
  return 1;
}

or_model* or_create(const or_cfg* c, const void* weights, uint64_t nbytes, int32_t trace,
                    int32_t* err) {
  *err = 0;
  if (!valid_cfg(c)) {
    *err = OR_ERR_CONFIG;
    return 0;
  }
  uint64_t es = c->bf16 ? 2 : 4;
  if (nbytes != or_weight_count(c) * es) {
    *err = OR_ERR_WEIGHTS_SIZE;
    return 0;
  }
  or_model* M = (or_model*)calloc(1, sizeof(or_model));
  M->c = *c;
  M->hd = 2 * c->half;
  M->H = c->kv * c->g;
  M->d = M->H * M->hd;
  M->kvw = c->kv * M->hd;
  M->f = c->ffn;
  M->V = c->vocab;
  M->L = c->layers;
  M->w = weights;
  uint64_t d = (uint64_t)M->d, kvw = (uint64_t)M->kvw, f = (uint64_t)M->f;
  M->layer_size = 2 * d + 2 * d * d + 2 * kvw * d + 3 * f * d;
  M->off_layer0 = (uint64_t)M->V * d;
  M->off_lnf = M->off_layer0 + (uint64_t)M->L * M->layer_size;
  M->off_head = c->tied ? 0 : M->off_lnf + d;
  M->cache_bf16 = c->bf16 && !c->kv_f32;
  uint64_t cn = (uint64_t)M->L * (uint64_t)c->batch * (uint64_t)c->kv * (uint64_t)c->cap * (uint64_t)M->hd;
  uint64_t ces = M->cache_bf16 ? 2 : 4;
  M->kc = calloc(cn, ces);
  M->vc = calloc(cn, ces);
  if (!M->kc || !M->vc) {
    free(M->kc);
    free(M->vc);
    free(M);
    *err = OR_ERR_OOM;
    return 0;
  }
  M->inv = (float*)malloc(sizeof(float) * (size_t)c->half);
  or_inv_freq(c, M->inv);
  int32_t mx = M->d > M->f ? M->d : M->f;
  float** bufs[] = {&M->x, &M->n1, &M->q, &M->k, &M->v, &M->qr, &M->kr, &M->att, &M->a,
                    &M->x1, &M->n2, &M->gg, &M->uu, &M->m, &M->y, &M->nf};
  for (size_t i = 0; i < sizeof(bufs) / sizeof(bufs[0]); ++i) *bufs[i] = (float*)calloc((size_t)mx, sizeof(float));
  M->sc = (float*)malloc(sizeof(float) * (size_t)c->cap);
  M->wt = (float*)malloc(sizeof(float) * (size_t)c->cap);
  M->trace = trace;
  M->act_w = mx;
  if (trace) M->act = (float*)calloc((size_t)M->L * A_COUNT * (size_t)mx, sizeof(float));
  return M;
}

void or_destroy(or_model* M) {
  if (!M) return;
  float* bufs[] = {M->x, M->n1, M->q, M->k, M->v, M->qr, M->kr, M->att, M->a,
                   M->x1, M->n2, M->gg, M->uu, M->m, M->y, M->nf, M->sc, M->wt, M->inv, M->act};
  for (size_t i = 0; i < sizeof(bufs) / sizeof(bufs[0]); ++i) free(bufs[i]);
  free(M->kc);
  free(M->vc);
  free(M);
}

void or_reset(or_model* M) {
  uint64_t cn = (uint64_t)M->L * (uint64_t)M->c.batch * (uint64_t)M->c.kv * (uint64_t)M->c.cap * (uint64_t)M->hd;
  uint64_t ces = M->cache_bf16 ? 2 : 4;
  memset(M->kc, 0, cn * ces);
  memset(M->vc, 0, cn * ces);
}

/*
 * [P1] attention / seq_att / group_att / head_att for one row: the rotated query heads q
 * [H][hd] at position t over cache positions 0..t of one layer and row (kc, vc point at
 * that layer's and row's [kv][cap][hd] block).  Group j holds query heads j*g .. j*g+g-1 and
 * reads key/value head j; the outputs are concatenated in head order.
 */
static void attend(const or_model* M, const float* q, const void* kc, const void* vc, int32_t t,
                   float* out) {
  const int32_t hd = M->hd, g = M->c.g, cap = M->c.cap;
  const float scale = 1.0f / sqrtf((float)hd);
  float* s = M->sc;
  float* w = M->wt;
  for (int32_t j = 0; j < M->c.kv; ++j) {
    uint64_t kb = (uint64_t)j * (uint64_t)cap * (uint64_t)hd;
    for (int32_t i = 0; i < g; ++i) {
      const int32_t h = j * g + i;
      const float* qh = q + (size_t)h * (size_t)hd;
      /* scores: q . K[p] for p = 0..t, then scale * s */
      for (int32_t p = 0; p <= t; ++p) {
        float acc = 0.0f;
        for (int32_t e = 0; e < hd; ++e) acc = acc + qh[e] * cget(M, kc, kb + (uint64_t)p * hd + e);
        s[p] = scale * acc;
      }
      /* list.softmax: max, exp(x - m), running sum from the left, divide */
      float mx = s[0];
      for (int32_t p = 1; p <= t; ++p) mx = fmaxf(mx, s[p]);
      float z = 0.0f;
      for (int32_t p = 0; p <= t; ++p) {
        w[p] = expf(s[p] - mx);
        z = z + w[p];
      }
      for (int32_t p = 0; p <= t; ++p) w[p] = w[p] / z;
      /* weighted: sum over p of w[p] * V[p] */
      float* o = out + (size_t)h * (size_t)hd;
      for (int32_t e = 0; e < hd; ++e) {
        float acc = 0.0f;
        for (int32_t p = 0; p <= t; ++p) acc = acc + w[p] * cget(M, vc, kb + (uint64_t)p * hd + e);
        o[e] = acc;
      }
    }
  }
}

int32_t or_attend(or_model* M, int32_t layer, int32_t b, const float* q, int32_t t, float* out) {
  if (layer < 0 || layer >= M->L || b < 0 || b >= M->c.batch || t < 0 || t >= M->c.cap) return OR_ERR_ARG;
  uint64_t base = cidx(M, layer, b, 0, 0);
  uint64_t es = M->cache_bf16 ? 2 : 4;
  attend(M, q, (const char*)M->kc + base * es, (const char*)M->vc + base * es, t, out);
  return 0;
}

static void keep(or_model* M, int32_t l, int32_t which, const float* src, int32_t n) {
  if (M->trace) memcpy(M->act + ((size_t)l * A_COUNT + (size_t)which) * (size_t)M->act_w, src, sizeof(float) * (size_t)n);
}

/* The pieces of one position, applied in P1 forward's order: or_embed (the embedding row of
 * tok into the residual stream), or_layer for l = 0..L-1 (P1 block at position t of row b), and
 * or_head (final norm and LM head).  or_forward runs them in that order. */
int32_t or_embed(or_model* M, int32_t tok) {
  if (tok < 0 || tok >= M->c.vocab) return OR_ERR_TOKEN_RANGE;
  for (int32_t i = 0; i < M->d; ++i) M->x[i] = W(M, (uint64_t)tok * (uint64_t)M->d + (uint64_t)i);
  return 0;
}

/* [P1] block: layer l at position t of row b on the residual stream x (in place), with the
 * row's cache holding positions 0..t-1 of that layer */
int32_t or_layer(or_model* M, int32_t l, int32_t b, int32_t t) {
  const or_cfg* c = &M->c;
  if (l < 0 || l >= M->L || b < 0 || b >= c->batch) return OR_ERR_ARG;
  if (t < 0 || t >= c->cap) return OR_ERR_POS_RANGE;
  const int32_t d = M->d, hd = M->hd, half = c->half, kvw = M->kvw, f = M->f;
  float cs[256], sn[256];
  for (int32_t i = 0; i < half; ++i) {
    float a = (float)t * M->inv[i];
    cs[i] = (float)cos((double)a);
    sn[i] = (float)sin((double)a);
  }
  float* g = (float*)malloc(sizeof(float) * (size_t)d);
  uint64_t es = M->cache_bf16 ? 2 : 4;
  keep(M, l, A_X, M->x, d);
  gains(M, toff(M, l, T_LN1), d, g);
  or_rmsnorm(M->x, g, d, c->eps, M->n1);
  matvec(M, toff(M, l, T_Q), d, d, M->n1, M->q);
  matvec(M, toff(M, l, T_K), kvw, d, M->n1, M->k);
  matvec(M, toff(M, l, T_V), kvw, d, M->n1, M->v);
  for (int32_t h = 0; h < M->H; ++h) or_rope_head(M->q + (size_t)h * hd, half, cs, sn, M->qr + (size_t)h * hd);
  for (int32_t j = 0; j < c->kv; ++j) or_rope_head(M->k + (size_t)j * hd, half, cs, sn, M->kr + (size_t)j * hd);
  /* KV.push at t: the rotated keys and the values, one array pair per key/value head */
  for (int32_t j = 0; j < c->kv; ++j)
    for (int32_t e = 0; e < hd; ++e) {
      uint64_t ci = cidx(M, l, b, j, t) + (uint64_t)e;
      cput(M, M->kc, ci, M->kr[j * hd + e]);
      cput(M, M->vc, ci, M->v[j * hd + e]);
    }
  uint64_t base = cidx(M, l, b, 0, 0);
  attend(M, M->qr, (const char*)M->kc + base * es, (const char*)M->vc + base * es, t, M->att);
  matvec(M, toff(M, l, T_O), d, d, M->att, M->a);
  for (int32_t i = 0; i < d; ++i) M->x1[i] = M->x[i] + M->a[i];
  gains(M, toff(M, l, T_LN2), d, g);
  or_rmsnorm(M->x1, g, d, c->eps, M->n2);
  matvec(M, toff(M, l, T_GATE), f, d, M->n2, M->gg);
  matvec(M, toff(M, l, T_UP), f, d, M->n2, M->uu);
  for (int32_t i = 0; i < f; ++i) M->uu[i] = silu(M->gg[i]) * M->uu[i];
  matvec(M, toff(M, l, T_DOWN), d, f, M->uu, M->m);
  for (int32_t i = 0; i < d; ++i) M->y[i] = M->x1[i] + M->m[i];
  keep(M, l, A_N1, M->n1, d);
  keep(M, l, A_Q, M->q, d);
  keep(M, l, A_K, M->k, kvw);
  keep(M, l, A_V, M->v, kvw);
  keep(M, l, A_QR, M->qr, d);
  keep(M, l, A_KR, M->kr, kvw);
  keep(M, l, A_ATTN, M->att, d);
  keep(M, l, A_A, M->a, d);
  keep(M, l, A_X1, M->x1, d);
  keep(M, l, A_N2, M->n2, d);
  keep(M, l, A_M, M->m, d);
  keep(M, l, A_Y, M->y, d);
  memcpy(M->x, M->y, sizeof(float) * (size_t)d);
  free(g);
  return 0;
}

/* [P1] head_of: the final norm, then logits = head . nf (head = the embedding when tied) */
void or_head(or_model* M, float* logits) {
  float* g = (float*)malloc(sizeof(float) * (size_t)M->d);
  gains(M, M->off_lnf, M->d, g);
  or_rmsnorm(M->x, g, M->d, M->c.eps, M->nf);
  matvec(M, M->off_head, M->V, M->d, M->nf, logits);
  free(g);
}

/* [P1] forward (logits != NULL) / forward_pre (logits == NULL): token tok at position t of
 * row b, with that row's caches holding positions 0..t-1. */
int32_t or_forward(or_model* M, int32_t b, int32_t tok, int32_t t, float* logits) {
  const or_cfg* c = &M->c;
  if (b < 0 || b >= c->batch) return OR_ERR_ARG;
  if (t < 0 || t >= c->cap) return OR_ERR_POS_RANGE;
  if (tok < 0 || tok >= c->vocab) return OR_ERR_TOKEN_RANGE;
  or_embed(M, tok);
  for (int32_t l = 0; l < M->L; ++l) or_layer(M, l, b, t);
  if (logits) or_head(M, logits);
  return 0;
}

/* P3 prefill semantics, as P1 runs a prompt: positions pos..pos+S-1 of row b through
 * forward_pre, then the final norm and head on the last one (logits may be NULL). */
int32_t or_prefill(or_model* M, int32_t b, const int32_t* toks, int32_t S, int32_t pos, float* logits) {
  if (S <= 0) return OR_ERR_ARG;
  if (pos < 0 || (int64_t)pos + S > M->c.cap) return OR_ERR_POS_RANGE;
  for (int32_t i = 0; i < S; ++i) {
    int32_t r = or_forward(M, b, toks[i], pos + i, i == S - 1 ? logits : 0);
    if (r) return r;
  }
  return 0;
}

/*
 * [P3] prefill_packed (lib.linnet "prefill_packed", its layer's prefill_packed): the tokens of
 * several prompts packed end to end, P in all.  Token p is position positions[p] of prompt
 * segments[p] and belongs to cache row rows[p].  Layer by layer, every token's rotated key
 * and its value go to its row at its position; then token i attends to the tokens j of its own
 * prompt (segments[j] == segments[i]) with positions[j] <= positions[i], in pack order, and to
 * nothing else: not to what its row's cache held before the pass.  The keys and values are
 * read back as the cache holds them (rounded to bf16 for bf16-weight models), as a decode step
 * reads its own.  logits [nlast][V] (may be NULL): after token last[m].  Two tokens may not
 * share a (row, position) slot.
 */
int32_t or_prefill_packed(or_model* M, const int32_t* toks, const int32_t* rows, const int32_t* positions,
                          const int32_t* segments, int32_t P, const int32_t* last, int32_t nlast, float* logits) {
  const or_cfg* c = &M->c;
  if (P <= 0 || nlast < 0) return OR_ERR_ARG;
  for (int32_t p = 0; p < P; ++p) {
    if (toks[p] < 0 || toks[p] >= c->vocab) return OR_ERR_TOKEN_RANGE;
    if (rows[p] < 0 || rows[p] >= c->batch) return OR_ERR_ARG;
    if (positions[p] < 0 || positions[p] >= c->cap) return OR_ERR_POS_RANGE;
    for (int32_t q = 0; q < p; ++q)
      if (rows[q] == rows[p] && positions[q] == positions[p]) return OR_ERR_ARG;
  }
  for (int32_t m = 0; m < nlast; ++m)
    if (last[m] < 0 || last[m] >= P) return OR_ERR_ARG;
  const int32_t d = M->d, hd = M->hd, half = c->half, kvw = M->kvw, f = M->f, g = c->g;
  const float scale = 1.0f / sqrtf((float)hd);
  float* X = (float*)malloc(sizeof(float) * (size_t)P * (size_t)d);    /* residual streams */
  float* QR = (float*)malloc(sizeof(float) * (size_t)P * (size_t)d);   /* rotated queries */
  float* ATT = (float*)malloc(sizeof(float) * (size_t)P * (size_t)d);  /* attention outputs */
  float* sc = (float*)malloc(sizeof(float) * (size_t)P);
  float* wt = (float*)malloc(sizeof(float) * (size_t)P);
  int32_t* own = (int32_t*)malloc(sizeof(int32_t) * (size_t)P);
  float* gn = (float*)malloc(sizeof(float) * (size_t)d);   /* ln1 gains of the layer */
  float* gn2 = (float*)malloc(sizeof(float) * (size_t)d);  /* ln2 gains */
  float cs[256], sn[256];
  for (int32_t p = 0; p < P; ++p)
    for (int32_t i = 0; i < d; ++i) X[(size_t)p * d + i] = W(M, (uint64_t)toks[p] * (uint64_t)d + (uint64_t)i);
  for (int32_t l = 0; l < M->L; ++l) {
    /* every token: norm, projections, rotation, and its key and value into the cache */
    gains(M, toff(M, l, T_LN1), d, gn);
    for (int32_t p = 0; p < P; ++p) {
      for (int32_t i = 0; i < half; ++i) {
        float a = (float)positions[p] * M->inv[i];
        cs[i] = (float)cos((double)a);
        sn[i] = (float)sin((double)a);
      }
      or_rmsnorm(X + (size_t)p * d, gn, d, c->eps, M->n1);
      matvec(M, toff(M, l, T_Q), d, d, M->n1, M->q);
      matvec(M, toff(M, l, T_K), kvw, d, M->n1, M->k);
      matvec(M, toff(M, l, T_V), kvw, d, M->n1, M->v);
      for (int32_t h = 0; h < M->H; ++h)
        or_rope_head(M->q + (size_t)h * hd, half, cs, sn, QR + (size_t)p * d + (size_t)h * hd);
      for (int32_t j = 0; j < c->kv; ++j) or_rope_head(M->k + (size_t)j * hd, half, cs, sn, M->kr + (size_t)j * hd);
      for (int32_t j = 0; j < c->kv; ++j)
        for (int32_t e = 0; e < hd; ++e) {
          uint64_t ci = cidx(M, l, rows[p], j, positions[p]) + (uint64_t)e;
          cput(M, M->kc, ci, M->kr[j * hd + e]);
          cput(M, M->vc, ci, M->v[j * hd + e]);
        }
    }
    /* every token attends to its own prompt's tokens up to its position, in pack order */
    for (int32_t i = 0; i < P; ++i) {
      int32_t n = 0;
      for (int32_t p = 0; p < P; ++p)
        if (segments[p] == segments[i] && positions[p] <= positions[i]) own[n++] = p;
      for (int32_t j = 0; j < c->kv; ++j)
        for (int32_t ih = 0; ih < g; ++ih) {
          const int32_t h = j * g + ih;
          const float* qh = QR + (size_t)i * d + (size_t)h * hd;
          for (int32_t a = 0; a < n; ++a) {
            const uint64_t kb = cidx(M, l, rows[own[a]], j, positions[own[a]]);
            float acc = 0.0f;
            for (int32_t e = 0; e < hd; ++e) acc = acc + qh[e] * cget(M, M->kc, kb + (uint64_t)e);
            sc[a] = scale * acc;
          }
          float mx = sc[0];
          for (int32_t a = 1; a < n; ++a) mx = fmaxf(mx, sc[a]);
          float z = 0.0f;
          for (int32_t a = 0; a < n; ++a) {
            wt[a] = expf(sc[a] - mx);
            z = z + wt[a];
          }
          for (int32_t a = 0; a < n; ++a) wt[a] = wt[a] / z;
          float* o = ATT + (size_t)i * d + (size_t)h * hd;
          for (int32_t e = 0; e < hd; ++e) {
            float acc = 0.0f;
            for (int32_t a = 0; a < n; ++a) {
              const uint64_t vb = cidx(M, l, rows[own[a]], j, positions[own[a]]);
              acc = acc + wt[a] * cget(M, M->vc, vb + (uint64_t)e);
            }
            o[e] = acc;
          }
        }
    }
    /* every token: o_proj and the residual, the norm, SwiGLU, down and the residual */
    gains(M, toff(M, l, T_LN2), d, gn2);
    for (int32_t p = 0; p < P; ++p) {
      float* x = X + (size_t)p * d;
      matvec(M, toff(M, l, T_O), d, d, ATT + (size_t)p * d, M->a);
      for (int32_t i = 0; i < d; ++i) M->x1[i] = x[i] + M->a[i];
      or_rmsnorm(M->x1, gn2, d, c->eps, M->n2);
      matvec(M, toff(M, l, T_GATE), f, d, M->n2, M->gg);
      matvec(M, toff(M, l, T_UP), f, d, M->n2, M->uu);
      for (int32_t i = 0; i < f; ++i) M->uu[i] = silu(M->gg[i]) * M->uu[i];
      matvec(M, toff(M, l, T_DOWN), d, f, M->uu, M->m);
      for (int32_t i = 0; i < d; ++i) x[i] = M->x1[i] + M->m[i];
    }
  }
  if (logits)
    for (int32_t m = 0; m < nlast; ++m) {
      memcpy(M->x, X + (size_t)last[m] * d, sizeof(float) * (size_t)d);
      or_head(M, logits + (size_t)m * (size_t)M->V);
    }
  free(X);
  free(QR);
  free(ATT);
  free(sc);
  free(wt);
  free(own);
  free(gn);
  free(gn2);
  return 0;
}

int32_t or_trace(const or_model* M, int32_t layer, const char* name, float* dst) {
  if (!M->trace || layer < 0 || layer >= M->L) return OR_ERR_ARG;
  for (int32_t i = 0; i < A_COUNT; ++i)
    if (strcmp(name, ACT_NAMES[i]) == 0) {
      int32_t n = (i == A_K || i == A_V || i == A_KR) ? M->kvw : M->d;
      memcpy(dst, M->act + ((size_t)layer * A_COUNT + (size_t)i) * (size_t)M->act_w, sizeof(float) * (size_t)n);
      return n;
    }
  return OR_ERR_ARG;
}

/* cache rows, element type of the cache (uint16 bf16 bits or f32), layout [kv][n][hd] */
int32_t or_kv_write(or_model* M, int32_t layer, int32_t b, int32_t pos0, int32_t n, const void* k, const void* v) {
  if (layer < 0 || layer >= M->L || b < 0 || b >= M->c.batch || pos0 < 0 || n < 0 || (int64_t)pos0 + n > M->c.cap)
    return OR_ERR_ARG;
  uint64_t es = M->cache_bf16 ? 2 : 4, hd = (uint64_t)M->hd;
  for (int32_t j = 0; j < M->c.kv; ++j) {
    uint64_t dst = cidx(M, layer, b, j, pos0) * es, src = ((uint64_t)j * (uint64_t)n) * hd * es;
    memcpy((char*)M->kc + dst, (const char*)k + src, (uint64_t)n * hd * es);
    memcpy((char*)M->vc + dst, (const char*)v + src, (uint64_t)n * hd * es);
  }
  return 0;
}

int32_t or_kv_read(const or_model* M, int32_t layer, int32_t b, int32_t pos0, int32_t n, void* k, void* v) {
  if (layer < 0 || layer >= M->L || b < 0 || b >= M->c.batch || pos0 < 0 || n < 0 || (int64_t)pos0 + n > M->c.cap)
    return OR_ERR_ARG;
  uint64_t es = M->cache_bf16 ? 2 : 4, hd = (uint64_t)M->hd;
  for (int32_t j = 0; j < M->c.kv; ++j) {
    uint64_t src = cidx(M, layer, b, j, pos0) * es, dst = ((uint64_t)j * (uint64_t)n) * hd * es;
    memcpy((char*)k + dst, (const char*)M->kc + src, (uint64_t)n * hd * es);
    memcpy((char*)v + dst, (const char*)M->vc + src, (uint64_t)n * hd * es);
  }
  return 0;
}

/* ------------------------------------------------------------------------------------ */
/* the full-sequence forward (P3 attention.linnet `forward`): an independent second path  */
/* ------------------------------------------------------------------------------------ */

/*
 * Logits for every position of one sequence of S tokens, computed as matrices with the
 * causal mask (query row i sees key rows s <= i; the others score -inf) and query head h
 * reading key/value head h / g.  Keys and values are used unrounded (f32), so for an f32
 * model this equals token-by-token decoding up to rounding order.
 */
int32_t or_forward_full(const or_cfg* c, const void* weights, uint64_t nbytes, const int32_t* toks,
                        int32_t S, float* logits) {
  int32_t err = 0;
  or_cfg c1 = *c;
  c1.batch = 1;
  c1.cap = S > 0 ? S : 1;
  or_model* M = or_create(&c1, weights, nbytes, 0, &err);
  if (!M) return err;
  const int32_t d = M->d, hd = M->hd, half = c->half, kvw = M->kvw, f = M->f, H = M->H, S_ = S;
  float* X = (float*)malloc(sizeof(float) * (size_t)S_ * d);
  float* N = (float*)malloc(sizeof(float) * (size_t)S_ * d);
  float* Q = (float*)malloc(sizeof(float) * (size_t)S_ * d);
  float* K = (float*)malloc(sizeof(float) * (size_t)S_ * kvw);
  float* Vv = (float*)malloc(sizeof(float) * (size_t)S_ * kvw);
  float* O = (float*)malloc(sizeof(float) * (size_t)S_ * d);
  float* G = (float*)malloc(sizeof(float) * (size_t)f);
  float* U = (float*)malloc(sizeof(float) * (size_t)f);
  float* T = (float*)malloc(sizeof(float) * (size_t)(d > f ? d : f));
  float* P = (float*)malloc(sizeof(float) * (size_t)S_);
  float* gn = (float*)malloc(sizeof(float) * (size_t)d);
  float* CS = (float*)malloc(sizeof(float) * (size_t)S_ * half);
  float* SN = (float*)malloc(sizeof(float) * (size_t)S_ * half);
  for (int32_t s = 0; s < S_; ++s) {
    for (int32_t i = 0; i < half; ++i) {
      float a = (float)s * M->inv[i];
      CS[s * half + i] = (float)cos((double)a);
      SN[s * half + i] = (float)sin((double)a);
    }
    if (toks[s] < 0 || toks[s] >= c->vocab) {
      err = OR_ERR_TOKEN_RANGE;
      goto done;
    }
    for (int32_t i = 0; i < d; ++i) X[(size_t)s * d + i] = W(M, (uint64_t)toks[s] * d + i);
  }
  const float scale = 1.0f / sqrtf((float)hd);
  for (int32_t l = 0; l < M->L; ++l) {
    gains(M, toff(M, l, T_LN1), d, gn);
    for (int32_t s = 0; s < S_; ++s) or_rmsnorm(X + (size_t)s * d, gn, d, c->eps, N + (size_t)s * d);
    for (int32_t s = 0; s < S_; ++s) {
      matvec(M, toff(M, l, T_Q), d, d, N + (size_t)s * d, T);
      for (int32_t h = 0; h < H; ++h) or_rope_head(T + h * hd, half, CS + s * half, SN + s * half, Q + (size_t)s * d + h * hd);
      matvec(M, toff(M, l, T_K), kvw, d, N + (size_t)s * d, T);
      for (int32_t j = 0; j < c->kv; ++j) or_rope_head(T + j * hd, half, CS + s * half, SN + s * half, K + (size_t)s * kvw + j * hd);
      matvec(M, toff(M, l, T_V), kvw, d, N + (size_t)s * d, Vv + (size_t)s * kvw);
    }
    for (int32_t h = 0; h < H; ++h) {
      int32_t j = or_gqa_kv_head(h, c->g);
      for (int32_t i = 0; i < S_; ++i) {
        for (int32_t s = 0; s < S_; ++s) {
          if (s > i) {
            P[s] = -INFINITY;
            continue;
          }
          float acc = 0.0f;
          for (int32_t e = 0; e < hd; ++e) acc = acc + Q[(size_t)i * d + h * hd + e] * K[(size_t)s * kvw + j * hd + e];
          P[s] = scale * acc;
        }
        float mx = P[0];
        for (int32_t s = 1; s < S_; ++s) mx = fmaxf(mx, P[s]);
        float z = 0.0f;
        for (int32_t s = 0; s < S_; ++s) {
          P[s] = expf(P[s] - mx);
          z = z + P[s];
        }
        for (int32_t s = 0; s < S_; ++s) P[s] = P[s] / z;
        for (int32_t e = 0; e < hd; ++e) {
          float acc = 0.0f;
          for (int32_t s = 0; s <= i; ++s) acc = acc + P[s] * Vv[(size_t)s * kvw + j * hd + e];
          O[(size_t)i * d + h * hd + e] = acc;
        }
      }
    }
    for (int32_t s = 0; s < S_; ++s) {
      float* x = X + (size_t)s * d;
      matvec(M, toff(M, l, T_O), d, d, O + (size_t)s * d, T);
      for (int32_t i = 0; i < d; ++i) x[i] = x[i] + T[i];
      gains(M, toff(M, l, T_LN2), d, gn);
      or_rmsnorm(x, gn, d, c->eps, N + (size_t)s * d);
      matvec(M, toff(M, l, T_GATE), f, d, N + (size_t)s * d, G);
      matvec(M, toff(M, l, T_UP), f, d, N + (size_t)s * d, U);
      for (int32_t i = 0; i < f; ++i) U[i] = silu(G[i]) * U[i];
      matvec(M, toff(M, l, T_DOWN), d, f, U, T);
      for (int32_t i = 0; i < d; ++i) x[i] = x[i] + T[i];
    }
  }
  gains(M, M->off_lnf, d, gn);
  for (int32_t s = 0; s < S_; ++s) {
    or_rmsnorm(X + (size_t)s * d, gn, d, c->eps, T);
    matvec(M, M->off_head, M->V, d, T, logits + (size_t)s * M->V);
  }
done:
  free(X); free(N); free(Q); free(K); free(Vv); free(O); free(G); free(U); free(T); free(P);
  free(gn); free(CS); free(SN);
  or_destroy(M);
  return err;
}
