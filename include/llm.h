/*
 * llm.h — C ABI of the GB300 KV-cached Llama decoder library (libllm.so).
 *
 * The library runs the KV-cached forward step of a Llama-architecture decoder and its
 * sampler on one GPU, in hand-written sm_103a kernels:
 *   embedding -> per layer { RMSNorm -> Q/K/V projections -> half-split RoPE (optionally
 *   with llama3 three-band frequency rescaling) -> KV-cache write -> grouped-query attention
 *   over cache positions 0..t -> o_proj + residual -> RMSNorm -> SwiGLU MLP + residual }
 *   -> final RMSNorm -> tied or untied LM head -> greedy or temperature/top-k/top-p sampling.
 *
 * Sources, by page title and section:
 *   "bend-ml-llama 0.2.1.0, main.bend" (P1): "The configuration" (Cfg), "A layer" (block),
 *     "The model" (forward, forward_pre, argmax), "Sampling" (sample), "Loading" (tensor order).
 *   "Llama 3.1 8B Instruct" model card (P3): README "Entries" (decode, prefill, next_token),
 *     rope.linnet (llama3 tables), attention.linnet (decode/prefill; cache [Batch, KvHeads,
 *     MaxSeq, hd]; the where-clauses on head counts).
 *   "needle-core v2 model.rs" (P5): the preallocated per-sequence state and the error results
 *     of forward (position beyond the cache, token beyond the vocabulary).
 *
 * Conventions for every function:
 *   - The return value is an llm_status; LLM_OK (0) on success.  On failure nothing on the
 *     device has been changed unless stated, and llm_last_error(h) holds a message.
 *   - Pointers named *_host are host memory; *_dev are device memory of the handle's GPU.
 *     Functions without a _dev suffix take host pointers and return after the result is in
 *     host memory.  _dev functions are ordered on the handle's CUDA stream and do not wait
 *     for the GPU; call llm_synchronize() to wait and to collect errors found on the device.
 *   - The library never frees or keeps caller memory after a call returns.
 *   - One handle is used by one host thread at a time.  Results are deterministic: the same
 *     inputs on the same GPU give bit-identical outputs.
 */
#ifndef LLM_GB300_H
#define LLM_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t llm_status;
enum {
  LLM_OK = 0,
  LLM_ERR_CONFIG = 1,         /* invalid llm_config (P3 attention.linnet where-clauses)      */
  LLM_ERR_WEIGHTS_SIZE = 2,   /* nbytes differs from the layout count (P1 layout laws)        */
  LLM_ERR_OOM = 3,            /* device allocation failed in llm_create                      */
  LLM_ERR_POS_RANGE = 4,      /* position outside the cache or past the filled length (P5)    */
  LLM_ERR_TOKEN_RANGE = 5,    /* token id < 0 or >= vocab (P5 forward)                        */
  LLM_ERR_BATCH = 6,          /* batch < 1 or > max_batch                                    */
  LLM_ERR_ARG = 7,            /* another argument out of its documented range, or NULL       */
  LLM_ERR_CUDA = 8,           /* a CUDA runtime call failed (message in llm_last_error)      */
  LLM_ERR_DEVICE_TIMEOUT = 9  /* a bounded device-side wait gave up                          */
};

enum { LLM_DTYPE_F32 = 0, LLM_DTYPE_BF16 = 1 };

/*
 * Model shape and capacity (P1 Cfg; P3 nest.toml generics and rope.linnet constants).
 * Derived: head size hd = 2*half, query heads H = kv_heads*group, hidden d = H*hd,
 * key width kvw = kv_heads*hd.
 */
typedef struct llm_config {
  int32_t kv_heads;     /* key/value heads                                    */
  int32_t group;        /* query heads per key/value head (g)                 */
  int32_t half;         /* half a head; a head has 2*half numbers             */
  int32_t ffn;          /* MLP inner width                                    */
  int32_t layers;
  int32_t vocab;
  float eps;            /* RMSNorm epsilon                                    */
  float theta;          /* RoPE base                                          */
  int32_t tied;         /* 1: LM head = embedding; 0: untied lm_head at the end of the blob */
  int32_t rope_llama3;  /* 1: llama3 rescaling of the [half] frequency table  */
  float rope_factor, rope_low_freq, rope_high_freq, rope_orig_max_pos;
  int32_t max_batch;    /* cache rows                                         */
  int32_t max_seq;      /* cache positions per row                            */
  int32_t dtype;        /* LLM_DTYPE_BF16: bf16 weights and bf16 cache; LLM_DTYPE_F32: both f32 */
  int32_t debug_trace;  /* 1: keep per-layer intermediates (slow path, for llm_debug_trace) */
  int32_t tc_min_batch; /* bf16 only: steps of at least this many rows run the projections on the
                           tensor cores (TMA-fed tcgen05 GEMM), fewer rows on the weight-streaming
                           GEMV; 0: the library default (2: only batch-1 steps stream through the
                           GEMV); above max(max_batch, max_tokens): never.  Models whose hidden
                           or MLP width exceeds 16384 keep every step on the GEMV */
  int32_t max_tokens;   /* prompt tokens one prefill pass processes together (llm_prefill with
                           S > 1, llm_prefill_packed): activations and attention scratch are sized
                           for max(max_batch, max_tokens) rows; 0: the library default (512) */
  int32_t step_kernel;  /* batch-1 steps with bf16 weights (head size 64 or 128, at most 8 query
                           heads per kv head): 1 run all layers and the head as one persistent
                           kernel where the device allows it; 0 one kernel per operation (the
                           default: faster at the 8B shape so far) */
} llm_config;

typedef struct llm_handle llm_handle;

/* Number of weight values the blob of cfg must hold:
 *   V*d + L*(2d + 2d^2 + 2*kvw*d + 3*f*d) + d (+ V*d if untied)   (P1 "The configuration",
 *   Cfg.layer_size and Cfg.size). */
uint64_t llm_weight_count(const llm_config* cfg);

/*
 * Create a model on the current CUDA device.
 * weights: the blob in the tensor order of P1 "Loading" (t_layer): emb[V][d]; for each layer
 *   ln1[d] q[d][d] k[kvw][d] v[kvw][d] o[d][d] ln2[d] gate[f][d] up[f][d] down[d][f]; lnf[d];
 *   then lm_head[V][d] when untied.  Matrices are row-major [out][in].  Elements are bf16 bit
 *   patterns (uint16) for LLM_DTYPE_BF16, f32 otherwise.  weights_on_device selects whether
 *   `weights` is a device pointer (1) or host pointer (0).  The library copies and repacks the
 *   weights into its own device memory; the caller keeps ownership of `weights`.
 * nbytes must equal llm_weight_count(cfg) * element size, else LLM_ERR_WEIGHTS_SIZE.
 * cuda_stream: the cudaStream_t every call is ordered on (NULL: the library creates one).
 * All device memory (weights, KV cache [layers][max_batch][kv][max_seq][hd], activations,
 * scratch) is allocated here; no later call allocates.
 */
llm_status llm_create(const llm_config* cfg, const void* weights, uint64_t nbytes,
                      int32_t weights_on_device, void* cuda_stream, llm_handle** out);
llm_status llm_destroy(llm_handle* h);

/* Mark every cache row empty (filled length 0); the cache memory is not cleared (P5 reset). */
llm_status llm_reset(llm_handle* h);

/*
 * Prefill (P3 "prefill<S>(tokens, pos)"; P1 forward_pre for every position but the last):
 * rows 0..B-1 take tokens[b*S + i] at positions pos+i, i < S; their keys and values are written
 * to the cache, and token i of row b attends to positions 0..pos+i of its row.  logits_host
 * [B][V] (may be NULL: no final norm / head) receives the logits after the last token.  The
 * B*S tokens run as passes of whole positions, at most max(B, max_tokens) tokens each: a pass is
 * one step whose rows are its tokens (projections on the tensor cores once a pass has
 * tc_min_batch tokens), and only the last tokens go through the final norm and the LM head.
 * Requires 1 <= B <= max_batch (else LLM_ERR_BATCH), S >= 1 (else LLM_ERR_ARG),
 * 0 <= pos <= filled length of every row b < B and pos + S <= max_seq (else LLM_ERR_POS_RANGE),
 * tokens in [0, vocab) (else LLM_ERR_TOKEN_RANGE).  On success the filled length of rows
 * b < B becomes pos + S (positions after it are dead and never read).
 */
llm_status llm_prefill(llm_handle* h, const int32_t* tokens_host, int32_t B, int32_t S,
                       int32_t pos, float* logits_host);

/*
 * One decode step (P3 "decode(token, pos)"; P1 forward): row b takes tokens[b] at position
 * pos, writes its key and value at pos and attends over cache positions 0..pos inclusive;
 * logits_host [B][V] receives the logits.  Same checks as llm_prefill with S = 1.  A pos
 * below the filled length rewinds the row.  After success the filled length is pos + 1.
 */
llm_status llm_decode(llm_handle* h, const int32_t* tokens_host, int32_t B, int32_t pos,
                      float* logits_host);

/*
 * Sampling (P1 "Sampling": sample(xs, temp, k, p, u); argmax).  For each row b of logits [B][V]:
 *   temp == 0: ids[b] = the first index of the largest logit (greedy; k, p and u unused);
 *   temp > 0: the k largest logits (k > V clamps to V; ties: lower id first) weigh
 *     exp(v/temp - top/temp); top-p keeps each candidate whose cumulative weight before it is
 *     below p * Z (the first is always kept); the draw u[b] in [0, 1) returns the first kept
 *     candidate whose cumulative weight is above u[b] * Zp, else the last kept.
 * Arguments: temp >= 0, k >= 1, 0 < p <= 1, 0 <= u[b] < 1, else LLM_ERR_ARG.  The exp of the
 * weights is a fixed sequence of IEEE operations, so ids can be reproduced bit for bit on a CPU.
 */
llm_status llm_sample(llm_handle* h, const float* logits_host, int32_t B, float temp, int32_t k,
                      float p, const float* u_host, int32_t* ids_host);

/*
 * A generation step: llm_decode then llm_sample on the device, without moving the logits.
 * ids_host [B] receives the drawn tokens; logits_host (may be NULL) the logits; u_host may be
 * NULL when temp == 0.  Same checks as the two calls.
 */
llm_status llm_step(llm_handle* h, const int32_t* tokens_host, int32_t B, int32_t pos, float temp,
                    int32_t k, float p, const float* u_host, int32_t* ids_host, float* logits_host);

/* Device-pointer variants: the same operations on device buffers, ordered on the handle's
 * stream, returning without waiting.  Position, batch and argument checks happen on the host
 * before launch; token ids are checked on the device (an out-of-range id is replaced by 0 and
 * LLM_ERR_TOKEN_RANGE is reported by the next llm_synchronize). */
llm_status llm_prefill_dev(llm_handle* h, const int32_t* tokens_dev, int32_t B, int32_t S,
                           int32_t pos, float* logits_dev);
llm_status llm_decode_dev(llm_handle* h, const int32_t* tokens_dev, int32_t B, int32_t pos,
                          float* logits_dev);
llm_status llm_sample_dev(llm_handle* h, const float* logits_dev, int32_t B, float temp, int32_t k,
                          float p, const float* u_dev, int32_t* ids_dev);
llm_status llm_step_dev(llm_handle* h, const int32_t* tokens_dev, int32_t B, int32_t pos, float temp,
                        int32_t k, float p, const float* u_dev, int32_t* ids_dev, float* logits_dev);

/*
 * Rows at their own positions (continuous batching; Llama 3.1 8B Instruct card, "Entries":
 * decode_rows(tokens, positions)):
 * row b takes tokens[b] at position positions_host[b], writes its key and value there and
 * attends over its own cache positions 0..positions_host[b] inclusive; the other rows' positions
 * do not affect it.  positions_host [B] is always host memory (read before the call returns).
 * Checks: 1 <= B <= max_batch (else LLM_ERR_BATCH); 0 <= positions_host[b] < max_seq and
 * positions_host[b] <= filled length of row b (else LLM_ERR_POS_RANGE); tokens in [0, vocab)
 * (host tokens: LLM_ERR_TOKEN_RANGE; device tokens: as llm_decode_dev).  After success the
 * filled length of row b is positions_host[b] + 1.  With every position equal these are
 * llm_decode / llm_step bit for bit.  llm_decode_rows writes logits [B][V]; llm_step_rows
 * samples as llm_step (ids [B], logits optional, u may be NULL when temp == 0).
 */
llm_status llm_decode_rows(llm_handle* h, const int32_t* tokens_host, int32_t B,
                           const int32_t* positions_host, float* logits_host);
llm_status llm_decode_rows_dev(llm_handle* h, const int32_t* tokens_dev, int32_t B,
                               const int32_t* positions_host, float* logits_dev);
llm_status llm_step_rows(llm_handle* h, const int32_t* tokens_host, int32_t B,
                         const int32_t* positions_host, float temp, int32_t k, float p,
                         const float* u_host, int32_t* ids_host, float* logits_host);
llm_status llm_step_rows_dev(llm_handle* h, const int32_t* tokens_dev, int32_t B,
                             const int32_t* positions_host, float temp, int32_t k, float p,
                             const float* u_dev, int32_t* ids_dev, float* logits_dev);

/*
 * Packed prefill (Llama 3.1 8B Instruct card, "Entries": prefill_packed(tokens, rows, positions,
 * segments, last)): P tokens of several prompts packed end to end; token p is position
 * positions_host[p] of prompt segments_host[p] (any int32 id) in cache row rows_host[p].  Every
 * token's key and value are written at its row and position, and each token attends to its own
 * prompt's tokens up to its position and to nothing else (not to its row's older cache).
 * logits_host [nlast][V] (may be NULL) receives the logits after token last_host[m].  Checks:
 * P >= 1 and nlast >= 0 (LLM_ERR_ARG); rows in
 * [0, max_batch) (LLM_ERR_BATCH); positions in [0, max_seq) (LLM_ERR_POS_RANGE); tokens in
 * [0, vocab) (LLM_ERR_TOKEN_RANGE); each prompt in one row at consecutive positions, each once,
 * prompts of a row not overlapping, no two tokens in one (row, position), last[m] in [0, P)
 * (LLM_ERR_ARG).  The tokens run in position order as passes of at most max(max_batch,
 * max_tokens) tokens, like llm_prefill's; on success each prompt's row is filled at least to its
 * last position + 1.  All arrays are host memory; the call returns when done.
 */
llm_status llm_prefill_packed(llm_handle* h, const int32_t* tokens_host, const int32_t* rows_host,
                              const int32_t* positions_host, const int32_t* segments_host, int32_t P,
                              const int32_t* last_host, int32_t nlast, float* logits_host);

/*
 * Paged caches (Llama 3.1 8B Instruct card, "Entries": decode_paged(tokens, positions, table)):
 * the key/value caches of a handle form one pool of max_batch * (max_seq / 64) pages of 64
 * positions (page q = positions (q % (max_seq/64))*64 .. +63 of cache row q / (max_seq/64)).
 * Row b takes tokens[b] at position positions_host[b]; its position p lies in pool page
 * table_host[b*pages_per_row + p/64], where the step writes its key and value and from which
 * attention reads positions 0..positions_host[b].  Which pages hold which sequence is the
 * caller's (a serving layer's) to manage: the filled lengths are not consulted or changed, and
 * pages written by earlier paged steps are read as they are.  Requires max_seq % 64 == 0 (else
 * LLM_ERR_CONFIG), 1 <= B <= max_batch (LLM_ERR_BATCH), 1 <= pages_per_row <= max_seq/64
 * (LLM_ERR_ARG), 0 <= positions_host[b] < pages_per_row*64 (LLM_ERR_POS_RANGE), every page
 * entry for positions 0..positions_host[b] inside the pool (LLM_ERR_ARG), tokens as llm_decode.
 * positions_host [B] and table_host [B][pages_per_row] are host memory, read before the call
 * returns.  With table[b][i] = b*(max_seq/64) + i (every row its own pages, in order) the step
 * is llm_decode_rows bit for bit.  llm_step_paged samples as llm_step.
 */
llm_status llm_decode_paged(llm_handle* h, const int32_t* tokens_host, int32_t B,
                            const int32_t* positions_host, const int32_t* table_host,
                            int32_t pages_per_row, float* logits_host);
llm_status llm_decode_paged_dev(llm_handle* h, const int32_t* tokens_dev, int32_t B,
                                const int32_t* positions_host, const int32_t* table_host,
                                int32_t pages_per_row, float* logits_dev);
llm_status llm_step_paged(llm_handle* h, const int32_t* tokens_host, int32_t B,
                          const int32_t* positions_host, const int32_t* table_host,
                          int32_t pages_per_row, float temp, int32_t k, float p,
                          const float* u_host, int32_t* ids_host, float* logits_host);
llm_status llm_step_paged_dev(llm_handle* h, const int32_t* tokens_dev, int32_t B,
                              const int32_t* positions_host, const int32_t* table_host,
                              int32_t pages_per_row, float temp, int32_t k, float p,
                              const float* u_dev, int32_t* ids_dev, float* logits_dev);

/*
 * Generation inside CUDA graphs (Llama 3.1 8B Instruct card, "Entries": generate<Steps>(token,
 * pos), sample<Steps>(...)): n_steps decode + draw steps; step s (0 <= s < n_steps) runs every row
 * b < B at position pos + s on the token drawn by step s - 1 (tokens[b] for s = 0) and draws
 * ids[s*B + b] as llm_step would with u[s*B + b] (u may be NULL when temp == 0).  The steps run
 * as graphs of 8 steps (then single steps) with no host work between the steps of a graph; the
 * ids equal those of n_steps chained llm_step calls bit for bit.  Checks as llm_step for every
 * step: n_steps >= 1 (else LLM_ERR_ARG), pos <= filled length of every row and pos + n_steps <=
 * max_seq (else LLM_ERR_POS_RANGE); handles created with debug_trace = 1 are refused
 * (LLM_ERR_ARG).  ids [n_steps][B]; after success the filled length of rows b < B is
 * pos + n_steps and the logits buffer holds the last step's logits.  llm_generate: host tokens,
 * draws and ids (returns when done); llm_generate_dev: device buffers, stream-ordered.
 */
llm_status llm_generate(llm_handle* h, const int32_t* tokens_host, int32_t B, int32_t pos,
                        int32_t n_steps, float temp, int32_t k, float p, const float* u_host,
                        int32_t* ids_host);
llm_status llm_generate_dev(llm_handle* h, const int32_t* tokens_dev, int32_t B, int32_t pos,
                            int32_t n_steps, float temp, int32_t k, float p, const float* u_dev,
                            int32_t* ids_dev);

/* Wait for the handle's stream; return the first error recorded on the device since the last
 * call (LLM_ERR_TOKEN_RANGE, LLM_ERR_DEVICE_TIMEOUT) and clear it. */
llm_status llm_synchronize(llm_handle* h);

/* The handle's stream (cudaStream_t) and its internal logits buffer [max_batch][V] (f32, device),
 * which decode writes; passing it back as logits_dev avoids a copy. */
void* llm_stream(llm_handle* h);
float* llm_logits_buffer(llm_handle* h);

/* Filled length of cache row b (-1 if b is out of range). */
int32_t llm_filled(const llm_handle* h, int32_t b);

/* A message for the last failure on h (owned by h; valid until the next call); with h == NULL,
 * why the last llm_create on the calling thread failed.  And a name for a status code. */
const char* llm_last_error(const llm_handle* h);
const char* llm_status_string(llm_status s);

/*
 * Test hooks.  kv_import / kv_export copy n positions starting at pos0 of one layer and cache
 * row, for every key/value head, from / to host memory laid out [kv][n][hd] in the cache element
 * type (bf16 bits or f32).  kv_import raises the row's filled length to at least pos0 + n.
 * Positions must satisfy 0 <= pos0, pos0 + n <= max_seq (else LLM_ERR_POS_RANGE).
 */
llm_status llm_kv_import(llm_handle* h, int32_t layer, int32_t row, int32_t pos0, int32_t n,
                         const void* k_host, const void* v_host);
llm_status llm_kv_export(llm_handle* h, int32_t layer, int32_t row, int32_t pos0, int32_t n,
                         void* k_host, void* v_host);

/*
 * Intermediates of the last decode step of layer `layer`, kept only when created with
 * debug_trace = 1 (the step then runs kernel by kernel on the weight-streaming path, not as a
 * graph).  Names after P1 "A layer" (Act): "n1" (attention_norm output [d]), "q" [d], "k" [kvw],
 * "v" [kvw] (projections before RoPE, heads in order), "qr" [d] and "kr" [kvw] (after RoPE; "kr"
 * in f32, before the cache's rounding), "attn" (attention output [d]), "a" (o_proj output
 * [d]), "x1" (x + a [d]), "n2" (ffn_norm output [d]), "swiglu" (silu(gate) * up [f]), "m" (down
 * projection output [d]), "y" (layer output x1 + m [d]).  dst_host receives [max_batch][width]
 * f32 (rows past the step's B are stale).  LLM_ERR_ARG for an unknown name or layer.
 */
llm_status llm_debug_trace(llm_handle* h, int32_t layer, const char* name, float* dst_host);

/*
 * Measurement hook: the mean duration of `reps` back-to-back launches of one kernel of the
 * decode step, timed alone with CUDA events on the handle's stream.  which: 0 Q/K/V projection
 * (with norm, RoPE and cache write), 1 attention, 2 o_proj + residual, 3 norm + gate/up +
 * SwiGLU, 4 down + residual, 5 final norm + LM head, 6 sampler.  Launch r uses layer r % layers,
 * so consecutive launches stream different weights from HBM.  B rows at position pos (pos <=
 * filled length; the cache entry at pos is rewritten).  *ms_per_launch receives the mean.
 */
llm_status llm_profile_kernel(llm_handle* h, int32_t which, int32_t B, int32_t pos, int32_t reps,
                              float* ms_per_launch);

/*
 * Test hook for the device-timeout report (needle-core v2 model.rs: forward returns an error
 * result instead of failing the process).  Launches, on the handle's stream, one small kernel
 * that waits on a shared-memory barrier nothing arrives on, with the same bounded wait the
 * kernels' copy rings use and a limit of limit_cycles SM cycles (1..1e9, else LLM_ERR_ARG).  The
 * wait runs out and the kernel records LLM_ERR_DEVICE_TIMEOUT in the handle's status word, which
 * the next llm_synchronize reports once (and clears, with the attention's merge counters).
 * Nothing faults or hangs; the handle stays usable.
 */
llm_status llm_check_wait_timeout(llm_handle* h, int64_t limit_cycles);

/*
 * How many kernels one llm_step / llm_step_dev of B rows launches at temperature temp and top-k
 * k (greedy when temp == 0; a draw with min(k, vocab) <= 1024 candidates is one selection
 * kernel, a larger one the sort of the whole row): the step prologue plus the kernels of the
 * step's CUDA graph, which this call captures if it does not exist yet (no kernel runs).
 * LLM_ERR_BATCH for B outside 1..max_batch; LLM_ERR_ARG for handles created with debug_trace
 * (they run without a graph).
 */
llm_status llm_step_kernels(llm_handle* h, int32_t B, float temp, int32_t k, int32_t* kernels);

/*
 * Sampling without a handle and without allocating: the same draw as llm_sample_dev (greedy
 * when temp == 0, else temperature / top-k / top-p with the draws u_dev), for callers that
 * cannot call cudaMalloc -- code running inside an allocator or memory-pool callback, plugins
 * whose host application owns all device memory, processes that reserved every byte up front.
 * The pages have no counterpart; this is a convenience of this library.
 * logits_dev [B][V] f32, u_dev [B] (may be NULL when temp == 0), ids_dev [B]: device memory of
 * the current device; the work is ordered on cuda_stream and the call returns without waiting.
 * The sort buffers live in one fixed device array inside the library, present on every GPU that
 * loads it until the process exits: B * (V rounded up to 32) must not exceed
 * LLM_SAMPLE_NOALLOC_MAX_ELEMS, else LLM_ERR_ARG (as for B < 1, V < 1, NULL pointers or the
 * argument ranges of llm_sample).  Calls share that array, so calls that overlap on the GPU race.
 * The array is created lazily, with the library's CUDA module that holds it: the first call on a
 * device (with it current) -- or llm_create on that device, which does the same set-up -- loads
 * that module, which reserves the array's memory, and looks up its device address.  Make that
 * first call (or llm_create) where allocating is allowed and before any stream capture on the
 * device.  Later calls allocate nothing; after cudaDeviceReset (a new context) the next call
 * looks the address up again and so counts as a first call.
 */
#define LLM_SAMPLE_NOALLOC_MAX_ELEMS 262144
llm_status llm_sample_noalloc(const float* logits_dev, int32_t B, int32_t V, float temp, int32_t k,
                              float p, const float* u_dev, int32_t* ids_dev, void* cuda_stream);

#ifdef __cplusplus
}
#endif
#endif
