// libllm: the C ABI (include/llm.h) over the decode-step kernels.
//
// One handle = one model on one GPU: weights repacked once into the layouts the kernels
// stream, the KV cache [layers][max_batch][kv][max_seq][hd], activations and scratch, all
// allocated in llm_create (needle-core v2 model.rs, V2State: the per-sequence state is
// preallocated so that a step does no allocation).  A decode step is captured once per
// (batch, mode) as a CUDA graph of programmatic-dependent launches:
//   step prologue (position, tokens, sampling parameters into device memory)
//   -> embedding -> per layer {QKV+norm+RoPE+KV write, attention, o_proj+residual,
//      norm+gate/up+SwiGLU, down+residual} -> final norm + LM head -> sampler.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <map>
#include <string>
#include <vector>

#include "attention.cuh"
#include "common.cuh"
#include "gemm.cuh"
#include "mega.cuh"
#include "gemv.cuh"
#include "llm.h"
#include "sampler.cuh"
#include "tc.cuh"

using namespace llm;

namespace {

constexpr int kInline = 64;  // rows whose token / draw travel inside the prologue's arguments

constexpr int kGenChunk = 8;  // steps per generation graph

constexpr int kDefaultTokens = 512;  // prompt tokens per prefill pass unless the config says

// where the steps of one generation graph launch read and write (set before each launch)
struct GenState {
  int32_t pos;          // position of the graph's first step
  int32_t B;
  float temp;
  int32_t k;
  float p;
  int32_t pad;
  const int32_t* prev;  // [B] tokens of the first step
  const float* u;       // [steps][B] draws (temp > 0)
  int32_t* ids;         // [steps][B] drawn tokens
};

struct BeginArgs {
  StepState* st;
  int32_t pos, B;          // pos: every row's position, unless the rows sit at their own:
  int32_t own_pos;         //   then pos_dev[b] (B > kInline) or pos_inline[b]
  const int32_t* pos_dev;
  const int32_t* table;    // paged step: [B][table_stride] pages, or null
  int32_t table_stride;
  const int32_t* ranges;   // prefill pass: [3][B] attention starts, first written positions, cache rows
  uint32_t* mega_bar;      // the persistent step kernel's barrier counter, reset here (or null)
  float temp;
  int32_t k;
  float p;
  int32_t vocab;
  const int32_t* tok_dev;  // token of row b at (b / tok_np) * tok_stride + b % tok_np + tok_col,
  int32_t tok_stride, tok_col, tok_np;  // or NULL: tok_inline
  const float* u_dev;      // or NULL: u_inline
  int32_t* tok_buf;        // [NT]
  float* u_buf;            // [NT]
  int32_t* status;
  int32_t tok_inline[kInline];
  float u_inline[kInline];
  int32_t pos_inline[kInline];
};

__global__ void step_begin_kernel(const BeginArgs a) {
  const int t = threadIdx.x;
  __shared__ int32_t s_max;
  if (t == 0) {
    s_max = 0;
    a.st->B = a.B;
    a.st->temp = a.temp;
    a.st->k = a.k;
    a.st->p = a.p;
    a.st->table = a.table;
    a.st->table_stride = a.table_stride;
    a.st->ranges = a.ranges ? 1 : 0;
    a.st->rowmap = a.ranges ? reinterpret_cast<int32_t*>(a.st + 1) + 3 * a.B : nullptr;
    if (a.mega_bar) *a.mega_bar = 0u;
  }
  __syncthreads();
  int32_t* rowpos = reinterpret_cast<int32_t*>(a.st + 1);
  for (int b = t; b < a.B; b += blockDim.x) {
    const int32_t pb = !a.own_pos ? a.pos : a.pos_dev ? a.pos_dev[b] : a.pos_inline[b];  // validated by the host
    rowpos[b] = pb;
    if (a.ranges) {
      rowpos[a.B + b] = a.ranges[b];
      rowpos[2 * a.B + b] = a.ranges[a.B + b];
      rowpos[3 * a.B + b] = a.ranges[2 * a.B + b];
    }
    atomicMax(&s_max, pb);
  }
  __syncthreads();
  if (t == 0) a.st->pos = s_max;
  for (int b = t; b < a.B; b += blockDim.x) {
    int tok = a.tok_dev ? a.tok_dev[(size_t)(b / a.tok_np) * a.tok_stride + b % a.tok_np + a.tok_col] : a.tok_inline[b];
    if (tok < 0 || tok >= a.vocab) {
      atomicCAS(a.status, 0, kErrTokenRange);
      tok = 0;
    }
    a.tok_buf[b] = tok;
    a.u_buf[b] = a.u_dev ? a.u_dev[b] : b < kInline ? a.u_inline[b] : 0.0f;
  }
}

// step i of a generation graph: the prologue of a step at position gen.pos + i whose tokens are
// the previous step's draws (gen.prev for i == 0) and whose draws are gen.u[i]
__global__ void gen_begin_kernel(StepState* st, const GenState* gen, int32_t* tok_buf, float* u_buf, int i,
                                 uint32_t* mega_bar) {
  const GenState g = *gen;
  const int t = threadIdx.x;
  if (t == 0) {
    if (mega_bar) *mega_bar = 0u;
    st->pos = g.pos + i;
    st->B = g.B;
    st->temp = g.temp;
    st->k = g.k;
    st->p = g.p;
    st->table = nullptr;
    st->table_stride = 0;
    st->ranges = 0;
    st->rowmap = nullptr;
  }
  int32_t* rowpos = reinterpret_cast<int32_t*>(st + 1);
  for (int b = t; b < g.B; b += blockDim.x) {
    rowpos[b] = g.pos + i;
    tok_buf[b] = i == 0 ? g.prev[b] : g.ids[(size_t)(i - 1) * g.B + b];
    u_buf[b] = g.temp > 0.0f ? g.u[(size_t)i * g.B + b] : 0.0f;
  }
}

// the end of step i: its draws into gen.ids[i]
__global__ void gen_end_kernel(const GenState* gen, const int32_t* ids_buf, int i) {
  const int B = gen->B;
  int32_t* out = gen->ids + (size_t)i * B;
  for (int b = threadIdx.x; b < B; b += blockDim.x) out[b] = ids_buf[b];
}

__global__ void gen_set_kernel(GenState* gen, const GenState v) { *gen = v; }

// a bounded wait that runs out: an mbarrier that nothing arrives on, waited on with the same
// bounded wait as the kernels' copy rings; on timeout the status word records it (needle-core
// v2 model.rs: a failed step is an error result, not a crash)
__global__ void wait_timeout_kernel(int32_t* status, uint64_t limit_cycles) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    mbar_fence_init();
  }
  __syncthreads();
  const bool ok = __all_sync(0xffffffffu, mbar_wait(b, 0, limit_cycles));
  if (!ok && threadIdx.x == 0) atomicCAS(status, 0, kErrDeviceTimeout);
}

template <int WT>
__global__ void embed_kernel(const void* emb, const int32_t* tok, float* x, int d, int x_stride) {
  grid_dep_wait();
  grid_dep_launch();
  const int b = blockIdx.y;
  const size_t row = (size_t)tok[b] * d;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < d; i += gridDim.x * blockDim.x)
    x[(size_t)b * x_stride + i] = load_elem<WT>(emb, row + i);
}

// row gather used by the repacking: dst row r = src row map[r], rows of `row_bytes` bytes
__global__ void gather_rows_kernel(char* dst, const char* src, const int64_t* map, int64_t nrows,
                                   int64_t row_bytes) {
  for (int64_t r = blockIdx.x; r < nrows; r += gridDim.x) {
    const uint4* s = reinterpret_cast<const uint4*>(src + map[r] * row_bytes);
    uint4* o = reinterpret_cast<uint4*>(dst + r * row_bytes);
    for (int64_t c = threadIdx.x; c < row_bytes / 16; c += blockDim.x) o[c] = s[c];
  }
}

template <int WT>
__global__ void widen_kernel(float* dst, const void* src, int64_t n) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    dst[i] = load_elem<WT>(src, (uint64_t)i);
}

// P1 inv_freq (1 / theta^(2i/hd)) and the llama3 band rescaling of the Llama 3.1 8B card
// (rope.linnet tables), every step an IEEE f32 operation; theta^e is the f32 rounding of the
// double power.  Then cos/sin of t * inv[i] (f32 product), rounded from double.
struct RopeArgs {
  float theta;
  int hd, half, cap, llama3;
  float factor, low, high, orig;
  float* cs;
  float* sn;
};

__device__ float rope_inv(const RopeArgs& a, int i) {
  const float PI = 3.14159265f;
  const float e = __fdiv_rn((float)(2 * i), (float)a.hd);
  const float pw = (float)pow((double)a.theta, (double)e);
  const float base = __fdiv_rn(1.0f, pw);
  if (!a.llama3) return base;
  const float wavelen = __fdiv_rn(__fmul_rn(2.0f, PI), base);
  const float low_wl = __fdiv_rn(a.orig, a.low), high_wl = __fdiv_rn(a.orig, a.high);
  const float smooth = __fdiv_rn(__fsub_rn(__fdiv_rn(a.orig, wavelen), a.low), __fsub_rn(a.high, a.low));
  const float smoothed = __fadd_rn(__fmul_rn(__fsub_rn(1.0f, smooth), __fdiv_rn(base, a.factor)),
                                   __fmul_rn(smooth, base));
  if (wavelen > low_wl) return __fdiv_rn(base, a.factor);
  if (wavelen < high_wl) return base;
  return smoothed;
}

__global__ void rope_table_kernel(const RopeArgs a) {
  const int64_t n = (int64_t)a.cap * a.half;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < n; idx += (int64_t)gridDim.x * blockDim.x) {
    const int t = (int)(idx / a.half), i = (int)(idx % a.half);
    const float ang = __fmul_rn((float)t, rope_inv(a, i));
    a.cs[idx] = (float)cos((double)ang);
    a.sn[idx] = (float)sin((double)ang);
  }
}

}  // namespace

// ---------------------------------------------------------------------------------------
// the handle
// ---------------------------------------------------------------------------------------

struct LayerW {
  void* qkv;   // packed [(H + 2kv) * hd][d], rows in RoPE pairs
  float* ln1;  // [d]
  void* o;     // [d][d]
  float* ln2;
  void* gu;    // packed [2f][d], rows (gate i, up i)
  void* down;  // [d][f]
};

struct TcMaps {
  CUtensorMap qkv, o, gu, down;
};

struct GraphKey {
  int B, mode, gen;  // gen: steps of a generation graph (0: one step after a host prologue)
  int pass;          // 1: a prefill pass (its rows are prompt tokens with attention ranges)
  bool operator<(const GraphKey& o) const {
    return B != o.B ? B < o.B : mode != o.mode ? mode < o.mode : gen != o.gen ? gen < o.gen : pass < o.pass;
  }
};


// the intermediates of a traced step, per layer (bend-ml-llama "A layer", Act: n1, q, k, v, qr,
// kr, attn, a, n2, m, y; plus x1 = x + a and the SwiGLU activations)
enum { TR_N1 = 0, TR_QKV, TR_QR, TR_KR, TR_ATTN, TR_A, TR_X1, TR_N2, TR_SWIGLU, TR_M, TR_Y, kTraceSlots };

// what follows the layers: nothing, the LM head, or the head and a greedy / top-k top-p draw
// (MODE_TOPK: top-k of at most sample_select_max() candidates, by a radix select; MODE_TOPP: a
// sort of the whole row)
enum { MODE_NOHEAD = 0, MODE_HEAD = 1, MODE_GREEDY = 2, MODE_TOPP = 3, MODE_TOPK = 4 };

struct llm_handle {
  llm_config cfg;
  int hd, H, d, kvw, f, V, L, wt, es;
  int NT;  // rows of the activation and attention buffers: max(max_batch, max_tokens)
  int dev, num_sms, smem_optin;
  cudaStream_t stream = nullptr, cap_stream = nullptr;
  bool own_stream = false;
  std::vector<void*> allocs;
  void* emb = nullptr;
  void* head = nullptr;
  float* lnf = nullptr;
  std::vector<LayerW> lw;
  void* kc = nullptr;  // [L][max_batch][kv][cap][hd]
  void* vc = nullptr;
  size_t layer_cache_elems = 0;
  float *rope_cos = nullptr, *rope_sin = nullptr;
  float *xa = nullptr, *xb = nullptr, *q = nullptr, *attn = nullptr, *m = nullptr, *logits = nullptr;
  float* part = nullptr;
  uint32_t* ticket = nullptr;
  int ticket_count = 0;
  int part_ns = 0;
  CUtensorMap kmap, vmap;  // the key and value caches as [layers * max_batch * kv * max_seq][hd]
  StepState* st = nullptr;
  int32_t* pos_buf = nullptr;  // [NT] positions of the rows of a step (or the entries of a pass) at their own positions
  GenState* gen = nullptr;     // generation: the state of the graph launch in flight
  int32_t* page_table = nullptr;  // paged steps: [max_batch][max_seq / kPage] (max_seq % kPage == 0)
  int32_t* range_buf = nullptr;   // prefill passes: [3][NT] attention starts, first written positions, cache rows
  int32_t* tile_buf = nullptr;    // prefill passes: the causal attention's tiles and units (attention.cuh)
  bool pf_attn = false;           // prefill passes run the tiled causal attention (bf16, head 64 / 128)
  float* xh = nullptr;            // [max_batch][d] final residual rows gathered for the LM head
  int32_t* head_map = nullptr;    // [max_batch] the entries those rows come from
  // batch-1 steps in one persistent kernel (bf16, supported shapes)
  bool mega = false;
  bool capturing_pass = false;  // the graph being captured is a prefill pass (never the persistent kernel)
  MegaLayer* mega_layers = nullptr;  // [L], device
  float* mega_part = nullptr;        // attention partials [H][kMegaMaxSplits][hd + 2]
  uint32_t* mega_ticket = nullptr;   // [kv + 1]
  uint32_t* mega_bar = nullptr;      // grid barrier counter (reset by each step's prologue)
  float* mega_cv = nullptr;          // [num_sms] argmax candidates
  int32_t* mega_ci = nullptr;
  float* u_gen = nullptr;      // [kGenChunk][max_batch] draws of one host-memory generation launch
  int32_t* ids_gen = nullptr;  // [kGenChunk][max_batch] its drawn tokens
  int32_t* status = nullptr;
  int32_t* tok_buf = nullptr;
  float* u_buf = nullptr;
  int32_t* ids_buf = nullptr;
  uint32_t* s_keys = nullptr;
  int32_t* s_idx = nullptr;
  float* s_pre = nullptr;
  uint32_t* s_hist = nullptr;
  int V_pad = 0;
  float* trace = nullptr;  // [L][kTraceSlots][max_batch][trace_w]: a traced handle's intermediates
  size_t trace_w = 0;      // max(d + 2 kvw, f)
  bool tracing = false;    // the kernels being launched write the trace
  // tensor-core projections (bf16, steps of at least tc_min rows)
  int tc_min = 0;          // 0: the tensor-core path is off for this handle
  std::vector<TcMaps> tmaps;
  CUtensorMap tmap_head;
  uint16_t* tc_xs = nullptr;    // split activations [2][Ntot][max(d, f)]
  float* tc_part = nullptr;     // split sums of the last projection [S][B][rows]
  std::map<std::pair<int, int>, CUtensorMap> xmaps;  // (K, B) -> map over tc_xs
  std::vector<int32_t> filled;
  std::map<GraphKey, std::pair<cudaGraphExec_t, int>> graphs;  // executable graph, kernels in it
  std::string err;
};

namespace {

thread_local std::string g_create_err;  // why the last llm_create on this thread failed

llm_status fail(llm_handle* h, llm_status s, const char* fmt, ...) {
  if (h) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    h->err = buf;
  }
  return s;
}

#define CUDA_TRY(h, call)                                                                     \
  do {                                                                                        \
    cudaError_t e_ = (call);                                                                  \
    if (e_ != cudaSuccess) return fail((h), LLM_ERR_CUDA, "%s: %s", #call, cudaGetErrorString(e_)); \
  } while (0)

uint64_t count_of(const llm_config* c) {
  const uint64_t hd = 2 * (uint64_t)c->half, H = (uint64_t)c->kv_heads * (uint64_t)c->group;
  const uint64_t d = H * hd, kvw = (uint64_t)c->kv_heads * hd, f = (uint64_t)c->ffn, V = (uint64_t)c->vocab;
  const uint64_t layer = 2 * d + 2 * d * d + 2 * kvw * d + 3 * f * d;
  return V * d + (uint64_t)c->layers * layer + d + (c->tied ? 0 : V * d);
}

const char* check_config(const llm_config* c) {
  if (c->kv_heads <= 0 || c->group <= 0 || c->half <= 0 || c->ffn <= 0 || c->layers <= 0 || c->vocab <= 0)
    return "kv_heads, group, half, ffn, layers and vocab must be positive";
  if (c->max_batch <= 0 || c->max_seq <= 0) return "max_batch and max_seq must be positive";
  if (c->max_tokens < 0 || c->max_tokens > 65535) return "max_tokens must be in 0..65535";
  if (c->dtype != LLM_DTYPE_F32 && c->dtype != LLM_DTYPE_BF16) return "dtype must be LLM_DTYPE_F32 or LLM_DTYPE_BF16";
  if (!(c->eps >= 0.0f) || !(c->theta > 0.0f)) return "eps must be >= 0 and theta > 0";
  if (c->rope_llama3 && !(c->rope_factor > 0.0f && c->rope_low_freq > 0.0f && c->rope_high_freq > c->rope_low_freq &&
                          c->rope_orig_max_pos > 0.0f))
    return "llama3 rope scaling needs factor > 0, 0 < low_freq < high_freq, orig_max_pos > 0";
  const int hd = 2 * c->half;
  if (!attn_supported(hd, c->group)) return "head size must be 16, 32, 64, 128 or 256 and group at most 16";
  const int per16 = c->dtype == LLM_DTYPE_BF16 ? 8 : 4;
  const int64_t d = (int64_t)c->kv_heads * c->group * hd;
  if (d % per16 || c->ffn % per16) return "hidden and ffn widths must fill whole 16-byte chunks";
  if ((int64_t)c->max_seq * c->max_batch > (int64_t)1 << 40) return "cache too large";
  return nullptr;
}

template <class T>
llm_status dalloc(llm_handle* h, T** p, size_t bytes) {
  void* v = nullptr;
  if (bytes == 0) bytes = 16;
  cudaError_t e = cudaMalloc(&v, bytes);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(h, LLM_ERR_OOM, "cudaMalloc(%zu bytes): %s", bytes, cudaGetErrorString(e));
  }
  h->allocs.push_back(v);
  *p = static_cast<T*>(v);
  return LLM_OK;
}

#define TRY(x)                  \
  do {                          \
    llm_status s_ = (x);        \
    if (s_ != LLM_OK) return s_; \
  } while (0)

// ---- repacking of one layer's tensors from the blob (device copy) ----
llm_status gather(llm_handle* h, void* dst, const char* src, const std::vector<int64_t>& map, int64_t row_bytes,
                  int64_t* dmap) {
  CUDA_TRY(h, cudaMemcpyAsync(dmap, map.data(), map.size() * 8, cudaMemcpyHostToDevice, h->stream));
  gather_rows_kernel<<<1024, 256, 0, h->stream>>>((char*)dst, src, dmap, (int64_t)map.size(), row_bytes);
  CUDA_TRY(h, cudaGetLastError());
  CUDA_TRY(h, cudaStreamSynchronize(h->stream));
  return LLM_OK;
}

llm_status widen(llm_handle* h, float* dst, const char* src, int64_t n) {
  if (h->wt) widen_kernel<1><<<64, 256, 0, h->stream>>>(dst, src, n);
  else widen_kernel<0><<<64, 256, 0, h->stream>>>(dst, src, n);
  CUDA_TRY(h, cudaGetLastError());
  return LLM_OK;
}

llm_status load_weights(llm_handle* h, const char* blob /* device */) {
  const int64_t d = h->d, kvw = h->kvw, f = h->f, V = h->V, hd = h->hd, half = hd / 2;
  const int64_t es = h->es, H = h->H, kv = h->cfg.kv_heads;
  const int64_t rowd = d * es;
  int64_t* dmap = nullptr;
  TRY(dalloc(h, &dmap, (size_t)std::max<int64_t>(std::max<int64_t>(V, 2 * f), (H + 2 * kv) * hd) * 8));
  // embedding and head: as given
  TRY(dalloc(h, &h->emb, (size_t)(V * d * es)));
  CUDA_TRY(h, cudaMemcpyAsync(h->emb, blob, (size_t)(V * d * es), cudaMemcpyDeviceToDevice, h->stream));
  int64_t off = V * d;  // elements
  h->lw.resize(h->L);
  for (int l = 0; l < h->L; ++l) {
    LayerW& w = h->lw[l];
    const int64_t o_ln1 = off, o_q = o_ln1 + d, o_k = o_q + d * d, o_v = o_k + kvw * d, o_o = o_v + kvw * d;
    const int64_t o_ln2 = o_o + d * d, o_g = o_ln2 + d, o_u = o_g + f * d, o_dn = o_u + f * d;
    off = o_dn + d * f;
    TRY(dalloc(h, &w.ln1, (size_t)d * 4));
    TRY(dalloc(h, &w.ln2, (size_t)d * 4));
    TRY(widen(h, w.ln1, blob + o_ln1 * es, d));
    TRY(widen(h, w.ln2, blob + o_ln2 * es, d));
    // QKV: q heads, then k heads, then v heads; inside a head the rows (i, i + half) side by side.
    // The source rows are addressed relative to o_q (q, k and v are adjacent in the blob).
    std::vector<int64_t> map;
    map.reserve((size_t)((H + 2 * kv) * hd));
    for (int64_t head = 0; head < H + 2 * kv; ++head) {
      int64_t base;  // first source row of this head, counted from o_q
      if (head < H) base = head * hd;
      else if (head < H + kv) base = d + (head - H) * hd;
      else base = d + kvw + (head - H - kv) * hd;
      for (int64_t i = 0; i < half; ++i) {
        map.push_back(base + i);
        map.push_back(base + i + half);
      }
    }
    TRY(dalloc(h, &w.qkv, (size_t)((H + 2 * kv) * hd * rowd)));
    TRY(gather(h, w.qkv, blob + o_q * es, map, rowd, dmap));
    TRY(dalloc(h, &w.o, (size_t)(d * d * es)));
    CUDA_TRY(h, cudaMemcpyAsync(w.o, blob + o_o * es, (size_t)(d * d * es), cudaMemcpyDeviceToDevice, h->stream));
    map.clear();
    for (int64_t i = 0; i < f; ++i) {
      map.push_back(i);      // gate row i (relative to o_g)
      map.push_back(f + i);  // up row i
    }
    TRY(dalloc(h, &w.gu, (size_t)(2 * f * rowd)));
    TRY(gather(h, w.gu, blob + o_g * es, map, rowd, dmap));
    TRY(dalloc(h, &w.down, (size_t)(d * f * es)));
    CUDA_TRY(h, cudaMemcpyAsync(w.down, blob + o_dn * es, (size_t)(d * f * es), cudaMemcpyDeviceToDevice, h->stream));
  }
  TRY(dalloc(h, &h->lnf, (size_t)d * 4));
  TRY(widen(h, h->lnf, blob + off * es, d));
  off += d;
  if (h->cfg.tied) {
    h->head = h->emb;
  } else {
    TRY(dalloc(h, &h->head, (size_t)(V * d * es)));
    CUDA_TRY(h, cudaMemcpyAsync(h->head, blob + off * es, (size_t)(V * d * es), cudaMemcpyDeviceToDevice, h->stream));
  }
  CUDA_TRY(h, cudaStreamSynchronize(h->stream));
  return LLM_OK;
}

// ---- the decode step ----

// K_SAMPLE is the temperature / top-k / top-p chain, K_SELECT the same draw for a small top-k,
// K_GREEDY the argmax
enum { K_QKV = 0, K_ATTN = 1, K_O = 2, K_GATEUP = 3, K_DOWN = 4, K_HEAD = 5, K_SAMPLE = 6, K_EMBED = 7, K_GREEDY = 8,
       K_SELECT = 9 };

SampleArgs sample_args(const llm_handle* h) {
  SampleArgs s = {};
  s.logits = h->logits; s.logits_stride = h->V; s.V = h->V; s.V_pad = h->V_pad;
  s.keys = h->s_keys; s.idx = h->s_idx; s.pre = h->s_pre; s.hist = h->s_hist; s.hist_per_row = kSampleHistPerRow;
  s.u = h->u_buf; s.ids = h->ids_buf; s.step = h->st;
  return s;
}

// the activation map of a B-row step over K-wide rows (built on first use; host only)
const CUtensorMap* tc_xmap(llm_handle* h, int K, int B) {
  auto key = std::make_pair(K, B);
  auto it = h->xmaps.find(key);
  if (it != h->xmaps.end()) return &it->second;
  const TcPlan p = plan_tc(kTcN, K, B, h->num_sms);
  CUtensorMap m;
  if (!tc_make_map(&m, h->tc_xs, (uint64_t)K, 2 * (uint64_t)p.Ntot, kTcK, (uint32_t)p.NP)) return nullptr;
  return &h->xmaps.emplace(key, m).first->second;
}

// the reader of a projection's split sums: x reduced (plus the residual, or SwiGLU), optionally
// written to xout and normalized, then split into bf16 halves for the next projection
struct PrepIn {
  const float* x = nullptr;  // plain rows (no split sums)
  int x_stride = 0;
  int src_rows = 0, src_K = 0;  // shape of the projection whose split sums are read
  bool swiglu = false;
  const float* resid = nullptr;
  float* xout = nullptr;
  const float* gain = nullptr;
};

llm_status launch_prep(llm_handle* h, const PrepIn& in, int K, int B, bool pdl) {
  TcPrepArgs pa = {};
  pa.x_in = in.x; pa.x_stride = in.x_stride;
  if (!in.x) {
    const TcPlan src = plan_tc(in.src_rows, in.src_K, B, h->num_sms);
    pa.part = h->tc_part; pa.S = src.S; pa.part_rows = in.src_rows;
  }
  pa.swiglu = in.swiglu ? 1 : 0;
  pa.resid = in.resid; pa.resid_stride = K;
  pa.xout = in.xout; pa.xout_stride = K;
  pa.gain = in.gain; pa.eps = h->cfg.eps;
  pa.K = K; pa.B = B; pa.Ntot = tc_ntot(B); pa.xs = h->tc_xs;
  CUDA_TRY(h, launch_tc_prep(pa, h->stream, pdl));
  return LLM_OK;
}

// out (split sums, [S][B][rows]) = W x' for the split activations of K-wide rows
llm_status launch_gemm(llm_handle* h, const CUtensorMap& tw, int rows, int K, int B, float* out, bool pdl,
                       bool whole = false) {
  const TcPlan p = plan_tc(rows, K, B, h->num_sms, whole);
  const CUtensorMap* tx = tc_xmap(h, K, B);
  if (!tx) return fail(h, LLM_ERR_CUDA, "tensor map of the activations (K %d, B %d)", K, B);
  TcArgs a = {};
  a.rows = rows; a.K = K; a.N = B; a.NP = p.NP; a.Ntot = p.Ntot; a.MT = p.MT; a.KB = p.KB; a.S = p.S;
  a.n_tile = p.n_tile;
  a.units = p.units; a.stages = p.stages; a.out = out; a.status = h->status;
  CUDA_TRY(h, launch_tc_gemm(tw, *tx, a, p, h->stream, pdl));
  return LLM_OK;
}

// trace slot `slot` of layer l ([max_batch][trace_w]), or null when the step is not traced
float* tr_slot(llm_handle* h, int l, int slot) {
  if (!h->tracing) return nullptr;
  return h->trace + ((size_t)l * kTraceSlots + slot) * h->cfg.max_batch * h->trace_w;
}

// launch one kernel of the decode step (layer l where it applies); on the tensor-core path a
// projection is two kernels (activation split, then the GEMM)
llm_status launch_one(llm_handle* h, int which, int l, int B, bool pdl) {
  const int wt = h->wt;
  const int cps = 2;
  const llm_config& c = h->cfg;
  if (which == K_EMBED) {
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3((h->d + 255) / 256, B);
    lc.blockDim = dim3(256);
    lc.stream = h->stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 0;
    lc.attrs = attr;
    lc.numAttrs = 1;
    if (wt) CUDA_TRY(h, cudaLaunchKernelEx(&lc, embed_kernel<1>, (const void*)h->emb, (const int32_t*)h->tok_buf, h->xa, h->d, h->d));
    else CUDA_TRY(h, cudaLaunchKernelEx(&lc, embed_kernel<0>, (const void*)h->emb, (const int32_t*)h->tok_buf, h->xa, h->d, h->d));
    return LLM_OK;
  }
  const bool tc = h->tc_min > 0 && B >= h->tc_min;
  if (which == K_HEAD && tc) {
    // x = the last layer's residual stream (its down projection's split sums + x1), final norm
    PrepIn in;
    in.src_rows = h->d; in.src_K = h->f; in.resid = h->xb; in.xout = h->xa; in.gain = h->lnf;
    TRY(launch_prep(h, in, h->d, B, pdl));
    // one K split: the GEMM writes the logits themselves
    return launch_gemm(h, h->tmap_head, h->V, h->d, B, h->logits, pdl, true);
  }
  if (which == K_HEAD) {
    const GemvPlan p_h = plan_gemv(h->V, h->d, 1, wt, B, h->num_sms, cps);
    GemvArgs hd = {};
    hd.step = h->st; hd.B = B; hd.eps = c.eps; hd.W = h->head; hd.rows = h->V; hd.cols = h->d; hd.rg = 1;
    hd.x = h->xa; hd.x_stride = h->d; hd.gain = h->lnf;
    hd.lpr = p_h.lpr; hd.seg_ch = p_h.seg_ch; hd.nseg = p_h.nseg; hd.rows_cap = p_h.rows_cap; hd.ws = p_h.ws;
    hd.out = h->logits; hd.out_stride = h->V;
    hd.status = h->status;
    CUDA_TRY(h, launch_gemv(hd, p_h, wt, EPI_STORE, true, h->stream, pdl));
    return LLM_OK;
  }
  if (which == K_SAMPLE || which == K_GREEDY || which == K_SELECT) {
    CUDA_TRY(h, launch_sample(sample_args(h), B, which == K_GREEDY, h->stream, pdl, which == K_SELECT));
    return LLM_OK;
  }
  const LayerW& w = h->lw[l];
  char* kcl = (char*)h->kc + (size_t)l * h->layer_cache_elems * h->es;
  char* vcl = (char*)h->vc + (size_t)l * h->layer_cache_elems * h->es;
  if (tc && which != K_ATTN) {
    const TcMaps& tm = h->tmaps[l];
    const int qkv_rows = (h->H + 2 * c.kv_heads) * h->hd;
    PrepIn in;
    if (which == K_QKV) {
      // x: the embedding (layer 0) or the previous layer's down split sums + x1; then norm 1
      if (l == 0) {
        in.x = h->xa; in.x_stride = h->d;
      } else {
        in.src_rows = h->d; in.src_K = h->f; in.resid = h->xb; in.xout = h->xa;
      }
      in.gain = w.ln1;
      TRY(launch_prep(h, in, h->d, B, pdl));
      TRY(launch_gemm(h, tm.qkv, qkv_rows, h->d, B, h->tc_part, pdl));
      TcQkvArgs qa = {};
      qa.part = h->tc_part; qa.S = plan_tc(qkv_rows, h->d, B, h->num_sms).S; qa.rows = qkv_rows; qa.B = B;
      qa.q_out = h->q; qa.q_stride = h->d; qa.kc = kcl; qa.vc = vcl;
      qa.H = h->H; qa.kv = c.kv_heads; qa.hd = h->hd; qa.cap = c.max_seq;
      qa.rope_cos = h->rope_cos; qa.rope_sin = h->rope_sin; qa.step = h->st;
      CUDA_TRY(h, launch_tc_qkv(qa, h->stream, pdl));
      return LLM_OK;
    }
    if (which == K_O) {
      in.x = h->attn; in.x_stride = h->d;
      TRY(launch_prep(h, in, h->d, B, pdl));
      return launch_gemm(h, tm.o, h->d, h->d, B, h->tc_part, pdl);
    }
    if (which == K_GATEUP) {
      // x1 = x + o_proj split sums (kept in xb for the down residual), norm 2
      in.src_rows = h->d; in.src_K = h->d; in.resid = h->xa; in.xout = h->xb; in.gain = w.ln2;
      TRY(launch_prep(h, in, h->d, B, pdl));
      return launch_gemm(h, tm.gu, 2 * h->f, h->d, B, h->tc_part, pdl);
    }
    if (which == K_DOWN) {
      // m = silu(gate) * up from the gate/up split sums
      in.src_rows = 2 * h->f; in.src_K = h->d; in.swiglu = true; in.xout = h->m;
      TRY(launch_prep(h, in, h->f, B, pdl));
      return launch_gemm(h, tm.down, h->d, h->f, B, h->tc_part, pdl);
    }
  }
  if (which == K_QKV) {
    const int qkv_rows = (h->H + 2 * c.kv_heads) * h->hd;
    const GemvPlan p = plan_gemv(qkv_rows, h->d, 2, wt, B, h->num_sms, cps);
    GemvArgs a = {};
    a.step = h->st; a.B = B; a.eps = c.eps;
    a.W = w.qkv; a.rows = qkv_rows; a.cols = h->d; a.rg = 2;
    a.x = h->xa; a.x_stride = h->d; a.gain = w.ln1;
    a.lpr = p.lpr; a.seg_ch = p.seg_ch; a.nseg = p.nseg; a.rows_cap = p.rows_cap; a.ws = p.ws;
    a.q_out = h->q; a.q_stride = h->d; a.kc = kcl; a.vc = vcl;
    a.H = h->H; a.kv = c.kv_heads; a.hd = h->hd; a.cap = c.max_seq;
    a.rope_cos = h->rope_cos; a.rope_sin = h->rope_sin;
    a.status = h->status;
    a.tr_in = tr_slot(h, l, TR_N1); a.tr_pre = tr_slot(h, l, TR_QKV); a.tr_rot = tr_slot(h, l, TR_KR);
    a.tr_stride = (int32_t)h->trace_w;
    CUDA_TRY(h, launch_gemv(a, p, wt, EPI_QKV, true, h->stream, pdl));
  } else if (which == K_ATTN && h->capturing_pass && h->pf_attn) {
    // a prefill pass: tiles of consecutive prompt tokens share each key/value stream
    AttnPrefillArgs pa = {};
    pa.q = h->q; pa.q_stride = h->d; pa.out = h->attn; pa.out_stride = h->d;
    pa.tiles = h->tile_buf; pa.max_tiles = h->NT;
    pa.krow0 = (int32_t)((size_t)l * c.max_batch * c.kv_heads * c.max_seq);
    pa.kv = c.kv_heads; pa.g = c.group; pa.hd = h->hd; pa.cap = c.max_seq; pa.scale = 1.0f / sqrtf((float)h->hd);
    pa.step = h->st; pa.status = h->status;
    CUDA_TRY(h, launch_attn_prefill(h->kmap, h->vmap, pa, h->num_sms, h->stream, pdl));
  } else if (which == K_ATTN) {
    const int ns = attn_splits(B, c.kv_heads, c.max_seq, h->num_sms);
    if (ns > h->part_ns) return fail(h, LLM_ERR_ARG, "internal: attention splits %d > %d", ns, h->part_ns);
    AttnArgs at = {};
    at.q = h->q; at.q_stride = h->d; at.vc = vcl; at.out = h->attn; at.out_stride = h->d;
    at.krow0 = (int32_t)((size_t)l * c.max_batch * c.kv_heads * c.max_seq); at.status = h->status;
    at.part = h->part; at.ticket = h->ticket; at.B = B; at.kv = c.kv_heads; at.g = c.group; at.hd = h->hd;
    at.cap = c.max_seq; at.ns = ns; at.scale = 1.0f / sqrtf((float)h->hd); at.step = h->st;
    CUDA_TRY(h, launch_attn(h->kmap, h->vmap, at, wt, h->stream, pdl));
  } else if (which == K_O) {
    // o_proj + residual: x1 (xb) = x (xa) + W_o attn
    const GemvPlan p = plan_gemv(h->d, h->d, 1, wt, B, h->num_sms, cps);
    GemvArgs o = {};
    o.step = h->st; o.B = B; o.W = w.o; o.rows = h->d; o.cols = h->d; o.rg = 1;
    o.x = h->attn; o.x_stride = h->d;
    o.lpr = p.lpr; o.seg_ch = p.seg_ch; o.nseg = p.nseg; o.rows_cap = p.rows_cap; o.ws = p.ws;
    o.out = h->xb; o.out_stride = h->d; o.resid = h->xa; o.resid_stride = h->d;
    o.status = h->status;
    o.tr_pre = tr_slot(h, l, TR_A); o.tr_stride = (int32_t)h->trace_w;
    CUDA_TRY(h, launch_gemv(o, p, wt, EPI_RESID, false, h->stream, pdl));
  } else if (which == K_GATEUP) {
    // RMSNorm + gate/up + SwiGLU: m = silu(W_g n2) * (W_u n2)
    const GemvPlan p = plan_gemv(2 * h->f, h->d, 2, wt, B, h->num_sms, cps);
    GemvArgs g = {};
    g.step = h->st; g.B = B; g.eps = c.eps; g.W = w.gu; g.rows = 2 * h->f; g.cols = h->d; g.rg = 2;
    g.x = h->xb; g.x_stride = h->d; g.gain = w.ln2;
    g.lpr = p.lpr; g.seg_ch = p.seg_ch; g.nseg = p.nseg; g.rows_cap = p.rows_cap; g.ws = p.ws;
    g.out = h->m; g.out_stride = h->f;
    g.status = h->status;
    g.tr_in = tr_slot(h, l, TR_N2); g.tr_stride = (int32_t)h->trace_w;
    CUDA_TRY(h, launch_gemv(g, p, wt, EPI_SWIGLU, true, h->stream, pdl));
  } else if (which == K_DOWN) {
    // down + residual: y (xa) = x1 (xb) + W_down m
    const GemvPlan p = plan_gemv(h->d, h->f, 1, wt, B, h->num_sms, cps);
    GemvArgs dn = {};
    dn.step = h->st; dn.B = B; dn.W = w.down; dn.rows = h->d; dn.cols = h->f; dn.rg = 1;
    dn.x = h->m; dn.x_stride = h->f;
    dn.lpr = p.lpr; dn.seg_ch = p.seg_ch; dn.nseg = p.nseg; dn.rows_cap = p.rows_cap; dn.ws = p.ws;
    dn.out = h->xa; dn.out_stride = h->d; dn.resid = h->xb; dn.resid_stride = h->d;
    dn.status = h->status;
    dn.tr_pre = tr_slot(h, l, TR_M); dn.tr_stride = (int32_t)h->trace_w;
    CUDA_TRY(h, launch_gemv(dn, p, wt, EPI_RESID, false, h->stream, pdl));
  } else {
    return fail(h, LLM_ERR_ARG, "unknown kernel %d", which);
  }
  return LLM_OK;
}

llm_status launch_layer_kernels(llm_handle* h, int B, int mode, bool pdl, bool trace) {
  const llm_config& c = h->cfg;
  TRY(launch_one(h, K_EMBED, 0, B, false));
  if (h->mega && B == 1 && !trace && !h->capturing_pass) {
    // every layer, the head and a greedy draw in one persistent kernel; a top-k top-p draw after
    MegaArgs a = {};
    a.layers = h->mega_layers; a.L = h->L; a.d = h->d; a.f = h->f; a.V = h->V; a.H = h->H; a.kv = c.kv_heads;
    a.g = c.group; a.hd = h->hd; a.cap = c.max_seq; a.max_batch = c.max_batch; a.eps = c.eps;
    a.scale = 1.0f / sqrtf((float)h->hd); a.lnf = h->lnf; a.head = h->head; a.kc = h->kc; a.vc = h->vc;
    a.rope_cos = h->rope_cos; a.rope_sin = h->rope_sin; a.step = h->st; a.x = h->xa; a.x1 = h->xb; a.q = h->q;
    a.attn = h->attn; a.m = h->m; a.logits = h->logits; a.apart = h->mega_part; a.ticket = h->mega_ticket;
    a.bar = h->mega_bar; a.cand_v = h->mega_cv; a.cand_i = h->mega_ci; a.ids = h->ids_buf; a.status = h->status;
    a.head_mode = mode == MODE_NOHEAD ? 0 : mode == MODE_GREEDY ? 2 : 1;
    CUDA_TRY(h, launch_mega(a, h->num_sms, h->stream));
    if (mode == MODE_TOPP) TRY(launch_one(h, K_SAMPLE, 0, B, false));
    if (mode == MODE_TOPK) TRY(launch_one(h, K_SELECT, 0, B, false));
    return LLM_OK;
  }
  const size_t tw = h->trace_w;
  h->tracing = trace;
  for (int l = 0; l < h->L; ++l) {
    for (int k = K_QKV; k <= K_DOWN; ++k) {
      llm_status s_ = launch_one(h, k, l, B, pdl);
      if (s_ != LLM_OK) {
        h->tracing = false;
        return s_;
      }
    }
    if (trace) {
      // the buffers that hold an intermediate whole after the layer (the GEMVs wrote the rest)
      const struct { int slot; const float* src; int width; } cp[] = {
          {TR_QR, h->q, h->d}, {TR_ATTN, h->attn, h->d}, {TR_X1, h->xb, h->d}, {TR_SWIGLU, h->m, h->f},
          {TR_Y, h->xa, h->d}};
      for (const auto& x : cp)
        CUDA_TRY(h, cudaMemcpy2DAsync(tr_slot(h, l, x.slot), tw * 4, x.src, (size_t)x.width * 4, (size_t)x.width * 4, B,
                                      cudaMemcpyDeviceToDevice, h->stream));
    }
  }
  h->tracing = false;
  if (mode >= MODE_HEAD) TRY(launch_one(h, K_HEAD, 0, B, pdl));
  if (mode == MODE_GREEDY) TRY(launch_one(h, K_GREEDY, 0, B, pdl));
  if (mode == MODE_TOPP) TRY(launch_one(h, K_SAMPLE, 0, B, pdl));
  if (mode == MODE_TOPK) TRY(launch_one(h, K_SELECT, 0, B, pdl));
  return LLM_OK;
}

// the step graph of (B, mode), captured on first use; with gen > 0, a generation graph of gen
// steps, each its own prologue (gen_begin_kernel), the step's kernels and gen_end_kernel
llm_status step_graph(llm_handle* h, int B, int mode, std::pair<cudaGraphExec_t, int>** out, int gen = 0,
                      bool pass = false) {
  GraphKey key{B, mode, gen, pass ? 1 : 0};
  auto it = h->graphs.find(key);
  if (it == h->graphs.end()) {
    // capture on a private stream, then replay on the handle's stream
    cudaStream_t saved = h->stream;
    h->stream = h->cap_stream;
    CUDA_TRY(h, cudaStreamBeginCapture(h->stream, cudaStreamCaptureModeThreadLocal));
    llm_status s = LLM_OK;
    h->capturing_pass = pass;
    if (gen == 0) {
      s = launch_layer_kernels(h, B, mode, true, false);
    } else {
      for (int i = 0; i < gen && s == LLM_OK; ++i) {
        gen_begin_kernel<<<1, 128, 0, h->stream>>>(h->st, h->gen, h->tok_buf, h->u_buf, i, h->mega_bar);
        s = launch_layer_kernels(h, B, mode, true, false);
        if (s == LLM_OK) gen_end_kernel<<<1, 128, 0, h->stream>>>(h->gen, h->ids_buf, i);
      }
    }
    h->capturing_pass = false;
    cudaGraph_t graph = nullptr;
    cudaError_t e = cudaStreamEndCapture(h->stream, &graph);
    h->stream = saved;
    if (s != LLM_OK) {
      if (graph) cudaGraphDestroy(graph);
      return s;
    }
    if (e != cudaSuccess) return fail(h, LLM_ERR_CUDA, "stream capture: %s", cudaGetErrorString(e));
    size_t nodes = 0;  // every node of the step graph is a kernel launch
    e = cudaGraphGetNodes(graph, nullptr, &nodes);
    cudaGraphExec_t exec = nullptr;
    if (e == cudaSuccess) e = cudaGraphInstantiate(&exec, graph, 0);
    cudaGraphDestroy(graph);
    if (e != cudaSuccess) return fail(h, LLM_ERR_CUDA, "graph instantiate: %s", cudaGetErrorString(e));
    it = h->graphs.emplace(key, std::make_pair(exec, (int)nodes)).first;
  }
  *out = &it->second;
  return LLM_OK;
}

llm_status run_step(llm_handle* h, int B, int mode, bool pass = false) {
  if (h->cfg.debug_trace) return launch_layer_kernels(h, B, mode, false, true);
  std::pair<cudaGraphExec_t, int>* g = nullptr;
  TRY(step_graph(h, B, mode, &g, 0, pass));
  CUDA_TRY(h, cudaGraphLaunch(g->first, h->stream));
  return LLM_OK;
}

// the step prologue; rows at their own positions when pos_host is given (copied to pos_buf)
llm_status begin(llm_handle* h, int pos, int B, const int32_t* tok_host, const int32_t* tok_dev, int tok_stride,
                 int tok_col, float temp, int k, float p, const float* u_host, const float* u_dev,
                 const int32_t* pos_host = nullptr, const int32_t* table_dev = nullptr, int table_stride = 0,
                 const int32_t* ranges_dev = nullptr, int tok_np = 1) {
  BeginArgs a = {};
  a.st = h->st; a.pos = pos; a.B = B; a.temp = temp; a.k = k; a.p = p; a.vocab = h->V;
  a.table = table_dev; a.table_stride = table_stride; a.ranges = ranges_dev; a.mega_bar = h->mega_bar;
  if (pos_host) {
    a.own_pos = 1;
    if (B <= kInline) {
      for (int b = 0; b < B; ++b) a.pos_inline[b] = pos_host[b];
    } else {
      CUDA_TRY(h, cudaMemcpyAsync(h->pos_buf, pos_host, (size_t)B * 4, cudaMemcpyHostToDevice, h->stream));
      a.pos_dev = h->pos_buf;
    }
  }
  a.tok_buf = h->tok_buf; a.u_buf = h->u_buf; a.status = h->status;
  a.tok_stride = tok_stride; a.tok_col = tok_col; a.tok_np = tok_np;
  auto tok_of = [&](int b) { return tok_host[(size_t)(b / tok_np) * tok_stride + b % tok_np + tok_col]; };
  if (tok_dev) {
    a.tok_dev = tok_dev;
  } else if (B <= kInline) {
    for (int b = 0; b < B; ++b) a.tok_inline[b] = tok_of(b);
  } else {
    std::vector<int32_t> col(B);
    for (int b = 0; b < B; ++b) col[b] = tok_of(b);
    CUDA_TRY(h, cudaMemcpyAsync(h->tok_buf, col.data(), (size_t)B * 4, cudaMemcpyHostToDevice, h->stream));
    a.tok_dev = h->tok_buf;
    a.tok_stride = 1;
    a.tok_col = 0;
    a.tok_np = 1;
  }
  if (u_dev) {
    a.u_dev = u_dev;
  } else if (u_host && B > kInline) {
    CUDA_TRY(h, cudaMemcpyAsync(h->u_buf, u_host, (size_t)B * 4, cudaMemcpyHostToDevice, h->stream));
    a.u_dev = h->u_buf;
  } else {
    for (int b = 0; b < B && b < kInline; ++b) a.u_inline[b] = u_host ? u_host[b] : 0.0f;
  }
  step_begin_kernel<<<1, 128, 0, h->stream>>>(a);
  CUDA_TRY(h, cudaGetLastError());
  return LLM_OK;
}

llm_status check_rows(llm_handle* h, int B, int pos, int S) {
  if (B < 1 || B > h->cfg.max_batch) return fail(h, LLM_ERR_BATCH, "batch %d outside 1..%d", B, h->cfg.max_batch);
  if (S < 1) return fail(h, LLM_ERR_ARG, "prompt length %d < 1", S);
  if (pos < 0 || (int64_t)pos + S > h->cfg.max_seq)
    return fail(h, LLM_ERR_POS_RANGE, "positions %d..%lld outside the cache of %d", pos, (long long)pos + S - 1, h->cfg.max_seq);
  for (int b = 0; b < B; ++b)
    if (pos > h->filled[b])
      return fail(h, LLM_ERR_POS_RANGE, "row %d: position %d after its filled length %d", b, pos, h->filled[b]);
  return LLM_OK;
}

llm_status check_tokens(llm_handle* h, const int32_t* toks, size_t n) {
  for (size_t i = 0; i < n; ++i)
    if (toks[i] < 0 || toks[i] >= h->V) return fail(h, LLM_ERR_TOKEN_RANGE, "token %d at %zu outside 0..%d", toks[i], i, h->V - 1);
  return LLM_OK;
}

llm_status check_sample_args(llm_handle* h, float temp, int k, float p) {
  if (!(temp >= 0.0f) || temp == INFINITY) return fail(h, LLM_ERR_ARG, "temperature must be finite and >= 0");
  if (temp > 0.0f) {
    if (k < 1) return fail(h, LLM_ERR_ARG, "top-k must be >= 1");
    if (!(p > 0.0f && p <= 1.0f)) return fail(h, LLM_ERR_ARG, "top-p must be in (0, 1]");
  }
  return LLM_OK;
}

// the mode of a step that draws with (temp, k): greedy, a small top-k, or the full sort
int draw_mode(const llm_handle* h, float temp, int k) {
  if (!(temp > 0.0f)) return MODE_GREEDY;
  return std::min(k, h->V) <= sample_select_max() ? MODE_TOPK : MODE_TOPP;
}

void set_filled(llm_handle* h, int B, int v) {
  for (int b = 0; b < B; ++b) h->filled[b] = v;
}

// rows at their own positions: 0 <= pos[b] <= filled length of row b, pos[b] < max_seq
llm_status check_row_positions(llm_handle* h, int B, const int32_t* pos) {
  if (B < 1 || B > h->cfg.max_batch) return fail(h, LLM_ERR_BATCH, "batch %d outside 1..%d", B, h->cfg.max_batch);
  for (int b = 0; b < B; ++b) {
    if (pos[b] < 0 || pos[b] >= h->cfg.max_seq)
      return fail(h, LLM_ERR_POS_RANGE, "row %d: position %d outside the cache of %d", b, pos[b], h->cfg.max_seq);
    if (pos[b] > h->filled[b])
      return fail(h, LLM_ERR_POS_RANGE, "row %d: position %d after its filled length %d", b, pos[b], h->filled[b]);
  }
  return LLM_OK;
}

}  // namespace

// ---------------------------------------------------------------------------------------
// C ABI
// ---------------------------------------------------------------------------------------

extern "C" {

uint64_t llm_weight_count(const llm_config* cfg) { return cfg ? count_of(cfg) : 0; }

const char* llm_status_string(llm_status s) {
  switch (s) {
    case LLM_OK: return "ok";
    case LLM_ERR_CONFIG: return "invalid config";
    case LLM_ERR_WEIGHTS_SIZE: return "weight blob size mismatch";
    case LLM_ERR_OOM: return "out of device memory";
    case LLM_ERR_POS_RANGE: return "position out of range";
    case LLM_ERR_TOKEN_RANGE: return "token out of range";
    case LLM_ERR_BATCH: return "batch out of range";
    case LLM_ERR_ARG: return "invalid argument";
    case LLM_ERR_CUDA: return "CUDA error";
    case LLM_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
  }
}

const char* llm_last_error(const llm_handle* h) { return h ? h->err.c_str() : g_create_err.c_str(); }

llm_status llm_destroy(llm_handle* h) {
  if (!h) return LLM_ERR_ARG;
  if (h->stream) cudaStreamSynchronize(h->stream);
  for (auto& kv : h->graphs) cudaGraphExecDestroy(kv.second.first);
  for (void* p : h->allocs) cudaFree(p);
  if (h->cap_stream) cudaStreamDestroy(h->cap_stream);
  if (h->own_stream && h->stream) cudaStreamDestroy(h->stream);
  delete h;
  return LLM_OK;
}

llm_status llm_create(const llm_config* cfg, const void* weights, uint64_t nbytes, int32_t weights_on_device,
                      void* cuda_stream, llm_handle** out) {
  if (!cfg || !weights || !out) {
    g_create_err = "NULL argument";
    return LLM_ERR_ARG;
  }
  *out = nullptr;
  if (const char* why = check_config(cfg)) {
    g_create_err = why;
    return LLM_ERR_CONFIG;
  }
  const uint64_t es = cfg->dtype == LLM_DTYPE_BF16 ? 2 : 4;
  if (nbytes != count_of(cfg) * es) {
    char buf[160];
    snprintf(buf, sizeof buf, "weights hold %llu bytes, the layout needs %llu",
             (unsigned long long)nbytes, (unsigned long long)(count_of(cfg) * es));
    g_create_err = buf;
    return LLM_ERR_WEIGHTS_SIZE;
  }
  g_create_err.clear();
  llm_handle* h = new llm_handle();
  h->cfg = *cfg;
  const llm_config& c = h->cfg;
  h->hd = 2 * c.half;
  h->H = c.kv_heads * c.group;
  h->d = h->H * h->hd;
  h->kvw = c.kv_heads * h->hd;
  h->f = c.ffn;
  h->V = c.vocab;
  h->L = c.layers;
  h->wt = c.dtype == LLM_DTYPE_BF16 ? 1 : 0;
  h->es = (int)es;
  h->filled.assign(c.max_batch, 0);
  h->NT = std::max(c.max_batch, c.max_tokens > 0 ? c.max_tokens : kDefaultTokens);
  llm_status st = LLM_OK;
  auto bail = [&](llm_status s) {
    cudaError_t ce = cudaGetLastError();
    g_create_err = h->err.empty() ? std::string(llm_status_string(s)) : h->err;
    if (ce != cudaSuccess) g_create_err += std::string(" (last CUDA error: ") + cudaGetErrorString(ce) + ")";
    llm_destroy(h);
    return s;
  };
  auto cuda_bail = [&](const char* what, cudaError_t e) {
    fail(h, LLM_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
    return bail(LLM_ERR_CUDA);
  };
  cudaError_t ce;
  if ((ce = cudaGetDevice(&h->dev)) != cudaSuccess) return cuda_bail("cudaGetDevice", ce);
  cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->dev);
  cudaDeviceGetAttribute(&h->smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, h->dev);
  if (cuda_stream) {
    h->stream = (cudaStream_t)cuda_stream;
  } else {
    if ((ce = cudaStreamCreateWithFlags(&h->stream, cudaStreamNonBlocking)) != cudaSuccess) return cuda_bail("stream", ce);
    h->own_stream = true;
  }
  if ((ce = cudaStreamCreateWithFlags(&h->cap_stream, cudaStreamNonBlocking)) != cudaSuccess) return cuda_bail("capture stream", ce);
  if ((ce = gemv_prepare(h->smem_optin)) != cudaSuccess) return cuda_bail("gemv kernel attributes", ce);
  // tensor-core path: bf16 weights, rows a whole number of 16-byte chunks (checked above)
  const int tc_min = c.tc_min_batch > 0 ? c.tc_min_batch : kTcDefaultMinBatch;
  // (debug_trace handles keep every step on the GEMV: the traced buffers are written in order there;
  // so do models whose hidden or MLP width exceeds what the prep kernels stage per row)
  if (h->wt && !c.debug_trace && tc_min <= h->NT && h->d <= kTcMaxK && h->f <= kTcMaxK && tc_available()) {
    if ((ce = tc_prepare(h->smem_optin)) != cudaSuccess) return cuda_bail("tensor-core kernel attributes", ce);
    h->tc_min = tc_min;
  }
  if ((ce = attn_prepare(h->smem_optin)) != cudaSuccess) return cuda_bail("attention kernel attributes", ce);
  h->pf_attn = attn_prefill_supported(h->wt, 2 * c.half, c.group);
  if (h->pf_attn && (ce = attn_prefill_prepare(h->smem_optin)) != cudaSuccess)
    return cuda_bail("prefill attention kernel attributes", ce);
  // the allocation-free sampler's array is reserved here, where allocating is allowed
  if ((ce = noalloc_prepare()) != cudaSuccess) return cuda_bail("allocation-free sampler set-up", ce);
  // weights: a device copy of the blob when it is on the host, then repacked
  const char* blob = (const char*)weights;
  char* staging = nullptr;
  if (!weights_on_device) {
    if ((ce = cudaMalloc(&staging, nbytes)) != cudaSuccess) {
      cudaGetLastError();
      fail(h, LLM_ERR_OOM, "cudaMalloc(%llu bytes) for the weight staging copy: %s", (unsigned long long)nbytes, cudaGetErrorString(ce));
      return bail(LLM_ERR_OOM);
    }
    if ((ce = cudaMemcpy(staging, weights, nbytes, cudaMemcpyHostToDevice)) != cudaSuccess) {
      cudaFree(staging);
      return cuda_bail("weights upload", ce);
    }
    blob = staging;
  }
  st = load_weights(h, blob);
  if (staging) cudaFree(staging);
  if (st != LLM_OK) return bail(st);
  // KV cache, RoPE table, activations, scratch
  h->layer_cache_elems = (size_t)c.max_batch * c.kv_heads * c.max_seq * h->hd;
  const size_t cache_bytes = (size_t)h->L * h->layer_cache_elems * es;
  if ((st = dalloc(h, &h->kc, cache_bytes)) || (st = dalloc(h, &h->vc, cache_bytes))) return bail(st);
  if ((uint64_t)h->L * c.max_batch * c.kv_heads * c.max_seq >= (1ull << 31) ||
      !attn_make_kmap(&h->kmap, h->kc, h->wt, h->hd, (uint64_t)h->L * c.max_batch * c.kv_heads * c.max_seq) ||
      !attn_make_kmap(&h->vmap, h->vc, h->wt, h->hd, (uint64_t)h->L * c.max_batch * c.kv_heads * c.max_seq)) {
    fail(h, LLM_ERR_CONFIG, "the key cache does not fit a tensor map (layers x rows x kv heads x positions < 2^31)");
    return bail(LLM_ERR_CONFIG);
  }
  if ((st = dalloc(h, &h->rope_cos, (size_t)c.max_seq * c.half * 4)) ||
      (st = dalloc(h, &h->rope_sin, (size_t)c.max_seq * c.half * 4)))
    return bail(st);
  const size_t B = c.max_batch;
  const size_t NT = h->NT;  // rows of a step or of a prefill pass
  if ((st = dalloc(h, &h->xa, NT * h->d * 4)) || (st = dalloc(h, &h->xb, NT * h->d * 4)) ||
      (st = dalloc(h, &h->q, NT * h->d * 4)) || (st = dalloc(h, &h->attn, NT * h->d * 4)) ||
      (st = dalloc(h, &h->m, NT * h->f * 4)) || (st = dalloc(h, &h->logits, B * h->V * 4)) ||
      (st = dalloc(h, &h->xh, B * h->d * 4)) || (st = dalloc(h, &h->head_map, B * 4)))
    return bail(st);
  int maxns = 1;
  for (int b = 1; b <= h->NT; ++b) {
    const int ns = attn_splits(b, c.kv_heads, c.max_seq, h->num_sms);
    maxns = std::max(maxns, ns);
    attn_cluster_merge(h->wt, h->hd, c.group, ns, b * c.kv_heads, c.max_seq);  // device queries before any capture
  }
  h->part_ns = maxns;
  h->ticket_count = (int)(NT * c.kv_heads);
  const int slots = attn_part_slots(h->wt, h->hd, maxns);
  if ((st = dalloc(h, &h->part, NT * h->H * slots * (h->hd + 2) * 4)) ||
      (st = dalloc(h, &h->ticket, NT * c.kv_heads * 4)) || (st = dalloc(h, &h->st, step_state_bytes((int)NT))) ||
      (st = dalloc(h, &h->pos_buf, NT * 4)) || (st = dalloc(h, &h->gen, sizeof(GenState))) ||
      (st = dalloc(h, &h->u_gen, (size_t)kGenChunk * B * 4)) || (st = dalloc(h, &h->ids_gen, (size_t)kGenChunk * B * 4)) ||
      (c.max_seq % kPage == 0 && (st = dalloc(h, &h->page_table, B * (size_t)(c.max_seq / kPage) * 4))) ||
      (st = dalloc(h, &h->range_buf, 3 * NT * 4)) ||
      (st = dalloc(h, &h->tile_buf, (4 + 4 * NT + 2 * NT * (size_t)c.kv_heads) * 4)) ||
      (st = dalloc(h, &h->status, 16)) || (st = dalloc(h, &h->tok_buf, NT * 4)) || (st = dalloc(h, &h->u_buf, NT * 4)) ||
      (st = dalloc(h, &h->ids_buf, B * 4)))
    return bail(st);
  h->V_pad = (h->V + 31) & ~31;
  if ((st = dalloc(h, &h->s_keys, B * 2 * h->V_pad * 4)) || (st = dalloc(h, &h->s_idx, B * 2 * h->V_pad * 4)) ||
      (st = dalloc(h, &h->s_pre, B * h->V_pad * 4)) || (st = dalloc(h, &h->s_hist, B * kSampleHistPerRow * 4)))
    return bail(st);
  if (h->tc_min) {
    // split activations for up to NT rows; split sums of the largest projection
    const int64_t qkv_rows = (int64_t)(h->H + 2 * c.kv_heads) * h->hd;
    size_t part = 0;
    for (int b = h->tc_min; b <= h->NT; ++b) {
      const int64_t shapes[4][2] = {{qkv_rows, h->d}, {h->d, h->d}, {2 * (int64_t)h->f, h->d}, {h->d, h->f}};
      for (auto& sh : shapes) {
        const TcPlan p = plan_tc((int)sh[0], (int)sh[1], b, h->num_sms);
        part = std::max(part, (size_t)p.S * b * (size_t)sh[0]);
      }
    }
    const size_t xs_elems = (size_t)2 * tc_ntot(h->NT) * std::max(h->d, h->f);
    if ((st = dalloc(h, &h->tc_xs, xs_elems * 2)) || (st = dalloc(h, &h->tc_part, part * 4))) return bail(st);
    if (cudaMemsetAsync(h->tc_xs, 0, xs_elems * 2, h->stream) != cudaSuccess ||
        cudaMemsetAsync(h->tc_part, 0, part * 4, h->stream) != cudaSuccess)
      return cuda_bail("clearing the tensor-core scratch", cudaGetLastError());
    h->tmaps.resize(h->L);
    bool ok = true;
    for (int l = 0; l < h->L && ok; ++l) {
      const LayerW& w = h->lw[l];
      TcMaps& m = h->tmaps[l];
      ok = tc_make_map(&m.qkv, w.qkv, h->d, (uint64_t)qkv_rows, kTcK, kTcN) &&
           tc_make_map(&m.o, w.o, h->d, h->d, kTcK, kTcN) && tc_make_map(&m.gu, w.gu, h->d, 2 * (uint64_t)h->f, kTcK, kTcN) &&
           tc_make_map(&m.down, w.down, h->f, h->d, kTcK, kTcN);
    }
    // a shape the tensor maps cannot describe keeps every step on the GEMV
    // the head runs unsplit; its tile height (the map's box) depends only on the vocabulary
    const int head_rows = plan_tc(h->V, h->d, 1, h->num_sms, true).n_tile;
    if (!ok || !tc_make_map(&h->tmap_head, h->head, h->d, h->V, kTcK, (uint32_t)head_rows)) h->tc_min = 0;
  }
  h->trace_w = (size_t)std::max(h->d + 2 * h->kvw, h->f);
  if (c.debug_trace && (st = dalloc(h, &h->trace, (size_t)h->L * kTraceSlots * B * h->trace_w * 4))) return bail(st);
  {
    // batch-1 steps as one persistent kernel where the shape allows it and every CTA can be resident
    int coop = 0;
    cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, h->dev);
    if (coop && !c.debug_trace && c.step_kernel == 1 && h->num_sms >= c.kv_heads &&
        mega_supported(h->wt, h->hd, c.group, h->d, h->f) &&
        mega_smem(h->d, h->f) + 1024 <= (size_t)h->smem_optin && mega_prepare(h->smem_optin) == cudaSuccess) {
      if ((st = dalloc(h, &h->mega_layers, sizeof(MegaLayer) * (size_t)h->L)) ||
          (st = dalloc(h, &h->mega_part, (size_t)h->H * kMegaMaxSplits * (h->hd + 2) * 4)) ||
          (st = dalloc(h, &h->mega_ticket, ((size_t)c.kv_heads + 1) * 4)) || (st = dalloc(h, &h->mega_bar, 4)) ||
          (st = dalloc(h, &h->mega_cv, (size_t)h->num_sms * 4)) || (st = dalloc(h, &h->mega_ci, (size_t)h->num_sms * 4)))
        return bail(st);
      std::vector<MegaLayer> ml(h->L);
      for (int l = 0; l < h->L; ++l)
        ml[l] = MegaLayer{h->lw[l].qkv, h->lw[l].ln1, h->lw[l].o, h->lw[l].ln2, h->lw[l].gu, h->lw[l].down};
      if (cudaMemcpy(h->mega_layers, ml.data(), sizeof(MegaLayer) * (size_t)h->L, cudaMemcpyHostToDevice) != cudaSuccess ||
          cudaMemsetAsync(h->mega_ticket, 0, ((size_t)c.kv_heads + 1) * 4, h->stream) != cudaSuccess ||
          cudaMemsetAsync(h->mega_bar, 0, 4, h->stream) != cudaSuccess)
        return cuda_bail("persistent step kernel setup", cudaGetLastError());
      h->mega = true;
    } else {
      cudaGetLastError();
    }
  }
  if (cudaMemsetAsync(h->ticket, 0, NT * c.kv_heads * 4, h->stream) != cudaSuccess ||
      cudaMemsetAsync(h->status, 0, 16, h->stream) != cudaSuccess ||
      cudaMemsetAsync(h->kc, 0, cache_bytes, h->stream) != cudaSuccess ||
      cudaMemsetAsync(h->vc, 0, cache_bytes, h->stream) != cudaSuccess)
    return cuda_bail("clearing the cache", cudaGetLastError());
  RopeArgs ra = {c.theta, h->hd, c.half, c.max_seq, c.rope_llama3, c.rope_factor, c.rope_low_freq, c.rope_high_freq,
                 c.rope_orig_max_pos, h->rope_cos, h->rope_sin};
  rope_table_kernel<<<1024, 256, 0, h->stream>>>(ra);
  if ((ce = cudaGetLastError()) != cudaSuccess || (ce = cudaStreamSynchronize(h->stream)) != cudaSuccess)
    return cuda_bail("RoPE tables", ce);
  *out = h;
  return LLM_OK;
}

llm_status llm_reset(llm_handle* h) {
  if (!h) return LLM_ERR_ARG;
  std::fill(h->filled.begin(), h->filled.end(), 0);
  return LLM_OK;
}

void* llm_stream(llm_handle* h) { return h ? (void*)h->stream : nullptr; }
float* llm_logits_buffer(llm_handle* h) { return h ? h->logits : nullptr; }
int32_t llm_filled(const llm_handle* h, int32_t b) {
  return (h && b >= 0 && b < h->cfg.max_batch) ? h->filled[b] : -1;
}

llm_status llm_synchronize(llm_handle* h) {
  if (!h) return LLM_ERR_ARG;
  CUDA_TRY(h, cudaStreamSynchronize(h->stream));
  int32_t s = 0;
  CUDA_TRY(h, cudaMemcpy(&s, h->status, 4, cudaMemcpyDeviceToHost));
  if (s != 0) {
    CUDA_TRY(h, cudaMemset(h->status, 0, 4));
    // a kernel that gave up may have left the attention's merge tickets short of their count
    if (s == LLM_ERR_DEVICE_TIMEOUT) {
      CUDA_TRY(h, cudaMemset(h->ticket, 0, (size_t)h->ticket_count * 4));
      if (h->mega_ticket) CUDA_TRY(h, cudaMemset(h->mega_ticket, 0, ((size_t)h->cfg.kv_heads + 1) * 4));
    }
    return fail(h, s, "device reported: %s", llm_status_string(s));
  }
  return LLM_OK;
}

llm_status llm_check_wait_timeout(llm_handle* h, int64_t limit_cycles) {
  if (!h) return LLM_ERR_ARG;
  if (limit_cycles < 1 || limit_cycles > 1000000000) return fail(h, LLM_ERR_ARG, "limit %lld outside 1..1e9 cycles", (long long)limit_cycles);
  wait_timeout_kernel<<<1, 32, 0, h->stream>>>(h->status, (uint64_t)limit_cycles);
  CUDA_TRY(h, cudaGetLastError());
  return LLM_OK;
}

// ---- prefill passes ----
//
// A pass is one step whose rows are prompt tokens ("entries"): entry e is token tokens[e] at
// position positions[e] of cache row rowmap[e], attending to positions start[e] .. positions[e]
// of that row.  The step prologue puts positions, starts, the first position the pass writes in
// each entry's row (wfirst: attention copies below it may start before the Q/K/V kernel ends) and
// the rows into the step state; the projections see n = entries rows (on the tensor cores once n
// reaches tc_min_batch) and the Q/K/V kernel writes every entry's key and value before the
// attention reads them.  No pass runs the LM head: the entries whose logits are wanted are
// gathered afterwards (pass_logits).

// gather rows of the final residual stream: dst[i] = src[map[i]] (width floats)
__global__ void gather_rows_f32_kernel(float* dst, const float* src, const int32_t* map, int width) {
  const float* s = src + (size_t)map[blockIdx.x] * width;
  float* o = dst + (size_t)blockIdx.x * width;
  for (int i = threadIdx.x; i < width; i += blockDim.x) o[i] = s[i];
}

// final norm + LM head over rows 0..m-1 of xh into the logits buffer
static llm_status head_rows(llm_handle* h, int m) {
  if (h->tc_min > 0 && m >= h->tc_min) {
    PrepIn in;
    in.x = h->xh; in.x_stride = h->d; in.gain = h->lnf;
    TRY(launch_prep(h, in, h->d, m, false));
    return launch_gemm(h, h->tmap_head, h->V, h->d, m, h->logits, false, true);
  }
  const GemvPlan p = plan_gemv(h->V, h->d, 1, h->wt, m, h->num_sms, 2);
  GemvArgs a = {};
  a.step = h->st; a.B = m; a.eps = h->cfg.eps; a.W = h->head; a.rows = h->V; a.cols = h->d; a.rg = 1;
  a.x = h->xh; a.x_stride = h->d; a.gain = h->lnf;
  a.lpr = p.lpr; a.seg_ch = p.seg_ch; a.nseg = p.nseg; a.rows_cap = p.rows_cap; a.ws = p.ws;
  a.out = h->logits; a.out_stride = h->V;
  a.status = h->status;
  CUDA_TRY(h, launch_gemv(a, p, h->wt, EPI_STORE, true, h->stream, false));
  return LLM_OK;
}

// logits after entries ents[i] of the pass of n entries just run, into dst rows dst_row[i]
// ([.][V], host or device memory)
static llm_status pass_logits(llm_handle* h, int n, const std::vector<int32_t>& ents, const std::vector<int>& dst_row,
                              float* dst, bool host) {
  if (ents.empty()) return LLM_OK;
  if (h->tc_min > 0 && n >= h->tc_min) {
    // the residual stream after the last layer: its down projection's split sums + x1
    PrepIn in;
    in.src_rows = h->d; in.src_K = h->f; in.resid = h->xb; in.xout = h->xa;
    TRY(launch_prep(h, in, h->d, n, false));
  }
  const int mb = h->cfg.max_batch;
  for (size_t c0 = 0; c0 < ents.size(); c0 += mb) {
    const int m = (int)std::min<size_t>(mb, ents.size() - c0);
    CUDA_TRY(h, cudaMemcpyAsync(h->head_map, ents.data() + c0, (size_t)m * 4, cudaMemcpyHostToDevice, h->stream));
    gather_rows_f32_kernel<<<m, 256, 0, h->stream>>>(h->xh, h->xa, h->head_map, h->d);
    CUDA_TRY(h, cudaGetLastError());
    TRY(head_rows(h, m));
    for (int i = 0; i < m; ++i)
      CUDA_TRY(h, cudaMemcpyAsync(dst + (size_t)dst_row[c0 + i] * h->V, h->logits + (size_t)i * h->V, (size_t)h->V * 4,
                                  host ? cudaMemcpyDeviceToHost : cudaMemcpyDeviceToDevice, h->stream));
  }
  return LLM_OK;
}

// one pass of n entries; ranges [3][n]: attention starts, first written positions, cache rows;
// tokens as for begin (host array, or device array read at (e / tok_np) * tok_stride + e % tok_np
// + tok_col)
static llm_status run_pass(llm_handle* h, int n, const int32_t* tok_host, const int32_t* tok_dev, int tok_stride,
                           int tok_col, int tok_np, const int32_t* pos_host, const int32_t* ranges_host) {
  CUDA_TRY(h, cudaMemcpyAsync(h->range_buf, ranges_host, (size_t)3 * n * 4, cudaMemcpyHostToDevice, h->stream));
  if (h->pf_attn) {
    // tiles: runs of at most qt entries of one cache row with one attention start at consecutive
    // positions; units (tile, kv head), longest key range first
    const int qt = attn_prefill_tile_tokens(h->cfg.group), kv = h->cfg.kv_heads, NT = h->NT;
    const int32_t* start = ranges_host;
    const int32_t* row = ranges_host + 2 * (size_t)n;
    std::vector<int32_t> tb(4 + 4 * (size_t)NT + 2 * (size_t)NT * kv, 0);
    int nt = 0;
    for (int e = 0; e < n; ++e) {
      int32_t* t = &tb[4 + 4 * (size_t)(nt - 1 >= 0 ? nt - 1 : 0)];
      if (nt > 0 && row[e] == t[2] && start[e] == t[3] && pos_host[e] == pos_host[e - 1] + 1 && t[1] < qt &&
          t[0] + t[1] == e) {
        ++t[1];
      } else {
        int32_t* nt_ = &tb[4 + 4 * (size_t)nt++];
        nt_[0] = e; nt_[1] = 1; nt_[2] = row[e]; nt_[3] = start[e];
      }
    }
    std::vector<int> order(nt);
    for (int i = 0; i < nt; ++i) order[i] = i;
    auto work = [&](int i) {
      const int32_t* t = &tb[4 + 4 * (size_t)i];
      return pos_host[t[0]] + t[1] - t[3];
    };
    std::stable_sort(order.begin(), order.end(), [&](int x, int y) { return work(x) > work(y); });
    int32_t* units = &tb[4 + 4 * (size_t)NT];
    int nu = 0;
    for (int i : order)
      for (int j = 0; j < kv; ++j) {
        units[2 * nu] = i;
        units[2 * nu + 1] = j;
        ++nu;
      }
    tb[0] = nu;
    tb[1] = nt;
    CUDA_TRY(h, cudaMemcpyAsync(h->tile_buf, tb.data(), (4 + 4 * (size_t)NT + 2 * (size_t)nu) * 4,
                                cudaMemcpyHostToDevice, h->stream));
  }
  TRY(begin(h, 0, n, tok_host, tok_dev, tok_stride, tok_col, 0.0f, 1, 1.0f, nullptr, nullptr, pos_host, nullptr, 0,
            h->range_buf, tok_np));
  return run_step(h, n, MODE_NOHEAD, true);
}

static llm_status prefill_impl(llm_handle* h, const int32_t* tok_host, const int32_t* tok_dev, int32_t B, int32_t S,
                               int32_t pos, float* logits, bool logits_on_host) {
  TRY(check_rows(h, B, pos, S));
  if (tok_host) TRY(check_tokens(h, tok_host, (size_t)B * S));
  if (S == 1 || h->cfg.debug_trace) {
    // single positions (a decode), or a traced handle: one step of all B rows per position
    for (int i = 0; i < S; ++i) {
      TRY(begin(h, pos + i, B, tok_host, tok_dev, S, i, 0.0f, 1, 1.0f, nullptr, nullptr));
      TRY(run_step(h, B, (i == S - 1 && logits) ? MODE_HEAD : MODE_NOHEAD));
    }
    if (logits) {
      if (logits_on_host) {
        CUDA_TRY(h, cudaMemcpyAsync(logits, h->logits, (size_t)B * h->V * 4, cudaMemcpyDeviceToHost, h->stream));
      } else if (logits != h->logits) {
        CUDA_TRY(h, cudaMemcpyAsync(logits, h->logits, (size_t)B * h->V * 4, cudaMemcpyDeviceToDevice, h->stream));
      }
    }
  } else {
    // passes of np whole positions of all B rows; entry e = b * cnt + i: row b, position
    // pos + p0 + i, token tokens[b * S + p0 + i]
    const int np = std::max(1, h->NT / B);
    std::vector<int32_t> epos, ranges, ents;
    std::vector<int> dst;
    for (int p0 = 0; p0 < S; p0 += np) {
      const int cnt = std::min(np, S - p0), n = B * cnt;
      epos.resize(n);
      ranges.resize(3 * (size_t)n);
      for (int b = 0; b < B; ++b)
        for (int i = 0; i < cnt; ++i) {
          const int e = b * cnt + i;
          epos[e] = pos + p0 + i;
          ranges[e] = 0;               // the whole cache of the row up to the position
          ranges[n + e] = pos + p0;    // this pass writes the row from pos + p0 on
          ranges[2 * n + e] = b;
        }
      TRY(run_pass(h, n, tok_host, tok_dev, S, p0, cnt, epos.data(), ranges.data()));
      if (p0 + cnt == S && logits) {
        ents.clear();
        dst.clear();
        for (int b = 0; b < B; ++b) {
          ents.push_back(b * cnt + cnt - 1);
          dst.push_back(b);
        }
        TRY(pass_logits(h, n, ents, dst, logits, logits_on_host));
      }
    }
  }
  if (logits_on_host) CUDA_TRY(h, cudaStreamSynchronize(h->stream));
  set_filled(h, B, pos + S);
  return LLM_OK;
}

llm_status llm_prefill(llm_handle* h, const int32_t* tokens_host, int32_t B, int32_t S, int32_t pos, float* logits_host) {
  if (!h || !tokens_host) return LLM_ERR_ARG;
  return prefill_impl(h, tokens_host, nullptr, B, S, pos, logits_host, true);
}

llm_status llm_prefill_dev(llm_handle* h, const int32_t* tokens_dev, int32_t B, int32_t S, int32_t pos, float* logits_dev) {
  if (!h || !tokens_dev) return LLM_ERR_ARG;
  return prefill_impl(h, nullptr, tokens_dev, B, S, pos, logits_dev, false);
}

llm_status llm_decode(llm_handle* h, const int32_t* tokens_host, int32_t B, int32_t pos, float* logits_host) {
  if (!h || !tokens_host || !logits_host) return LLM_ERR_ARG;
  return prefill_impl(h, tokens_host, nullptr, B, 1, pos, logits_host, true);
}

llm_status llm_decode_dev(llm_handle* h, const int32_t* tokens_dev, int32_t B, int32_t pos, float* logits_dev) {
  if (!h || !tokens_dev || !logits_dev) return LLM_ERR_ARG;
  return prefill_impl(h, nullptr, tokens_dev, B, 1, pos, logits_dev, false);
}

// one token per row, each row at its own position; logits of every row
static llm_status decode_rows_impl(llm_handle* h, const int32_t* tok_host, const int32_t* tok_dev, int32_t B,
                                   const int32_t* pos, float* logits, bool host) {
  TRY(check_row_positions(h, B, pos));
  if (tok_host) TRY(check_tokens(h, tok_host, (size_t)B));
  TRY(begin(h, 0, B, tok_host, tok_dev, 1, 0, 0.0f, 1, 1.0f, nullptr, nullptr, pos));
  TRY(run_step(h, B, MODE_HEAD));
  if (host) {
    CUDA_TRY(h, cudaMemcpyAsync(logits, h->logits, (size_t)B * h->V * 4, cudaMemcpyDeviceToHost, h->stream));
    CUDA_TRY(h, cudaStreamSynchronize(h->stream));
  } else if (logits != h->logits) {
    CUDA_TRY(h, cudaMemcpyAsync(logits, h->logits, (size_t)B * h->V * 4, cudaMemcpyDeviceToDevice, h->stream));
  }
  for (int b = 0; b < B; ++b) h->filled[b] = pos[b] + 1;
  return LLM_OK;
}

llm_status llm_decode_rows(llm_handle* h, const int32_t* tokens_host, int32_t B, const int32_t* positions_host,
                           float* logits_host) {
  if (!h || !tokens_host || !positions_host || !logits_host) return LLM_ERR_ARG;
  return decode_rows_impl(h, tokens_host, nullptr, B, positions_host, logits_host, true);
}

llm_status llm_decode_rows_dev(llm_handle* h, const int32_t* tokens_dev, int32_t B, const int32_t* positions_host,
                               float* logits_dev) {
  if (!h || !tokens_dev || !positions_host || !logits_dev) return LLM_ERR_ARG;
  return decode_rows_impl(h, nullptr, tokens_dev, B, positions_host, logits_dev, false);
}

// a paged step: rows at their own positions, every position found through the row's pages
static llm_status paged_impl(llm_handle* h, const int32_t* tok_host, const int32_t* tok_dev, int32_t B,
                             const int32_t* pos, const int32_t* table, int32_t pages_per_row, int mode, float temp,
                             int32_t k, float p, const float* u_host, const float* u_dev, int32_t* ids, float* logits,
                             bool host) {
  if (!h->page_table)
    return fail(h, LLM_ERR_CONFIG, "paged steps need max_seq (%d) to be a multiple of %d", h->cfg.max_seq, kPage);
  if (B < 1 || B > h->cfg.max_batch) return fail(h, LLM_ERR_BATCH, "batch %d outside 1..%d", B, h->cfg.max_batch);
  const int per_row = h->cfg.max_seq / kPage;
  if (pages_per_row < 1 || pages_per_row > per_row)
    return fail(h, LLM_ERR_ARG, "pages per row %d outside 1..%d", pages_per_row, per_row);
  const int64_t pool = (int64_t)h->cfg.max_batch * per_row;
  for (int b = 0; b < B; ++b) {
    if (pos[b] < 0 || pos[b] >= pages_per_row * kPage)
      return fail(h, LLM_ERR_POS_RANGE, "row %d: position %d outside its %d pages", b, pos[b], pages_per_row);
    for (int i = 0; i <= pos[b] / kPage; ++i) {
      const int32_t q = table[(size_t)b * pages_per_row + i];
      if (q < 0 || q >= pool) return fail(h, LLM_ERR_ARG, "row %d: page %d is %d, outside the pool of %lld", b, i, q, (long long)pool);
    }
  }
  TRY(check_sample_args(h, temp, k, p));
  if (temp > 0.0f && !u_host && !u_dev) return fail(h, LLM_ERR_ARG, "sampling needs uniform draws u");
  if (tok_host) TRY(check_tokens(h, tok_host, (size_t)B));
  if (u_host && temp > 0.0f)
    for (int b = 0; b < B; ++b)
      if (!(u_host[b] >= 0.0f && u_host[b] < 1.0f)) return fail(h, LLM_ERR_ARG, "u[%d] outside [0, 1)", b);
  CUDA_TRY(h, cudaMemcpyAsync(h->page_table, table, (size_t)B * pages_per_row * 4, cudaMemcpyHostToDevice, h->stream));
  TRY(begin(h, 0, B, tok_host, tok_dev, 1, 0, temp, k, p, u_host, u_dev, pos, h->page_table, pages_per_row));
  TRY(run_step(h, B, mode));
  if (host) {
    if (logits) CUDA_TRY(h, cudaMemcpyAsync(logits, h->logits, (size_t)B * h->V * 4, cudaMemcpyDeviceToHost, h->stream));
    if (ids) CUDA_TRY(h, cudaMemcpyAsync(ids, h->ids_buf, (size_t)B * 4, cudaMemcpyDeviceToHost, h->stream));
    CUDA_TRY(h, cudaStreamSynchronize(h->stream));
  } else {
    if (logits && logits != h->logits)
      CUDA_TRY(h, cudaMemcpyAsync(logits, h->logits, (size_t)B * h->V * 4, cudaMemcpyDeviceToDevice, h->stream));
    if (ids && ids != h->ids_buf) CUDA_TRY(h, cudaMemcpyAsync(ids, h->ids_buf, (size_t)B * 4, cudaMemcpyDeviceToDevice, h->stream));
  }
  return LLM_OK;
}

llm_status llm_decode_paged(llm_handle* h, const int32_t* tokens_host, int32_t B, const int32_t* positions_host,
                            const int32_t* table_host, int32_t pages_per_row, float* logits_host) {
  if (!h || !tokens_host || !positions_host || !table_host || !logits_host) return LLM_ERR_ARG;
  return paged_impl(h, tokens_host, nullptr, B, positions_host, table_host, pages_per_row, MODE_HEAD, 0.0f, 1, 1.0f,
                    nullptr, nullptr, nullptr, logits_host, true);
}

llm_status llm_decode_paged_dev(llm_handle* h, const int32_t* tokens_dev, int32_t B, const int32_t* positions_host,
                                const int32_t* table_host, int32_t pages_per_row, float* logits_dev) {
  if (!h || !tokens_dev || !positions_host || !table_host || !logits_dev) return LLM_ERR_ARG;
  return paged_impl(h, nullptr, tokens_dev, B, positions_host, table_host, pages_per_row, MODE_HEAD, 0.0f, 1, 1.0f,
                    nullptr, nullptr, nullptr, logits_dev, false);
}

llm_status llm_step_paged(llm_handle* h, const int32_t* tokens_host, int32_t B, const int32_t* positions_host,
                          const int32_t* table_host, int32_t pages_per_row, float temp, int32_t k, float p,
                          const float* u_host, int32_t* ids_host, float* logits_host) {
  if (!h || !tokens_host || !positions_host || !table_host || !ids_host) return LLM_ERR_ARG;
  return paged_impl(h, tokens_host, nullptr, B, positions_host, table_host, pages_per_row,
                    draw_mode(h, temp, k), temp, k, p, u_host, nullptr, ids_host, logits_host, true);
}

llm_status llm_step_paged_dev(llm_handle* h, const int32_t* tokens_dev, int32_t B, const int32_t* positions_host,
                              const int32_t* table_host, int32_t pages_per_row, float temp, int32_t k, float p,
                              const float* u_dev, int32_t* ids_dev, float* logits_dev) {
  if (!h || !tokens_dev || !positions_host || !table_host || !ids_dev) return LLM_ERR_ARG;
  return paged_impl(h, nullptr, tokens_dev, B, positions_host, table_host, pages_per_row,
                    draw_mode(h, temp, k), temp, k, p, nullptr, u_dev, ids_dev, logits_dev, false);
}

// Prompts packed end to end (Llama 3.1 8B Instruct card, "Entries": prefill_packed): token p is
// position positions[p] of prompt segments[p], in cache row rows[p]; each token attends to its
// own prompt's tokens up to itself.  The tokens run as the entries of prefill passes of at most
// NT entries, in position order: entry e reads and writes cache row rows[e], attends to positions
// start .. its position (start: its prompt's first position), and reads nothing its pass writes
// before the Q/K/V kernel has finished.
static llm_status packed_impl(llm_handle* h, const int32_t* toks, const int32_t* rows, const int32_t* positions,
                              const int32_t* segments, int32_t P, const int32_t* last, int32_t nlast, float* logits) {
  if (P < 1 || nlast < 0) return fail(h, LLM_ERR_ARG, "tokens %d < 1 or last count %d < 0", P, nlast);
  if (h->cfg.debug_trace) return fail(h, LLM_ERR_ARG, "debug_trace handles run without graphs");
  TRY(check_tokens(h, toks, (size_t)P));
  for (int i = 0; i < P; ++i) {
    if (rows[i] < 0 || rows[i] >= h->cfg.max_batch)
      return fail(h, LLM_ERR_BATCH, "token %d: row %d outside 0..%d", i, rows[i], h->cfg.max_batch - 1);
    if (positions[i] < 0 || positions[i] >= h->cfg.max_seq)
      return fail(h, LLM_ERR_POS_RANGE, "token %d: position %d outside the cache of %d", i, positions[i], h->cfg.max_seq);
  }
  for (int m = 0; m < nlast; ++m)
    if (last[m] < 0 || last[m] >= P) return fail(h, LLM_ERR_ARG, "last[%d] = %d names no token", m, last[m]);
  // each prompt: one row, consecutive positions first..first+n-1, each once; prompts of one row
  // do not overlap
  struct Span { int row, lo, hi, n; };
  std::map<int32_t, Span> span;
  for (int i = 0; i < P; ++i) {
    auto it = span.find(segments[i]);
    if (it == span.end()) {
      span[segments[i]] = Span{rows[i], positions[i], positions[i], 1};
    } else {
      Span& sp = it->second;
      if (sp.row != rows[i]) return fail(h, LLM_ERR_ARG, "prompt %d spans rows %d and %d", segments[i], sp.row, rows[i]);
      sp.lo = std::min(sp.lo, positions[i]);
      sp.hi = std::max(sp.hi, positions[i]);
      ++sp.n;
    }
  }
  {
    std::map<std::pair<int, int>, int> slot;  // (row, position) -> token
    for (int i = 0; i < P; ++i)
      if (!slot.emplace(std::make_pair(rows[i], positions[i]), i).second)
        return fail(h, LLM_ERR_ARG, "tokens %d and %d share row %d position %d", slot[{rows[i], positions[i]}], i,
                    rows[i], positions[i]);
    for (auto& kv : span)
      if (kv.second.hi - kv.second.lo + 1 != kv.second.n)
        return fail(h, LLM_ERR_ARG, "prompt %d does not fill positions %d..%d", kv.first, kv.second.lo, kv.second.hi);
    for (auto& a : span)
      for (auto& b : span)
        if (a.first < b.first && a.second.row == b.second.row && a.second.lo <= b.second.hi && b.second.lo <= a.second.hi)
          return fail(h, LLM_ERR_ARG, "prompts %d and %d overlap in row %d", a.first, b.first, a.second.row);
  }
  // position order, then passes of at most NT entries
  std::vector<int> order(P);
  for (int i = 0; i < P; ++i) order[i] = i;
  std::stable_sort(order.begin(), order.end(), [&](int x, int y) { return positions[x] < positions[y]; });
  std::vector<std::vector<int>> last_of(P);  // token -> the indices m of last naming it
  for (int m = 0; m < nlast; ++m) last_of[last[m]].push_back(m);
  const int cap_e = h->NT;
  std::vector<int32_t> etok, epos, eranges, ents;
  std::vector<int> dst;
  for (int p0 = 0; p0 < P; p0 += cap_e) {
    const int n = std::min(cap_e, P - p0);
    // inside a pass, the entries of one row in position order (runs of one prompt form the
    // attention's tiles)
    std::vector<int> pe(order.begin() + p0, order.begin() + p0 + n);
    std::stable_sort(pe.begin(), pe.end(), [&](int x, int y) {
      return rows[x] != rows[y] ? rows[x] < rows[y] : positions[x] < positions[y];
    });
    etok.assign(n, 0);
    epos.assign(n, 0);
    eranges.assign(3 * (size_t)n, 0);
    ents.clear();
    dst.clear();
    std::map<int, int> wfirst;  // row -> first position this pass writes in it
    for (int e = 0; e < n; ++e) {
      const int i = pe[e];
      etok[e] = toks[i];
      epos[e] = positions[i];
      eranges[e] = span[segments[i]].lo;
      eranges[2 * (size_t)n + e] = rows[i];
      auto w = wfirst.find(rows[i]);
      if (w == wfirst.end() || positions[i] < w->second) wfirst[rows[i]] = positions[i];
      for (int m : last_of[i]) {
        ents.push_back(e);
        dst.push_back(m);
      }
    }
    for (int e = 0; e < n; ++e) eranges[n + e] = wfirst[rows[pe[e]]];
    TRY(run_pass(h, n, etok.data(), nullptr, 1, 0, 1, epos.data(), eranges.data()));
    if (logits) TRY(pass_logits(h, n, ents, dst, logits, true));
    // (the host vectors are refilled for the next pass: its copies read them first)
    CUDA_TRY(h, cudaStreamSynchronize(h->stream));
  }
  for (auto& kv : span) h->filled[kv.second.row] = std::max(h->filled[kv.second.row], kv.second.hi + 1);
  return LLM_OK;
}

llm_status llm_prefill_packed(llm_handle* h, const int32_t* tokens_host, const int32_t* rows_host,
                              const int32_t* positions_host, const int32_t* segments_host, int32_t P,
                              const int32_t* last_host, int32_t nlast, float* logits_host) {
  if (!h || !tokens_host || !rows_host || !positions_host || !segments_host || (nlast > 0 && !last_host))
    return LLM_ERR_ARG;
  return packed_impl(h, tokens_host, rows_host, positions_host, segments_host, P, last_host, nlast, logits_host);
}

// n decode steps, each feeding its draws to the next as tokens, as CUDA graphs of kGenChunk
// steps (then single steps): no host round trip between the steps of a graph
static llm_status generate_impl(llm_handle* h, const int32_t* tok_host, const int32_t* tok_dev, int32_t B,
                                int32_t pos, int32_t n, float temp, int32_t k, float p, const float* u_host,
                                const float* u_dev, int32_t* ids, bool host) {
  if (n < 1) return fail(h, LLM_ERR_ARG, "steps %d < 1", n);
  if (h->cfg.debug_trace) return fail(h, LLM_ERR_ARG, "debug_trace handles run without graphs");
  TRY(check_rows(h, B, pos, n));
  TRY(check_sample_args(h, temp, k, p));
  const bool sampled = temp > 0.0f;
  if (sampled && !u_host && !u_dev) return fail(h, LLM_ERR_ARG, "sampling needs uniform draws u");
  if (tok_host) TRY(check_tokens(h, tok_host, (size_t)B));
  if (u_host && sampled)
    for (size_t i = 0; i < (size_t)n * B; ++i)
      if (!(u_host[i] >= 0.0f && u_host[i] < 1.0f)) return fail(h, LLM_ERR_ARG, "u[%zu] outside [0, 1)", i);
  const int mode = draw_mode(h, temp, k);
  const int32_t* prev = tok_dev;
  if (tok_host) {
    CUDA_TRY(h, cudaMemcpyAsync(h->tok_buf, tok_host, (size_t)B * 4, cudaMemcpyHostToDevice, h->stream));
    prev = h->tok_buf;
  }
  for (int done = 0; done < n;) {
    const int c = n - done >= kGenChunk ? kGenChunk : 1;
    GenState v = {};
    v.pos = pos + done; v.B = B; v.temp = temp; v.k = k; v.p = p; v.prev = prev;
    if (host) {
      if (sampled)
        CUDA_TRY(h, cudaMemcpyAsync(h->u_gen, u_host + (size_t)done * B, (size_t)c * B * 4, cudaMemcpyHostToDevice,
                                    h->stream));
      v.u = h->u_gen;
      v.ids = h->ids_gen;
    } else {
      v.u = sampled ? u_dev + (size_t)done * B : nullptr;
      v.ids = ids + (size_t)done * B;
    }
    gen_set_kernel<<<1, 1, 0, h->stream>>>(h->gen, v);
    CUDA_TRY(h, cudaGetLastError());
    std::pair<cudaGraphExec_t, int>* g = nullptr;
    TRY(step_graph(h, B, mode, &g, c));
    CUDA_TRY(h, cudaGraphLaunch(g->first, h->stream));
    if (host) {
      CUDA_TRY(h, cudaMemcpyAsync(ids + (size_t)done * B, h->ids_gen, (size_t)c * B * 4, cudaMemcpyDeviceToHost,
                                  h->stream));
      prev = h->ids_gen + (size_t)(c - 1) * B;  // read by the next launch's first step before it is rewritten
    } else {
      prev = ids + (size_t)(done + c - 1) * B;
    }
    done += c;
  }
  if (host) CUDA_TRY(h, cudaStreamSynchronize(h->stream));
  set_filled(h, B, pos + n);
  return LLM_OK;
}

llm_status llm_generate(llm_handle* h, const int32_t* tokens_host, int32_t B, int32_t pos, int32_t n_steps,
                        float temp, int32_t k, float p, const float* u_host, int32_t* ids_host) {
  if (!h || !tokens_host || !ids_host) return LLM_ERR_ARG;
  return generate_impl(h, tokens_host, nullptr, B, pos, n_steps, temp, k, p, u_host, nullptr, ids_host, true);
}

llm_status llm_generate_dev(llm_handle* h, const int32_t* tokens_dev, int32_t B, int32_t pos, int32_t n_steps,
                            float temp, int32_t k, float p, const float* u_dev, int32_t* ids_dev) {
  if (!h || !tokens_dev || !ids_dev) return LLM_ERR_ARG;
  return generate_impl(h, nullptr, tokens_dev, B, pos, n_steps, temp, k, p, nullptr, u_dev, ids_dev, false);
}

static llm_status sample_impl(llm_handle* h, const float* logits, bool logits_on_host, int32_t B, float temp, int32_t k,
                              float p, const float* u, bool u_on_host, int32_t* ids, bool ids_on_host) {
  if (B < 1 || B > h->cfg.max_batch) return fail(h, LLM_ERR_BATCH, "batch %d outside 1..%d", B, h->cfg.max_batch);
  TRY(check_sample_args(h, temp, k, p));
  if (temp > 0.0f && !u) return fail(h, LLM_ERR_ARG, "sampling needs uniform draws u");
  if (u && u_on_host && temp > 0.0f)
    for (int b = 0; b < B; ++b)
      if (!(u[b] >= 0.0f && u[b] < 1.0f)) return fail(h, LLM_ERR_ARG, "u[%d] outside [0, 1)", b);
  if (logits != h->logits)
    CUDA_TRY(h, cudaMemcpyAsync(h->logits, logits, (size_t)B * h->V * 4,
                                logits_on_host ? cudaMemcpyHostToDevice : cudaMemcpyDeviceToDevice, h->stream));
  // the prologue also carries temp, k, p and u; its tokens are unused here
  std::vector<int32_t> toks(B, 0);
  TRY(begin(h, 0, B, toks.data(), nullptr, 1, 0, temp, k, p, u_on_host ? u : nullptr, u_on_host ? nullptr : u));
  CUDA_TRY(h, launch_sample(sample_args(h), B, !(temp > 0.0f), h->stream, false, draw_mode(h, temp, k) == MODE_TOPK));
  if (ids_on_host) {
    CUDA_TRY(h, cudaMemcpyAsync(ids, h->ids_buf, (size_t)B * 4, cudaMemcpyDeviceToHost, h->stream));
    CUDA_TRY(h, cudaStreamSynchronize(h->stream));
  } else if (ids != h->ids_buf) {
    CUDA_TRY(h, cudaMemcpyAsync(ids, h->ids_buf, (size_t)B * 4, cudaMemcpyDeviceToDevice, h->stream));
  }
  return LLM_OK;
}

llm_status llm_sample(llm_handle* h, const float* logits_host, int32_t B, float temp, int32_t k, float p,
                      const float* u_host, int32_t* ids_host) {
  if (!h || !logits_host || !ids_host) return LLM_ERR_ARG;
  return sample_impl(h, logits_host, true, B, temp, k, p, u_host, true, ids_host, true);
}

llm_status llm_sample_dev(llm_handle* h, const float* logits_dev, int32_t B, float temp, int32_t k, float p,
                          const float* u_dev, int32_t* ids_dev) {
  if (!h || !logits_dev || !ids_dev) return LLM_ERR_ARG;
  return sample_impl(h, logits_dev, false, B, temp, k, p, u_dev, false, ids_dev, false);
}

static llm_status step_impl(llm_handle* h, const int32_t* tok_host, const int32_t* tok_dev, int32_t B, int32_t pos,
                            float temp, int32_t k, float p, const float* u_host, const float* u_dev, int32_t* ids,
                            float* logits, bool host, const int32_t* pos_rows = nullptr) {
  if (pos_rows) TRY(check_row_positions(h, B, pos_rows));
  else TRY(check_rows(h, B, pos, 1));
  TRY(check_sample_args(h, temp, k, p));
  if (temp > 0.0f && !u_host && !u_dev) return fail(h, LLM_ERR_ARG, "sampling needs uniform draws u");
  if (tok_host) TRY(check_tokens(h, tok_host, (size_t)B));
  if (u_host && temp > 0.0f)
    for (int b = 0; b < B; ++b)
      if (!(u_host[b] >= 0.0f && u_host[b] < 1.0f)) return fail(h, LLM_ERR_ARG, "u[%d] outside [0, 1)", b);
  TRY(begin(h, pos, B, tok_host, tok_dev, 1, 0, temp, k, p, u_host, u_dev, pos_rows));
  TRY(run_step(h, B, draw_mode(h, temp, k)));
  if (host) {
    if (logits) CUDA_TRY(h, cudaMemcpyAsync(logits, h->logits, (size_t)B * h->V * 4, cudaMemcpyDeviceToHost, h->stream));
    CUDA_TRY(h, cudaMemcpyAsync(ids, h->ids_buf, (size_t)B * 4, cudaMemcpyDeviceToHost, h->stream));
    CUDA_TRY(h, cudaStreamSynchronize(h->stream));
  } else {
    if (logits && logits != h->logits)
      CUDA_TRY(h, cudaMemcpyAsync(logits, h->logits, (size_t)B * h->V * 4, cudaMemcpyDeviceToDevice, h->stream));
    if (ids != h->ids_buf) CUDA_TRY(h, cudaMemcpyAsync(ids, h->ids_buf, (size_t)B * 4, cudaMemcpyDeviceToDevice, h->stream));
  }
  if (pos_rows) {
    for (int b = 0; b < B; ++b) h->filled[b] = pos_rows[b] + 1;
  } else {
    set_filled(h, B, pos + 1);
  }
  return LLM_OK;
}

llm_status llm_step(llm_handle* h, const int32_t* tokens_host, int32_t B, int32_t pos, float temp, int32_t k, float p,
                    const float* u_host, int32_t* ids_host, float* logits_host) {
  if (!h || !tokens_host || !ids_host) return LLM_ERR_ARG;
  return step_impl(h, tokens_host, nullptr, B, pos, temp, k, p, u_host, nullptr, ids_host, logits_host, true);
}

llm_status llm_step_dev(llm_handle* h, const int32_t* tokens_dev, int32_t B, int32_t pos, float temp, int32_t k,
                        float p, const float* u_dev, int32_t* ids_dev, float* logits_dev) {
  if (!h || !tokens_dev || !ids_dev) return LLM_ERR_ARG;
  return step_impl(h, nullptr, tokens_dev, B, pos, temp, k, p, nullptr, u_dev, ids_dev, logits_dev, false);
}

llm_status llm_step_rows(llm_handle* h, const int32_t* tokens_host, int32_t B, const int32_t* positions_host,
                         float temp, int32_t k, float p, const float* u_host, int32_t* ids_host, float* logits_host) {
  if (!h || !tokens_host || !positions_host || !ids_host) return LLM_ERR_ARG;
  return step_impl(h, tokens_host, nullptr, B, 0, temp, k, p, u_host, nullptr, ids_host, logits_host, true,
                   positions_host);
}

llm_status llm_step_rows_dev(llm_handle* h, const int32_t* tokens_dev, int32_t B, const int32_t* positions_host,
                             float temp, int32_t k, float p, const float* u_dev, int32_t* ids_dev, float* logits_dev) {
  if (!h || !tokens_dev || !positions_host || !ids_dev) return LLM_ERR_ARG;
  return step_impl(h, nullptr, tokens_dev, B, 0, temp, k, p, nullptr, u_dev, ids_dev, logits_dev, false,
                   positions_host);
}

static llm_status kv_copy(llm_handle* h, int32_t layer, int32_t row, int32_t pos0, int32_t n, void* k, void* v,
                          bool import) {
  if (!h || !k || !v) return LLM_ERR_ARG;
  if (layer < 0 || layer >= h->L) return fail(h, LLM_ERR_ARG, "layer %d outside 0..%d", layer, h->L - 1);
  if (row < 0 || row >= h->cfg.max_batch) return fail(h, LLM_ERR_BATCH, "row %d outside 0..%d", row, h->cfg.max_batch - 1);
  if (pos0 < 0 || n < 0 || (int64_t)pos0 + n > h->cfg.max_seq)
    return fail(h, LLM_ERR_POS_RANGE, "positions %d..+%d outside the cache of %d", pos0, n, h->cfg.max_seq);
  const size_t es = h->es, hd = h->hd, kv = h->cfg.kv_heads, cap = h->cfg.max_seq;
  const size_t bytes = (size_t)n * hd * es;
  for (size_t j = 0; j < kv; ++j) {
    const size_t elem = (size_t)layer * h->layer_cache_elems + (((size_t)row * kv + j) * cap + pos0) * hd;
    char* dk = (char*)h->kc + elem * es;
    char* dv = (char*)h->vc + elem * es;
    char* hk = (char*)k + j * bytes;
    char* hv = (char*)v + j * bytes;
    if (import) {
      CUDA_TRY(h, cudaMemcpyAsync(dk, hk, bytes, cudaMemcpyHostToDevice, h->stream));
      CUDA_TRY(h, cudaMemcpyAsync(dv, hv, bytes, cudaMemcpyHostToDevice, h->stream));
    } else {
      CUDA_TRY(h, cudaMemcpyAsync(hk, dk, bytes, cudaMemcpyDeviceToHost, h->stream));
      CUDA_TRY(h, cudaMemcpyAsync(hv, dv, bytes, cudaMemcpyDeviceToHost, h->stream));
    }
  }
  CUDA_TRY(h, cudaStreamSynchronize(h->stream));
  if (import && h->filled[row] < pos0 + n) h->filled[row] = pos0 + n;
  return LLM_OK;
}

llm_status llm_kv_import(llm_handle* h, int32_t layer, int32_t row, int32_t pos0, int32_t n, const void* k_host,
                         const void* v_host) {
  return kv_copy(h, layer, row, pos0, n, (void*)k_host, (void*)v_host, true);
}

llm_status llm_kv_export(llm_handle* h, int32_t layer, int32_t row, int32_t pos0, int32_t n, void* k_host, void* v_host) {
  return kv_copy(h, layer, row, pos0, n, k_host, v_host, false);
}

llm_status llm_step_kernels(llm_handle* h, int32_t B, float temp, int32_t k, int32_t* kernels) {
  if (!h || !kernels) return LLM_ERR_ARG;
  if (B < 1 || B > h->cfg.max_batch) return fail(h, LLM_ERR_BATCH, "batch %d outside 1..%d", B, h->cfg.max_batch);
  if (h->cfg.debug_trace) return fail(h, LLM_ERR_ARG, "debug_trace handles run without a step graph");
  std::pair<cudaGraphExec_t, int>* g = nullptr;
  TRY(step_graph(h, B, draw_mode(h, temp, k), &g));
  *kernels = 1 + g->second;  // the step prologue, then the graph
  return LLM_OK;
}

llm_status llm_profile_kernel(llm_handle* h, int32_t which, int32_t B, int32_t pos, int32_t reps, float* ms_per_launch) {
  if (!h || !ms_per_launch || reps < 1) return LLM_ERR_ARG;
  if (which < K_QKV || which > K_SAMPLE) return fail(h, LLM_ERR_ARG, "kernel id %d outside 0..6", which);
  TRY(check_rows(h, B, pos, 1));
  std::vector<int32_t> toks(B, 0);
  std::vector<float> u(B, 0.5f);
  TRY(begin(h, pos, B, toks.data(), nullptr, 1, 0, 1.0f, h->V, 1.0f, u.data(), nullptr));
  TRY(launch_one(h, K_EMBED, 0, B, false));
  cudaEvent_t e0, e1;
  CUDA_TRY(h, cudaEventCreate(&e0));
  CUDA_TRY(h, cudaEventCreate(&e1));
  CUDA_TRY(h, cudaEventRecord(e0, h->stream));
  for (int r = 0; r < reps; ++r) TRY(launch_one(h, which, r % h->L, B, false));
  CUDA_TRY(h, cudaEventRecord(e1, h->stream));
  CUDA_TRY(h, cudaEventSynchronize(e1));
  float ms = 0.f;
  CUDA_TRY(h, cudaEventElapsedTime(&ms, e0, e1));
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  *ms_per_launch = ms / reps;
  return LLM_OK;
}

llm_status llm_debug_trace(llm_handle* h, int32_t layer, const char* name, float* dst_host) {
  if (!h || !name || !dst_host) return LLM_ERR_ARG;
  if (!h->cfg.debug_trace) return fail(h, LLM_ERR_ARG, "the handle was created without debug_trace");
  if (layer < 0 || layer >= h->L) return fail(h, LLM_ERR_ARG, "layer %d outside 0..%d", layer, h->L - 1);
  // name -> (slot, first element, width)
  const int d = h->d, kvw = h->kvw;
  const struct { const char* name; int slot, off, width; } names[] = {
      {"n1", TR_N1, 0, d},     {"q", TR_QKV, 0, d},       {"k", TR_QKV, d, kvw},   {"v", TR_QKV, d + kvw, kvw},
      {"qr", TR_QR, 0, d},     {"kr", TR_KR, 0, kvw},     {"attn", TR_ATTN, 0, d}, {"a", TR_A, 0, d},
      {"x1", TR_X1, 0, d},     {"n2", TR_N2, 0, d},       {"swiglu", TR_SWIGLU, 0, h->f},
      {"m", TR_M, 0, d},       {"y", TR_Y, 0, d}};
  int which = -1;
  for (int i = 0; i < (int)(sizeof names / sizeof names[0]); ++i)
    if (!strcmp(name, names[i].name)) which = i;
  if (which < 0) return fail(h, LLM_ERR_ARG, "unknown trace name %s", name);
  const size_t maxw = h->trace_w;
  const size_t width = (size_t)names[which].width;
  const float* src = h->trace + ((size_t)layer * kTraceSlots + names[which].slot) * h->cfg.max_batch * maxw +
                     names[which].off;
  CUDA_TRY(h, cudaStreamSynchronize(h->stream));
  CUDA_TRY(h, cudaMemcpy2D(dst_host, width * 4, src, maxw * 4, width * 4, h->cfg.max_batch, cudaMemcpyDeviceToHost));
  return LLM_OK;
}

}  // extern "C"
