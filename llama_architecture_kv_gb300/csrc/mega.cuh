// One kernel for all layers of a batch-1 decode step (declarations).
#pragma once
#include "common.cuh"

namespace llm {

struct MegaLayer {
  const void* qkv;   // [(H + 2kv) * hd][d] bf16, rows in RoPE pairs
  const float* ln1;  // [d]
  const void* o;     // [d][d]
  const float* ln2;  // [d]
  const void* gu;    // [2f][d], rows (gate i, up i)
  const void* down;  // [d][f]
};

struct MegaArgs {
  const MegaLayer* layers;  // [L], device memory
  int32_t L, d, f, V, H, kv, g, hd, cap, max_batch;
  float eps, scale;
  const float* lnf;         // [d]
  const void* head;         // [V][d] bf16 (the embedding when tied)
  void* kc;                 // key cache [L][max_batch][kv][cap][hd] bf16 (row 0 is used)
  void* vc;                 // value cache
  const float* rope_cos;    // [cap][hd / 2]
  const float* rope_sin;
  const StepState* step;
  float* x;                 // residual stream [d]: the embedding on entry, the last layer's output after
  float* x1;                // [d]
  float* q;                 // rotated queries [H * hd]
  float* attn;              // attention output [H * hd]
  float* m;                 // SwiGLU output [f]
  float* logits;            // [V]
  float* apart;             // attention partials [H][kMegaMaxSplits][hd + 2]
  uint32_t* ticket;         // [kv + 1], zero between launches: attention merges, then the argmax
  uint32_t* bar;            // grid barrier counter, zero on entry
  float* cand_v;            // [grid] per-CTA argmax candidates
  int32_t* cand_i;
  int32_t* ids;             // the greedy id (head_mode 2)
  int32_t head_mode;        // 0: no head, 1: logits, 2: logits and the greedy id
  int32_t* status;
};

constexpr int kMegaMaxSplits = 64;

// bf16 weights and cache, head size 64 or 128, at most 8 query heads per kv head, widths that
// are multiples of 8
bool mega_supported(int wt, int hd, int g, int d, int f);
// shared memory of one CTA for hidden size d and MLP width f
size_t mega_smem(int d, int f);
cudaError_t mega_prepare(int max_smem_optin);
// cooperative launch of `grid` CTAs (one per SM)
cudaError_t launch_mega(const MegaArgs& a, int grid, cudaStream_t s);

}  // namespace llm
