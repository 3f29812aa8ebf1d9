// Split-K decode attention over the KV cache (declarations).
#pragma once
#include "common.cuh"

namespace llm {

struct AttnArgs {
  const float* q;      // rotated queries [B][q_stride]
  int32_t q_stride;
  const void* kc;      // this layer's key cache [max_batch][kv][cap][hd]
  const void* vc;      // this layer's value cache
  float* out;          // attention output [B][out_stride], heads concatenated
  int32_t out_stride;
  float* part;         // partials [B][H][ns][hd + 2]: unnormalized o, running max, running sum
  uint32_t* ticket;    // [B][kv], zero between launches
  int32_t B, kv, g, hd, cap, ns;
  float scale;         // 1 / sqrt(hd), rounded to f32
  const StepState* step;
};

constexpr int kAttnMaxCluster = 16;  // most splits merged inside one thread-block cluster

bool attn_supported(int hd, int g);
// splits per (row, kv head); at most attn_max_cluster() means the splits form one cluster
int attn_max_cluster();
int attn_splits(int B, int kv, int cap, int num_sms);
cudaError_t attn_prepare(int max_smem_optin);
cudaError_t launch_attn(const AttnArgs& a, int kt, cudaStream_t s, bool pdl);

}  // namespace llm
