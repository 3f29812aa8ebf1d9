// Greedy and temperature / top-k / top-p sampling (declarations).
#pragma once
#include "common.cuh"

namespace llm {

struct SampleArgs {
  const float* logits;   // [B][logits_stride]
  int32_t logits_stride;
  int32_t V;
  int32_t V_pad;         // row pitch of the scratch arrays
  uint32_t* keys;        // scratch [B][2][V_pad]
  int32_t* idx;          // scratch [B][2][V_pad]
  float* pre;            // scratch [B][V_pad]: weights, then their running sums
  const float* u;        // [B] uniform draws
  int32_t* ids;          // [B] drawn ids
  const StepState* step; // temp, k, p
};

size_t sample_smem();
cudaError_t sample_prepare();
cudaError_t launch_sample(const SampleArgs& a, int B, cudaStream_t s, bool pdl);

}  // namespace llm
