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
  uint32_t* hist;        // scratch [B][digits][sample_slices(V)]: digit counts, then offsets, per CTA slice
  size_t hist_per_row;   // uint32 entries of hist per row: 256 digits (8-bit) need 256 * slices
  const float* u;        // [B] uniform draws
  int32_t* ids;          // [B] drawn ids
  const StepState* step; // temp, k, p
};

constexpr int kSortMaxSlicesPerRow = 64;
constexpr size_t kSampleHistPerRow = 256 * kSortMaxSlicesPerRow;  // uint32 entries a row needs at most (8-bit digits)

int sample_slices(int V);
// greedy: one argmax kernel; select (top-k with k <= sample_select_max()): one radix-select
// kernel per row; otherwise the sort chain and the draw (temp, k, p from *step)
cudaError_t launch_sample(const SampleArgs& a, int B, bool greedy, cudaStream_t s, bool pdl, bool select = false);
int sample_select_max();
// loads the allocation-free sampler's fixed array on the current device and records its address
cudaError_t noalloc_prepare();

}  // namespace llm
