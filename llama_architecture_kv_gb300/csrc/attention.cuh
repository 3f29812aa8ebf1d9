// Split-K decode attention over the KV cache (declarations).
#pragma once
#include <cuda.h>

#include "common.cuh"

namespace llm {

struct AttnArgs {
  const float* q;      // rotated queries [B][q_stride]
  int32_t q_stride;
  const void* vc;      // this layer's value cache [max_batch][kv][cap][hd]
  int32_t krow0;       // row of this layer's position 0 of (row 0, kv head 0) in the key map
  float* out;          // attention output [B][out_stride], heads concatenated
  int32_t out_stride;
  float* part;         // partials [B][H][ns][hd + 2]: unnormalized o, running max, running sum
  uint32_t* ticket;    // [B][kv], zero between launches
  int32_t B, kv, g, hd, cap, ns;
  float scale;         // 1 / sqrt(hd), rounded to f32
  const StepState* step;
  int32_t* status;     // device error flag
  int32_t cluster;     // set by launch_attn: the splits form one thread-block cluster
};

constexpr int kAttnMaxCluster = 16;  // most splits merged inside one thread-block cluster

bool attn_supported(int hd, int g);
// splits per (row, kv head); at most attn_max_cluster() means the splits form one cluster
int attn_max_cluster();
int attn_splits(int B, int kv, int cap, int num_sms);
cudaError_t attn_prepare(int max_smem_optin);
// tensor map over a whole key (or value) cache viewed as [rows][hd]
// (rows = layers * max_batch * kv * cap), boxes of 32 rows
bool attn_make_kmap(CUtensorMap* map, const void* kc, int kt, int hd, uint64_t rows);
// bf16 caches with hd 64 or 128 run the tensor-core kernel (which also reads the values by map)
bool attn_uses_mma(int kt, int hd);
// partial slots per (row, kv head) the kernels need for ns splits
int attn_part_slots(int kt, int hd, int ns);
// whether ns splits of `clusters` (row, kv head) pairs merge inside thread-block clusters (the
// tensor-core kernel: clusters of its own size, for caches of at most cap positions); the first
// call for a shape queries the device (make it outside stream capture)
bool attn_cluster_merge(int kt, int hd, int g, int ns, int clusters, int cap);
cudaError_t launch_attn(const CUtensorMap& kmap, const CUtensorMap& vmap, const AttnArgs& a, int kt, cudaStream_t s,
                        bool pdl);

// Causal attention of a prefill pass over tiles of consecutive prompt tokens (bf16 caches, head
// size 64 or 128, at most 8 query heads per kv head).  tiles: int32 [4 + 4 * max_tiles + 2 *
// max_tiles * kv] = {units, tiles, 0, 0}, then per tile {first entry, tokens, cache row,
// attention start}, then per unit {tile, kv head}, units longest first.  A tile holds at most
// attn_prefill_tile_tokens(g) tokens of one cache row at consecutive positions.
struct AttnPrefillArgs {
  const float* q;        // rotated queries of the pass's entries [n][q_stride]
  int32_t q_stride;
  float* out;            // [n][out_stride]
  int32_t out_stride;
  const int32_t* tiles;  // device memory, layout above
  int32_t max_tiles;
  int32_t krow0;         // row of this layer's position 0 of (cache row 0, kv head 0) in the maps
  int32_t kv, g, hd, cap;
  float scale;
  const StepState* step; // entry positions (row_pos)
  int32_t* status;
};
bool attn_prefill_supported(int kt, int hd, int g);
int attn_prefill_tile_tokens(int g);
cudaError_t attn_prefill_prepare(int max_smem_optin);
cudaError_t launch_attn_prefill(const CUtensorMap& kmap, const CUtensorMap& vmap, const AttnPrefillArgs& a, int grid,
                                cudaStream_t s, bool pdl);

}  // namespace llm
