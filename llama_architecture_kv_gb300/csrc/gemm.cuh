// Tensor-core (tcgen05) projections for batched decode (declarations).
#pragma once
#include <cuda.h>

#include "common.cuh"
#include "gemv.cuh"

namespace llm {

constexpr int kTcThreads = 192;   // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int kTcM = 128;         // weight rows per tile (TMEM lanes)
constexpr int kTcK = 64;          // K elements per stage (one 128-byte swizzle row)
constexpr int kTcMaxNP = 256;     // columns per tile
constexpr int kTcDefaultMinBatch = 16;  // rows from which a step uses the tensor cores

struct TcArgs {
  int32_t rows, K;        // W [rows][K] bf16, row-major
  int32_t N;              // valid columns (batch rows) in total
  int32_t NP;             // columns per tile: a multiple of 16, at most 256
  int32_t Ntot;           // columns of the split activations per half (a multiple of NP)
  int32_t MT, KB;         // 128-row tiles, 64-element K blocks
  int32_t stages;         // shared-memory pipeline depth
  uint32_t tmem_cols;     // tensor-memory columns allocated (two accumulators of NP)
  float* part;            // split partials [n tiles][grid][2][128 rows][NP]
  uint32_t* ticket;       // [n tiles][MT], zero between launches
  int32_t* status;        // device error flag
  const StepState* step;
  // epilogue (as GemvArgs)
  float* out;
  int32_t out_stride;
  const float* resid;
  int32_t resid_stride;
  float* q_out;
  int32_t q_stride;
  void* kc;
  void* vc;
  int32_t H, kv, hd, cap;
  const float* rope_cos;
  const float* rope_sin;
};

struct TcSplitArgs {
  const float* x;         // [B][x_stride] f32
  int32_t x_stride;
  const float* gain;      // RMSNorm gains [K] or nullptr (no norm)
  float eps;
  int32_t K, B, Ntot;
  uint16_t* xs;           // [2][Ntot][K] bf16: hi rows, then lo rows
};

struct TcPlan {
  int NP, Ntot, MT, KB, grid, ntiles, stages;
  uint32_t tmem_cols;
  size_t smem;
};

// the tensor-core path needs bf16 weights and rows of K a multiple of 8 elements (16 bytes)
bool tc_available();
cudaError_t tc_prepare(int max_smem_optin);
TcPlan plan_tc(int rows, int K, int B, int num_sms);
// 2D bf16 tensor map over [outer][inner] (row pitch inner elements), box box_inner x box_outer,
// 128-byte swizzle
bool tc_make_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
                 uint32_t box_outer);
// general 2D tensor map (elements of elem_bytes: 2 = bf16, 4 = f32) with the given swizzle
bool make_map_2d(CUtensorMap* map, const void* base, int elem_bytes, uint64_t inner, uint64_t outer,
                 uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle);
cudaError_t launch_tc_split(const TcSplitArgs& a, cudaStream_t s, bool pdl);
cudaError_t launch_tc_gemm(const CUtensorMap& tw, const CUtensorMap& tx, const TcArgs& a, const TcPlan& p, int epi,
                           cudaStream_t s, bool pdl);

}  // namespace llm
