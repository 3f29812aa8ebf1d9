// Tensor-core (tcgen05) projections for batched decode (declarations).
#pragma once
#include <cuda.h>

#include "common.cuh"

namespace llm {

constexpr int kTcThreads = 192;   // warp 0 TMA, warp 1 MMA, warps 2..5 read the accumulators
constexpr int kTcN = 256;         // weight rows per tile (the MMA's N)
constexpr int kTcK = 64;          // K elements per stage (one 128-byte swizzle row)
constexpr int kTcRows = 64;       // activation rows per tile (hi in MMA rows 0..63, lo in 64..127)
constexpr int kTcDefaultMinBatch = 2;   // rows from which a step uses the tensor cores
constexpr int kTcMaxK = 16384;          // widest projection input the prep kernels stage (hidden, MLP)

// out[s][j][r] = sum over K block range s of W[r][c] * x'[j][c]: raw split sums, f32
struct TcArgs {
  int32_t rows, K;        // W [rows][K] bf16, row-major
  int32_t N;              // activation rows (batch)
  int32_t NP;             // activation rows per tile: a multiple of 16, at most 64
  int32_t Ntot;           // rows of each half (hi, lo) of the split activations (ntiles * NP)
  int32_t MT, KB, S;      // weight tiles, 64-element K blocks, K splits
  int32_t n_tile;         // weight rows per tile (the MMA's N): 256 or 128
  int32_t units;          // ntiles * MT * S
  int32_t stages;         // shared-memory pipeline depth
  float* out;             // [S][N][rows]
  int32_t* status;        // device error flag
};

// the activations of a projection, reduced and normalized, split into bf16 hi and lo:
//   x = resid + sum_s part[s]         (part given; resid optional)
//   x = silu(g) * u, (g, u) = sum_s part[s] rows (2i, 2i + 1)   (swiglu)
//   x = x_in                          (part null)
// then optionally x is written to xout, and x' = norm ? gain * (x * inv_rms) : x is split
struct TcPrepArgs {
  const float* x_in;
  int32_t x_stride;
  const float* part;      // [S][B][part_rows]
  int32_t S, part_rows;
  int32_t swiglu;
  const float* resid;
  int32_t resid_stride;
  float* xout;
  int32_t xout_stride;
  const float* gain;      // RMSNorm gains [K] or null
  float eps;
  int32_t K, B, Ntot;
  uint16_t* xs;           // [2][Ntot][K]
};

// Q/K/V from split sums: RoPE on q and k, q to q_out, k and v into the cache at pos
struct TcQkvArgs {
  const float* part;      // [S][B][rows], rows in RoPE pairs (q heads, k heads, v heads)
  int32_t S, rows, B;
  float* q_out;
  int32_t q_stride;
  void* kc;
  void* vc;
  int32_t H, kv, hd, cap;
  const float* rope_cos;
  const float* rope_sin;
  const StepState* step;
};

struct TcPlan {
  int NP, Ntot, ntiles, MT, KB, S, units, grid, stages, n_tile;
  size_t smem;
};

bool tc_available();
cudaError_t tc_prepare(int max_smem_optin);
// whole: one split (the output is final); the tile height is chosen for an even fill
TcPlan plan_tc(int rows, int K, int B, int num_sms, bool whole = false);
// rows of the split activations buffer for B rows, per half
int tc_ntot(int B);
// 2D bf16 tensor map over [outer][inner] (row pitch inner elements), box box_inner x box_outer,
// 128-byte swizzle
bool tc_make_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
                 uint32_t box_outer);
// general 2D tensor map (elements of elem_bytes: 2 = bf16, 4 = f32) with the given swizzle
bool make_map_2d(CUtensorMap* map, const void* base, int elem_bytes, uint64_t inner, uint64_t outer,
                 uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle);
cudaError_t launch_tc_prep(const TcPrepArgs& a, cudaStream_t s, bool pdl);
cudaError_t launch_tc_gemm(const CUtensorMap& tw, const CUtensorMap& tx, const TcArgs& a, const TcPlan& p,
                           cudaStream_t s, bool pdl);
cudaError_t launch_tc_qkv(const TcQkvArgs& a, cudaStream_t s, bool pdl);

}  // namespace llm
