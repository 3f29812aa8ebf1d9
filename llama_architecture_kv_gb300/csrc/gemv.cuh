// Weight-streaming matrix-vector products of the decode step (declarations).
#pragma once
#include "common.cuh"

namespace llm {

enum GemvEpi : int {
  EPI_QKV = 0,     // rows are RoPE pairs of q/k/v heads: rotate, store q, write k and v to the cache
  EPI_RESID = 1,   // out = resid + W x
  EPI_SWIGLU = 2,  // rows are (gate, up) pairs: out = silu(gate) * up
  EPI_STORE = 3,   // out = W x
};

struct GemvArgs {
  const void* W;        // [rows][cols], row-major, element type WT
  int32_t rows, cols;
  int32_t rg;           // rows per work unit (2 for pair epilogues, else 1)
  const float* x;       // input activations [B][x_stride]
  int32_t x_stride;
  const float* gain;    // RMSNorm gains [cols] (prologue norm only)
  float eps;
  int32_t B;            // batch rows
  int32_t lpr;          // threads that share one row (power of two dividing seg_ch)
  int32_t seg_ch;       // 16-byte chunks per staged column segment
  int32_t nseg;         // segments per row (seg_ch * nseg = chunks per row)
  int32_t rows_cap;     // upper bound of rows per CTA (sizes the accumulator)
  int32_t ws;           // 1: per-warp row partials in shared memory, summed once at the end
  const StepState* step;
  float* out;           // [B][out_stride]
  int32_t out_stride;
  const float* resid;   // [B][resid_stride]
  int32_t resid_stride;
  // EPI_QKV
  float* q_out;         // rotated queries [B][q_stride]
  int32_t q_stride;
  void* kc;             // this layer's key cache [max_batch][kv][cap][hd]
  void* vc;             // this layer's value cache
  int32_t H, kv, hd, cap;
  const float* rope_cos;  // [cap][hd/2]
  const float* rope_sin;
  int32_t* status;      // device error flag (a bounded wait that ran out)
  // intermediates for a traced step (null otherwise; set, the launch runs gemv_kernel):
  float* tr_in;         // the (normalized) input [B][cols], written by CTA 0
  float* tr_pre;        // EPI_QKV: q|k|v before RoPE [B][rows] in head order; EPI_RESID: W x [B][rows]
  float* tr_rot;        // EPI_QKV: the rotated keys in f32 [B][kv * hd]
  int32_t tr_stride;    // floats between two rows of a trace
};

struct GemvPlan {
  int bt, lpr, seg_ch, nseg, grid, rows_cap, ws;
  size_t smem;
  // batch 1 with bf16 weights: the bulk-copy kernel (tma_ns > 0 steps in flight per warp)
  int tma_ns, tma_grid;
  size_t tma_smem;
};

constexpr int kGemvThreads = 256;

GemvPlan plan_gemv(int rows, int cols, int rg, int wt, int B, int num_sms, int ctas_per_sm);
cudaError_t launch_gemv(const GemvArgs& a, const GemvPlan& p, int wt, int epi, bool norm,
                        cudaStream_t s, bool pdl);
cudaError_t gemv_prepare(int max_smem_optin);

}  // namespace llm
