// Weight-streaming matrix-vector products of the decode step.
//
// y[b][r] = sum_c W[r][c] * x'[b][c] for a batch of B activation rows, W bf16 (or f32)
// row-major [out][in] ("row = output", bend-ml-llama "A layer", LW), accumulated in f32.
// The input x' is either x itself or RMSNorm(x) (bend-ml-llama "The numeric pieces",
// rmsnorm: g * (x * (1 / sqrt(mean(x^2) + eps)))), computed in the prologue of every CTA.
// Epilogues fuse what follows each projection in the layer (bend-ml-llama "A layer", block):
//   EPI_QKV    rows come in RoPE pairs (element i and i + half of one head): rotate q and k
//              (rot_lo = lo*cos - hi*sin, rot_hi = hi*cos + lo*sin) at the row's position,
//              store the rotated q, and write the rotated k and the plain v into the KV cache
//              there (KV.push; through the row's page table in a paged step), rounding to the
//              cache element type;
//   EPI_RESID  x1 = x + W_o attn, y = x1 + W_down m;
//   EPI_SWIGLU rows come in (gate, up) pairs: m = silu(gate) * up, silu(v) = v / (1 + exp(-v));
//   EPI_STORE  logits = W_head nf.
//
// Design: the decode step is bound by HBM bandwidth (each weight byte is read once per step),
// so both kernels here are streaming engines.  gemv_kernel (any batch, bf16 or f32 weights):
// each CTA owns a contiguous, balanced range of rows (whole work units, so RoPE and SwiGLU pairs
// stay in one CTA) and reads them with 16-byte non-allocating loads in groups of 8 per thread,
// two groups in flight (double buffered); the threads of a row split its columns; the
// (normalized) input lives in shared memory as f32; partial dot products are reduced with warp
// shuffles and a fixed-order sum across warps, so results are deterministic.  gemv_tma_kernel
// (batch 1, bf16) streams the rows through per-warp rings of bulk copies instead (see below).
#include "gemv.cuh"
#include "tc.cuh"

namespace llm {

template <int BT> struct GemvTile {
  static constexpr int RB = BT >= 8 ? 1 : 8 / BT;  // rows per thread per batch
};

template <int WT, int BT, int EPI, bool NORM>
__global__ void __launch_bounds__(kGemvThreads, 2) gemv_kernel(const GemvArgs a) {
  constexpr int E = Elem<WT>::per16;
  constexpr int RB = GemvTile<BT>::RB;
  constexpr int MU = 8 / RB;  // chunks of a row per load group (8 loads per group)
  constexpr int NW = kGemvThreads / 32;
  extern __shared__ __align__(16) float sm[];
  const int seg_cols = a.seg_ch * E;
  float* xs = sm;                            // [BT][seg_cols]
  float* acc = xs + BT * seg_cols;           // [rows_cap][BT]
  float* wpart = acc + a.rows_cap * BT;      // [2][NW][RB][BT]
  float* inv = wpart + 2 * NW * RB * BT;     // [BT]
  float* red = inv + BT;                     // [NW][BT]
  float* wsum = red + NW * BT;               // [lpr/32][rows_cap][BT] per-warp row partials (a.ws)

  const int tid = threadIdx.x;
  const int units = a.rows / a.rg;
  const int u0 = (int)(((long long)units * blockIdx.x) / gridDim.x);
  const int u1 = (int)(((long long)units * (blockIdx.x + 1)) / gridDim.x);
  const int r0 = u0 * a.rg;
  const int nrows = (u1 - u0) * a.rg;
  const size_t row_bytes = (size_t)a.cols * Elem<WT>::bytes;
  const char* Wb = (const char*)a.W + (size_t)r0 * row_bytes;

  // the weights do not depend on the previous kernel: start pulling them into L2
  if (tid == 0 && nrows > 0) {
    size_t bytes = (size_t)nrows * row_bytes;
    if (bytes > 131072) bytes = 131072;
    prefetch_l2(Wb, (uint32_t)bytes);
  }
  grid_dep_wait();
  grid_dep_launch();

  const int lpr = a.lpr;
  const int RP = kGemvThreads / lpr;  // rows processed side by side
  const int rs = tid / lpr, li = tid - (tid / lpr) * lpr;
  const int nch = a.seg_ch / lpr;     // chunks per thread per row per segment
  const int warp = tid >> 5, lane = tid & 31;
  const int c4 = a.cols >> 2;          // float4 per input row
  const int seg4 = seg_cols >> 2;

  for (int b0 = 0; b0 < a.B; b0 += BT) {
    const int nb = min(BT, a.B - b0);
    if constexpr (NORM) {
      // sum of squares of every input row, all threads, 16-byte loads issued together
      float ss[BT];
#pragma unroll
      for (int b = 0; b < BT; ++b) ss[b] = 0.f;
#pragma unroll
      for (int b = 0; b < BT; ++b) {
        if (b < nb) {
          const float4* xr = reinterpret_cast<const float4*>(a.x + (size_t)(b0 + b) * a.x_stride);
#pragma unroll 4
          for (int i = tid; i < c4; i += kGemvThreads) {
            const float4 v = __ldg(xr + i);
            ss[b] = fmaf(v.x, v.x, ss[b]);
            ss[b] = fmaf(v.y, v.y, ss[b]);
            ss[b] = fmaf(v.z, v.z, ss[b]);
            ss[b] = fmaf(v.w, v.w, ss[b]);
          }
        }
      }
#pragma unroll
      for (int b = 0; b < BT; ++b) {
        const float v = warp_sum(ss[b]);
        if (lane == 0) red[warp * BT + b] = v;
      }
      __syncthreads();
      if (tid < nb) {
        float s = 0.f;
        for (int w = 0; w < NW; ++w) s += red[w * BT + tid];
        inv[tid] = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(s, (float)a.cols), a.eps)));
      }
    }
    for (int i = tid; i < nrows * BT; i += kGemvThreads) acc[i] = 0.f;
    if (a.ws)
      for (int i = tid; i < (lpr >> 5) * a.rows_cap * BT; i += kGemvThreads) wsum[i] = 0.f;
    int buf = 0;
    // the loads of one "group": RB rows x MU chunks per thread; groups are double buffered, so
    // the next group is in flight while this one is multiplied and its batch reduced
    const int ngrp = (nch + MU - 1) / MU;                 // groups per batch of RP*RB rows
    const int nbat = (nrows + RP * RB - 1) / (RP * RB);
    const int G = nbat * ngrp;                            // groups per segment
    float av[RB][BT];
#pragma unroll
    for (int k = 0; k < RB; ++k)
#pragma unroll
      for (int b = 0; b < BT; ++b) av[k][b] = 0.f;
    for (int seg = 0; seg < a.nseg; ++seg) {
      __syncthreads();
      const int c0 = seg * seg_cols;
      // stage this segment of the (normalized) inputs, 16 bytes at a time
#pragma unroll 4
      for (int i = tid; i < BT * seg4; i += kGemvThreads) {
        const int b = i / seg4, c = (i - b * seg4) * 4;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (b < nb) {
          v = __ldg(reinterpret_cast<const float4*>(a.x + (size_t)(b0 + b) * a.x_stride + c0 + c));
          if constexpr (NORM) {
            const float4 gv = __ldg(reinterpret_cast<const float4*>(a.gain + c0 + c));
            const float iv = inv[b];
            v.x = __fmul_rn(gv.x, __fmul_rn(iv, v.x));
            v.y = __fmul_rn(gv.y, __fmul_rn(iv, v.y));
            v.z = __fmul_rn(gv.z, __fmul_rn(iv, v.z));
            v.w = __fmul_rn(gv.w, __fmul_rn(iv, v.w));
          }
        }
        *reinterpret_cast<float4*>(xs + b * seg_cols + c) = v;
        if (a.tr_in && blockIdx.x == 0 && b < nb)
          *reinterpret_cast<float4*>(a.tr_in + (size_t)(b0 + b) * a.tr_stride + c0 + c) = v;
      }
      __syncthreads();
      const char* Wseg = Wb + (size_t)seg * a.seg_ch * 16;

      auto load_group = [&](uint4 (&w)[MU][RB], int g) {
        const int bi = g / ngrp, m0 = (g - bi * ngrp) * MU;
        const int rbase = bi * RP * RB;
#pragma unroll
        for (int mu = 0; mu < MU; ++mu) {
          const int ch = li + (m0 + mu) * lpr;
#pragma unroll
          for (int k = 0; k < RB; ++k) {
            const int rl = rbase + rs + k * RP;
            w[mu][k] = (rl < nrows && m0 + mu < nch)
                           ? ld_stream(Wseg + (size_t)rl * row_bytes + (size_t)ch * 16)
                           : make_uint4(0u, 0u, 0u, 0u);
          }
        }
      };
      auto fma_group = [&](const uint4 (&w)[MU][RB], int g) {
        const int bi = g / ngrp, m0 = (g - bi * ngrp) * MU;
#pragma unroll
        for (int mu = 0; mu < MU; ++mu) {
          if (m0 + mu >= nch) break;
          const int ch = li + (m0 + mu) * lpr;
          float xv[BT][E];
#pragma unroll
          for (int b = 0; b < BT; ++b) {
            const float4* xp = reinterpret_cast<const float4*>(xs + b * seg_cols + ch * E);
#pragma unroll
            for (int e4 = 0; e4 < E / 4; ++e4) {
              const float4 t = xp[e4];
              xv[b][4 * e4 + 0] = t.x;
              xv[b][4 * e4 + 1] = t.y;
              xv[b][4 * e4 + 2] = t.z;
              xv[b][4 * e4 + 3] = t.w;
            }
          }
#pragma unroll
          for (int k = 0; k < RB; ++k) {
            float wf[E];
            unpack16<WT>(w[mu][k], wf);
#pragma unroll
            for (int b = 0; b < BT; ++b)
#pragma unroll
              for (int e = 0; e < E; ++e) av[k][b] = fmaf(wf[e], xv[b][e], av[k][b]);
          }
        }
      };
      auto reduce_batch = [&](int bi) {
        const int rbase = bi * RP * RB;
        if (lpr >= 32 && a.ws) {
          // each warp keeps its own partial of each row; the warps are summed once at the end
          const int wi = warp % (lpr >> 5);
#pragma unroll
          for (int k = 0; k < RB; ++k) {
            const int rl = rbase + rs + k * RP;
#pragma unroll
            for (int b = 0; b < BT; ++b) {
              const float v = warp_sum(av[k][b]);
              if (lane == 0 && rl < nrows) wsum[((size_t)wi * a.rows_cap + rl) * BT + b] += v;
            }
          }
        } else if (lpr >= 32) {
#pragma unroll
          for (int k = 0; k < RB; ++k)
#pragma unroll
            for (int b = 0; b < BT; ++b) {
              const float v = warp_sum(av[k][b]);
              if (lane == 0) wpart[((buf * NW + warp) * RB + k) * BT + b] = v;
            }
          __syncthreads();
          const int wpr = lpr >> 5;
          for (int i = tid; i < RP * RB * BT; i += kGemvThreads) {
            const int b = i % BT, k = (i / BT) % RB, r = i / (BT * RB);
            const int rl = rbase + r + k * RP;
            if (rl < nrows && b < nb) {
              float sum = 0.f;
              for (int wi = 0; wi < wpr; ++wi) sum += wpart[((buf * NW + r * wpr + wi) * RB + k) * BT + b];
              acc[rl * BT + b] += sum;
            }
          }
          buf ^= 1;
        } else {
#pragma unroll
          for (int k = 0; k < RB; ++k)
#pragma unroll
            for (int b = 0; b < BT; ++b) {
              float v = av[k][b];
              for (int o = lpr >> 1; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
              av[k][b] = v;
            }
          if (li == 0) {
#pragma unroll
            for (int k = 0; k < RB; ++k) {
              const int rl = rbase + rs + k * RP;
              if (rl < nrows)
#pragma unroll
                for (int b = 0; b < BT; ++b)
                  if (b < nb) acc[rl * BT + b] += av[k][b];
            }
          }
        }
#pragma unroll
        for (int k = 0; k < RB; ++k)
#pragma unroll
          for (int b = 0; b < BT; ++b) av[k][b] = 0.f;
      };

      uint4 wa[MU][RB], wb[MU][RB];
      if (G > 0) load_group(wa, 0);
      for (int g = 0; g < G; g += 2) {
        if (g + 1 < G) load_group(wb, g + 1);
        fma_group(wa, g);
        if (g % ngrp == ngrp - 1) reduce_batch(g / ngrp);
        if (g + 1 >= G) break;
        if (g + 2 < G) load_group(wa, g + 2);
        fma_group(wb, g + 1);
        if ((g + 1) % ngrp == ngrp - 1) reduce_batch((g + 1) / ngrp);
      }
    }
    __syncthreads();
    if (a.ws) {
      const int wpr = lpr >> 5;
      for (int i = tid; i < nrows * BT; i += kGemvThreads) {
        float sum = 0.f;
        for (int wi = 0; wi < wpr; ++wi) sum += wsum[(size_t)wi * a.rows_cap * BT + i];
        acc[i] = sum;
      }
      __syncthreads();
    }

    // ---- epilogue ----
    if constexpr (EPI == EPI_QKV) {
      const int half = a.hd >> 1;
      const int npairs = nrows >> 1;
      for (int i = tid; i < npairs * nb; i += kGemvThreads) {
        const int b = i / npairs, p = i - b * npairs;
        const int pos = row_pos(a.step, b0 + b);
        const int R = r0 + 2 * p;
        const int head = R / a.hd, e = (R - head * a.hd) >> 1;
        const float x0 = acc[(2 * p) * BT + b], x1 = acc[(2 * p + 1) * BT + b];
        const size_t row = (size_t)(b0 + b);
        if (a.tr_pre) {
          a.tr_pre[row * a.tr_stride + (size_t)head * a.hd + e] = x0;
          a.tr_pre[row * a.tr_stride + (size_t)head * a.hd + e + half] = x1;
        }
        if (head < a.H + a.kv) {
          const float c = a.rope_cos[(size_t)pos * half + e], s = a.rope_sin[(size_t)pos * half + e];
          const float lo = __fadd_rn(__fmul_rn(x0, c), __fmul_rn(-x1, s));
          const float hi = __fadd_rn(__fmul_rn(x1, c), __fmul_rn(x0, s));
          if (head < a.H) {
            float* q = a.q_out + row * a.q_stride + (size_t)head * a.hd;
            q[e] = lo;
            q[e + half] = hi;
          } else {
            if (a.tr_rot) {
              a.tr_rot[row * a.tr_stride + (size_t)(head - a.H) * a.hd + e] = lo;
              a.tr_rot[row * a.tr_stride + (size_t)(head - a.H) * a.hd + e + half] = hi;
            }
            int r, pp;
            cache_slot(a.step, a.cap, (int)row, pos, r, pp);
            const size_t ci = (((size_t)r * a.kv + (size_t)(head - a.H)) * a.cap + pp) * a.hd;
            store_elem<WT>(a.kc, ci + e, lo);
            store_elem<WT>(a.kc, ci + e + half, hi);
          }
        } else {
          int r, pp;
          cache_slot(a.step, a.cap, (int)row, pos, r, pp);
          const size_t ci = (((size_t)r * a.kv + (size_t)(head - a.H - a.kv)) * a.cap + pp) * a.hd;
          store_elem<WT>(a.vc, ci + e, x0);
          store_elem<WT>(a.vc, ci + e + half, x1);
        }
      }
    } else if constexpr (EPI == EPI_SWIGLU) {
      const int npairs = nrows >> 1;
      for (int i = tid; i < npairs * nb; i += kGemvThreads) {
        const int b = i / npairs, p = i - b * npairs;
        const float gt = acc[(2 * p) * BT + b], up = acc[(2 * p + 1) * BT + b];
        const float si = __fdiv_rn(gt, __fadd_rn(1.0f, expf(-gt)));
        a.out[(size_t)(b0 + b) * a.out_stride + (r0 >> 1) + p] = __fmul_rn(si, up);
      }
    } else if constexpr (EPI == EPI_RESID) {
      for (int i = tid; i < nrows * nb; i += kGemvThreads) {
        const int b = i / nrows, r = i - b * nrows;
        const float rv = a.resid[(size_t)(b0 + b) * a.resid_stride + r0 + r];
        a.out[(size_t)(b0 + b) * a.out_stride + r0 + r] = __fadd_rn(rv, acc[r * BT + b]);
        if (a.tr_pre) a.tr_pre[(size_t)(b0 + b) * a.tr_stride + r0 + r] = acc[r * BT + b];
      }
    } else {
      for (int i = tid; i < nrows * nb; i += kGemvThreads) {
        const int b = i / nrows, r = i - b * nrows;
        a.out[(size_t)(b0 + b) * a.out_stride + r0 + r] = acc[r * BT + b];
      }
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------------------
// batch 1, bf16: each warp streams its rows through its own ring of bulk copies
// ---------------------------------------------------------------------------------------
// Rows are taken two at a time (a "group": a RoPE pair, a (gate, up) pair, or two neighbouring
// rows); a CTA owns a contiguous, balanced range of groups.  A step is the same 4 KB piece of
// both rows of a group; the CTA's steps (group-major) are dealt to its warps in turn, so warps
// differ by at most one step.  Lane 0 of a warp copies its steps into a private ring of slots
// (two cp.async.bulk copies on one mbarrier per slot), `ns` steps ahead, so the bytes in flight
// no longer depend on registers; the first steps are requested before the wait on the previous
// kernel (the weights do not depend on it).  Lane l multiplies 16-byte chunks l, l + 32, ... of
// both pieces with the (normalized) input, which sits in shared memory as f32 in two planes
// (elements 0-3 and 4-7 of every 8-element chunk) so that the loads of a warp are contiguous and
// each serves both rows.  A step's two sums (warp reductions) go to shared memory; at the end the
// threads add each row's pieces in order and run the epilogues of gemv_kernel.
constexpr int kTmaWarps = 8;
constexpr int kPiece = 4096;              // bytes of one row per step
constexpr int kStepBytes = 2 * kPiece;    // both rows of a group
constexpr int kTmaMaxSteps = 2;           // steps in flight per warp
constexpr int kTmaXr = 4;                 // float4s of the input a thread keeps in registers
constexpr uint64_t kTmaWaitCycles = 4000000000ull;  // SM cycles: about 2 s at 2 GHz
static int g_smem_optin = 0;              // set by gemv_prepare

static LLM_HD size_t gemv_tma_x_bytes(int cols) { return ((size_t)cols * 4 + 1023) & ~(size_t)1023; }
static LLM_HD int gemv_tma_ppr(int cols) { return (int)(((size_t)cols * 2 + kPiece - 1) / kPiece); }
// input planes, ring slots, their mbarriers, and two partial sums per step of at most maxg groups
static size_t gemv_tma_smem(int cols, int ns, int maxg) {
  return gemv_tma_x_bytes(cols) + (size_t)kTmaWarps * ns * (kStepBytes + 8) + (size_t)maxg * gemv_tma_ppr(cols) * 8;
}

template <int EPI, bool NORM>
__global__ void __launch_bounds__(kTmaWarps * 32, 1) gemv_tma_kernel(const GemvArgs a, const int ns) {
  extern __shared__ __align__(1024) uint8_t gsm[];
  constexpr int NW = kTmaWarps;
  const int cols = a.cols;
  float* xlo = reinterpret_cast<float*>(gsm);  // [cols / 2]: elements 0..3 of each chunk
  float* xhi = xlo + (cols >> 1);              // elements 4..7
  uint8_t* ring = gsm + gemv_tma_x_bytes(cols);
  const uint32_t ring_s = smem_u32(ring);
  const uint32_t bars = ring_s + (uint32_t)(NW * ns * kStepBytes);
  float* part = reinterpret_cast<float*>(ring + (size_t)NW * ns * (kStepBytes + 8));  // [steps][2]
  __shared__ float red[NW];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const int groups = (a.rows + 1) >> 1;
  const int g0 = (int)(((long long)groups * blockIdx.x) / gridDim.x);
  const int g1 = (int)(((long long)groups * (blockIdx.x + 1)) / gridDim.x);
  const size_t row_bytes = (size_t)cols * 2;
  const int ppr = gemv_tma_ppr(cols);  // pieces per row
  const int nsteps = (g1 - g0) * ppr;  // steps of the CTA; this warp's are warp, warp + NW, ...
  const int total = nsteps > warp ? (nsteps - warp + NW - 1) / NW : 0;
  const char* W = (const char*)a.W;

  if (tid == 0) {
    for (int i = 0; i < NW * ns; ++i) mbar_init(bars + 8u * i, 1);
    mbar_fence_init();
  }
  __syncthreads();
  // step t of this warp: CTA step q = warp + t * NW, piece q % ppr of the rows of group g0 + q / ppr
  auto issue = [&](int t) {
    const int q = warp + t * NW;
    const int ig = q / ppr, pc = q - ig * ppr;
    const size_t r0 = 2 * (size_t)(g0 + ig);
    const size_t r1 = r0 + 1 < (size_t)a.rows ? r0 + 1 : r0;  // an odd last row is read twice
    const size_t off = (size_t)pc * kPiece;
    const uint32_t bytes = (uint32_t)(row_bytes - off < (size_t)kPiece ? row_bytes - off : (size_t)kPiece);
    const int slot = t % ns;
    const uint32_t bar = bars + 8u * (warp * ns + slot);
    const uint32_t dst = ring_s + (uint32_t)((warp * ns + slot) * kStepBytes);
    mbar_expect_tx(bar, 2 * bytes);
    bulk_load(dst, W + r0 * row_bytes + off, bytes, bar);
    bulk_load(dst + kPiece, W + r1 * row_bytes + off, bytes, bar);
  };
  if (lane == 0)
    for (int t = 0; t < ns && t < total; ++t) issue(t);

  // the (normalized) input, f32, in its two planes.  Up to kTmaXr float4s per thread stay in
  // registers, so the input is read once (one round trip after the wait); the gains are constant
  // and are read before the wait.  Thread i owns float4s i, i + NT, ... in both paths, so the sum
  // of squares has the same order either way.
  constexpr int NT = NW * 32;
  const int c4 = cols >> 2;
  const float4* xr = reinterpret_cast<const float4*>(a.x);
  const float4* gr4 = reinterpret_cast<const float4*>(a.gain);
  const bool in_regs = c4 <= kTmaXr * NT;
  float4 gv[kTmaXr];
  if constexpr (NORM) {
    if (in_regs) {
#pragma unroll
      for (int k = 0; k < kTmaXr; ++k)
        if (tid + k * NT < c4) gv[k] = __ldg(gr4 + tid + k * NT);
    }
  }
  // the epilogue's other inputs of group g: the residual rows (EPI_RESID), or the step's
  // position, its RoPE factors and the cache slot (EPI_QKV).  For this thread's first group they
  // are read before the wait: the RoPE tables are constant, the step state was written by the
  // step prologue, and the residual two kernels back (o_proj: the previous layer's down; down:
  // o_proj), all complete before this kernel can start; the residual is read through L2.
  struct EpiIn {
    float r0, r1, c, s;
    int pos, r, pp;
  };
  auto epi_in = [&](int g, bool early) {
    EpiIn in = {0.f, 0.f, 0.f, 0.f, 0, 0, 0};
    if constexpr (EPI == EPI_RESID) {
      in.r0 = early ? __ldcg(a.resid + 2 * g) : a.resid[2 * g];
      if (2 * g + 1 < a.rows) in.r1 = early ? __ldcg(a.resid + 2 * g + 1) : a.resid[2 * g + 1];
    } else if constexpr (EPI == EPI_QKV) {
      const int R = 2 * g, half = a.hd >> 1;
      const int head = R / a.hd, e = (R - head * a.hd) >> 1;
      in.pos = row_pos(a.step, 0);
      if (head < a.H + a.kv) {
        in.c = __ldg(a.rope_cos + (size_t)in.pos * half + e);
        in.s = __ldg(a.rope_sin + (size_t)in.pos * half + e);
      }
      if (head >= a.H) cache_slot(a.step, a.cap, 0, in.pos, in.r, in.pp);
    }
    return in;
  };
  EpiIn pre = {0.f, 0.f, 0.f, 0.f, 0, 0, 0};
  if (tid < g1 - g0) pre = epi_in(g0 + tid, true);
  grid_dep_wait();
  grid_dep_launch();

  auto put = [&](int i, float4 v) { reinterpret_cast<float4*>((i & 1) ? xhi : xlo)[i >> 1] = v; };
  auto scale = [](float4 v, float4 g, float inv) {
    v.x = __fmul_rn(g.x, __fmul_rn(inv, v.x));
    v.y = __fmul_rn(g.y, __fmul_rn(inv, v.y));
    v.z = __fmul_rn(g.z, __fmul_rn(inv, v.z));
    v.w = __fmul_rn(g.w, __fmul_rn(inv, v.w));
    return v;
  };
  // 1 / rms from the warps' sums of squares (every thread adds them in the same order)
  auto inv_rms = [&](float ss) {
    ss = warp_sum(ss);
    if (lane == 0) red[warp] = ss;
    __syncthreads();
    float t = 0.f;
    for (int w = 0; w < NW; ++w) t += red[w];
    return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(t, (float)cols), a.eps)));
  };
  if (in_regs) {
    float4 xv[kTmaXr];
#pragma unroll
    for (int k = 0; k < kTmaXr; ++k)
      if (tid + k * NT < c4) xv[k] = __ldg(xr + tid + k * NT);
    if constexpr (NORM) {
      float ss = 0.f;
#pragma unroll
      for (int k = 0; k < kTmaXr; ++k)
        if (tid + k * NT < c4) {
          ss = fmaf(xv[k].x, xv[k].x, ss);
          ss = fmaf(xv[k].y, xv[k].y, ss);
          ss = fmaf(xv[k].z, xv[k].z, ss);
          ss = fmaf(xv[k].w, xv[k].w, ss);
        }
      const float inv = inv_rms(ss);
#pragma unroll
      for (int k = 0; k < kTmaXr; ++k)
        if (tid + k * NT < c4) xv[k] = scale(xv[k], gv[k], inv);
    }
#pragma unroll
    for (int k = 0; k < kTmaXr; ++k)
      if (tid + k * NT < c4) put(tid + k * NT, xv[k]);
  } else {
    float inv = 1.f;
    if constexpr (NORM) {
      float ss = 0.f;
      for (int i = tid; i < c4; i += NT) {
        const float4 v = __ldg(xr + i);
        ss = fmaf(v.x, v.x, ss);
        ss = fmaf(v.y, v.y, ss);
        ss = fmaf(v.z, v.z, ss);
        ss = fmaf(v.w, v.w, ss);
      }
      inv = inv_rms(ss);
    }
#pragma unroll 4
    for (int i = tid; i < c4; i += NT) {
      float4 v = __ldg(xr + i);
      if constexpr (NORM) v = scale(v, __ldg(gr4 + i), inv);
      put(i, v);
    }
  }
  __syncthreads();

  bool ok = true;
  int consumed = 0;
  float a0[2] = {0.f, 0.f}, a1[2] = {0.f, 0.f};  // the group's two rows
  auto chunk = [&](const uint8_t* w0, const float* xl, const float* xh, int j, int par) {
    float f0[8], f1[8];
    unpack16<1>(*reinterpret_cast<const uint4*>(w0 + j * 16), f0);
    unpack16<1>(*reinterpret_cast<const uint4*>(w0 + kPiece + j * 16), f1);
    const float4 lo = *reinterpret_cast<const float4*>(xl + j * 4);
    const float4 hi = *reinterpret_cast<const float4*>(xh + j * 4);
    const float xv[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      a0[par] = fmaf(f0[e], xv[e], a0[par]);
      a1[par] = fmaf(f1[e], xv[e], a1[par]);
    }
  };
  for (int t = 0; t < total; ++t) {
    const int slot = t % ns;
    ok = __all_sync(0xffffffffu, mbar_wait(bars + 8u * (warp * ns + slot), (uint32_t)(t / ns) & 1u, kTmaWaitCycles));
    if (!ok) break;
    consumed = t + 1;
    const int q = warp + t * NW;
    const int pc = q - (q / ppr) * ppr;
    const size_t off = (size_t)pc * kPiece;
    const int nch = (int)((row_bytes - off < (size_t)kPiece ? row_bytes - off : (size_t)kPiece) >> 4);
    const uint8_t* w0 = ring + (size_t)(warp * ns + slot) * kStepBytes;
    const float* xl = xlo + (size_t)pc * (kPiece / 4);
    const float* xh = xhi + (size_t)pc * (kPiece / 4);
    if (nch == kPiece / 16) {
#pragma unroll
      for (int i = 0; i < kPiece / 16 / 32; ++i) chunk(w0, xl, xh, lane + 32 * i, i & 1);
    } else {
      for (int j = lane; j < nch; j += 32) chunk(w0, xl, xh, j, 0);
    }
    __syncwarp();
    if (lane == 0 && t + ns < total) {
      fence_proxy_async_smem();  // this slot's reads come before the copy that refills it
      issue(t + ns);
    }
    {
      const float v0 = warp_sum(a0[0] + a0[1]);
      const float v1 = warp_sum(a1[0] + a1[1]);
      a0[0] = a0[1] = a1[0] = a1[1] = 0.f;
      if (lane == 0) {
        part[2 * q] = v0;
        part[2 * q + 1] = v1;
      }
    }
  }
  if (!ok && lane == 0) {
    atomicCAS(a.status, 0, kErrDeviceTimeout);
    // no copy may still be writing shared memory when the CTA exits
    for (int t = consumed; t < total && t < consumed + ns; ++t)
      mbar_wait(bars + 8u * (warp * ns + t % ns), (uint32_t)(t / ns) & 1u, kTmaWaitCycles);
  }
  __syncthreads();
  // ---- epilogue: each group's two rows, pieces added in order ----
  for (int i = tid; i < g1 - g0; i += NW * 32) {
    float v0 = 0.f, v1 = 0.f;
    for (int pc = 0; pc < ppr; ++pc) {
      v0 += part[2 * (i * ppr + pc)];
      v1 += part[2 * (i * ppr + pc) + 1];
    }
    const int g = g0 + i;
    if constexpr (EPI == EPI_STORE) {
      const int r0 = 2 * g;
      a.out[r0] = v0;
      if (r0 + 1 < a.rows) a.out[r0 + 1] = v1;
    } else if constexpr (EPI == EPI_RESID) {
      const EpiIn in = i == tid ? pre : epi_in(g, false);
      const int r0 = 2 * g;
      a.out[r0] = __fadd_rn(in.r0, v0);
      if (r0 + 1 < a.rows) a.out[r0 + 1] = __fadd_rn(in.r1, v1);
    } else if constexpr (EPI == EPI_SWIGLU) {
      const float si = __fdiv_rn(v0, __fadd_rn(1.0f, expf(-v0)));
      a.out[g] = __fmul_rn(si, v1);
    } else {
      const EpiIn in = i == tid ? pre : epi_in(g, false);
      const int R = 2 * g, half = a.hd >> 1;
      const int head = R / a.hd, e = (R - head * a.hd) >> 1;
      if (head < a.H + a.kv) {
        const float lo = __fadd_rn(__fmul_rn(v0, in.c), __fmul_rn(-v1, in.s));
        const float hi = __fadd_rn(__fmul_rn(v1, in.c), __fmul_rn(v0, in.s));
        if (head < a.H) {
          float* qo = a.q_out + (size_t)head * a.hd;
          qo[e] = lo;
          qo[e + half] = hi;
        } else {
          const size_t ci = (((size_t)in.r * a.kv + (size_t)(head - a.H)) * a.cap + in.pp) * a.hd;
          store_elem<1>(a.kc, ci + e, lo);
          store_elem<1>(a.kc, ci + e + half, hi);
        }
      } else {
        const size_t ci = (((size_t)in.r * a.kv + (size_t)(head - a.H - a.kv)) * a.cap + in.pp) * a.hd;
        store_elem<1>(a.vc, ci + e, v0);
        store_elem<1>(a.vc, ci + e + half, v1);
      }
    }
  }
}

// ---------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------

GemvPlan plan_gemv(int rows, int cols, int rg, int wt, int B, int num_sms, int ctas_per_sm) {
  GemvPlan p{};
  const int E = wt ? 8 : 4;
  const int CH = cols / E;
  p.bt = B <= 1 ? 1 : B <= 2 ? 2 : B <= 4 ? 4 : 8;
  int lpr = 1;
  while (lpr < kGemvThreads && CH % (lpr * 2) == 0) lpr *= 2;
  const size_t budget = 64 * 1024;
  for (;;) {
    const int q = CH / lpr;
    int best = -1;
    for (int k = 1; k <= q; ++k)
      if (q % k == 0 && (size_t)(CH / k) * E * p.bt * 4 <= budget) {
        best = k;
        break;
      }
    if (best > 0) {
      p.seg_ch = CH / best;
      p.nseg = best;
      break;
    }
    lpr /= 2;
  }
  p.lpr = lpr;
  const int units = rows / rg;
  const int RP = kGemvThreads / lpr;
  int grid = num_sms * ctas_per_sm;
  const int by_rows = (rows + RP - 1) / RP;  // at least one row per row slot
  if (grid > by_rows) grid = by_rows;
  if (grid > units) grid = units;
  if (grid < 1) grid = 1;
  p.grid = grid;
  p.rows_cap = ((units + grid - 1) / grid) * rg;
  const int RB = p.bt >= 8 ? 1 : 8 / p.bt;
  // per-warp row partials (no CTA barrier per batch) when they fit
  const size_t ws_floats = lpr >= 32 ? (size_t)(lpr / 32) * p.rows_cap * p.bt : 0;
  p.ws = (lpr >= 32 && ws_floats * 4 <= 48 * 1024) ? 1 : 0;
  p.smem = ((size_t)p.bt * p.seg_ch * E + (size_t)p.rows_cap * p.bt + 2 * 8 * RB * p.bt + 8 + 8 * 8 +
            (p.ws ? ws_floats : 0)) * 4;
  // batch 1, bf16, rows of whole 16-byte chunks: kTmaMaxSteps steps in flight per warp (fewer
  // if shared memory does not hold them; two measured faster than three at the 8B shape, the
  // smaller footprint leaving room for the next kernel's CTAs); one CTA per SM
  p.tma_ns = 0;
  if (B == 1 && wt == 1 && cols % 8 == 0 && g_smem_optin > 0) {
    const int groups = (rows + 1) / 2;
    const int grid = groups < num_sms ? groups : num_sms;
    const int maxg = (groups + grid - 1) / grid;
    int ns = kTmaMaxSteps;
    while (ns >= 2 && gemv_tma_smem(cols, ns, maxg) + 1024 > (size_t)g_smem_optin) --ns;
    if (ns >= 2) {
      p.tma_ns = ns;
      p.tma_grid = grid;
      p.tma_smem = gemv_tma_smem(cols, ns, maxg);
    }
  }
  return p;
}

using GemvFn = void (*)(const GemvArgs);

template <int WT, int BT>
static GemvFn pick_epi(int epi, bool norm) {
  switch (epi) {
    case EPI_QKV: return gemv_kernel<WT, BT, EPI_QKV, true>;
    case EPI_SWIGLU: return gemv_kernel<WT, BT, EPI_SWIGLU, true>;
    case EPI_RESID: return gemv_kernel<WT, BT, EPI_RESID, false>;
    default: return norm ? gemv_kernel<WT, BT, EPI_STORE, true> : gemv_kernel<WT, BT, EPI_STORE, false>;
  }
}

template <int WT>
static GemvFn pick_bt(int bt, int epi, bool norm) {
  switch (bt) {
    case 1: return pick_epi<WT, 1>(epi, norm);
    case 2: return pick_epi<WT, 2>(epi, norm);
    case 4: return pick_epi<WT, 4>(epi, norm);
    default: return pick_epi<WT, 8>(epi, norm);
  }
}

static GemvFn pick(int wt, int bt, int epi, bool norm) {
  return wt ? pick_bt<1>(bt, epi, norm) : pick_bt<0>(bt, epi, norm);
}

using GemvTmaFn = void (*)(const GemvArgs, const int);

static GemvTmaFn pick_tma(int epi, bool norm) {
  switch (epi) {
    case EPI_QKV: return gemv_tma_kernel<EPI_QKV, true>;
    case EPI_SWIGLU: return gemv_tma_kernel<EPI_SWIGLU, true>;
    case EPI_RESID: return gemv_tma_kernel<EPI_RESID, false>;
    default: return norm ? gemv_tma_kernel<EPI_STORE, true> : gemv_tma_kernel<EPI_STORE, false>;
  }
}

cudaError_t gemv_prepare(int max_smem_optin) {
  for (int wt = 0; wt < 2; ++wt)
    for (int bt : {1, 2, 4, 8})
      for (int epi = 0; epi < 4; ++epi)
        for (int norm = 0; norm < 2; ++norm) {
          GemvFn fn = pick(wt, bt, epi, norm != 0);
          cudaFuncAttributes fa;
          cudaError_t e = cudaFuncGetAttributes(&fa, fn);
          if (e != cudaSuccess) return e;
          e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   max_smem_optin - (int)fa.sharedSizeBytes);
          if (e != cudaSuccess) return e;
        }
  for (int epi = 0; epi < 4; ++epi)
    for (int norm = 0; norm < 2; ++norm) {
      GemvTmaFn fn = pick_tma(epi, norm != 0);
      cudaFuncAttributes fa;
      cudaError_t e = cudaFuncGetAttributes(&fa, fn);
      if (e != cudaSuccess) return e;
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               max_smem_optin - (int)fa.sharedSizeBytes);
      if (e != cudaSuccess) return e;
    }
  g_smem_optin = max_smem_optin;
  return cudaSuccess;
}

cudaError_t launch_gemv(const GemvArgs& a, const GemvPlan& p, int wt, int epi, bool norm,
                        cudaStream_t s, bool pdl) {
  if (p.tma_ns > 0 && a.B == 1 && !a.tr_in && !a.tr_pre) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.tma_grid);
    cfg.blockDim = dim3(kTmaWarps * 32);
    cfg.dynamicSmemBytes = p.tma_smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, pick_tma(epi, norm), a, p.tma_ns);
  }
  GemvFn fn = pick(wt, p.bt, epi, norm);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(kGemvThreads);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fn, a);
}

}  // namespace llm
