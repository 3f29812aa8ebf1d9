// Tensor-core projections of batched decode: out[j][r] = sum_c W[r][c] * x'[j][c] for B >= 16
// activation rows, on the 5th-generation tensor core (tcgen05.mma, accumulators in tensor memory,
// operands staged by TMA), with the same fused epilogues as the weight-streaming GEMV
// (bend-ml-llama "A layer", block: RoPE + KV write after Q/K/V, residual adds, SwiGLU; the LM
// head after the final norm).
//
// Precision.  The weights are bf16; the activations are f32.  Each activation is split into
// two bf16 numbers, hi = bf16(x') and lo = bf16(x' - hi), and the product runs as W*hi + W*lo
// into one f32 accumulator: x' is represented to about 2^-17 relative, close to the f32 inputs
// of the plain matrix-vector product, at twice the tensor work (still far below the weight
// stream's time).  x' is x or RMSNorm(x) (bend-ml-llama "The numeric pieces", rmsnorm),
// computed by tc_split_kernel before the product.
//
// Work split.  The weight tiles (128 rows x 64 K) of all row tiles, K innermost, form one
// sequence; each CTA (one per SM) takes an equal contiguous run of it (stream-K).  A CTA whose
// run covers a whole row tile applies the epilogue from tensor memory; row tiles shared by
// several CTAs are finished by the last CTA to arrive (atomic ticket, nobody waits), which adds
// the partials in CTA order, so results do not depend on timing.
//
// Roles: warp 0 issues TMA copies into a ring of shared-memory stages (mbarrier full/empty),
// warp 1 issues the MMAs (one thread) into two tensor-memory accumulators so the epilogue of one
// run overlaps the next, warps 2..5 read the accumulator (tcgen05.ld, one row per thread) and
// run the epilogue.  Every wait is bounded: on timeout the kernel records kErrDeviceTimeout,
// lets its copies and MMAs drain (bounded again), frees its tensor memory and returns.
#include <cudaTypedefs.h>

#include <mutex>

#include "gemm.cuh"
#include "tc.cuh"

namespace llm {

constexpr uint64_t kTcWaitNs = 4000000000ull;  // SM cycles: about 2 s at 2 GHz

LLM_HD int tc_owner(int64_t it, int64_t T, int G) { return (int)(((it + 1) * G + T - 1) / T - 1); }
LLM_HD int64_t tc_first(int64_t T, int G, int c) { return T * c / G; }

// epilogue of column j (batch row), weight row R, accumulated value v; lanes hold consecutive
// rows, so RoPE and SwiGLU partners (rows 2i, 2i+1) are neighbouring lanes
template <int EPI>
LLM_D void tc_epi(const TcArgs& a, int R, int j, float v) {
  const bool ok = R < a.rows;
  if constexpr (EPI == EPI_STORE) {
    if (ok) a.out[(size_t)j * a.out_stride + R] = v;
  } else if constexpr (EPI == EPI_RESID) {
    if (ok) a.out[(size_t)j * a.out_stride + R] = __fadd_rn(a.resid[(size_t)j * a.resid_stride + R], v);
  } else if constexpr (EPI == EPI_SWIGLU) {
    const float up = __shfl_xor_sync(0xffffffffu, v, 1);
    if (ok && !(R & 1)) {
      const float si = __fdiv_rn(v, __fadd_rn(1.0f, expf(-v)));
      a.out[(size_t)j * a.out_stride + (R >> 1)] = __fmul_rn(si, up);
    }
  } else {
    const float other = __shfl_xor_sync(0xffffffffu, v, 1);
    if (ok) {
      const bool odd = (R & 1) != 0;
      const float x0 = odd ? other : v, x1 = odd ? v : other;
      const int head = R / a.hd, e = (R - head * a.hd) >> 1, half = a.hd >> 1;
      const int pos = a.step->pos;
      const int ee = odd ? e + half : e;
      const size_t row = (size_t)j;
      if (head < a.H + a.kv) {
        const float c = a.rope_cos[(size_t)pos * half + e], s = a.rope_sin[(size_t)pos * half + e];
        const float r = odd ? __fadd_rn(__fmul_rn(x1, c), __fmul_rn(x0, s))
                            : __fadd_rn(__fmul_rn(x0, c), __fmul_rn(-x1, s));
        if (head < a.H) {
          a.q_out[row * a.q_stride + (size_t)head * a.hd + ee] = r;
        } else {
          const size_t ci = ((row * a.kv + (size_t)(head - a.H)) * a.cap + pos) * a.hd;
          store_elem<1>(a.kc, ci + ee, r);
        }
      } else {
        const size_t ci = ((row * a.kv + (size_t)(head - a.H - a.kv)) * a.cap + pos) * a.hd;
        store_elem<1>(a.vc, ci + ee, v);
      }
    }
  }
}

template <int EPI>
__global__ void __launch_bounds__(kTcThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tw, const __grid_constant__ CUtensorMap tx, const TcArgs a) {
  extern __shared__ uint8_t tc_smem[];
  const uint32_t s_raw = smem_u32(tc_smem);
  const uint32_t s_base = (s_raw + 1023u) & ~1023u;  // the 128-byte swizzle repeats every 1024 bytes
  uint8_t* g_base = tc_smem + (s_base - s_raw);
  const int NP = a.NP, S = a.stages, KB = a.KB;
  const uint32_t bB = (uint32_t)NP * 128u;
  const uint32_t stage = 16384u + 2u * bB;
  const uint32_t bars = s_base + (uint32_t)S * stage;
  // barriers: full[S], empty[S], acc_full[2], acc_empty[2], drain
  const uint32_t FULL0 = bars, EMPTY0 = bars + 8u * S, ACCF0 = bars + 16u * S, ACCE0 = ACCF0 + 16u,
                 DRAIN = ACCE0 + 16u;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(g_base + (size_t)S * stage + 16u * S + 40u);
  volatile int* flags = reinterpret_cast<volatile int*>(tmem_slot + 2);  // [0] abort, [1] last arrival

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x, G = gridDim.x, nt = blockIdx.y;
  const int64_t T = (int64_t)a.MT * KB;
  const int64_t it0 = tc_first(T, G, c), it1 = tc_first(T, G, c + 1);
  const int64_t n_it = it1 - it0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(FULL0 + 8u * i, 1);
      mbar_init(EMPTY0 + 8u * i, 1);
    }
    mbar_init(ACCF0, 1);
    mbar_init(ACCF0 + 8u, 1);
    mbar_init(ACCE0, 128);
    mbar_init(ACCE0 + 8u, 128);
    mbar_init(DRAIN, 1);
    flags[0] = 0;
    flags[1] = 0;
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32((const void*)tmem_slot), a.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  auto fail = [&]() {
    flags[0] = 1;
    atomicCAS(a.status, 0, kErrDeviceTimeout);
  };

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_map(&tw);
      tma_prefetch_map(&tx);
      const int n = (int)n_it;
      const int npre = n < S ? n : S;
      const int m0 = (int)(it0 / KB), kb00 = (int)(it0 - (int64_t)m0 * KB);
      // the weight tiles of the first stages do not depend on the previous kernel
      int m = m0, kb = kb00;
      for (int i = 0; i < npre; ++i) {
        mbar_expect_tx(FULL0 + 8u * i, stage);
        tma_load_2d(s_base + (uint32_t)i * stage, &tw, FULL0 + 8u * i, kb * kTcK, m * kTcM);
        if (++kb == KB) kb = 0, ++m;
      }
      grid_dep_wait();
      grid_dep_launch();
      kb = kb00;
      for (int i = 0; i < npre; ++i) {
        const uint32_t sb = s_base + (uint32_t)i * stage + 16384u;
        tma_load_2d(sb, &tx, FULL0 + 8u * i, kb * kTcK, nt * NP);
        tma_load_2d(sb + bB, &tx, FULL0 + 8u * i, kb * kTcK, a.Ntot + nt * NP);
        if (++kb == KB) kb = 0;
      }
      // m, kb: the tile of iteration npre; (s, ph): its stage and round parity
      int s = npre == S ? 0 : npre;
      uint32_t ph = npre == S ? 1u : 0u;
      int issued = npre;
      for (int i = npre; i < n; ++i) {
        if (flags[0] || !mbar_wait(EMPTY0 + 8u * s, ph ^ 1u, kTcWaitNs)) {
          fail();
          break;
        }
        const uint32_t sa = s_base + (uint32_t)s * stage;
        mbar_expect_tx(FULL0 + 8u * s, stage);
        tma_load_2d(sa, &tw, FULL0 + 8u * s, kb * kTcK, m * kTcM);
        tma_load_2d(sa + 16384u, &tx, FULL0 + 8u * s, kb * kTcK, nt * NP);
        tma_load_2d(sa + 16384u + bB, &tx, FULL0 + 8u * s, kb * kTcK, a.Ntot + nt * NP);
        issued = i + 1;
        if (++kb == KB) kb = 0, ++m;
        if (++s == S) s = 0, ph ^= 1u;
      }
      // no copy may still be writing shared memory when the CTA exits
      for (int i = issued > S ? issued - S : 0; i < issued; ++i)
        if (!mbar_wait(FULL0 + 8u * (uint32_t)(i % S), (uint32_t)(i / S) & 1u, kTcWaitNs)) fail();
    } else {
      grid_dep_wait();
      grid_dep_launch();
    }
  } else if (warp == 1) {
    grid_dep_wait();
    grid_dep_launch();
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kTcM, NP);
      int s = 0;
      uint32_t ph = 0;
      int si = 0;
      bool ok = true;
      const int n = (int)n_it;
      int kb0 = (int)(it0 % KB);
      for (int done = 0; done < n && ok; ++si) {
        const int kb1 = KB < kb0 + (n - done) ? KB : kb0 + (n - done);
        const int buf = si & 1, use = si >> 1;
        if (use > 0 && !mbar_wait(ACCE0 + 8u * buf, (uint32_t)(use - 1) & 1u, kTcWaitNs)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(buf * NP);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (flags[0] || !mbar_wait(FULL0 + 8u * s, ph, kTcWaitNs)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = s_base + (uint32_t)s * stage, sb = sa + 16384u;
          const uint64_t ad = sw128_kmajor_desc(sa), bh = sw128_kmajor_desc(sb), bl = sw128_kmajor_desc(sb + bB);
#pragma unroll
          for (int k = 0; k < kTcK / 16; ++k) {
            // 16 K elements = 32 bytes = 2 in the descriptor's address field
            tc_mma_bf16(d, ad + 2 * k, bh + 2 * k, idesc, (kb > kb0 || k > 0) ? 1u : 0u);
            tc_mma_bf16(d, ad + 2 * k, bl + 2 * k, idesc, 1u);
          }
          tc_commit(EMPTY0 + 8u * s);
          if (++s == S) s = 0, ph ^= 1u;
        }
        if (!ok) break;
        tc_commit(ACCF0 + 8u * buf);
        done += kb1 - kb0;
        kb0 = 0;
      }
      if (!ok) fail();
      // every MMA has completed before tensor memory is freed
      tc_commit(DRAIN);
      if (!mbar_wait(DRAIN, 0, kTcWaitNs)) fail();
    }
  } else {
    grid_dep_wait();
    grid_dep_launch();
    const int q = warp & 3;  // this warp's quarter of the tensor-memory lanes
    const int rl = q * 32 + lane;
    int si = 0;
    for (int64_t it = it0; it < it1; ++si) {
      const int m = (int)(it / KB), kb0 = (int)(it - (int64_t)m * KB);
      const int kb1 = (int)((int64_t)KB < kb0 + (it1 - it) ? KB : kb0 + (it1 - it));
      const int buf = si & 1, use = si >> 1;
      bool ok = !flags[0] && mbar_wait(ACCF0 + 8u * buf, (uint32_t)use & 1u, kTcWaitNs);
      ok = named_sync_and(1, 128, ok);
      if (!ok) {
        if (threadIdx.x == 64) fail();
        break;
      }
      tc_fence_after();
      const bool whole = kb0 == 0 && kb1 == KB;
      const int R = m * kTcM + rl;
      const int j0 = nt * NP;
      const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * NP);
      float* mine = a.part + ((size_t)(nt * G + c) * 2 + (si == 0 ? 0 : 1)) * (size_t)NP * kTcM + (size_t)rl * NP;
      for (int jc = 0; jc < NP; jc += 16) {
        float v[16];
        tc_ld16(taddr + (uint32_t)jc, v);
        tc_wait_ld();
        if (whole) {
#pragma unroll
          for (int jj = 0; jj < 16; ++jj)
            if (j0 + jc + jj < a.N) tc_epi<EPI>(a, R, j0 + jc + jj, v[jj]);
        } else {
#pragma unroll
          for (int jj = 0; jj < 16; jj += 4)
            *reinterpret_cast<float4*>(mine + jc + jj) = make_float4(v[jj], v[jj + 1], v[jj + 2], v[jj + 3]);
        }
      }
      tc_fence_before();
      mbar_arrive(ACCE0 + 8u * buf);
      if (!whole) {
        __threadfence();
        named_sync(1, 128);
        const int cf = tc_owner((int64_t)m * KB, T, G), cl = tc_owner((int64_t)m * KB + KB - 1, T, G);
        if (threadIdx.x == 64) {
          uint32_t* tk = a.ticket + (size_t)nt * a.MT + m;
          const uint32_t old = atomicAdd(tk, 1u);
          const int last = old == (uint32_t)(cl - cf) ? 1 : 0;
          if (last) *tk = 0u;  // ready for the next launch
          flags[1] = last;
        }
        named_sync(1, 128);
        if (flags[1]) {
          __threadfence();
          // 16 columns at a time; the loads of two contributors are in flight together, and each
          // column adds the contributors in CTA order
          for (int jc = 0; jc < NP && j0 + jc < a.N; jc += 16) {
            float acc[16];
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) acc[jj] = 0.f;
            for (int cc = cf; cc <= cl; cc += 2) {
              float4 p0[4], p1[4];
              const int slot0 = tc_first(T, G, cc) >= (int64_t)m * KB ? 0 : 1;
              const float4* q0 = reinterpret_cast<const float4*>(
                  a.part + ((size_t)(nt * G + cc) * 2 + slot0) * (size_t)NP * kTcM + (size_t)rl * NP + jc);
#pragma unroll
              for (int u = 0; u < 4; ++u) p0[u] = __ldcg(q0 + u);
              const bool two = cc + 1 <= cl;
              if (two) {
                const int slot1 = tc_first(T, G, cc + 1) >= (int64_t)m * KB ? 0 : 1;
                const float4* q1 = reinterpret_cast<const float4*>(
                    a.part + ((size_t)(nt * G + cc + 1) * 2 + slot1) * (size_t)NP * kTcM + (size_t)rl * NP + jc);
#pragma unroll
                for (int u = 0; u < 4; ++u) p1[u] = __ldcg(q1 + u);
              }
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                acc[4 * u] += p0[u].x;
                acc[4 * u + 1] += p0[u].y;
                acc[4 * u + 2] += p0[u].z;
                acc[4 * u + 3] += p0[u].w;
              }
              if (two) {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                  acc[4 * u] += p1[u].x;
                  acc[4 * u + 1] += p1[u].y;
                  acc[4 * u + 2] += p1[u].z;
                  acc[4 * u + 3] += p1[u].w;
                }
              }
            }
#pragma unroll
            for (int jj = 0; jj < 16; ++jj)
              if (j0 + jc + jj < a.N) tc_epi<EPI>(a, R, j0 + jc + jj, acc[jj]);
          }
        }
        named_sync(1, 128);
      }
      it += kb1 - kb0;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, a.tmem_cols);
  }
}

// x' = x or RMSNorm(x), split into bf16 hi and lo rows; one CTA per activation row
constexpr int kSplitThreads = 256;

__global__ void __launch_bounds__(kSplitThreads) tc_split_kernel(const TcSplitArgs a) {
  grid_dep_wait();
  grid_dep_launch();
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (b >= a.B) return;
  const float4* xr = reinterpret_cast<const float4*>(a.x + (size_t)b * a.x_stride);
  const int k4 = a.K >> 2;
  __shared__ float red[kSplitThreads / 32];
  __shared__ float s_inv;
  float inv = 1.0f;
  if (a.gain) {
    float ss = 0.f;
    for (int i = tid; i < k4; i += kSplitThreads) {
      const float4 v = __ldg(xr + i);
      ss = fmaf(v.x, v.x, ss);
      ss = fmaf(v.y, v.y, ss);
      ss = fmaf(v.z, v.z, ss);
      ss = fmaf(v.w, v.w, ss);
    }
    ss = warp_sum(ss);
    if (lane == 0) red[warp] = ss;
    __syncthreads();
    if (tid == 0) {
      float s = 0.f;
      for (int w = 0; w < kSplitThreads / 32; ++w) s += red[w];
      s_inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(s, (float)a.K), a.eps)));
    }
    __syncthreads();
    inv = s_inv;
  }
  uint16_t* hi = a.xs + (size_t)b * a.K;
  uint16_t* lo = a.xs + ((size_t)a.Ntot + b) * a.K;
  for (int i = tid; i < k4; i += kSplitThreads) {
    float4 v = __ldg(xr + i);
    if (a.gain) {
      const float4 g = __ldg(reinterpret_cast<const float4*>(a.gain) + i);
      v.x = __fmul_rn(g.x, __fmul_rn(inv, v.x));
      v.y = __fmul_rn(g.y, __fmul_rn(inv, v.y));
      v.z = __fmul_rn(g.z, __fmul_rn(inv, v.z));
      v.w = __fmul_rn(g.w, __fmul_rn(inv, v.w));
    }
    const float f[4] = {v.x, v.y, v.z, v.w};
    uint16_t h[4], l[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      h[e] = f32_to_bf16(f[e]);
      l[e] = f32_to_bf16(__fsub_rn(f[e], bf16_to_f32(h[e])));
    }
    reinterpret_cast<uint2*>(hi)[i] = make_uint2(h[0] | ((uint32_t)h[1] << 16), h[2] | ((uint32_t)h[3] << 16));
    reinterpret_cast<uint2*>(lo)[i] = make_uint2(l[0] | ((uint32_t)l[1] << 16), l[2] | ((uint32_t)l[3] << 16));
  }
}

// ---------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------

static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
static std::once_flag g_encode_once;

bool tc_available() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess && fn)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

bool make_map_2d(CUtensorMap* map, const void* base, int elem_bytes, uint64_t inner, uint64_t outer,
                 uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle) {
  if (!tc_available()) return false;
  if ((inner * elem_bytes) % 16 != 0 || ((uintptr_t)base & 15u) != 0) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * (uint64_t)elem_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  return g_encode(map, elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                  const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tc_make_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
                 uint32_t box_outer) {
  return make_map_2d(map, base, 2, inner, outer, box_inner, box_outer, CU_TENSOR_MAP_SWIZZLE_128B);
}

TcPlan plan_tc(int rows, int K, int B, int num_sms) {
  TcPlan p{};
  p.NP = (B + 15) / 16 * 16;
  if (p.NP > kTcMaxNP) p.NP = kTcMaxNP;
  p.ntiles = (B + p.NP - 1) / p.NP;
  p.Ntot = p.ntiles * p.NP;
  p.MT = (rows + kTcM - 1) / kTcM;
  p.KB = (K + kTcK - 1) / kTcK;
  const int64_t T = (int64_t)p.MT * p.KB;
  p.grid = (int)(T < num_sms ? T : num_sms);
  const size_t stage = 16384 + 2 * (size_t)p.NP * 128;
  int st = (int)((200 * 1024) / stage);
  p.stages = st > 8 ? 8 : st < 2 ? 2 : st;
  uint32_t cols = 32;
  while (cols < 2u * (uint32_t)p.NP) cols <<= 1;
  p.tmem_cols = cols;
  // at least 116 KB keeps one CTA per SM, so tensor-memory allocations never queue
  size_t smem = 1024 + (size_t)p.stages * stage + 16 * (size_t)p.stages + 64;
  if (smem < 116 * 1024) smem = 116 * 1024;
  p.smem = smem;
  return p;
}

using TcFn = void (*)(const CUtensorMap, const CUtensorMap, const TcArgs);

static TcFn pick_tc(int epi) {
  switch (epi) {
    case EPI_QKV: return tc_gemm_kernel<EPI_QKV>;
    case EPI_SWIGLU: return tc_gemm_kernel<EPI_SWIGLU>;
    case EPI_RESID: return tc_gemm_kernel<EPI_RESID>;
    default: return tc_gemm_kernel<EPI_STORE>;
  }
}

cudaError_t tc_prepare(int max_smem_optin) {
  for (int epi = 0; epi < 4; ++epi) {
    cudaError_t e = cudaFuncSetAttribute(pick_tc(epi), cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem_optin);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_tc_split(const TcSplitArgs& a, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.B);
  cfg.blockDim = dim3(kSplitThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, tc_split_kernel, a);
}

cudaError_t launch_tc_gemm(const CUtensorMap& tw, const CUtensorMap& tx, const TcArgs& a, const TcPlan& p, int epi,
                           cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.grid, p.ntiles);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, pick_tc(epi), tw, tx, a);
}

}  // namespace llm
