// Tensor-core projections of batched decode: out[j][r] = sum_c W[r][c] * x'[j][c] for batches of
// activation rows, on the 5th-generation tensor core (tcgen05.mma, accumulators in tensor memory,
// operands staged by TMA).  The steps around each projection (bend-ml-llama "A layer", block:
// RMSNorm before Q/K/V and gate/up, RoPE and the KV write after Q/K/V, the residual adds, SwiGLU;
// the final norm before the LM head) run in the small kernels that read the projection's output.
//
// Precision.  The weights are bf16; the activations are f32.  Each activation is split into two
// bf16 numbers, hi = bf16(x') and lo = bf16(x' - hi) (about 2^-17 relative together), and both
// multiply the weights in one MMA: hi rows sit in MMA rows 0..63, lo rows in 64..127, and the two
// accumulator rows of an activation are added in the epilogue.
//
// Shape of the MMA: M = 128 (the stacked activation rows), N = 256 (weight rows), K = 16; the
// weights are the N operand, so one MMA covers 256 weight rows and a 64-element K block of a
// 32 KB weight tile takes four MMAs.
//
// Work split.  The K range of every 256-row weight tile is cut into S equal splits (S chosen per
// shape so that tiles x splits fills the GPU's SMs evenly); a unit (activation tile, weight tile,
// split) writes its raw sums to out[s].  CTAs are persistent, one per SM, and take units
// c, c + grid, ...; the reader of the projection adds the S splits in split order, so results do
// not depend on timing.
//
// Roles: warp 0 issues TMA copies into a ring of shared-memory stages (mbarrier full/empty),
// warp 1 issues the MMAs (one thread) into two tensor-memory accumulators so the epilogue of one
// unit overlaps the next, warps 2..5 read the accumulators (tcgen05.ld, one MMA row per thread):
// the lo rows pass their values through shared memory to the hi rows, which add and store.  Every
// wait is bounded: on timeout the kernel records kErrDeviceTimeout, lets its copies and MMAs
// drain (bounded again), frees its tensor memory and returns.
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "gemm.cuh"
#include "tc.cuh"

namespace llm {

constexpr uint64_t kTcWaitCycles = 4000000000ull;  // SM cycles: about 2 s at 2 GHz
constexpr int kTcStages = 4;
constexpr uint32_t kTcA = 128 * 128;               // activation tile: 128 MMA rows x 128 bytes
constexpr int kXchgPitch = 33;                     // floats per exchange row (conflict-free)

__global__ void __launch_bounds__(kTcThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tw, const __grid_constant__ CUtensorMap tx, const TcArgs a) {
  extern __shared__ uint8_t tc_smem[];
  const uint32_t s_raw = smem_u32(tc_smem);
  const uint32_t s_base = (s_raw + 1023u) & ~1023u;  // the 128-byte swizzle repeats every 1024 bytes
  uint8_t* g_base = tc_smem + (s_base - s_raw);
  const int NP = a.NP, KB = a.KB, S = a.S, NT = a.n_tile;
  const uint32_t kTcW = (uint32_t)NT * 128u;   // weight tile: NT rows x 128 bytes
  const uint32_t kTcStage = kTcA + kTcW;
  float* xchg = reinterpret_cast<float*>(g_base + kTcStages * kTcStage);  // [64][kXchgPitch]
  const uint32_t bars = s_base + kTcStages * kTcStage + kTcRows * kXchgPitch * 4;
  // barriers: full[stages], empty[stages], acc_full[2], acc_empty[2], drain
  const uint32_t FULL0 = bars, EMPTY0 = bars + 8u * kTcStages, ACCF0 = bars + 16u * kTcStages, ACCE0 = ACCF0 + 16u,
                 DRAIN = ACCE0 + 16u;
  volatile uint32_t* tmem_slot =
      reinterpret_cast<volatile uint32_t*>(g_base + kTcStages * kTcStage + kTcRows * kXchgPitch * 4 + 16 * kTcStages + 40);
  volatile int* flags = reinterpret_cast<volatile int*>(tmem_slot + 2);  // [0] abort

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x, G = gridDim.x;
  const uint32_t xbytes = 2u * (uint32_t)NP * 128u;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kTcStages; ++i) {
      mbar_init(FULL0 + 8u * i, 1);
      mbar_init(EMPTY0 + 8u * i, 1);
    }
    mbar_init(ACCF0, 1);
    mbar_init(ACCF0 + 8u, 1);
    mbar_init(ACCE0, 128);
    mbar_init(ACCE0 + 8u, 128);
    mbar_init(DRAIN, 1);
    flags[0] = 0;
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32((const void*)tmem_slot), 2 * kTcN);
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
  // unit u = (m * T + t) * S + s: weight tile m, activation tile t, split s.  The activation
  // tiles of one weight tile are neighbours, so the CTAs that run them at the same time share
  // the weight tile through L2 (a pass of many prompt tokens reads its weights from HBM once).
  const int T = a.Ntot / NP;
  auto unit = [&](int u, int& t, int& m, int& kb0, int& kb1) {
    const int s = u % S, tm = u / S;
    t = tm % T;
    m = tm / T;
    kb0 = KB * s / S;
    kb1 = KB * (s + 1) / S;
  };

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_map(&tw);
      tma_prefetch_map(&tx);
      // the weight tiles of the first stages do not depend on the previous kernel
      int u = c, t = 0, m = 0, kb0 = 0, kb1 = 0, kb = 0;
      if (u < a.units) unit(u, t, m, kb0, kb1), kb = kb0;
      int npre = 0;
      {
        int pu = u, pt = t, pm = m, pk0 = kb0, pk1 = kb1, pk = kb;
        while (npre < kTcStages && pu < a.units) {
          mbar_expect_tx(FULL0 + 8u * npre, kTcW + xbytes);
          tma_load_2d(s_base + (uint32_t)npre * kTcStage + kTcA, &tw, FULL0 + 8u * npre, pk * kTcK, pm * NT);
          ++npre;
          if (++pk == pk1) {
            pu += G;
            if (pu < a.units) unit(pu, pt, pm, pk0, pk1), pk = pk0;
          }
        }
      }
      grid_dep_wait();
      grid_dep_launch();
      int stg = 0;
      uint32_t ph = 0;
      int issued = 0;
      bool ok = true;
      while (u < a.units && ok) {
        if (issued >= kTcStages && (flags[0] || !mbar_wait(EMPTY0 + 8u * stg, ph ^ 1u, kTcWaitCycles))) {
          fail();
          ok = false;
          break;
        }
        const uint32_t sa = s_base + (uint32_t)stg * kTcStage;
        if (issued >= npre) {
          mbar_expect_tx(FULL0 + 8u * stg, kTcW + xbytes);
          tma_load_2d(sa + kTcA, &tw, FULL0 + 8u * stg, kb * kTcK, m * NT);
        }
        tma_load_2d(sa, &tx, FULL0 + 8u * stg, kb * kTcK, t * NP);                       // hi rows
        tma_load_2d(sa + 64u * 128u, &tx, FULL0 + 8u * stg, kb * kTcK, a.Ntot + t * NP);  // lo rows
        ++issued;
        if (++stg == kTcStages) stg = 0, ph ^= 1u;
        if (++kb == kb1) {
          u += G;
          if (u < a.units) unit(u, t, m, kb0, kb1), kb = kb0;
        }
      }
      // no copy may still be writing shared memory when the CTA exits
      for (int i = issued > kTcStages ? issued - kTcStages : 0; i < issued; ++i)
        if (!mbar_wait(FULL0 + 8u * (uint32_t)(i % kTcStages), (uint32_t)(i / kTcStages) & 1u, kTcWaitCycles)) fail();
    } else {
      grid_dep_wait();
      grid_dep_launch();
    }
  } else if (warp == 1) {
    grid_dep_wait();
    grid_dep_launch();
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, NT);
      int stg = 0;
      uint32_t ph = 0;
      bool ok = true;
      int si = 0;
      for (int u = c; u < a.units && ok; u += G, ++si) {
        int t, m, kb0, kb1;
        unit(u, t, m, kb0, kb1);
        const int buf = si & 1, use = si >> 1;
        if (use > 0 && !mbar_wait(ACCE0 + 8u * buf, (uint32_t)(use - 1) & 1u, kTcWaitCycles)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(buf * kTcN);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (flags[0] || !mbar_wait(FULL0 + 8u * stg, ph, kTcWaitCycles)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = s_base + (uint32_t)stg * kTcStage;
          const uint64_t ad = sw128_kmajor_desc(sa), bd = sw128_kmajor_desc(sa + kTcA);
#pragma unroll
          for (int k = 0; k < kTcK / 16; ++k)  // 16 K elements = 32 bytes = 2 in the address field
            tc_mma_bf16(d, ad + 2 * k, bd + 2 * k, idesc, (kb > kb0 || k > 0) ? 1u : 0u);
          tc_commit(EMPTY0 + 8u * stg);
          if (++stg == kTcStages) stg = 0, ph ^= 1u;
        }
        if (!ok) break;
        tc_commit(ACCF0 + 8u * buf);
      }
      if (!ok) fail();
      // every MMA has completed before tensor memory is freed
      tc_commit(DRAIN);
      if (!mbar_wait(DRAIN, 0, kTcWaitCycles)) fail();
    }
  } else {
    grid_dep_wait();
    grid_dep_launch();
    const int q = warp & 3;          // this warp's quarter of the tensor-memory lanes
    const bool hi = q < 2;           // MMA rows 0..63: hi halves; 64..127: lo halves
    const int j = (q & 1) * 32 + lane;  // activation row within the tile
    const bool active = (q & 1) == 0 || NP > 32;
    const bool vec = (a.rows & 3) == 0;
    int si = 0;
    for (int u = c; u < a.units; u += G, ++si) {
      int t, m, kb0, kb1;
      unit(u, t, m, kb0, kb1);
      const int s = u % S;
      const int buf = si & 1, use = si >> 1;
      bool ok = !flags[0] && mbar_wait(ACCF0 + 8u * buf, (uint32_t)use & 1u, kTcWaitCycles);
      ok = named_sync_and(1, 128, ok);
      if (!ok) {
        if (threadIdx.x == 64) fail();
        break;
      }
      tc_fence_after();
      const int row = t * NP + j;  // activation (batch) row
      const bool valid = j < NP && row < a.N;
      float* orow = a.out + ((size_t)s * a.N + (size_t)(valid ? row : 0)) * a.rows;
      const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * kTcN);
      for (int cc = 0; cc < NT / 32; ++cc) {
        float v[32];
        if (active) {
          float w[16];
          tc_ld16(taddr + (uint32_t)(cc * 32), w);
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = w[i];
          tc_ld16(taddr + (uint32_t)(cc * 32 + 16), w);
#pragma unroll
          for (int i = 0; i < 16; ++i) v[16 + i] = w[i];
          tc_wait_ld();
          if (!hi)
#pragma unroll
            for (int i = 0; i < 32; ++i) xchg[j * kXchgPitch + i] = v[i];
        }
        named_sync(1, 128);
        if (hi && active && valid) {
          const int col0 = m * NT + cc * 32;
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __fadd_rn(v[i], xchg[j * kXchgPitch + i]);
          if (vec && col0 + 32 <= a.rows) {
#pragma unroll
            for (int i = 0; i < 32; i += 4)
              *reinterpret_cast<float4*>(orow + col0 + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (col0 + i < a.rows) orow[col0 + i] = v[i];
          }
        }
        named_sync(1, 128);
      }
      tc_fence_before();
      mbar_arrive(ACCE0 + 8u * buf);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 2 * kTcN);
  }
}

// ---------------------------------------------------------------------------------------
// the readers of the split sums
// ---------------------------------------------------------------------------------------

constexpr int kPrepThreads = 128;
constexpr int kPrepCluster = 8;   // CTAs sharing one activation row (a thread-block cluster)
constexpr int kPrepMaxV = 4;      // float4 of the row per thread (K <= 8 * 128 * 4 * 4 = kTcMaxK)
constexpr int kMaxSplits = 16;  // K splits a reader adds (plan_tc stays within it)

LLM_D float silu_mul(float g, float u) { return __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, expf(-g))), u); }

// sum_s p[s * stride] in split order; the loads are issued together
LLM_D float4 sum_splits4(const float* p, size_t stride, int S) {
  float4 t[kMaxSplits];
#pragma unroll
  for (int s = 0; s < kMaxSplits; ++s)
    if (s < S) t[s] = *reinterpret_cast<const float4*>(p + s * stride);
  float4 v = t[0];
#pragma unroll
  for (int s = 1; s < kMaxSplits; ++s)
    if (s < S) {
      v.x = __fadd_rn(v.x, t[s].x); v.y = __fadd_rn(v.y, t[s].y); v.z = __fadd_rn(v.z, t[s].z); v.w = __fadd_rn(v.w, t[s].w);
    }
  return v;
}

// grid (kPrepCluster, B): the CTAs of one row form a cluster and exchange their parts of the
// sum of squares through distributed shared memory (added in rank order)
__global__ void __launch_bounds__(kPrepThreads) tc_prep_kernel(const TcPrepArgs a) {
  __shared__ float red[kPrepThreads / 32];
  __shared__ float s_part;
  grid_dep_wait();
  grid_dep_launch();
  const int rank = blockIdx.x, b = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int k4 = a.K >> 2;
  const int per = (k4 + kPrepCluster - 1) / kPrepCluster;  // float4 of this CTA
  const int i0 = rank * per, i1 = min(k4, i0 + per);
  const size_t split = (size_t)a.B * a.part_rows;
  float4 xv[kPrepMaxV];
  float ss = 0.f;
#pragma unroll
  for (int r = 0; r < kPrepMaxV; ++r) {
    const int i = i0 + tid + r * kPrepThreads;
    if (i < i1) {
      float4 v;
      if (!a.part) {
        v = *reinterpret_cast<const float4*>(a.x_in + (size_t)b * a.x_stride + 4 * i);
      } else if (a.swiglu) {
        const float* p = a.part + (size_t)b * a.part_rows + 8 * i;  // (g, u) pairs of 4 outputs
        const float4 s0 = sum_splits4(p, split, a.S), s1 = sum_splits4(p + 4, split, a.S);
        v = make_float4(silu_mul(s0.x, s0.y), silu_mul(s0.z, s0.w), silu_mul(s1.x, s1.y), silu_mul(s1.z, s1.w));
      } else {
        v = sum_splits4(a.part + (size_t)b * a.part_rows + 4 * i, split, a.S);
        if (a.resid) {
          const float4 rr = *reinterpret_cast<const float4*>(a.resid + (size_t)b * a.resid_stride + 4 * i);
          v.x = __fadd_rn(rr.x, v.x); v.y = __fadd_rn(rr.y, v.y); v.z = __fadd_rn(rr.z, v.z); v.w = __fadd_rn(rr.w, v.w);
        }
      }
      if (a.xout) *reinterpret_cast<float4*>(a.xout + (size_t)b * a.xout_stride + 4 * i) = v;
      ss = fmaf(v.x, v.x, ss);
      ss = fmaf(v.y, v.y, ss);
      ss = fmaf(v.z, v.z, ss);
      ss = fmaf(v.w, v.w, ss);
      xv[r] = v;
    }
  }
  float inv = 1.0f;
  if (a.gain) {
    ss = warp_sum(ss);
    if (lane == 0) red[warp] = ss;
    __syncthreads();
    if (tid == 0) {
      float t = 0.f;
      for (int w = 0; w < kPrepThreads / 32; ++w) t += red[w];
      s_part = t;
    }
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
    // lane r fetches rank r's part; the parts are then added in rank order
    float pr = 0.f;
    if (lane < kPrepCluster) {
      uint32_t remote;
      asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(&s_part)), "r"(lane));
      asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(pr) : "r"(remote) : "memory");
    }
    float tot = 0.f;
#pragma unroll
    for (int r = 0; r < kPrepCluster; ++r) tot += __shfl_sync(0xffffffffu, pr, r);
    inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(tot, (float)a.K), a.eps)));
    // no CTA leaves while another may still read its part
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
  }
  uint16_t* hi = a.xs + (size_t)b * a.K;
  uint16_t* lo = a.xs + ((size_t)a.Ntot + b) * a.K;
#pragma unroll
  for (int r = 0; r < kPrepMaxV; ++r) {
    const int i = i0 + tid + r * kPrepThreads;
    if (i < i1) {
      float4 v = xv[r];
      if (a.gain) {
        const float4 g = *reinterpret_cast<const float4*>(a.gain + 4 * i);
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
}

// one thread per (row, RoPE pair): the split sums added in order, then as the GEMV's Q/K/V
// epilogue (rot_lo = lo*cos - hi*sin, rot_hi = hi*cos + lo*sin; v unrotated; the cache element
// rounded on write)
__global__ void tc_qkv_kernel(const TcQkvArgs a) {
  grid_dep_wait();
  grid_dep_launch();
  const int npairs = a.rows >> 1;
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= a.B * npairs) return;
  const int b = idx / npairs, pr = idx - b * npairs;
  const int R = 2 * pr;
  const size_t split = (size_t)a.B * a.rows;
  const float* p = a.part + (size_t)b * a.rows + R;
  float2 t[kMaxSplits];
#pragma unroll
  for (int s = 0; s < kMaxSplits; ++s)
    if (s < a.S) t[s] = *reinterpret_cast<const float2*>(p + s * split);
  float2 x = t[0];
#pragma unroll
  for (int s = 1; s < kMaxSplits; ++s)
    if (s < a.S) {
      x.x = __fadd_rn(x.x, t[s].x);
      x.y = __fadd_rn(x.y, t[s].y);
    }
  const float x0 = x.x, x1 = x.y;
  const int pos = row_pos(a.step, b), half = a.hd >> 1;
  const int head = R / a.hd, e = (R - head * a.hd) >> 1;
  const size_t row = (size_t)b;
  if (head < a.H + a.kv) {
    const float c = a.rope_cos[(size_t)pos * half + e], s = a.rope_sin[(size_t)pos * half + e];
    const float lo = __fadd_rn(__fmul_rn(x0, c), __fmul_rn(-x1, s));
    const float hi = __fadd_rn(__fmul_rn(x1, c), __fmul_rn(x0, s));
    if (head < a.H) {
      float* q = a.q_out + row * a.q_stride + (size_t)head * a.hd;
      q[e] = lo;
      q[e + half] = hi;
    } else {
      int r, pp;
      cache_slot(a.step, a.cap, b, pos, r, pp);
      const size_t ci = (((size_t)r * a.kv + (size_t)(head - a.H)) * a.cap + pp) * a.hd;
      store_elem<1>(a.kc, ci + e, lo);
      store_elem<1>(a.kc, ci + e + half, hi);
    }
  } else {
    int r, pp;
    cache_slot(a.step, a.cap, b, pos, r, pp);
    const size_t ci = (((size_t)r * a.kv + (size_t)(head - a.H - a.kv)) * a.cap + pp) * a.hd;
    store_elem<1>(a.vc, ci + e, x0);
    store_elem<1>(a.vc, ci + e + half, x1);
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

int tc_ntot(int B) {
  const int np = B >= kTcRows ? kTcRows : (B + 15) / 16 * 16;
  return (B + np - 1) / np * np;
}

TcPlan plan_tc(int rows, int K, int B, int num_sms, bool whole) {
  TcPlan p{};
  p.NP = B >= kTcRows ? kTcRows : (B + 15) / 16 * 16;
  p.ntiles = (B + p.NP - 1) / p.NP;
  p.Ntot = p.ntiles * p.NP;
  p.KB = (K + kTcK - 1) / kTcK;
  auto eff = [&](long long U) {
    const long long waves = (U + num_sms - 1) / num_sms;
    return (double)U / (double)(waves * num_sms);
  };
  if (whole) {
    // no K split (the reader takes the output as it is): 256- or 128-row tiles, whichever fills
    // the SMs more evenly
    const int m256 = (rows + 255) / 256, m128 = (rows + 127) / 128;
    p.n_tile = eff((long long)m128 * p.ntiles) > eff((long long)m256 * p.ntiles) + 1e-9 ? 128 : 256;
    p.S = 1;
  } else {
    // splits: the most even fill of the SMs (units / (waves * SMs)), at least 4 K blocks a split.
    // Split sums cost S * B * rows * 4 bytes written and read again: never more than a quarter
    // of the weight bytes (many activation rows, as in a prefill pass, have tiles enough).
    p.n_tile = kTcN;
    const int base = p.ntiles * ((rows + kTcN - 1) / kTcN);
    double best = -1.0;
    p.S = 1;
    const int smax = std::max(1, std::min(kMaxSplits, K / (8 * B)));
    for (int S = 1; S <= smax && S <= p.KB; ++S) {
      if (S > 1 && p.KB / S < 4) break;
      const double e = eff((long long)base * S);
      if (e > best + 1e-9) {
        best = e;
        p.S = S;
      }
    }
  }
  p.MT = (rows + p.n_tile - 1) / p.n_tile;
  p.units = p.ntiles * p.MT * p.S;
  p.grid = p.units < num_sms ? p.units : num_sms;
  p.stages = kTcStages;
  p.smem = 1024 + (size_t)kTcStages * (kTcA + (size_t)p.n_tile * 128) + (size_t)kTcRows * kXchgPitch * 4 + 16 * kTcStages + 64;
  return p;
}

__global__ void tc_prep_rows_kernel(const TcPrepArgs a);
constexpr int kPrepRowMaxKDecl = kTcMaxK;

cudaError_t tc_prepare(int max_smem_optin) {
  cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem_optin);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(tc_prep_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPrepRowMaxKDecl * 4);
  return e;
}

static cudaLaunchConfig_t cfg_of(dim3 grid, int threads, size_t smem, cudaStream_t s, bool pdl,
                                 cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

// The same reader for many rows (a prefill pass): one CTA of kPrepRowThreads per row keeps the
// whole row in shared memory, so the sum of squares needs no cluster; the rows themselves fill
// the GPU.
constexpr int kPrepRowThreads = 256;
constexpr int kPrepRowMaxK = kPrepRowMaxKDecl;  // floats of a row in shared memory (64 KB)
constexpr int kPrepRowsFrom = 128;   // rows from which the per-row kernel is used

__global__ void __launch_bounds__(kPrepRowThreads) tc_prep_rows_kernel(const TcPrepArgs a) {
  extern __shared__ float4 rowv[];  // [K / 4]
  __shared__ float red[kPrepRowThreads / 32];
  __shared__ float s_inv;
  grid_dep_wait();
  grid_dep_launch();
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int k4 = a.K >> 2;
  const size_t split = (size_t)a.B * a.part_rows;
  float ss = 0.f;
  for (int i = tid; i < k4; i += kPrepRowThreads) {
    float4 v;
    if (!a.part) {
      v = *reinterpret_cast<const float4*>(a.x_in + (size_t)b * a.x_stride + 4 * i);
    } else if (a.swiglu) {
      const float* p = a.part + (size_t)b * a.part_rows + 8 * i;
      const float4 s0 = sum_splits4(p, split, a.S), s1 = sum_splits4(p + 4, split, a.S);
      v = make_float4(silu_mul(s0.x, s0.y), silu_mul(s0.z, s0.w), silu_mul(s1.x, s1.y), silu_mul(s1.z, s1.w));
    } else {
      v = sum_splits4(a.part + (size_t)b * a.part_rows + 4 * i, split, a.S);
      if (a.resid) {
        const float4 rr = *reinterpret_cast<const float4*>(a.resid + (size_t)b * a.resid_stride + 4 * i);
        v.x = __fadd_rn(rr.x, v.x); v.y = __fadd_rn(rr.y, v.y); v.z = __fadd_rn(rr.z, v.z); v.w = __fadd_rn(rr.w, v.w);
      }
    }
    if (a.xout) *reinterpret_cast<float4*>(a.xout + (size_t)b * a.xout_stride + 4 * i) = v;
    ss = fmaf(v.x, v.x, ss);
    ss = fmaf(v.y, v.y, ss);
    ss = fmaf(v.z, v.z, ss);
    ss = fmaf(v.w, v.w, ss);
    rowv[i] = v;
  }
  float inv = 1.0f;
  if (a.gain) {
    ss = warp_sum(ss);
    if (lane == 0) red[warp] = ss;
    __syncthreads();
    if (tid == 0) {
      float t = 0.f;
      for (int w = 0; w < kPrepRowThreads / 32; ++w) t += red[w];
      s_inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(t, (float)a.K), a.eps)));
    }
  }
  __syncthreads();
  if (a.gain) inv = s_inv;
  uint16_t* hi = a.xs + (size_t)b * a.K;
  uint16_t* lo = a.xs + ((size_t)a.Ntot + b) * a.K;
  for (int i = tid; i < k4; i += kPrepRowThreads) {
    float4 v = rowv[i];
    if (a.gain) {
      const float4 g = *reinterpret_cast<const float4*>(a.gain + 4 * i);
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

cudaError_t launch_tc_prep(const TcPrepArgs& a, cudaStream_t s, bool pdl) {
  if (a.K > kPrepCluster * kPrepThreads * kPrepMaxV * 4 || (a.K & 3) || a.S > kMaxSplits) return cudaErrorInvalidValue;
  if (a.B >= kPrepRowsFrom && a.K <= kPrepRowMaxK) {
    cudaLaunchAttribute attr1[1];
    const cudaLaunchConfig_t cfg = cfg_of(dim3(a.B), kPrepRowThreads, (size_t)a.K * 4, s, pdl, attr1);
    return cudaLaunchKernelEx(&cfg, tc_prep_rows_kernel, a);
  }
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = cfg_of(dim3(kPrepCluster, a.B), kPrepThreads, 0, s, pdl, attr);
  if (a.gain) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = kPrepCluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  return cudaLaunchKernelEx(&cfg, tc_prep_kernel, a);
}

cudaError_t launch_tc_gemm(const CUtensorMap& tw, const CUtensorMap& tx, const TcArgs& a, const TcPlan& p,
                           cudaStream_t s, bool pdl) {
  cudaLaunchAttribute attr[1];
  const cudaLaunchConfig_t cfg = cfg_of(dim3(p.grid), kTcThreads, p.smem, s, pdl, attr);
  return cudaLaunchKernelEx(&cfg, tc_gemm_kernel, tw, tx, a);
}

cudaError_t launch_tc_qkv(const TcQkvArgs& a, cudaStream_t s, bool pdl) {
  cudaLaunchAttribute attr[1];
  const int n = a.B * (a.rows >> 1);
  const cudaLaunchConfig_t cfg = cfg_of(dim3((n + 255) / 256), 256, 0, s, pdl, attr);
  return cudaLaunchKernelEx(&cfg, tc_qkv_kernel, a);
}


}  // namespace llm
