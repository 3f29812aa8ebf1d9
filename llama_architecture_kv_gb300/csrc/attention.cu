// Grouped-query attention of one decode step over the KV cache (split-K flash decode).
//
// Computes, for every batch row b and query head h = j*g + i (group j reads key/value head j:
// bend-ml-llama "Grouped-query attention", gqa_head), the output
//   o_h = sum_{p=0..t} softmax_p(scale * q_h . K_j[p]) V_j[p],  scale = 1/sqrt(hd),
// over exactly the cache positions 0..t, t = pos (bend-ml-llama law causal; Llama 3.1 8B card,
// attention.linnet decode: seen[s] = s <= pos).
//
// Layout: the cache of one layer is [max_batch][kv][cap][hd] (attention.linnet cache_k), so the
// positions of one (row, key/value head) are contiguous.  Grid: (splits, kv, B).  A CTA takes
// one contiguous slice of positions of one (row, kv head), stages its keys and values in shared
// memory once (cp.async, double buffered) and serves all g query heads of the group from them:
// the cache is read from HBM exactly once per step.  Each CTA keeps an online softmax (running
// max m, sum l, unnormalized output) and writes a partial (o, m, l).  The last CTA of a (row,
// kv head) to finish -- found with an atomic ticket, nobody waits -- merges the partials in
// split order (log-sum-exp), so the result does not depend on which CTA finished last.
#include "attention.cuh"

namespace llm {

constexpr int kAttnThreads = 128;
constexpr int kAttnWarps = kAttnThreads / 32;
constexpr int kMaxHeadsPerWarp = 4;
constexpr int kMinChunk = 64;  // fewest positions a split takes

LLM_D void cp_async16(void* smem, const void* gmem) {
  const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
LLM_D void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N> LLM_D void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

template <int KT> LLM_D float2 load2(const void* base, int idx) {
  if constexpr (KT == 0) {
    return *reinterpret_cast<const float2*>((const float*)base + idx);
  } else {
    const uint32_t u = *reinterpret_cast<const uint32_t*>((const uint16_t*)base + idx);
    return make_float2(bf16_lo(u), bf16_hi(u));
  }
}

// KT: cache element type (0 f32, 1 bf16); HD: head size
template <int KT, int HD>
__global__ void __launch_bounds__(kAttnThreads) attn_decode_kernel(const AttnArgs a) {
  constexpr int ES = Elem<KT>::bytes;
  constexpr int ROWB = HD * ES;             // bytes of one cached row
  constexpr int KPAD = ROWB + 16;           // padded key row (conflict-free per-lane rows)
  constexpr int NE = HD >= 64 ? HD / 64 : 1;  // column pairs per lane in P.V
  extern __shared__ __align__(16) unsigned char smraw[];

  const int split = blockIdx.x, j = blockIdx.y, b = blockIdx.z;
  const int g = a.g, H = a.kv * a.g;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // warp roles: hw = head lane (heads hw, hw+HW, ...), pw = position lane
  const int HW = g < kAttnWarps ? g : kAttnWarps;
  const int PW = (kAttnWarps % HW == 0) ? kAttnWarps / HW : 1;
  const int TILE = 32 * PW;
  const int hw = warp % HW, pw = warp / HW;
  const bool active = warp < HW * PW;

  float* qs = reinterpret_cast<float*>(smraw);                         // [g][HD]
  unsigned char* kbuf = smraw + (size_t)g * HD * 4;                    // [2][TILE][KPAD]
  unsigned char* vbuf = kbuf + 2 * (size_t)TILE * KPAD;                // [2][TILE][ROWB]
  float* red = reinterpret_cast<float*>(vbuf + 2 * (size_t)TILE * ROWB);  // [warps][MAXH][HD+2]
  __shared__ int s_last;

  grid_dep_wait();
  grid_dep_launch();

  // positions 0..t in contiguous slices of at least kMinChunk: the number of active splits
  // follows t, so a short context is not cut into slivers whose merge would cost more than them
  const int t = a.step->pos;
  const int npos = t + 1;
  int chunk = (npos + a.ns - 1) / a.ns;
  chunk = (chunk + 31) & ~31;
  if (chunk < kMinChunk) chunk = kMinChunk;
  const int nact = (npos + chunk - 1) / chunk;
  if (split >= nact) return;
  const int p0 = split * chunk;
  const int p1 = min(npos, p0 + chunk);

  for (int i = tid; i < g * HD; i += kAttnThreads)
    qs[i] = a.q[(size_t)b * a.q_stride + (size_t)j * g * HD + i];

  const size_t head_off = (((size_t)b * a.kv + j) * a.cap) * HD;  // element offset of position 0
  const unsigned char* kg = (const unsigned char*)a.kc + head_off * ES;
  const unsigned char* vg = (const unsigned char*)a.vc + head_off * ES;

  auto stage = [&](int buf, int tb) {
    // rows tb .. tb+TILE-1 (clamped to p1), 16-byte pieces
    constexpr int PIECES = ROWB / 16;
    const int rows = min(TILE, p1 - tb);
    for (int i = tid; i < rows * PIECES; i += kAttnThreads) {
      const int r = i / PIECES, c = i - r * PIECES;
      cp_async16(kbuf + ((size_t)buf * TILE + r) * KPAD + c * 16, kg + (size_t)(tb + r) * ROWB + c * 16);
      cp_async16(vbuf + ((size_t)buf * TILE + r) * ROWB + c * 16, vg + (size_t)(tb + r) * ROWB + c * 16);
    }
  };

  float m[kMaxHeadsPerWarp], l[kMaxHeadsPerWarp], o[kMaxHeadsPerWarp][NE][2];
#pragma unroll
  for (int hh = 0; hh < kMaxHeadsPerWarp; ++hh) {
    m[hh] = -INFINITY;
    l[hh] = 0.f;
#pragma unroll
    for (int n = 0; n < NE; ++n) o[hh][n][0] = o[hh][n][1] = 0.f;
  }

  const int ntiles = p0 < p1 ? (p1 - p0 + TILE - 1) / TILE : 0;
  if (ntiles > 0) stage(0, p0);
  cp_async_commit();
  for (int it = 0; it < ntiles; ++it) {
    const int tb = p0 + it * TILE;
    if (it + 1 < ntiles) stage((it + 1) & 1, tb + TILE);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const int buf = it & 1;
    if (active) {
      const int p = tb + pw * 32 + lane;  // this lane's position
      const bool valid = p < p1;
      const unsigned char* krow = kbuf + ((size_t)buf * TILE + pw * 32 + lane) * KPAD;
      const int nh = (g - hw + HW - 1) / HW;  // heads this warp serves
      // scores of every head of this warp: each key row is read from shared memory once
      float s[kMaxHeadsPerWarp];
#pragma unroll
      for (int hh = 0; hh < kMaxHeadsPerWarp; ++hh) s[hh] = 0.f;
      if (valid) {
#pragma unroll 2
        for (int c = 0; c < ROWB / 16; ++c) {
          const uint4 kv4 = *reinterpret_cast<const uint4*>(krow + c * 16);
          float kf[16 / ES];
          unpack16<KT>(kv4, kf);
#pragma unroll
          for (int hh = 0; hh < kMaxHeadsPerWarp; ++hh) {
            if (hh < nh) {
              const float4* q4 = reinterpret_cast<const float4*>(qs + (hw + hh * HW) * HD + c * (16 / ES));
#pragma unroll
              for (int e4 = 0; e4 < 16 / ES / 4; ++e4) {
                const float4 qv = q4[e4];
                s[hh] = fmaf(qv.x, kf[4 * e4 + 0], s[hh]);
                s[hh] = fmaf(qv.y, kf[4 * e4 + 1], s[hh]);
                s[hh] = fmaf(qv.z, kf[4 * e4 + 2], s[hh]);
                s[hh] = fmaf(qv.w, kf[4 * e4 + 3], s[hh]);
              }
            }
          }
        }
      }
      // online softmax per head (running max m, running sum l)
      float w[kMaxHeadsPerWarp];
#pragma unroll
      for (int hh = 0; hh < kMaxHeadsPerWarp; ++hh) {
        w[hh] = 0.f;
        if (hh < nh) {
          const float sc = valid ? s[hh] * a.scale : -INFINITY;
          const float mnew = fmaxf(m[hh], warp_max(sc));
          if (mnew != -INFINITY) {  // uniform across the warp
            const float corr = expf(m[hh] - mnew);
            w[hh] = valid ? expf(sc - mnew) : 0.f;
            l[hh] = l[hh] * corr + warp_sum(w[hh]);
            m[hh] = mnew;
#pragma unroll
            for (int n = 0; n < NE; ++n) {
              o[hh][n][0] *= corr;
              o[hh][n][1] *= corr;
            }
          }
        }
      }
      // weighted values: each value row is read from shared memory once for all heads
      const unsigned char* vt = vbuf + ((size_t)buf * TILE + pw * 32) * ROWB;
      const int nv = min(32, p1 - (tb + pw * 32));
      for (int pp = 0; pp < nv; ++pp) {
        float2 v2[NE];
#pragma unroll
        for (int n = 0; n < NE; ++n) {
          const int e = 2 * lane + 64 * n;
          v2[n] = e < HD ? load2<KT>(vt + (size_t)pp * ROWB, e) : make_float2(0.f, 0.f);
        }
#pragma unroll
        for (int hh = 0; hh < kMaxHeadsPerWarp; ++hh) {
          if (hh < nh) {
            const float wp = __shfl_sync(0xffffffffu, w[hh], pp);
#pragma unroll
            for (int n = 0; n < NE; ++n) {
              o[hh][n][0] = fmaf(wp, v2[n].x, o[hh][n][0]);
              o[hh][n][1] = fmaf(wp, v2[n].y, o[hh][n][1]);
            }
          }
        }
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();

  // ---- merge the position lanes of each head inside the CTA, write this split's partial ----
  if (active) {
#pragma unroll
    for (int hh = 0; hh < kMaxHeadsPerWarp; ++hh) {
      const int i = hw + hh * HW;
      if (i >= g) break;
      float* r = red + ((size_t)warp * kMaxHeadsPerWarp + hh) * (HD + 2);
#pragma unroll
      for (int n = 0; n < NE; ++n) {
        const int e = 2 * lane + 64 * n;
        if (e < HD) {
          r[e] = o[hh][n][0];
          r[e + 1] = o[hh][n][1];
        }
      }
      if (lane == 0) {
        r[HD] = m[hh];
        r[HD + 1] = l[hh];
      }
    }
  }
  __syncthreads();
  for (int idx = tid; idx < g * HD; idx += kAttnThreads) {
    const int i = idx / HD, e = idx - i * HD;
    const int hwi = i % HW, hh = i / HW;
    float M = -INFINITY;
    for (int q = 0; q < PW; ++q) M = fmaxf(M, red[((size_t)(q * HW + hwi) * kMaxHeadsPerWarp + hh) * (HD + 2) + HD]);
    float L = 0.f, O = 0.f;
    if (M != -INFINITY) {
      for (int q = 0; q < PW; ++q) {
        const float* r = red + ((size_t)(q * HW + hwi) * kMaxHeadsPerWarp + hh) * (HD + 2);
        const float f = expf(r[HD] - M);
        L += r[HD + 1] * f;
        O += r[e] * f;
      }
    }
    float* part = a.part + (((size_t)b * H + (size_t)j * g + i) * a.ns + split) * (HD + 2);
    part[e] = O;
    if (e == 0) {
      part[HD] = M;
      part[HD + 1] = L;
    }
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const unsigned int prev = atomicAdd(a.ticket + (size_t)b * a.kv + j, 1u);
    s_last = (prev == (unsigned int)(nact - 1));
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // ---- the last CTA of this (row, kv head): merge the splits in order ----
  // weights f[i][s] = exp(m_s - M_i) / L_i per head and split (one warp per head, fixed order),
  // then out[i][e] = sum_s f[i][s] o_s[e] with the o loads issued together
  float* fw = reinterpret_cast<float*>(kbuf);  // [g][nact] (the tiles are no longer needed)
  const float* pbase = a.part + (((size_t)b * H + (size_t)j * g) * a.ns) * (HD + 2);
  for (int i = warp; i < g; i += kAttnWarps) {
    const float* pb = pbase + (size_t)i * a.ns * (HD + 2);
    float M = -INFINITY;
    for (int s2 = lane; s2 < nact; s2 += 32) M = fmaxf(M, __ldcg(pb + (size_t)s2 * (HD + 2) + HD));
    M = warp_max(M);
    float L = 0.f;
    for (int s2 = lane; s2 < nact; s2 += 32) {
      const float ms = __ldcg(pb + (size_t)s2 * (HD + 2) + HD);
      const float f = ms == -INFINITY ? 0.f : expf(ms - M);
      fw[i * nact + s2] = f;
      L += __ldcg(pb + (size_t)s2 * (HD + 2) + HD + 1) * f;
    }
    L = warp_sum(L);
    const float rl = 1.0f / L;
    for (int s2 = lane; s2 < nact; s2 += 32) fw[i * nact + s2] *= rl;
  }
  __syncthreads();
  for (int idx = tid; idx < g * HD; idx += kAttnThreads) {
    const int i = idx / HD, e = idx - i * HD;
    const float* pb = pbase + (size_t)i * a.ns * (HD + 2) + e;
    float O = 0.f;
    int s2 = 0;
    for (; s2 + 8 <= nact; s2 += 8) {
      float ov[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) ov[q] = __ldcg(pb + (size_t)(s2 + q) * (HD + 2));
#pragma unroll
      for (int q = 0; q < 8; ++q) O = fmaf(fw[i * nact + s2 + q], ov[q], O);
    }
    for (; s2 < nact; ++s2) O = fmaf(fw[i * nact + s2], __ldcg(pb + (size_t)s2 * (HD + 2)), O);
    a.out[(size_t)b * a.out_stride + ((size_t)j * g + i) * HD + e] = O;
  }
  if (tid == 0) a.ticket[(size_t)b * a.kv + j] = 0u;
}

// ---------------------------------------------------------------------------------------

template <int KT, int HD>
static size_t smem_for(int g, int ns) {
  const int HW = g < kAttnWarps ? g : kAttnWarps;
  const int PW = (kAttnWarps % HW == 0) ? kAttnWarps / HW : 1;
  const int TILE = 32 * PW;
  const int ROWB = HD * Elem<KT>::bytes;
  size_t tiles = 2 * (size_t)TILE * (ROWB + 16) + 2 * (size_t)TILE * ROWB;
  if (tiles < (size_t)g * ns * 4) tiles = (size_t)g * ns * 4;  // the merge reuses the tile space
  return (size_t)g * HD * 4 + tiles + (size_t)kAttnWarps * kMaxHeadsPerWarp * (HD + 2) * 4;
}

using AttnFn = void (*)(const AttnArgs);

template <int KT>
static AttnFn pick_hd(int hd, size_t* smem, int g, int ns) {
  switch (hd) {
    case 16: *smem = smem_for<KT, 16>(g, ns); return attn_decode_kernel<KT, 16>;
    case 32: *smem = smem_for<KT, 32>(g, ns); return attn_decode_kernel<KT, 32>;
    case 64: *smem = smem_for<KT, 64>(g, ns); return attn_decode_kernel<KT, 64>;
    case 128: *smem = smem_for<KT, 128>(g, ns); return attn_decode_kernel<KT, 128>;
    case 256: *smem = smem_for<KT, 256>(g, ns); return attn_decode_kernel<KT, 256>;
    default: return nullptr;
  }
}

bool attn_supported(int hd, int g) { return (hd == 16 || hd == 32 || hd == 64 || hd == 128 || hd == 256) && g >= 1 && g <= 16; }

cudaError_t attn_prepare(int max_smem_optin) {
  for (int kt = 0; kt < 2; ++kt)
    for (int hd : {16, 32, 64, 128, 256}) {
      size_t sm = 0;
      AttnFn fn = kt ? pick_hd<1>(hd, &sm, 1, 1) : pick_hd<0>(hd, &sm, 1, 1);
      cudaFuncAttributes fa;
      cudaError_t e = cudaFuncGetAttributes(&fa, fn);
      if (e != cudaSuccess) return e;
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem_optin - (int)fa.sharedSizeBytes);
      if (e != cudaSuccess) return e;
    }
  return cudaSuccess;
}

int attn_splits(int B, int kv, int cap, int num_sms) {
  // enough CTAs to cover the GPU twice, but at least 32 positions per split at full capacity
  int ns = (2 * num_sms + B * kv - 1) / (B * kv);
  const int by_cap = (cap + 31) / 32;
  if (ns > by_cap) ns = by_cap;
  if (ns > 1024) ns = 1024;
  if (ns < 1) ns = 1;
  return ns;
}

cudaError_t launch_attn(const AttnArgs& a, int kt, cudaStream_t s, bool pdl) {
  size_t smem = 0;
  AttnFn fn = kt ? pick_hd<1>(a.hd, &smem, a.g, a.ns) : pick_hd<0>(a.hd, &smem, a.g, a.ns);
  if (!fn) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.ns, a.kv, a.B);
  cfg.blockDim = dim3(kAttnThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fn, a);
}

}  // namespace llm
