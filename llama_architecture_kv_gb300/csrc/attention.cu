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
// one contiguous slice of positions of one (row, kv head) and streams it through shared memory
// in tiles (cp.async, a ring of 2..4 tiles, all but one in flight); the g query heads of the
// group are served from the same tile, so the cache is read from HBM once.  Inside a tile all eight warps work on it together,
// which keeps the dependent chains short (decode attention at small batch is latency-bound):
//   scores   one thread per (head, position): a dot product of hd with four accumulators;
//   softmax  one warp per head: tile maximum, running max m, weights exp(s - m), running sum l;
//   values   one thread per (head, two dimensions), or a few threads splitting the positions
//            when heads x dimensions is small; outputs stay in registers across tiles.
// Merging the splits of one (row, kv head) (log-sum-exp, in split order, so the result does not
// depend on timing):
//   up to attn_max_cluster() splits (8, or 16 where the device allows) form one cluster; each CTA leaves its partial in
//   its shared memory and, after a cluster barrier, CTA 0 of the cluster reads the others'
//   through distributed shared memory;
//   more splits (long contexts) write partials to global memory, and the last CTA to finish --
//   found with an atomic ticket, nobody waits -- merges them.
#include "attention.cuh"

namespace llm {

constexpr int kAttnThreads = 256;
constexpr int kAttnWarps = kAttnThreads / 32;
constexpr int kMinChunk = 64;   // fewest positions a split takes
constexpr int kMaxPairs = 4;    // output pairs (two dimensions each) per thread

// Tile shape: about 256 (head, position) scores per tile, and a ring of 2..4 tile buffers
// (ring - 1 tiles in flight ahead of the one in use) within 160 KB of shared memory.
struct TileCfg {
  int tp, ring;
};
LLM_HD TileCfg tile_cfg(int g, int rowb) {
  int tp = g >= 8 ? 32 : g >= 2 ? 32 * (8 / g) : 128;
  const size_t per = 2 * (size_t)rowb + 16;  // a padded key row and a value row
  const size_t budget = 160 * 1024;
  int ring = 4;
  while (ring > 2 && ring * tp * per > budget) --ring;
  while (tp > 32 && ring * tp * per > budget) tp -= 32;
  return {tp, ring};
}

LLM_D void cp_async16(void* smem, const void* gmem) {
  const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
LLM_D void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N> LLM_D void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

LLM_D void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
LLM_D uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// a float in the shared memory of CTA `rank` of this cluster, at the address `p` has here
LLM_D float ld_cluster(const float* p, uint32_t rank) {
  uint32_t local = (uint32_t)__cvta_generic_to_shared(p), remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}

template <int KT> LLM_D float2 load2(const void* base, int idx) {
  if constexpr (KT == 0) {
    return *reinterpret_cast<const float2*>((const float*)base + idx);
  } else {
    const uint32_t u = *reinterpret_cast<const uint32_t*>((const uint16_t*)base + idx);
    return make_float2(bf16_lo(u), bf16_hi(u));
  }
}

template <int KT, int HD>
struct AttnSmem {
  static constexpr int ES = Elem<KT>::bytes;
  static constexpr int ROWB = HD * ES;    // bytes of one cached row
  static constexpr int KPAD = ROWB + 16;  // padded key row: lanes reading different rows do not collide
  // qs [g][HD] | tiles: kbuf [ring][TP][KPAD], vbuf [ring][TP][ROWB] | sw [g][TP] | m, l, corr [g] |
  // part [g][HD+2] | fac [g][kAttnMaxCluster]
  static LLM_HD size_t tiles(int g, int ns) {
    const TileCfg tc = tile_cfg(g, ROWB);
    size_t t = (size_t)tc.ring * tc.tp * KPAD + (size_t)tc.ring * tc.tp * ROWB;
    if (t < (size_t)g * ns * 8) t = (size_t)g * ns * 8;  // the global merge reuses the tile space
    return t;
  }
  static LLM_HD size_t bytes(int g, int ns) {
    return (size_t)g * HD * 4 + tiles(g, ns) + (size_t)g * tile_cfg(g, ROWB).tp * 4 + 3 * (size_t)g * 4 +
           (size_t)g * (HD + 2) * 4 + (size_t)g * kAttnMaxCluster * 4;
  }
};

// KT: cache element type (0 f32, 1 bf16); HD: head size; CLUSTER: splits merged in a cluster
template <int KT, int HD, bool CLUSTER>
__global__ void __launch_bounds__(kAttnThreads) attn_decode_kernel(const AttnArgs a) {
  using S = AttnSmem<KT, HD>;
  constexpr int ROWB = S::ROWB, KPAD = S::KPAD, CPR = ROWB / 16, EPC = 16 / S::ES;
  extern __shared__ __align__(16) unsigned char smraw[];

  const int split = blockIdx.x, j = blockIdx.y, b = blockIdx.z;
  const int g = a.g, H = a.kv * a.g;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const TileCfg tc = tile_cfg(g, ROWB);
  const int TP = tc.tp, NR = tc.ring;

  float* qs = reinterpret_cast<float*>(smraw);
  unsigned char* kbuf = smraw + (size_t)g * HD * 4;
  unsigned char* vbuf = kbuf + (size_t)NR * TP * KPAD;
  float* sw = reinterpret_cast<float*>(kbuf + S::tiles(g, a.ns));  // scores, then weights [g][TP]
  float* mst = sw + g * TP;
  float* lst = mst + g;
  float* cst = lst + g;
  float* mypart = cst + g;                // [g][HD+2]: unnormalized o, m, l
  float* fac = mypart + g * (HD + 2);     // [g][kAttnMaxCluster]
  __shared__ int s_last;

  grid_dep_wait();
  grid_dep_launch();

  // positions 0..t in contiguous slices of at least kMinChunk
  const int t = a.step->pos;
  const int npos = t + 1;
  int chunk = (npos + a.ns - 1) / a.ns;
  chunk = (chunk + 31) & ~31;
  if (chunk < kMinChunk) chunk = kMinChunk;
  const int nact = (npos + chunk - 1) / chunk;
  if (!CLUSTER && split >= nact) return;  // (a cluster's CTAs all take part in its barriers)
  const int p0 = split * chunk;
  const int p1 = min(npos, p0 + chunk);

  // output ownership: pairs (head, 2 dimensions); T threads per pair split the positions
  const int pairs = g * HD / 2;
  int T = 1;
  while (T * 2 * pairs <= kAttnThreads) T *= 2;
  const int npt = pairs > kAttnThreads ? (pairs + kAttnThreads - 1) / kAttnThreads : 1;
  const int sub = tid % T;
  float o[kMaxPairs][2];
#pragma unroll
  for (int k = 0; k < kMaxPairs; ++k) o[k][0] = o[k][1] = 0.f;

  const size_t head_off = (((size_t)b * a.kv + j) * a.cap) * HD;  // element offset of position 0
  const unsigned char* kg = (const unsigned char*)a.kc + head_off * S::ES;
  const unsigned char* vg = (const unsigned char*)a.vc + head_off * S::ES;
  auto stage = [&](int buf, int tb) {
    const int rows = min(TP, p1 - tb);
    for (int i = tid; i < rows * CPR; i += kAttnThreads) {
      const int r = i / CPR, c = i - r * CPR;
      cp_async16(kbuf + ((size_t)buf * TP + r) * KPAD + c * 16, kg + (size_t)(tb + r) * ROWB + c * 16);
      cp_async16(vbuf + ((size_t)buf * TP + r) * ROWB + c * 16, vg + (size_t)(tb + r) * ROWB + c * 16);
    }
  };

  // the first NR - 1 tiles go out before anything else, then the queries
  const int ntiles = p0 < p1 ? (p1 - p0 + TP - 1) / TP : 0;
  for (int r = 0; r < NR - 1; ++r) {
    if (r < ntiles) stage(r, p0 + r * TP);
    cp_async_commit();
  }
  // queries of the group: 16-byte loads issued together
  {
    const float4* src = reinterpret_cast<const float4*>(a.q + (size_t)b * a.q_stride + (size_t)j * g * HD);
    float4* dst = reinterpret_cast<float4*>(qs);
    const int n4 = g * HD / 4;
    float4 v[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int i = tid + r * kAttnThreads;
      if (i < n4) v[r] = src[i];
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int i = tid + r * kAttnThreads;
      if (i < n4) dst[i] = v[r];
    }
  }
  for (int h = tid; h < g; h += kAttnThreads) {
    mst[h] = -INFINITY;
    lst[h] = 0.f;
  }

  __syncthreads();
  for (int it = 0; it < ntiles; ++it) {
    const int tb = p0 + it * TP;
    const int nv = min(TP, p1 - tb);
    if (it + NR - 1 < ntiles) stage((it + NR - 1) % NR, tb + (NR - 1) * TP);
    cp_async_commit();
    // tile it has landed once at most NR - 1 of the groups committed so far are pending
    if (NR == 4) cp_async_wait<3>();
    else if (NR == 3) cp_async_wait<2>();
    else cp_async_wait<1>();
    __syncthreads();
    const int buf = it % NR;
    // scores: one (head, position) per thread
    for (int item = tid; item < g * TP; item += kAttnThreads) {
      const int h = item / TP, p = item - h * TP;
      float s = -INFINITY;
      if (p < nv) {
        const unsigned char* krow = kbuf + ((size_t)buf * TP + p) * KPAD;
        const float* qh = qs + h * HD;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
        for (int c = 0; c < CPR; ++c) {
          const uint4 kv4 = *reinterpret_cast<const uint4*>(krow + c * 16);
          float kf[EPC];
          unpack16<KT>(kv4, kf);
          const float4* q4 = reinterpret_cast<const float4*>(qh + c * EPC);
#pragma unroll
          for (int e4 = 0; e4 < EPC / 4; ++e4) {
            const float4 qv = q4[e4];
            float& r = acc[(c * (EPC / 4) + e4) & 3];
            r = fmaf(qv.x, kf[4 * e4 + 0], r);
            r = fmaf(qv.y, kf[4 * e4 + 1], r);
            r = fmaf(qv.z, kf[4 * e4 + 2], r);
            r = fmaf(qv.w, kf[4 * e4 + 3], r);
          }
        }
        s = ((acc[0] + acc[1]) + (acc[2] + acc[3])) * a.scale;
      }
      sw[h * TP + p] = s;
    }
    __syncthreads();
    // online softmax: one warp per head
    for (int h = warp; h < g; h += kAttnWarps) {
      float mx = -INFINITY;
      for (int p = lane; p < TP; p += 32) mx = fmaxf(mx, sw[h * TP + p]);
      mx = warp_max(mx);
      const float mold = mst[h];
      const float mnew = fmaxf(mold, mx);  // finite: the tile holds at least one position
      const float corr = mold == -INFINITY ? 0.f : expf(mold - mnew);
      float sum = 0.f;
      for (int p = lane; p < TP; p += 32) {
        const float sc = sw[h * TP + p];
        const float w = sc == -INFINITY ? 0.f : expf(sc - mnew);
        sw[h * TP + p] = w;
        sum += w;
      }
      sum = warp_sum(sum);
      if (lane == 0) {
        mst[h] = mnew;
        lst[h] = lst[h] * corr + sum;
        cst[h] = corr;
      }
    }
    __syncthreads();
    // weighted values
#pragma unroll
    for (int k = 0; k < kMaxPairs; ++k) {
      if (k >= npt) break;
      const int pi = T == 1 ? tid + k * kAttnThreads : tid / T;
      if (pi < pairs) {
        const int h = pi / (HD / 2), e = 2 * (pi - h * (HD / 2));
        const float c = cst[h];
        float o0 = o[k][0] * c, o1 = o[k][1] * c;
        const float* wh = sw + h * TP;
        const unsigned char* vb = vbuf + (size_t)buf * TP * ROWB;
#pragma unroll 4
        for (int p = sub; p < nv; p += T) {
          const float w = wh[p];
          const float2 v2 = load2<KT>(vb + (size_t)p * ROWB, e);
          o0 = fmaf(w, v2.x, o0);
          o1 = fmaf(w, v2.y, o1);
        }
        o[k][0] = o0;
        o[k][1] = o1;
      }
    }
    __syncthreads();  // this buffer is refilled NR - 1 tiles later
  }
  cp_async_wait<0>();

  // the CTA's partial: sum the position sub-splits, then (o, m, l) per head
  if (T > 1) {
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      float v = o[0][r];
      for (int off = T >> 1; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      o[0][r] = v;
    }
  }
  if (sub == 0) {
#pragma unroll
    for (int k = 0; k < kMaxPairs; ++k) {
      if (k >= npt) break;
      const int pi = T == 1 ? tid + k * kAttnThreads : tid / T;
      if (pi < pairs) {
        const int h = pi / (HD / 2), e = 2 * (pi - h * (HD / 2));
        mypart[h * (HD + 2) + e] = o[k][0];
        mypart[h * (HD + 2) + e + 1] = o[k][1];
      }
    }
  }
  for (int h = tid; h < g; h += kAttnThreads) {
    mypart[h * (HD + 2) + HD] = mst[h];
    mypart[h * (HD + 2) + HD + 1] = lst[h];
  }
  float* outb = a.out + (size_t)b * a.out_stride + (size_t)j * g * HD;

  if constexpr (CLUSTER) {
    // ---- merge inside the cluster (CTA rank = split) through distributed shared memory ----
    const int nr = a.ns;
    cluster_sync_all();
    if (cluster_rank() == 0) {
      for (int h = tid; h < g; h += kAttnThreads) {
        float M = -INFINITY;
        for (int r = 0; r < nr; ++r) M = fmaxf(M, ld_cluster(mypart + h * (HD + 2) + HD, r));
        float L = 0.f;
        for (int r = 0; r < nr; ++r) {
          const float mr = ld_cluster(mypart + h * (HD + 2) + HD, r);
          const float f = mr == -INFINITY ? 0.f : expf(mr - M);
          fac[h * kAttnMaxCluster + r] = f;
          L += ld_cluster(mypart + h * (HD + 2) + HD + 1, r) * f;
        }
        const float rl = 1.0f / L;
        for (int r = 0; r < nr; ++r) fac[h * kAttnMaxCluster + r] *= rl;
      }
      __syncthreads();
      for (int idx = tid; idx < g * HD; idx += kAttnThreads) {
        const int h = idx / HD, e = idx - h * HD;
        float ov[kAttnMaxCluster];
#pragma unroll
        for (int r = 0; r < kAttnMaxCluster; ++r)
          if (r < nr) ov[r] = ld_cluster(mypart + h * (HD + 2) + e, r);
        float O = 0.f;
#pragma unroll
        for (int r = 0; r < kAttnMaxCluster; ++r)
          if (r < nr) O = fmaf(fac[h * kAttnMaxCluster + r], ov[r], O);
        outb[(size_t)h * HD + e] = O;
      }
    }
    cluster_sync_all();  // the other CTAs keep their shared memory until CTA 0 has read it
    return;
  } else {
    // ---- global partials; the last CTA of this (row, kv head) merges them in order ----
    __syncthreads();
    float* pglob = a.part + (((size_t)b * H + (size_t)j * g) * a.ns) * (HD + 2);
    for (int idx = tid; idx < g * (HD + 2); idx += kAttnThreads) {
      const int h = idx / (HD + 2), e = idx - h * (HD + 2);
      pglob[((size_t)h * a.ns + split) * (HD + 2) + e] = mypart[idx];
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
    float* fm = reinterpret_cast<float*>(kbuf);  // [g][nact] maxima, then factors
    float* fl = fm + g * nact;                   // [g][nact] sums
    for (int idx = tid; idx < g * nact; idx += kAttnThreads) {
      const int h = idx / nact, s2 = idx - h * nact;
      const float* pp = pglob + ((size_t)h * a.ns + s2) * (HD + 2);
      fm[idx] = __ldcg(pp + HD);
      fl[idx] = __ldcg(pp + HD + 1);
    }
    __syncthreads();
    for (int h = warp; h < g; h += kAttnWarps) {
      float M = -INFINITY;
      for (int s2 = lane; s2 < nact; s2 += 32) M = fmaxf(M, fm[h * nact + s2]);
      M = warp_max(M);
      float L = 0.f;
      for (int s2 = lane; s2 < nact; s2 += 32) {
        const float ms = fm[h * nact + s2];
        const float f = ms == -INFINITY ? 0.f : expf(ms - M);
        fm[h * nact + s2] = f;
        L += fl[h * nact + s2] * f;
      }
      L = warp_sum(L);
      const float rl = 1.0f / L;
      for (int s2 = lane; s2 < nact; s2 += 32) fm[h * nact + s2] *= rl;
    }
    __syncthreads();
    for (int idx = tid; idx < g * HD; idx += kAttnThreads) {
      const int h = idx / HD, e = idx - h * HD;
      const float* pb = pglob + (size_t)h * a.ns * (HD + 2) + e;
      float O = 0.f;
      int s2 = 0;
      for (; s2 + 8 <= nact; s2 += 8) {
        float ov[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) ov[q] = __ldcg(pb + (size_t)(s2 + q) * (HD + 2));
#pragma unroll
        for (int q = 0; q < 8; ++q) O = fmaf(fm[h * nact + s2 + q], ov[q], O);
      }
      for (; s2 < nact; ++s2) O = fmaf(fm[h * nact + s2], __ldcg(pb + (size_t)s2 * (HD + 2)), O);
      outb[(size_t)h * HD + e] = O;
    }
    if (tid == 0) a.ticket[(size_t)b * a.kv + j] = 0u;
  }
}

// ---------------------------------------------------------------------------------------

using AttnFn = void (*)(const AttnArgs);

template <int KT, bool CL>
static AttnFn pick_hd(int hd, size_t* smem, int g, int ns) {
  switch (hd) {
    case 16: *smem = AttnSmem<KT, 16>::bytes(g, ns); return attn_decode_kernel<KT, 16, CL>;
    case 32: *smem = AttnSmem<KT, 32>::bytes(g, ns); return attn_decode_kernel<KT, 32, CL>;
    case 64: *smem = AttnSmem<KT, 64>::bytes(g, ns); return attn_decode_kernel<KT, 64, CL>;
    case 128: *smem = AttnSmem<KT, 128>::bytes(g, ns); return attn_decode_kernel<KT, 128, CL>;
    case 256: *smem = AttnSmem<KT, 256>::bytes(g, ns); return attn_decode_kernel<KT, 256, CL>;
    default: return nullptr;
  }
}

static AttnFn pick(int kt, bool cl, int hd, size_t* smem, int g, int ns) {
  if (kt) return cl ? pick_hd<1, true>(hd, smem, g, ns) : pick_hd<1, false>(hd, smem, g, ns);
  return cl ? pick_hd<0, true>(hd, smem, g, ns) : pick_hd<0, false>(hd, smem, g, ns);
}

static int g_max_cluster = 8;  // 16 once attn_prepare finds the device can schedule it
int attn_max_cluster() { return g_max_cluster; }

bool attn_supported(int hd, int g) {
  return (hd == 16 || hd == 32 || hd == 64 || hd == 128 || hd == 256) && g >= 1 && g <= 16 &&
         g * hd <= 2 * kAttnThreads * kMaxPairs;
}

cudaError_t attn_prepare(int max_smem_optin) {
  for (int kt = 0; kt < 2; ++kt)
    for (int cl = 0; cl < 2; ++cl)
      for (int hd : {16, 32, 64, 128, 256}) {
        size_t sm = 0;
        AttnFn fn = pick(kt, cl != 0, hd, &sm, 1, 1);
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, fn);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem_optin - (int)fa.sharedSizeBytes);
        if (e != cudaSuccess) return e;
      }
  // clusters of 16 (beyond the portable 8) where the device can run them with this kernel
  g_max_cluster = 8;
  for (int kt = 0; kt < 2; ++kt)
    for (int hd : {16, 32, 64, 128, 256}) {
      size_t sm = 0;
      AttnFn fn = pick(kt, true, hd, &sm, 1, 1);
      if (cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
        cudaGetLastError();
        return cudaSuccess;
      }
    }
  {
    size_t sm = 0;
    AttnFn fn = pick(1, true, 128, &sm, 4, 16);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(16, 8, 1);
    cfg.blockDim = dim3(kAttnThreads);
    cfg.dynamicSmemBytes = sm;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 16;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int nclusters = 0;
    if (cudaOccupancyMaxActiveClusters(&nclusters, fn, &cfg) == cudaSuccess && nclusters >= 1) g_max_cluster = 16;
    cudaGetLastError();
  }
  return cudaSuccess;
}

int attn_splits(int B, int kv, int cap, int num_sms) {
  // enough CTAs to cover the GPU twice, each split at least kMinChunk positions of the capacity;
  // up to kAttnMaxCluster splits merge inside a cluster, which is cheaper than a global merge,
  // so a short cache uses one cluster of kAttnMaxCluster splits instead of more global ones
  int ns = (2 * num_sms + B * kv - 1) / (B * kv);
  int by_cap = cap / kMinChunk;
  if (by_cap < 1) by_cap = 1;
  if (ns > by_cap) ns = by_cap;
  const int mc = attn_max_cluster();
  if (ns > mc && cap / mc <= 4096) ns = mc;
  if (ns > 1024) ns = 1024;
  if (ns < 1) ns = 1;
  return ns;
}

cudaError_t launch_attn(const AttnArgs& a, int kt, cudaStream_t s, bool pdl) {
  const bool cl = a.ns <= attn_max_cluster();
  size_t smem = 0;
  AttnFn fn = pick(kt, cl, a.hd, &smem, a.g, a.ns);
  if (!fn) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.ns, a.kv, a.B);
  cfg.blockDim = dim3(kAttnThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  int na = 1;
  if (cl) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = a.ns;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    na = 2;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, fn, a);
}

}  // namespace llm
