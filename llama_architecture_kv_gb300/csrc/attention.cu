// Grouped-query attention of one decode step over the KV cache (split-K flash decode).
//
// Computes, for every batch row b and query head h = j*g + i (group j reads key/value head j:
// bend-ml-llama "Grouped-query attention", gqa_head), the output
//   o_h = sum_{p=0..t} softmax_p(scale * q_h . K_j[p]) V_j[p],  scale = 1/sqrt(hd),
// over exactly the cache positions 0..t, t = the row's position (bend-ml-llama law causal;
// Llama 3.1 8B card, attention.linnet decode: seen[s] = s <= pos).
//
// Layout: the cache of one layer is [max_batch][kv][cap][hd] (attention.linnet cache_k), so the
// positions of one (row, key/value head) are contiguous; in a paged step a row's positions are
// found 64 at a time through its page table (cache_slot), and no chunk crosses a page.
// Two kernels: attn_mma_kernel (bf16 caches, head size 64 or 128; warp-level tensor-core MMAs,
// described further down) and attn_decode_kernel (everything else), described here.
// attn_decode_kernel grid: (splits, kv, B); a CTA takes a
// contiguous slice of positions of one (row, kv head) and its warps take 32-position chunks of
// it in turn.  Each warp streams its own chunks through a private ring of shared-memory buffers
// (a TMA tensor copy of the keys with the 128-byte swizzle, a bulk copy of the values; one
// mbarrier per buffer), so warps never wait for one another inside the loop.  Per chunk:
//   scores   lane = position: the g dot products q_h . K[p] (the key row is read once for the
//            whole group; the queries are shared-memory broadcasts; the swizzle keeps the 32
//            lanes' row reads on distinct banks);
//   softmax  per head, across the warp: chunk maximum, running max m, weights exp(s - m),
//            per-lane running sums l, rescaled when m grows;
//   values   lane = hd/32 consecutive dimensions of every head; per position one value load and
//            one broadcast of the g weights.
// The warps' (o, m, l) merge in warp order, then the splits of one (row, kv head) merge by
// log-sum-exp in split order (the result does not depend on timing): up to attn_max_cluster()
// splits form one thread-block cluster and CTA 0 reads the others' partials through distributed
// shared memory; more splits (long contexts) write partials to global memory and the last CTA to
// finish -- found with an atomic ticket, nobody waits -- merges them.
// Chunks that lie entirely below position t were written by earlier steps, so their copies start
// before the wait on the previous kernel (which writes position t).
#include <map>
#include <mutex>
#include <tuple>

#include "attention.cuh"
#include "gemm.cuh"
#include "tc.cuh"

namespace llm {

constexpr int kChunk = 32;      // positions per chunk: one per lane
constexpr int kMinChunk = 64;   // fewest positions a split takes
constexpr int kAttnMaxThreads = 128;
constexpr uint64_t kAttnWaitCycles = 1000000000ull;  // about 0.5 s at 2 GHz

template <int KT, int HD>
struct AttnShape {
  static constexpr int ES = Elem<KT>::bytes;
  static constexpr int ROWB = HD * ES;               // bytes of one cached row
  static constexpr bool SWZ = ROWB >= 128;           // keys staged with the 128-byte swizzle
  static constexpr int BOXB = SWZ ? 128 : ROWB;      // bytes of a key row inside one copy box
  static constexpr int NBOX = ROWB / BOXB;           // boxes per key chunk
  static constexpr int BUF = 2 * kChunk * ROWB;      // one chunk: keys, then values
  static constexpr int CPR = ROWB / 16;              // 16-byte pieces of a row
  static constexpr int EPC = 16 / ES;                // elements per piece
  static constexpr int DPL = HD >= 32 ? HD / 32 : 1; // value dimensions per lane
  static constexpr int VL = HD >= 32 ? 32 : HD;      // lanes that hold value dimensions
};

// warps per CTA and buffers per warp for a chunk of buf bytes (within 192 KB)
struct AttnGeom {
  int nw, nr;
};
LLM_HD AttnGeom attn_geom(int buf) {
  const int budget = 192 * 1024;
  int nw = 4;
  while (nw > 1 && nw * 2 * buf > budget) nw >>= 1;
  int nr = 3;
  while (nr > 2 && nw * nr * buf > budget) --nr;
  return {nw, nr};
}

template <int KT, int HD>
LLM_HD size_t attn_region(int g, int ns) {  // ring buffers; the global merge reuses them
  const AttnGeom geo = attn_geom(AttnShape<KT, HD>::BUF);
  size_t r = (size_t)geo.nw * geo.nr * AttnShape<KT, HD>::BUF;
  if (r < (size_t)g * ns * 8) r = (size_t)g * ns * 8;
  return (r + 1023) & ~(size_t)1023;
}

template <int KT, int HD, int GM>
LLM_HD size_t attn_smem(int g, int ns) {
  const AttnGeom geo = attn_geom(AttnShape<KT, HD>::BUF);
  size_t s = 1024 + attn_region<KT, HD>(g, ns);
  s += (size_t)g * HD * 4;                    // queries
  s += (size_t)geo.nw * kChunk * GM * 4;      // weights of the chunk in use, per warp
  s += (size_t)geo.nw * g * (HD + 2) * 4;     // warp partials
  s += (size_t)g * (HD + 2) * 4;              // CTA partial
  s += (size_t)g * kAttnMaxCluster * 4;       // merge factors
  s = (s + 7) & ~(size_t)7;
  s += (size_t)geo.nw * geo.nr * 8;           // mbarriers
  return s;
}

LLM_D void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
LLM_D uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
LLM_D void cluster_arrive_relaxed() { asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory"); }
LLM_D void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
LLM_D void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
// the address in CTA `rank`'s shared memory of the one `local` has here
LLM_D uint32_t map_rank(uint32_t local, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
  return remote;
}
LLM_D void st_cluster(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
// a float in the shared memory of CTA `rank` of this cluster, at the address `p` has here
LLM_D float ld_cluster(const float* p, uint32_t rank) {
  uint32_t local = (uint32_t)__cvta_generic_to_shared(p), remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}

// DPL consecutive cached elements as f32
template <int KT, int DPL>
LLM_D void load_dims(const unsigned char* p, float (&v)[DPL]) {
  if constexpr (KT == 1) {
    if constexpr (DPL == 1) {
      v[0] = bf16_to_f32(*reinterpret_cast<const uint16_t*>(p));
    } else if constexpr (DPL == 2) {
      const uint32_t u = *reinterpret_cast<const uint32_t*>(p);
      v[0] = bf16_lo(u);
      v[1] = bf16_hi(u);
    } else if constexpr (DPL == 4) {
      const uint2 u = *reinterpret_cast<const uint2*>(p);
      v[0] = bf16_lo(u.x); v[1] = bf16_hi(u.x); v[2] = bf16_lo(u.y); v[3] = bf16_hi(u.y);
    } else {
#pragma unroll
      for (int q = 0; q < DPL; q += 8) {
        const uint4 u = *reinterpret_cast<const uint4*>(p + q * 2);
        v[q + 0] = bf16_lo(u.x); v[q + 1] = bf16_hi(u.x); v[q + 2] = bf16_lo(u.y); v[q + 3] = bf16_hi(u.y);
        v[q + 4] = bf16_lo(u.z); v[q + 5] = bf16_hi(u.z); v[q + 6] = bf16_lo(u.w); v[q + 7] = bf16_hi(u.w);
      }
    }
  } else {
    if constexpr (DPL == 1) {
      v[0] = *reinterpret_cast<const float*>(p);
    } else if constexpr (DPL == 2) {
      const float2 f = *reinterpret_cast<const float2*>(p);
      v[0] = f.x; v[1] = f.y;
    } else {
#pragma unroll
      for (int q = 0; q < DPL; q += 4) {
        const float4 f = *reinterpret_cast<const float4*>(p + q * 4);
        v[q] = f.x; v[q + 1] = f.y; v[q + 2] = f.z; v[q + 3] = f.w;
      }
    }
  }
}

// Combines the warps' partials (wpart [NW][g][HD+2]: o, m, l) into the CTA's partial, then
// merges the splits of this (row, kv head) and writes the output.  Every thread calls it.
template <int HD>
LLM_D void attn_finish(const AttnArgs& a, unsigned char* base, const float* wpart, float* mypart, float* fac, int nact,
                       int split, int b, int j) {
  const int g = a.g, H = a.kv * a.g;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int NT = blockDim.x, NW = NT >> 5;
  __shared__ int s_last;
  for (int idx = tid; idx < g * (HD + 2); idx += NT) {
    const int h = idx / (HD + 2), e = idx - h * (HD + 2);
    float M = -INFINITY;
    for (int w = 0; w < NW; ++w) M = fmaxf(M, wpart[(w * g + h) * (HD + 2) + HD]);
    float r = M;
    if (e != HD) {
      r = 0.f;
      for (int w = 0; w < NW; ++w) {
        const float mw = wpart[(w * g + h) * (HD + 2) + HD];
        const float f = mw == -INFINITY ? 0.f : expf(mw - M);
        r = fmaf(f, wpart[(w * g + h) * (HD + 2) + e], r);
      }
    }
    mypart[idx] = r;
  }
  __syncthreads();
  float* outb = a.out + (size_t)b * a.out_stride + (size_t)j * g * HD;

  if (a.cluster) {
    // ---- merge inside the cluster (CTA rank = split) through distributed shared memory ----
    const int nr = a.ns;
    cluster_sync_all();
    if (cluster_rank() == 0) {
      // every rank's (m, l) of every head, fetched together (the ring is idle scratch now)
      float* cm = reinterpret_cast<float*>(base);  // [g][nr]
      float* cl = cm + g * nr;                     // [g][nr]
      for (int idx = tid; idx < g * nr; idx += NT) {
        const int h = idx / nr, r = idx - h * nr;
        cm[idx] = ld_cluster(mypart + h * (HD + 2) + HD, r);
        cl[idx] = ld_cluster(mypart + h * (HD + 2) + HD + 1, r);
      }
      __syncthreads();
      for (int h = tid; h < g; h += NT) {
        float M = -INFINITY;
        for (int r = 0; r < nr; ++r) M = fmaxf(M, cm[h * nr + r]);
        float L = 0.f;
        for (int r = 0; r < nr; ++r) {
          const float mr = cm[h * nr + r];
          const float f = mr == -INFINITY ? 0.f : expf(mr - M);
          fac[h * kAttnMaxCluster + r] = f;
          L += cl[h * nr + r] * f;
        }
        const float rl = 1.0f / L;
        for (int r = 0; r < nr; ++r) fac[h * kAttnMaxCluster + r] *= rl;
      }
      __syncthreads();
      for (int idx = tid; idx < g * HD; idx += NT) {
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
  }
  // ---- global partials; the last CTA of this (row, kv head) merges them in order ----
  float* pglob = a.part + (((size_t)b * H + (size_t)j * g) * a.ns) * (HD + 2);
  for (int idx = tid; idx < g * (HD + 2); idx += NT) {
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
  float* fm = reinterpret_cast<float*>(base);  // [g][nact] maxima, then factors (the ring is idle)
  float* fl = fm + g * nact;                   // [g][nact] sums
  for (int idx = tid; idx < g * nact; idx += NT) {
    const int h = idx / nact, s2 = idx - h * nact;
    const float* pp = pglob + ((size_t)h * a.ns + s2) * (HD + 2);
    fm[idx] = __ldcg(pp + HD);
    fl[idx] = __ldcg(pp + HD + 1);
  }
  __syncthreads();
  for (int h = warp; h < g; h += NW) {
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
  for (int idx = tid; idx < g * HD; idx += NT) {
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

// KT: cache element type (0 f32, 1 bf16); HD: head size; GM: group size bound (g <= GM)
template <int KT, int HD, int GM>
__global__ void __launch_bounds__(kAttnMaxThreads)
    attn_decode_kernel(const __grid_constant__ CUtensorMap kmap, const AttnArgs a) {
  using S = AttnShape<KT, HD>;
  constexpr int ROWB = S::ROWB, BUF = S::BUF, DPL = S::DPL;
  extern __shared__ unsigned char araw[];
  const uint32_t s_raw = smem_u32(araw);
  unsigned char* base = araw + (((s_raw + 1023u) & ~1023u) - s_raw);
  const uint32_t s_base = smem_u32(base);

  const int split = blockIdx.x, j = blockIdx.y, b = blockIdx.z;
  const int g = a.g;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int NT = blockDim.x, NW = NT >> 5;
  const int NR = attn_geom(BUF).nr;
  const size_t region = attn_region<KT, HD>(g, a.ns);
  float* qs = reinterpret_cast<float*>(base + region);  // [g][HD]
  float* wb = qs + g * HD;                               // [NW][32][GM]
  float* wpart = wb + NW * kChunk * GM;                  // [NW][g][HD+2]
  float* mypart = wpart + NW * g * (HD + 2);             // [g][HD+2]: unnormalized o, m, l
  float* fac = mypart + g * (HD + 2);                    // [g][kAttnMaxCluster]
  const uint32_t bars = (smem_u32(fac + g * kAttnMaxCluster) + 7u) & ~7u;

  // positions ts..t of row b (ts = 0 but in packed passes) in contiguous slices of at least
  // kMinChunk (multiples of 32), starting from ts rounded down to 32 so that chunks stay aligned
  // (and inside pages); positions below ts are masked
  const int t = row_pos(a.step, b);
  const int ts = row_start(a.step, b), tw = row_wfirst(a.step, b);
  const int pbase = ts & ~(kChunk - 1);
  const int npos = t + 1 - pbase;
  int chunk = (npos + a.ns - 1) / a.ns;
  chunk = (chunk + 31) & ~31;
  if (chunk < kMinChunk) chunk = kMinChunk;
  const int nact = (npos + chunk - 1) / chunk;
  if (!a.cluster && split >= nact) return;  // (a cluster's CTAs all take part in its barriers)
  const int p0 = pbase + split * chunk;
  const int p1 = min(t + 1, p0 + chunk);
  const int nch = p0 < p1 ? (p1 - p0 + kChunk - 1) / kChunk : 0;
  const int cnt = nch > warp ? (nch - warp + NW - 1) / NW : 0;  // chunks of this warp

  if (tid == 0) {
    for (int i = 0; i < NW * NR; ++i) mbar_init(bars + 8u * i, 1);
    mbar_fence_init();
  }
  __syncthreads();

  auto issue = [&](int k) {  // lane 0: chunk k of this warp into its ring slot
    const int slot = k % NR;
    const int pb = p0 + (warp + k * NW) * kChunk;
    const int nv = min(kChunk, p1 - pb);
    // the cache row and position holding position pb (a chunk never crosses a page)
    int r, pp;
    cache_slot(a.step, a.cap, b, pb, r, pp);
    const int krow = a.krow0 + (r * a.kv + j) * a.cap + pp;  // key-map row
    const unsigned char* vsrc = (const unsigned char*)a.vc + ((size_t)(r * a.kv + j) * a.cap + pp) * ROWB;
    const uint32_t bar = bars + 8u * (warp * NR + slot);
    const uint32_t dst = s_base + (uint32_t)((warp * NR + slot) * BUF);
    fence_proxy_async_smem();
    mbar_expect_tx(bar, (uint32_t)(kChunk * ROWB + nv * ROWB));
#pragma unroll
    for (int bx = 0; bx < S::NBOX; ++bx)
      tma_load_2d(dst + (uint32_t)(bx * kChunk * S::BOXB), &kmap, bar, bx * (S::BOXB / S::ES), krow);
    bulk_load(dst + (uint32_t)(kChunk * ROWB), vsrc, (uint32_t)(nv * ROWB), bar);
  };
  // chunks below the first position this step writes in the row do not depend on the previous
  // kernel
  const int npre = cnt < NR ? cnt : NR;
  int issued = 0;
  if (lane == 0) {
    while (issued < npre) {
      const int pb = p0 + (warp + issued * NW) * kChunk;
      if (pb + min(kChunk, p1 - pb) > tw) break;  // holds a position written by this step
      issue(issued++);
    }
  }
  grid_dep_wait();
  grid_dep_launch();
  if (lane == 0)
    while (issued < npre) issue(issued++);
  {
    const float4* src = reinterpret_cast<const float4*>(a.q + (size_t)b * a.q_stride + (size_t)j * g * HD);
    float4* dst = reinterpret_cast<float4*>(qs);
    for (int i = tid; i < g * HD / 4; i += NT) dst[i] = src[i];
  }
  __syncthreads();

  float m[GM], l[GM], o[GM][DPL];
#pragma unroll
  for (int h = 0; h < GM; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.f;
#pragma unroll
    for (int e = 0; e < DPL; ++e) o[h][e] = 0.f;
  }
  float* wme = wb + warp * kChunk * GM;
  bool ok = true;
  int consumed = 0;
  for (int k = 0; k < cnt; ++k) {
    const int slot = k % NR;
    const uint32_t bar = bars + 8u * (warp * NR + slot);
    ok = __all_sync(0xffffffffu, mbar_wait(bar, (uint32_t)(k / NR) & 1u, kAttnWaitCycles));
    if (!ok) break;
    consumed = k + 1;
    const int pb = p0 + (warp + k * NW) * kChunk;
    const int nv = min(kChunk, p1 - pb);
    const unsigned char* kreg = base + (size_t)(warp * NR + slot) * BUF;
    const unsigned char* vreg = kreg + kChunk * ROWB;
    const bool valid = lane < nv && pb + lane >= ts;
    // scores: lane = position
    float acc[GM][2];
#pragma unroll
    for (int h = 0; h < GM; ++h) acc[h][0] = acc[h][1] = 0.f;
#pragma unroll
    for (int c = 0; c < S::CPR; ++c) {
      const unsigned char* kp;
      if constexpr (S::SWZ)
        kp = kreg + (c >> 3) * (kChunk * 128) + lane * 128 + (((c & 7) ^ (lane & 7)) << 4);
      else
        kp = kreg + lane * ROWB + c * 16;
      float kf[S::EPC];
      unpack16<KT>(*reinterpret_cast<const uint4*>(kp), kf);
#pragma unroll
      for (int h = 0; h < GM; ++h) {
        if (h < g) {
          const float4* q4 = reinterpret_cast<const float4*>(qs + h * HD + c * S::EPC);
#pragma unroll
          for (int e4 = 0; e4 < S::EPC / 4; ++e4) {
            const float4 qv = q4[e4];
            float& r = acc[h][c & 1];
            r = fmaf(qv.x, kf[4 * e4 + 0], r);
            r = fmaf(qv.y, kf[4 * e4 + 1], r);
            r = fmaf(qv.z, kf[4 * e4 + 2], r);
            r = fmaf(qv.w, kf[4 * e4 + 3], r);
          }
        }
      }
    }
    // online softmax, per head across the warp
#pragma unroll
    for (int h = 0; h < GM; ++h) {
      if (h < g) {
        const float s = valid ? (acc[h][0] + acc[h][1]) * a.scale : -INFINITY;
        const float mnew = fmaxf(m[h], warp_max(s));  // finite: every chunk holds a position of the range
        const float corr = m[h] == -INFINITY ? 0.f : expf(m[h] - mnew);
        const float w = valid ? expf(s - mnew) : 0.f;
        l[h] = fmaf(l[h], corr, w);
#pragma unroll
        for (int e = 0; e < DPL; ++e) o[h][e] *= corr;
        m[h] = mnew;
        wme[lane * GM + h] = w;
      }
    }
    __syncwarp();
    // values: lane = DPL dimensions of every head
    if (lane < S::VL) {
      const unsigned char* vp = vreg + lane * DPL * S::ES;
#pragma unroll 2
      for (int pp = ts > pb ? ts - pb : 0; pp < nv; ++pp) {  // (rows below ts may not be finite)
        float wv[GM];
#pragma unroll
        for (int h4 = 0; h4 < GM; h4 += 4) {
          const float4 w4 = *reinterpret_cast<const float4*>(wme + pp * GM + h4);
          wv[h4] = w4.x; wv[h4 + 1] = w4.y; wv[h4 + 2] = w4.z; wv[h4 + 3] = w4.w;
        }
        float v[DPL];
        load_dims<KT, DPL>(vp + (size_t)pp * ROWB, v);
#pragma unroll
        for (int h = 0; h < GM; ++h)
          if (h < g)
#pragma unroll
            for (int e = 0; e < DPL; ++e) o[h][e] = fmaf(wv[h], v[e], o[h][e]);
      }
    }
    __syncwarp();
    if (lane == 0 && issued < cnt) issue(issued++);
  }
  if (!ok) {
    if (lane == 0) atomicCAS(a.status, 0, kErrDeviceTimeout);
  }
  // no copy may still be writing shared memory when the CTA moves on or exits
  if (lane == 0)
    for (int k = consumed; k < issued; ++k)
      if (!mbar_wait(bars + 8u * (warp * NR + k % NR), (uint32_t)(k / NR) & 1u, kAttnWaitCycles))
        atomicCAS(a.status, 0, kErrDeviceTimeout);
  __syncwarp();

  // the warp's partial, then the CTA's: warps merged in order
#pragma unroll
  for (int h = 0; h < GM; ++h) {
    if (h < g) {
      const float lsum = warp_sum(l[h]);
      float* wp = wpart + (warp * g + h) * (HD + 2);
      if (lane < S::VL)
#pragma unroll
        for (int e = 0; e < DPL; ++e) wp[lane * DPL + e] = o[h][e];
      if (lane == 0) {
        wp[HD] = m[h];
        wp[HD + 1] = lsum;
      }
    }
  }
  __syncthreads();
  attn_finish<HD>(a, base, wpart, mypart, fac, nact, split, b, j);
}


// ---------------------------------------------------------------------------------------
// bf16 caches, hd 64 or 128: the two contractions of a chunk on warp-level tensor-core MMAs
// (m16n8k16, bf16 in, f32 accumulate).  Rows of the MMA are the chunk's 16 positions, columns
// the query heads of the group (one 8-column tile for g <= 8, two for g <= 16), so a small group
// wastes at most half of each MMA:
//   scores  S^T[16][8] = K Q^T: K fragments by ldmatrix from the swizzled key tile, Q as bf16
//           hi + lo fragments kept in registers for the whole segment (two MMAs into separate
//           accumulators, so each query enters to about 2^-17 relative);
//   softmax per head = per column: 16 positions over the 8 lanes of one quad column;
//   values  O^T[hd][8] += V^T P^T: V fragments by transposing ldmatrix from the swizzled value
//           tile, the weights P as bf16 hi + lo B fragments gathered from the score fragments
//           with shuffles.
// ---------------------------------------------------------------------------------------

LLM_D void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
LLM_D void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
// d += a * b, m16n8k16, bf16 inputs, f32 accumulators
LLM_D void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// two f32 as bf16 hi parts (x0 in the low half) and the bf16 of what they leave over
LLM_D void split_bf16x2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(hi) : "f"(x1), "f"(x0));
  const float h0 = __uint_as_float(hi << 16), h1 = __uint_as_float(hi & 0xffff0000u);
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(lo) : "f"(__fsub_rn(x1, h1)), "f"(__fsub_rn(x0, h0)));
}

constexpr int kMmaChunk = 16;   // positions per chunk of a warp (one MMA k-step of the values)
constexpr int kMmaWarps = 8;

template <int HD>
struct MmaShape {
  static constexpr int ROWB = HD * 2;
  static constexpr int NBOX = ROWB / 128;   // 128-byte column boxes per row
  static constexpr int BUF = 2 * kMmaChunk * ROWB;
  static constexpr int QP = HD + 8;         // padded query row (elements): ldmatrix rows on distinct banks
  static constexpr int DT = HD / 16;        // 16-dimension tiles of the output
  static constexpr int KS = HD / 16;        // k-steps of the scores
};

constexpr int kMmaCluster = 8;     // CTAs per (row, kv head) in cluster mode (portable size)

// shared memory of the kernel with nr ring slots per warp
template <int HD>
LLM_HD size_t attn_mma_smem_nr(int g, int nr, bool cluster = false) {
  using M = MmaShape<HD>;
  size_t s = 1024 + (size_t)kMmaWarps * nr * M::BUF;
  s += 2 * 16 * (size_t)M::QP * 2;            // queries hi, lo
  s += (size_t)kMmaWarps * g * (HD + 2) * 4;  // warp partials
  s += (size_t)g * (HD + 2) * 4;              // CTA partial
  s += (size_t)g * 64 * 4;                    // merge factors
  if (cluster) s += (size_t)kMmaCluster * g * (HD + 2) * 4;  // cluster mode: every rank's partial
  s = (s + 7) & ~(size_t)7;
  s += (size_t)kMmaWarps * nr * 8;            // mbarriers
  return s;
}
// ring slots per warp: three for 64-dimension heads, two for 128 (measured faster than three at
// both batch 1 and 32 on the 8B shape), two wherever three would not fit
template <int HD>
LLM_HD int attn_mma_nr(int g) { return HD <= 64 && attn_mma_smem_nr<HD>(g, 3) <= 232448 - 1024 ? 3 : 2; }

constexpr int kMmaMaxSplits = 64;  // splits of one (row, kv head) the persistent kernel merges
constexpr size_t kMmaClusterMaxBytes = 1u << 20;  // most cache bytes per CTA in cluster mode

template <int HD>
LLM_HD size_t attn_mma_smem(int g, bool cluster = false) { return attn_mma_smem_nr<HD>(g, attn_mma_nr<HD>(g), cluster); }

// byte offset of 16-byte piece c of row r in a chunk tile stored as 128-byte-wide swizzled boxes
// of kMmaChunk rows
LLM_D uint32_t swz_off(int r, int c) {
  return (uint32_t)((c >> 3) * (kMmaChunk * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// Persistent and evenly split: the (row, kv head, 16-position chunk) sequence, rows and heads
// outermost, is cut into one contiguous run per CTA; a run crosses into at most a few
// (row, kv head) segments, and each warp's ring runs ahead across segment boundaries, so copies
// never stop.  A (row, kv head) shared by several CTAs is finished by the last of them (atomic
// ticket), which merges their partials in CTA order (the order of the positions).
template <int HD, int NG>
__global__ void __launch_bounds__(kMmaWarps * 32, 1)
    attn_mma_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap, const AttnArgs a) {
  using M = MmaShape<HD>;
  constexpr int ROWB = M::ROWB, BUF = M::BUF, QP = M::QP, DT = M::DT, KS = M::KS;
  constexpr int CH = kMmaChunk;
  const int NR = attn_mma_nr<HD>(a.g);
  extern __shared__ unsigned char araw[];
  const uint32_t s_raw = smem_u32(araw);
  unsigned char* base = araw + (((s_raw + 1023u) & ~1023u) - s_raw);
  const uint32_t s_base = smem_u32(base);

  const int g = a.g, H = a.kv * a.g, ns = kMmaMaxSplits;  // partial slots per (row, kv head)
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int NT = blockDim.x, NW = NT >> 5;
  const int c = blockIdx.x, G = gridDim.x;
  uint16_t* qbase = reinterpret_cast<uint16_t*>(base + (size_t)kMmaWarps * NR * BUF);  // [hi, lo][16][QP]
  float* wpart = reinterpret_cast<float*>(qbase + 2 * 16 * QP);                       // [NW][g][HD+2]
  float* mypart = wpart + NW * g * (HD + 2);                                           // [g][HD+2]
  float* fac = mypart + g * (HD + 2);                                                  // [g][kMmaMaxSplits]
  float* cpart = fac + g * kMmaMaxSplits;  // cluster mode: [rank][g][HD+2], filled in rank 0
  const uint32_t bars = (smem_u32(cpart + (a.cluster ? kMmaCluster * g * (HD + 2) : 0)) + 7u) & ~7u;
  __shared__ int s_last;
  __shared__ float wfac[kMmaWarps * 16];   // per head, each warp's factor exp(m_w - M)

  // Every (row, kv head) gets the chunk count of the longest row (rows may sit at different
  // positions); a row's chunks past its own position are empty: never copied, never computed,
  // but their CTAs still take part in the merge (with empty partials).
  const int nchk = (a.step->pos + 1 + CH - 1) / CH;   // chunks of one (row, kv head)
  const long long T = (long long)a.B * a.kv * nchk;   // chunks of the launch
  // cluster mode: cluster bj takes (row, kv head) bj and its CTA of rank r the r-th of a.ns
  // even parts of the chunks (possibly none)
  const bool clus = a.cluster != 0;
  const int crank = clus ? (int)cluster_rank() : 0;
  const long long cbj = clus ? c / a.ns : 0;
  const long long c0 = clus ? cbj * nchk + (long long)nchk * crank / a.ns : T * c / G;
  const long long c1 = clus ? cbj * nchk + (long long)nchk * (crank + 1) / a.ns : T * (c + 1) / G;
  auto owner = [&](long long it) { return (int)(((it + 1) * G + T - 1) / T - 1); };
  // the segment starting at chunk st of the sequence: (row b, kv head j), chunks [k0, k1), of
  // which [kv0, kv1) hold positions of row b's range ts..tb (tw: the first position this step
  // writes in the row)
  struct Seg {
    int b, j, k0, k1, kv0, kv1, tb, ts, tw;
    int kbase;  // key-map row of position 0 of (b, j) when the step has no page table, else -1
  };
  auto seg = [&](long long st, Seg& sg, long long& next) {
    const long long bj = st / nchk;
    sg.k0 = (int)(st - bj * nchk);
    const long long end = c1 < (bj + 1) * nchk ? c1 : (bj + 1) * nchk;
    sg.k1 = sg.k0 + (int)(end - st);
    sg.j = (int)(bj % a.kv);
    sg.b = (int)(bj / a.kv);
    sg.tb = row_pos(a.step, sg.b);
    sg.ts = row_start(a.step, sg.b);
    sg.tw = row_wfirst(a.step, sg.b);
    const int nb = (sg.tb + 1 + CH - 1) / CH, cs = sg.ts / CH;
    sg.kv0 = sg.k0 > cs ? sg.k0 : cs;
    sg.kv1 = sg.k1 < nb ? sg.k1 : nb;
    if (sg.kv1 < sg.kv0) sg.kv1 = sg.kv0;
    sg.kbase = -1;
    if (!a.step->table) {
      int r, pp;
      cache_slot(a.step, a.cap, sg.b, 0, r, pp);
      sg.kbase = a.krow0 + (r * a.kv + sg.j) * a.cap;
    }
    next = end;
  };

  if (tid == 0) {
    for (int i = 0; i < NW * NR; ++i) mbar_init(bars + 8u * i, 1);
    mbar_fence_init();
  }
  __syncthreads();
  if (clus) cluster_arrive_relaxed();  // waited for before the first access to another CTA

  // the issuing side of this warp (lane 0): cursor over (segment, chunk) pairs
  long long ist = c0, inext = c0;
  int iq = warp, issued = 0;
  Seg is = {};
  if (ist < c1) seg(ist, is, inext);
  auto settle = [&]() {  // move the cursor to a pair that exists (or past the run)
    while (ist < c1 && iq >= is.kv1 - is.kv0) {
      ist = inext;
      iq = warp;
      if (ist < c1) seg(ist, is, inext);
    }
  };
  settle();
  int islot = 0;  // issued % NR
  auto issue = [&]() {
    const int slot = islot;
    if (++islot == NR) islot = 0;
    const int pb = (is.kv0 + iq) * CH;
    // the key-map row holding position pb (a chunk never crosses a page)
    int krow;
    if (is.kbase >= 0) {
      krow = is.kbase + pb;
    } else {
      int r, pp;
      cache_slot(a.step, a.cap, is.b, pb, r, pp);
      krow = a.krow0 + (r * a.kv + is.j) * a.cap + pp;
    }
    const uint32_t bar = bars + 8u * (warp * NR + slot);
    const uint32_t dst = s_base + (uint32_t)((warp * NR + slot) * BUF);
    fence_proxy_async_smem();
    mbar_expect_tx(bar, (uint32_t)(2 * CH * ROWB));
#pragma unroll
    for (int bx = 0; bx < M::NBOX; ++bx) {
      tma_load_2d(dst + (uint32_t)(bx * CH * 128), &kmap, bar, bx * 64, krow);
      tma_load_2d(dst + (uint32_t)(CH * ROWB + bx * CH * 128), &vmap, bar, bx * 64, krow);
    }
    ++issued;
    iq += NW;
    settle();
  };
  // the first segment, from the step state (written by the step prologue, long complete): before
  // the wait, so that no dependent read of it lies on the path after the previous kernel
  Seg s0 = {};
  long long nx0 = c0;
  if (c0 < c1) seg(c0, s0, nx0);
  if (lane == 0) {
    tma_prefetch_map(&kmap);
    tma_prefetch_map(&vmap);
    // chunks below the first position this step writes in the row do not depend on the
    // previous kernel
    while (issued < NR && ist < c1 && (is.kv0 + iq) * CH + min(CH, is.tb + 1 - (is.kv0 + iq) * CH) <= is.tw) issue();
  }
  grid_dep_wait();
  grid_dep_launch();
  if (lane == 0)
    while (issued < NR && ist < c1) issue();
  auto load_q = [&](int b, int j) {  // queries of (b, j) as bf16 hi + lo, rows g..15 zero
    uint16_t* qh = qbase;
    uint16_t* ql = qh + 16 * QP;
    const float* qsrc = a.q + (size_t)b * a.q_stride + (size_t)j * g * HD;
    for (int i = tid; i < 16 * HD / 2; i += NT) {
      const int r = (2 * i) / HD, e = (2 * i) - r * HD;
      float x0 = 0.f, x1 = 0.f;
      if (r < g) {
        const float2 v = *reinterpret_cast<const float2*>(qsrc + (size_t)r * HD + e);
        x0 = v.x;
        x1 = v.y;
      }
      uint32_t hi, lo;
      split_bf16x2(x0, x1, hi, lo);
      *reinterpret_cast<uint32_t*>(qh + r * QP + e) = hi;
      *reinterpret_cast<uint32_t*>(ql + r * QP + e) = lo;
    }
  };
  if (c0 < c1) load_q(s0.b, s0.j);
  __syncthreads();

  const int mi = lane >> 3, mr = lane & 7;
  bool ok = true;
  int consumed = 0;
  int cslot = 0;       // consumed % NR
  uint32_t cpar = 0u;  // (consumed / NR) & 1

  // the splits of (row b, kv head j) merge in rank 0: every CTA stores its partial into rank 0's
  // shared memory (distributed shared memory), one cluster barrier publishes them, and rank 0
  // merges them in rank order (the order of the positions) and writes the output
  auto cluster_merge = [&](int b, int j) {
    const int cs = a.ns;
    cluster_wait();  // every CTA of the cluster has started
    const uint32_t dst = map_rank(smem_u32(cpart + crank * g * (HD + 2)), 0);
    for (int idx = tid; idx < g * (HD + 2); idx += NT) st_cluster(dst + 4u * idx, mypart[idx]);
    cluster_arrive();
    cluster_wait();  // every partial is in rank 0 (and no CTA leaves with its stores in flight)
    if (crank != 0) return;
    for (int h = tid; h < g; h += NT) {
      float Mx = -INFINITY;
      for (int r = 0; r < cs; ++r) Mx = fmaxf(Mx, cpart[(r * g + h) * (HD + 2) + HD]);
      float L = 0.f;
      for (int r = 0; r < cs; ++r) {
        const float mr = cpart[(r * g + h) * (HD + 2) + HD];
        const float f = mr == -INFINITY ? 0.f : expf(mr - Mx);
        fac[h * kMmaMaxSplits + r] = f;
        L += cpart[(r * g + h) * (HD + 2) + HD + 1] * f;
      }
      const float rl = 1.0f / L;
      for (int r = 0; r < cs; ++r) fac[h * kMmaMaxSplits + r] *= rl;
    }
    __syncthreads();
    float* outb = a.out + (size_t)b * a.out_stride + (size_t)j * g * HD;
    for (int idx = tid; idx < g * HD; idx += NT) {
      const int h = idx / HD, e = idx - h * HD;
      float O = 0.f;
      for (int r = 0; r < cs; ++r) O = fmaf(fac[h * kMmaMaxSplits + r], cpart[(r * g + h) * (HD + 2) + e], O);
      outb[(size_t)h * HD + e] = O;
    }
  };
  if (clus && c0 == c1) {
    // no chunks here: an empty part (o = 0, m = -inf, l = 0) joins the merge
    for (int idx = tid; idx < g * (HD + 2); idx += NT) mypart[idx] = (idx % (HD + 2)) == HD ? -INFINITY : 0.f;
    __syncthreads();
    cluster_merge((int)(cbj / a.kv), (int)(cbj % a.kv));
  }

  int lu = 0;
  long long next = c0;
  for (long long st = c0; st < c1; st = next, ++lu) {
    Seg sg;
    if (st == c0) {
      sg = s0;
      next = nx0;
    } else {
      seg(st, sg, next);
    }
    const int b = sg.b, j = sg.j, k0 = sg.k0, ts = sg.ts;
    const int p0 = sg.kv0 * CH, p1 = min(sg.tb + 1, sg.kv1 * CH), nch = sg.kv1 - sg.kv0;  // nch may be 0
    // this segment's queries as B fragments (k = dimensions, n = heads), hi and lo, kept in
    // registers: x4 loads give (b0, b1) of two consecutive k-steps
    uint32_t qfh[NG][KS][2], qfl[NG][KS][2];
#pragma unroll
    for (int n = 0; n < NG; ++n)
#pragma unroll
      for (int ks = 0; ks < KS; ks += 2) {
        const uint32_t off = (uint32_t)(((n * 8 + mr) * QP + ks * 16 + mi * 8) * 2);
        uint32_t r[4];
        ldsm_x4(smem_u32(qbase) + off, r);
        qfh[n][ks][0] = r[0]; qfh[n][ks][1] = r[1]; qfh[n][ks + 1][0] = r[2]; qfh[n][ks + 1][1] = r[3];
        ldsm_x4(smem_u32(qbase + 16 * QP) + off, r);
        qfl[n][ks][0] = r[0]; qfl[n][ks][1] = r[1]; qfl[n][ks + 1][0] = r[2]; qfl[n][ks + 1][1] = r[3];
      }
    // O^T tiles: o[n][dt] = (dims dt*16 + gid (+8), heads n*8 + 2 tig (+1))
    float o[NG][DT][4];
#pragma unroll
    for (int n = 0; n < NG; ++n)
#pragma unroll
      for (int dt = 0; dt < DT; ++dt) o[n][dt][0] = o[n][dt][1] = o[n][dt][2] = o[n][dt][3] = 0.f;
    // running max and this lane's share of the running sum, per head n*8 + 2 tig + hc
    float mrow[NG][2], lrow[NG][2];
#pragma unroll
    for (int n = 0; n < NG; ++n) mrow[n][0] = mrow[n][1] = -INFINITY, lrow[n][0] = lrow[n][1] = 0.f;
    for (int ci = warp; ci < nch && ok; ci += NW) {
      const int slot = cslot;
      const uint32_t bar = bars + 8u * (warp * NR + slot);
      ok = __all_sync(0xffffffffu, mbar_wait(bar, cpar, kAttnWaitCycles));
      if (!ok) break;
      ++consumed;
      if (++cslot == NR) cslot = 0, cpar ^= 1u;
      const int pb = p0 + ci * CH;
      const int nv = min(CH, p1 - pb);
      const uint32_t kreg = s_base + (uint32_t)((warp * NR + slot) * BUF);
      const uint32_t vreg = kreg + (uint32_t)(CH * ROWB);
      const int r0 = ts > pb ? ts - pb : 0;  // rows below the range's start (first chunk only)
      if (nv < CH || r0 > 0) {
        // rows outside the range hold other data (possibly not finite): zero the values
        unsigned char* vz = base + (size_t)(warp * NR + slot) * BUF + CH * ROWB;
        for (int i = lane; i < CH * (ROWB / 16); i += 32) {
          const int r = i / (ROWB / 16), cc = i - r * (ROWB / 16);
          if (r >= nv || r < r0) *reinterpret_cast<uint4*>(vz + swz_off(r, cc)) = make_uint4(0u, 0u, 0u, 0u);
        }
        __syncwarp();
      }
      // ---- scores S^T = K Q^T: rows = the 16 positions, columns = heads; separate hi and lo
      // accumulators ----
      float sh[NG][4], sl[NG][4];
#pragma unroll
      for (int n = 0; n < NG; ++n)
#pragma unroll
        for (int i = 0; i < 4; ++i) sh[n][i] = sl[n][i] = 0.f;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        // matrices: positions 0-7 and 8-15 of dims ks*16 + 0..7, then of dims ks*16 + 8..15
        uint32_t ka[4];
        ldsm_x4(kreg + swz_off((mi & 1) * 8 + mr, 2 * ks + (mi >> 1)), ka);
#pragma unroll
        for (int n = 0; n < NG; ++n) mma_bf16_16816(sh[n], ka, qfh[n][ks][0], qfh[n][ks][1]);
#pragma unroll
        for (int n = 0; n < NG; ++n) mma_bf16_16816(sl[n], ka, qfl[n][ks][0], qfl[n][ks][1]);
      }
      // ---- online softmax per head (a column: the 8 lanes of one tig, two rows each) ----
      float p[NG][4], corr[NG][2];
#pragma unroll
      for (int n = 0; n < NG; ++n) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int pos = gid + 8 * (i >> 1), hh = n * 8 + 2 * tig + (i & 1);
          p[n][i] = (pos < nv && pos >= r0 && hh < g) ? (sh[n][i] + sl[n][i]) * a.scale : -INFINITY;
        }
#pragma unroll
        for (int hc = 0; hc < 2; ++hc) {
          float mx = fmaxf(p[n][hc], p[n][2 + hc]);
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          const float mnew = fmaxf(mrow[n][hc], mx);  // -inf only for a padding head
          corr[n][hc] = mrow[n][hc] == -INFINITY ? 0.f : expf(mrow[n][hc] - mnew);
          mrow[n][hc] = mnew;
          const float w0 = p[n][hc] == -INFINITY ? 0.f : expf(p[n][hc] - mnew);
          const float w1 = p[n][2 + hc] == -INFINITY ? 0.f : expf(p[n][2 + hc] - mnew);
          p[n][hc] = w0;
          p[n][2 + hc] = w1;
          lrow[n][hc] = fmaf(lrow[n][hc], corr[n][hc], w0 + w1);
        }
      }
      // the outputs need rescaling only when a running maximum moved
      bool same = true;
#pragma unroll
      for (int n = 0; n < NG; ++n) same = same && corr[n][0] == 1.f && corr[n][1] == 1.f;
      if (!__all_sync(0xffffffffu, same)) {
#pragma unroll
        for (int n = 0; n < NG; ++n)
#pragma unroll
          for (int dt = 0; dt < DT; ++dt) {
            o[n][dt][0] *= corr[n][0];
            o[n][dt][1] *= corr[n][1];
            o[n][dt][2] *= corr[n][0];
            o[n][dt][3] *= corr[n][1];
          }
      }
      // ---- values O^T += V^T P^T: the weights as the B operand (k = positions, n = heads),
      // gathered from the score fragments: lane (gid = head, tig = t) takes positions 2t, 2t + 1
      // from lane 8t + gid/2 and lane 8t + 4 + gid/2, rows gid and gid + 8 ----
      uint32_t pfh[NG][2], pfl[NG][2];
      {
        const int sa = 8 * tig + (gid >> 1), sb = sa + 4;
        const bool odd = gid & 1;
#pragma unroll
        for (int n = 0; n < NG; ++n) {
          const float a0 = __shfl_sync(0xffffffffu, p[n][0], sa), a1 = __shfl_sync(0xffffffffu, p[n][1], sa);
          const float a2 = __shfl_sync(0xffffffffu, p[n][2], sa), a3 = __shfl_sync(0xffffffffu, p[n][3], sa);
          const float b0 = __shfl_sync(0xffffffffu, p[n][0], sb), b1 = __shfl_sync(0xffffffffu, p[n][1], sb);
          const float b2 = __shfl_sync(0xffffffffu, p[n][2], sb), b3 = __shfl_sync(0xffffffffu, p[n][3], sb);
          split_bf16x2(odd ? a1 : a0, odd ? b1 : b0, pfh[n][0], pfl[n][0]);  // positions 2t, 2t + 1
          split_bf16x2(odd ? a3 : a2, odd ? b3 : b2, pfh[n][1], pfl[n][1]);  // positions 2t + 8, 2t + 9
        }
      }
#pragma unroll
      for (int dt = 0; dt < DT; ++dt) {
        // matrices (transposed): positions 0-7 of dims dt*16 + 0..7 and + 8..15, then 8-15
        uint32_t va[4];
        ldsm_x4_t(vreg + swz_off((mi >> 1) * 8 + mr, 2 * dt + (mi & 1)), va);
#pragma unroll
        for (int n = 0; n < NG; ++n) mma_bf16_16816(o[n][dt], va, pfh[n][0], pfh[n][1]);
#pragma unroll
        for (int n = 0; n < NG; ++n) mma_bf16_16816(o[n][dt], va, pfl[n][0], pfl[n][1]);
      }
      __syncwarp();
      if (lane == 0)
        while (issued - consumed < NR && ist < c1) issue();
    }
    // ---- the unit's end: warp partials, the CTA's partial, the split merge ----
#pragma unroll
    for (int n = 0; n < NG; ++n)
#pragma unroll
      for (int hc = 0; hc < 2; ++hc) {
        float l = lrow[n][hc];
        l += __shfl_xor_sync(0xffffffffu, l, 4);
        l += __shfl_xor_sync(0xffffffffu, l, 8);
        l += __shfl_xor_sync(0xffffffffu, l, 16);
        const int h = n * 8 + 2 * tig + hc;
        if (h < g) {
          float* wp = wpart + (warp * g + h) * (HD + 2);
#pragma unroll
          for (int dt = 0; dt < DT; ++dt) {
            wp[dt * 16 + gid] = o[n][dt][hc];
            wp[dt * 16 + gid + 8] = o[n][dt][2 + hc];
          }
          if (gid == 0) {
            wp[HD] = mrow[n][hc];
            wp[HD + 1] = l;
          }
        }
      }
    __syncthreads();
    // the CTA's partial: per head the maximum M over the warps and each warp's factor
    // exp(m_w - M), then the factor-weighted sums of o and l in warp order
    for (int i = tid; i < g * NW; i += NT) {
      const int h = i / NW, w = i - h * NW;
      float Mx = -INFINITY;
      for (int w2 = 0; w2 < NW; ++w2) Mx = fmaxf(Mx, wpart[(w2 * g + h) * (HD + 2) + HD]);
      const float mw = wpart[(w * g + h) * (HD + 2) + HD];
      wfac[i] = mw == -INFINITY ? 0.f : expf(mw - Mx);
      if (w == 0) mypart[h * (HD + 2) + HD] = Mx;
    }
    __syncthreads();
    for (int idx = tid; idx < g * (HD + 2); idx += NT) {
      const int h = idx / (HD + 2), e = idx - h * (HD + 2);
      if (e == HD) continue;
      float r = 0.f;
      for (int w = 0; w < NW; ++w) r = fmaf(wfac[h * NW + w], wpart[(w * g + h) * (HD + 2) + e], r);
      mypart[idx] = r;
    }
    if (next < c1) {  // (every warp is past this segment's chunks: the query buffer is free)
      Seg s2;
      long long nx2;
      seg(next, s2, nx2);
      load_q(s2.b, s2.j);
    }
    __syncthreads();
    if (clus) {
      cluster_merge(b, j);
      continue;
    }
    float* outb = a.out + (size_t)b * a.out_stride + (size_t)j * g * HD;
    // the CTAs holding chunks of this (row, kv head): with at least one chunk per CTA they are
    // first..last; with fewer chunks than CTAs each holds one chunk
    const long long bj0 = ((long long)b * a.kv + j) * nchk;
    const int first = owner(bj0), last = owner(bj0 + nchk - 1);
    const int nc = T >= G ? last - first + 1 : nchk, sp = T >= G ? c - first : k0;
    if (nc == 1) {
      // this CTA holds all positions: the output is o / l (the merge's factor for one part)
      for (int idx = tid; idx < g * HD; idx += NT) {
        const int h = idx / HD, e = idx - h * HD;
        const float rl = 1.0f / mypart[h * (HD + 2) + HD + 1];
        outb[(size_t)h * HD + e] = fmaf(rl, mypart[h * (HD + 2) + e], 0.f);
      }
    } else {
      // global partials; the last CTA of this (row, kv head) merges them in CTA order
      float* pglob = a.part + (((size_t)b * H + (size_t)j * g) * ns) * (HD + 2);
      for (int idx = tid; idx < g * (HD + 2); idx += NT) {
        const int h = idx / (HD + 2), e = idx - h * (HD + 2);
        pglob[((size_t)h * ns + sp) * (HD + 2) + e] = mypart[idx];
      }
      __threadfence();
      __syncthreads();
      if (tid == 0) {
        const unsigned int prev = atomicAdd(a.ticket + (size_t)b * a.kv + j, 1u);
        s_last = (prev == (unsigned int)(nc - 1));
      }
      __syncthreads();
      if (s_last) {
        __threadfence();
        for (int h = warp; h < g; h += NW) {
          float Mx = -INFINITY;
          for (int s2 = lane; s2 < nc; s2 += 32) Mx = fmaxf(Mx, __ldcg(pglob + ((size_t)h * ns + s2) * (HD + 2) + HD));
          Mx = warp_max(Mx);
          float L = 0.f;
          for (int s2 = lane; s2 < nc; s2 += 32) {
            const float* pp = pglob + ((size_t)h * ns + s2) * (HD + 2);
            const float ms = __ldcg(pp + HD);
            const float f = ms == -INFINITY ? 0.f : expf(ms - Mx);
            fac[h * kMmaMaxSplits + s2] = f;
            L += __ldcg(pp + HD + 1) * f;
          }
          L = warp_sum(L);
          const float rl = 1.0f / L;
          for (int s2 = lane; s2 < nc; s2 += 32) fac[h * kMmaMaxSplits + s2] *= rl;
        }
        __syncthreads();
        for (int idx = tid; idx < g * HD; idx += NT) {
          const int h = idx / HD, e = idx - h * HD;
          const float* pb = pglob + (size_t)h * ns * (HD + 2) + e;
          float O = 0.f;
          int s2 = 0;
          for (; s2 + 8 <= nc; s2 += 8) {
            float ov[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) ov[q] = __ldcg(pb + (size_t)(s2 + q) * (HD + 2));
#pragma unroll
            for (int q = 0; q < 8; ++q) O = fmaf(fac[h * kMmaMaxSplits + s2 + q], ov[q], O);
          }
          for (; s2 < nc; ++s2) O = fmaf(fac[h * kMmaMaxSplits + s2], __ldcg(pb + (size_t)s2 * (HD + 2)), O);
          outb[(size_t)h * HD + e] = O;
        }
        if (tid == 0) a.ticket[(size_t)b * a.kv + j] = 0u;
      }
      __syncthreads();
    }
  }
  if (!ok && lane == 0) atomicCAS(a.status, 0, kErrDeviceTimeout);
  // no copy may still be writing shared memory when the CTA exits
  if (lane == 0)
    for (int k = consumed; k < issued; ++k)
      if (!mbar_wait(bars + 8u * (warp * NR + k % NR), (uint32_t)(k / NR) & 1u, kAttnWaitCycles))
        atomicCAS(a.status, 0, kErrDeviceTimeout);
}

// ---------------------------------------------------------------------------------------

using AttnFn = void (*)(const CUtensorMap, const AttnArgs);
using MmaFn = void (*)(const CUtensorMap, const CUtensorMap, const AttnArgs);

// the tensor-core kernel for a head size (64 or 128) and group size (one or two 8-head tiles)
static MmaFn mma_fn(int hd, int g) {
  if (hd == 64) return g <= 8 ? attn_mma_kernel<64, 1> : attn_mma_kernel<64, 2>;
  return g <= 8 ? attn_mma_kernel<128, 1> : attn_mma_kernel<128, 2>;
}

template <int KT, int HD>
static AttnFn pick_gm(int g, size_t* smem, int ns, int* nw) {
  *nw = attn_geom(AttnShape<KT, HD>::BUF).nw;
  if (g <= 4) {
    *smem = attn_smem<KT, HD, 4>(g, ns);
    return attn_decode_kernel<KT, HD, 4>;
  }
  if constexpr (HD <= 128) {
    if (g <= 8) {
      *smem = attn_smem<KT, HD, 8>(g, ns);
      return attn_decode_kernel<KT, HD, 8>;
    }
  }
  if constexpr (HD <= 64) {
    if (g <= 16) {
      *smem = attn_smem<KT, HD, 16>(g, ns);
      return attn_decode_kernel<KT, HD, 16>;
    }
  }
  return nullptr;
}

template <int KT>
static AttnFn pick_hd(int hd, int g, size_t* smem, int ns, int* nw) {
  switch (hd) {
    case 16: return pick_gm<KT, 16>(g, smem, ns, nw);
    case 32: return pick_gm<KT, 32>(g, smem, ns, nw);
    case 64: return pick_gm<KT, 64>(g, smem, ns, nw);
    case 128: return pick_gm<KT, 128>(g, smem, ns, nw);
    case 256: return pick_gm<KT, 256>(g, smem, ns, nw);
    default: return nullptr;
  }
}

static AttnFn pick(int kt, int hd, int g, size_t* smem, int ns, int* nw) {
  return kt ? pick_hd<1>(hd, g, smem, ns, nw) : pick_hd<0>(hd, g, smem, ns, nw);
}

static int g_max_cluster = 8;  // 16 once attn_prepare finds the device can schedule it
static int g_smem_limit = 0;   // dynamic shared memory a kernel of this file may use
int attn_max_cluster() { return g_max_cluster; }

bool attn_supported(int hd, int g) {
  return (hd == 16 || hd == 32 || hd == 64 || hd == 128 || hd == 256) && g >= 1 && g <= 16 && g * hd <= 1024;
}

cudaError_t attn_prepare(int max_smem_optin) {
  for (int kt = 0; kt < 2; ++kt)
    for (int hd : {16, 32, 64, 128, 256})
      for (int g : {4, 8, 16}) {
        if (!attn_supported(hd, g)) continue;
        size_t sm = 0;
        int nw = 0;
        AttnFn fn = pick(kt, hd, g, &sm, 1, &nw);
        if (!fn) continue;
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem_optin - 64);
        if (e != cudaSuccess) return e;
        if (cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) cudaGetLastError();
      }
  g_smem_limit = max_smem_optin - 1024;  // (the kernels' static shared memory is far below this margin)
  for (auto fn : {attn_mma_kernel<64, 1>, attn_mma_kernel<64, 2>, attn_mma_kernel<128, 1>, attn_mma_kernel<128, 2>}) {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, fn);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem_optin - (int)fa.sharedSizeBytes);
    if (e != cudaSuccess) return e;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) cudaGetLastError();
  }
  // clusters of 16 (beyond the portable 8) where the device can run them with this kernel
  g_max_cluster = 8;
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(16, 8, 1);
    cfg.blockDim = dim3(kMmaWarps * 32);
    cfg.dynamicSmemBytes = attn_mma_smem<128>(4);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 16;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int nclusters = 0;
    if (cudaOccupancyMaxActiveClusters(&nclusters, attn_mma_kernel<128, 1>, &cfg) == cudaSuccess && nclusters >= 1)
      g_max_cluster = 16;
    cudaGetLastError();
  }
  return cudaSuccess;
}

bool attn_make_kmap(CUtensorMap* map, const void* kc, int kt, int hd, uint64_t rows) {
  const int es = kt ? 2 : 4;
  const int rowb = hd * es;
  const bool swz = rowb >= 128;
  const int boxb = swz ? 128 : rowb;
  const int box_rows = attn_uses_mma(kt, hd) ? kMmaChunk : kChunk;
  return make_map_2d(map, kc, es, (uint64_t)hd, rows, (uint32_t)(boxb / es), (uint32_t)box_rows,
                     swz ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE);
}

int attn_splits(int B, int kv, int cap, int num_sms) {
  // about two CTAs per SM, each split at least kMinChunk positions of the capacity; among nearby
  // counts the one whose CTAs fill whole waves of one CTA per SM
  const int units = B * kv;
  int by_cap = cap / kMinChunk;
  if (by_cap < 1) by_cap = 1;
  if (by_cap > 64) by_cap = 64;  // (the persistent kernel merges at most 64 splits)
  const int ns0 = (2 * num_sms + units - 1) / units;
  int best = 1;
  double best_eff = -1.0;
  int lo = ns0 / 2 > 1 ? ns0 / 2 : 1;
  if (lo > by_cap) lo = by_cap;
  for (int ns = lo; ns <= 2 * ns0 && ns <= by_cap; ++ns) {
    const long long ctas = (long long)units * ns;
    const long long waves = (ctas + num_sms - 1) / num_sms;
    const double eff = (double)ctas / (double)(waves * num_sms);
    if (eff > best_eff + 1e-9) {
      best_eff = eff;
      best = ns;
    }
  }
  return best;
}

bool attn_uses_mma(int kt, int hd) { return kt == 1 && (hd == 64 || hd == 128); }

int attn_part_slots(int kt, int hd, int ns) { return attn_uses_mma(kt, hd) ? kMmaMaxSplits : ns; }

// clusters of cs CTAs of this kernel that the device runs at once (queried once per shape)
static int max_active_clusters(const void* fn, size_t smem, int threads, int cs) {
  static std::mutex mu;
  static std::map<std::tuple<const void*, size_t, int, int>, int> cache;
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_tuple(fn, smem, threads, cs);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cs, 1, 1);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  cache.emplace(key, n);
  return n;
}

// The splits merge inside a cluster only when every cluster of the launch runs at once (a second
// wave of clusters would double the time); otherwise through global partials.
bool attn_cluster_merge(int kt, int hd, int g, int ns, int clusters, int cap) {
  if (attn_uses_mma(kt, hd)) {
    // the tensor-core kernel: clusters of kMmaCluster CTAs per (row, kv head) when they all run at
    // once and each CTA's share of a full cache is small (a long cache wants every SM streaming
    // it), else the persistent split over every SM with global partials
    if ((size_t)cap * hd * 2 * 2 / kMmaCluster > kMmaClusterMaxBytes) return false;
    const void* f = (const void*)mma_fn(hd, g);
    const size_t smem = hd == 64 ? attn_mma_smem<64>(g, true) : attn_mma_smem<128>(g, true);
    if (smem > (size_t)g_smem_limit) return false;
    return clusters <= max_active_clusters(f, smem, kMmaWarps * 32, kMmaCluster);
  }
  if (ns == 1) return true;
  if (ns > attn_max_cluster()) return false;
  size_t smem = 0;
  int nw = 0;
  const void* f = (const void*)pick(kt, hd, g, &smem, ns, &nw);
  if (!f) return false;
  return clusters <= max_active_clusters(f, smem, nw * 32, ns);
}

cudaError_t launch_attn(const CUtensorMap& kmap, const CUtensorMap& vmap, const AttnArgs& a0, int kt, cudaStream_t s,
                        bool pdl) {
  AttnArgs a = a0;
  size_t smem = 0;
  int nw = 0;
  AttnFn fn = nullptr;
  MmaFn mfn = nullptr;
  if (attn_uses_mma(kt, a.hd)) {
    mfn = mma_fn(a.hd, a.g);
    smem = a.hd == 64 ? attn_mma_smem<64>(a.g) : attn_mma_smem<128>(a.g);
    nw = kMmaWarps;
  } else {
    fn = pick(kt, a.hd, a.g, &smem, a.ns, &nw);
    if (!fn) return cudaErrorInvalidValue;
  }
  a.cluster = attn_cluster_merge(kt, a.hd, a.g, a.ns, a.B * a.kv, a.cap) ? 1 : 0;
  if (mfn && a.cluster) smem = a.hd == 64 ? attn_mma_smem<64>(a.g, true) : attn_mma_smem<128>(a.g, true);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.ns, a.kv, a.B);
  if (mfn && a.cluster) {
    // one cluster per (row, kv head)
    a.ns = kMmaCluster;
    cfg.gridDim = dim3(a.B * a.kv * kMmaCluster);
  } else if (mfn) {
    // persistent: one CTA per SM, each walking (row, kv head, split) units
    static int sms = 0;
    if (!sms) {
      int dev = 0;
      cudaGetDevice(&dev);
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      if (sms < 1) sms = 1;
    }
    // at most kMmaMaxSplits - 1 CTAs per (row, kv head) keeps every one's parts within its slots
    const int cap = (kMmaMaxSplits - 1) * a.B * a.kv;
    cfg.gridDim = dim3(cap < sms ? cap : sms);
  }
  cfg.blockDim = dim3(nw * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  int na = 1;
  if (a.cluster) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = a.ns;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    na = 2;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  if (mfn) return cudaLaunchKernelEx(&cfg, mfn, kmap, vmap, a);
  return cudaLaunchKernelEx(&cfg, fn, kmap, a);
}

// ---------------------------------------------------------------------------------------
// Causal attention of a prefill pass (Llama 3.1 8B Instruct card, attention.linnet prefill<S>:
// token i of a prompt at position pos + i sees the positions s <= pos + i; bend-ml-llama law
// causal).  The entries of a pass come in tiles: up to 64 / g consecutive prompt tokens of one
// cache row, at consecutive positions, with one attention start (0, or the prompt's first
// position for packed prompts).  A unit is (tile, kv head j): its columns are the (token, head)
// pairs t * g + h, and the keys and values of positions start .. the tile's last position are
// streamed once for all of them -- instead of once per token as a decode step would.
//
// One CTA per SM walks the units (the host sorts them longest first, CTA c takes c, c + G, ...).
// A producer warp streams 16-position chunks of the unit's keys and values through a ring of
// shared-memory stages (TMA tensor copies, 128-byte swizzle; full / empty mbarriers), running on
// into the next unit; eight consumer warps each own kPfNT 8-column MMA tiles of the tile's
// columns and read every chunk: scores S^T = K Q^T (rows = the chunk's 16 positions, columns =
// the warp's (token, head) pairs; the queries as bf16 hi + lo B fragments), an online softmax
// per column with the
// causal mask start <= s <= that token's position, and O^T += V^T P^T (the weights as hi + lo B
// fragments).  A warp owns its columns' whole key range, so it writes o / l straight to the
// output; nothing is merged across CTAs.  Every wait is bounded; after one runs out the CTA
// records kErrDeviceTimeout and its warps stop waiting (they still pass the same barriers).
// ---------------------------------------------------------------------------------------

constexpr int kPfWarps = 8;              // consumer warps
constexpr int kPfNT = 1;                 // 8-column MMA tiles per warp (two measured slower: fewer, longer units)
constexpr int kPfCols = kPfWarps * 8 * kPfNT;  // (token, head) columns of a tile
constexpr int kPfStages = 8;             // ring stages (16 positions of keys and values each)

template <int HD>
struct PfShape {
  static constexpr int ROWB = HD * 2;
  static constexpr int NBOX = ROWB / 128;
  static constexpr int STAGE = 2 * kMmaChunk * ROWB;  // keys, then values
  static constexpr int QP = HD + 8;                    // padded query row (elements)
  static constexpr int KS = HD / 16;
  static constexpr int DT = HD / 16;
};

template <int HD>
LLM_HD size_t attn_prefill_smem() {
  using P = PfShape<HD>;
  return 1024 + (size_t)kPfStages * P::STAGE + 2 * (size_t)kPfCols * P::QP * 2 + 2 * kPfStages * 8;
}

int attn_prefill_tile_tokens(int g) { return kPfCols / g; }

template <int HD>
__global__ void __launch_bounds__((kPfWarps + 1) * 32, 1)
    attn_prefill_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                        const AttnPrefillArgs a) {
  using P = PfShape<HD>;
  constexpr int ROWB = P::ROWB, STAGE = P::STAGE, QP = P::QP, KS = P::KS, DT = P::DT;
  constexpr int CH = kMmaChunk;
  extern __shared__ unsigned char praw[];
  const uint32_t s_raw = smem_u32(praw);
  unsigned char* base = praw + (((s_raw + 1023u) & ~1023u) - s_raw);
  const uint32_t s_base = smem_u32(base);
  uint16_t* qbase = reinterpret_cast<uint16_t*>(base + (size_t)kPfStages * STAGE);  // [hi, lo][64][QP]
  const uint32_t FULL0 = smem_u32(qbase + 2 * kPfCols * QP);
  const uint32_t EMPTY0 = FULL0 + 8u * kPfStages;
  __shared__ volatile int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2, tig = lane & 3, mi = lane >> 3, mr = lane & 7;
  const int g = a.g;
  const int nunits = a.tiles[0];
  const int4* tiles = reinterpret_cast<const int4*>(a.tiles + 4);
  const int2* units = reinterpret_cast<const int2*>(a.tiles + 4 + 4 * a.max_tiles);

  if (tid == 0) {
    for (int s = 0; s < kPfStages; ++s) {
      mbar_init(FULL0 + 8u * s, 1);
      mbar_init(EMPTY0 + 8u * s, kPfWarps);
    }
    s_abort = 0;
    mbar_fence_init();
  }
  __syncthreads();
  // the queries and the cache positions of this pass are written by the Q/K/V kernel
  grid_dep_wait();
  grid_dep_launch();

  // unit u: tile (first entry e0, tokens nq, cache row, attention start), kv head j, positions
  // P0 .. P0 + nq - 1, chunks [k0, k1) covering positions start .. P0 + nq - 1
  struct Unit {
    int e0, nq, row, start, j, P0, k0, k1;
  };
  auto unit = [&](int u) {
    Unit U;
    const int2 uj = units[u];
    const int4 t = tiles[uj.x];
    U.e0 = t.x; U.nq = t.y; U.row = t.z; U.start = t.w; U.j = uj.y;
    U.P0 = row_pos(a.step, U.e0);
    U.k0 = U.start / CH;
    U.k1 = (U.P0 + U.nq - 1) / CH + 1;
    return U;
  };
  auto fail = [&]() {
    if (!s_abort) {
      s_abort = 1;
      atomicCAS(a.status, 0, kErrDeviceTimeout);
    }
  };

  if (warp == kPfWarps) {
    // ---- producer ----
    if (lane == 0) {
      tma_prefetch_map(&kmap);
      tma_prefetch_map(&vmap);
      int it = 0;
      for (int u = blockIdx.x; u < nunits; u += gridDim.x) {
        const Unit U = unit(u);
        for (int k = U.k0; k < U.k1; ++k, ++it) {
          const int s = it % kPfStages;
          if (it >= kPfStages && !s_abort &&
              !mbar_wait(EMPTY0 + 8u * s, (uint32_t)(it / kPfStages - 1) & 1u, kAttnWaitCycles))
            fail();
          if (s_abort) break;
          const int krow = a.krow0 + (U.row * a.kv + U.j) * a.cap + k * CH;
          const uint32_t dst = s_base + (uint32_t)(s * STAGE);
          fence_proxy_async_smem();
          mbar_expect_tx(FULL0 + 8u * s, (uint32_t)STAGE);
#pragma unroll
          for (int bx = 0; bx < P::NBOX; ++bx) {
            tma_load_2d(dst + (uint32_t)(bx * CH * 128), &kmap, FULL0 + 8u * s, bx * 64, krow);
            tma_load_2d(dst + (uint32_t)(CH * ROWB + bx * CH * 128), &vmap, FULL0 + 8u * s, bx * 64, krow);
          }
        }
        if (s_abort) break;
      }
      // no copy may still be writing shared memory when the CTA exits
      for (int i = it > kPfStages ? it - kPfStages : 0; i < it; ++i)
        mbar_wait(FULL0 + 8u * (i % kPfStages), (uint32_t)(i / kPfStages) & 1u, kAttnWaitCycles);
    }
    return;
  }

  // ---- consumers: warp w owns columns 8 kPfNT w .. 8 kPfNT (w + 1) - 1 (MMA tiles n) ----
  constexpr int NT = kPfNT;
  int it = 0;
  for (int u = blockIdx.x; u < nunits; u += gridDim.x) {
    const Unit U = unit(u);
    named_sync(1, kPfWarps * 32);  // the previous unit's readers of the queries are done
    {
      // the tile's queries as bf16 hi + lo, columns t * g + h, padding columns zero
      uint16_t* qh = qbase;
      uint16_t* ql = qh + kPfCols * QP;
      for (int i = tid; i < kPfCols * HD / 2; i += kPfWarps * 32) {
        const int col = (2 * i) / HD, e = (2 * i) - col * HD;
        const int t = col / g, h = col - t * g;
        float x0 = 0.f, x1 = 0.f;
        if (t < U.nq) {
          const float2 v = *reinterpret_cast<const float2*>(a.q + (size_t)(U.e0 + t) * a.q_stride +
                                                            (size_t)(U.j * g + h) * HD + e);
          x0 = v.x;
          x1 = v.y;
        }
        uint32_t hi, lo;
        split_bf16x2(x0, x1, hi, lo);
        *reinterpret_cast<uint32_t*>(qh + col * QP + e) = hi;
        *reinterpret_cast<uint32_t*>(ql + col * QP + e) = lo;
      }
    }
    named_sync(1, kPfWarps * 32);
    uint32_t qfh[NT][KS][2], qfl[NT][KS][2];
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int ks = 0; ks < KS; ks += 2) {
        const uint32_t off = (uint32_t)((((warp * NT + n) * 8 + mr) * QP + ks * 16 + mi * 8) * 2);
        uint32_t r[4];
        ldsm_x4(smem_u32(qbase) + off, r);
        qfh[n][ks][0] = r[0]; qfh[n][ks][1] = r[1]; qfh[n][ks + 1][0] = r[2]; qfh[n][ks + 1][1] = r[3];
        ldsm_x4(smem_u32(qbase + kPfCols * QP) + off, r);
        qfl[n][ks][0] = r[0]; qfl[n][ks][1] = r[1]; qfl[n][ks + 1][0] = r[2]; qfl[n][ks + 1][1] = r[3];
      }
    // this lane's columns (n, hc): token, its position (the last key it sees), whether it exists
    int pc[NT][2];
    bool cv[NT][2];
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int hc = 0; hc < 2; ++hc) {
        const int col = (warp * NT + n) * 8 + 2 * tig + hc, t = col / g;
        cv[n][hc] = t < U.nq;
        pc[n][hc] = U.P0 + t;
      }
    const int plast = U.P0 + U.nq - 1;
    float o[NT][DT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int dt = 0; dt < DT; ++dt) o[n][dt][0] = o[n][dt][1] = o[n][dt][2] = o[n][dt][3] = 0.f;
    float mrow[NT][2], lrow[NT][2];
#pragma unroll
    for (int n = 0; n < NT; ++n) mrow[n][0] = mrow[n][1] = -INFINITY, lrow[n][0] = lrow[n][1] = 0.f;
    for (int k = U.k0; k < U.k1; ++k, ++it) {
      const int s = it % kPfStages;
      if (!s_abort) {
        const bool w = __all_sync(0xffffffffu, mbar_wait(FULL0 + 8u * s, (uint32_t)(it / kPfStages) & 1u, kAttnWaitCycles));
        if (!w && lane == 0) fail();
        __syncwarp();
      }
      const int kb = k * CH;
      const uint32_t kreg = s_base + (uint32_t)(s * STAGE);
      const uint32_t vreg = kreg + (uint32_t)(CH * ROWB);
      // scores: rows = positions kb + 0..15, columns = this warp's; even / odd k-steps in
      // separate accumulators (shorter dependency chains)
      float sh[NT][2][4], sl[NT][2][4];
#pragma unroll
      for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int par = 0; par < 2; ++par)
#pragma unroll
          for (int i = 0; i < 4; ++i) sh[n][par][i] = sl[n][par][i] = 0.f;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        uint32_t ka[4];
        ldsm_x4(kreg + swz_off((mi & 1) * 8 + mr, 2 * ks + (mi >> 1)), ka);
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          mma_bf16_16816(sh[n][ks & 1], ka, qfh[n][ks][0], qfh[n][ks][1]);
          mma_bf16_16816(sl[n][ks & 1], ka, qfl[n][ks][0], qfl[n][ks][1]);
        }
      }
      float p[NT][4];
      bool same = true;
#pragma unroll
      for (int n = 0; n < NT; ++n) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int pos = kb + gid + 8 * (i >> 1), hc = i & 1;
          const float sc = (sh[n][0][i] + sh[n][1][i]) + (sl[n][0][i] + sl[n][1][i]);
          p[n][i] = (cv[n][hc] && pos >= U.start && pos <= pc[n][hc]) ? sc * a.scale : -INFINITY;
        }
        float corr[2];
#pragma unroll
        for (int hc = 0; hc < 2; ++hc) {
          float mx = fmaxf(p[n][hc], p[n][2 + hc]);
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          const float mnew = fmaxf(mrow[n][hc], mx);  // -inf while the column has seen no position
          corr[hc] = mrow[n][hc] == -INFINITY ? 0.f : expf(mrow[n][hc] - mnew);
          mrow[n][hc] = mnew;
          const float w0 = p[n][hc] == -INFINITY ? 0.f : expf(p[n][hc] - mnew);
          const float w1 = p[n][2 + hc] == -INFINITY ? 0.f : expf(p[n][2 + hc] - mnew);
          p[n][hc] = w0;
          p[n][2 + hc] = w1;
          lrow[n][hc] = fmaf(lrow[n][hc], corr[hc], w0 + w1);
        }
        if (!__all_sync(0xffffffffu, corr[0] == 1.f && corr[1] == 1.f)) {
          same = false;
#pragma unroll
          for (int dt = 0; dt < DT; ++dt) {
            o[n][dt][0] *= corr[0];
            o[n][dt][1] *= corr[1];
            o[n][dt][2] *= corr[0];
            o[n][dt][3] *= corr[1];
          }
        }
      }
      (void)same;
      // the weights as B fragments (k = positions, n = columns), gathered from the score
      // fragments: lane (gid = column, tig = t) takes positions 2t, 2t + 1 (and + 8)
      uint32_t pfh[NT][2], pfl[NT][2];
      {
        const int sa = 8 * tig + (gid >> 1), sb = sa + 4;
        const bool odd = gid & 1;
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          const float a0 = __shfl_sync(0xffffffffu, p[n][0], sa), a1 = __shfl_sync(0xffffffffu, p[n][1], sa);
          const float a2 = __shfl_sync(0xffffffffu, p[n][2], sa), a3 = __shfl_sync(0xffffffffu, p[n][3], sa);
          const float b0 = __shfl_sync(0xffffffffu, p[n][0], sb), b1 = __shfl_sync(0xffffffffu, p[n][1], sb);
          const float b2 = __shfl_sync(0xffffffffu, p[n][2], sb), b3 = __shfl_sync(0xffffffffu, p[n][3], sb);
          split_bf16x2(odd ? a1 : a0, odd ? b1 : b0, pfh[n][0], pfl[n][0]);
          split_bf16x2(odd ? a3 : a2, odd ? b3 : b2, pfh[n][1], pfl[n][1]);
        }
      }
      // positions outside start .. plast hold other data (possibly not finite): their value
      // elements are zeroed in the A fragments (keys 2 tig, 2 tig + 1 in a0 / a1, + 8 in a2 / a3)
      const bool edge = kb < U.start || kb + CH - 1 > plast;
      uint32_t km0 = 0xffffffffu, km1 = 0xffffffffu;
      if (edge) {
        const int p0 = kb + 2 * tig, p8 = p0 + 8;
        km0 = (p0 >= U.start && p0 <= plast ? 0x0000ffffu : 0u) | (p0 + 1 >= U.start && p0 + 1 <= plast ? 0xffff0000u : 0u);
        km1 = (p8 >= U.start && p8 <= plast ? 0x0000ffffu : 0u) | (p8 + 1 >= U.start && p8 + 1 <= plast ? 0xffff0000u : 0u);
      }
#pragma unroll
      for (int dt = 0; dt < DT; ++dt) {
        uint32_t va[4];
        ldsm_x4_t(vreg + swz_off((mi >> 1) * 8 + mr, 2 * dt + (mi & 1)), va);
        va[0] &= km0;
        va[1] &= km0;
        va[2] &= km1;
        va[3] &= km1;
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          mma_bf16_16816(o[n][dt], va, pfh[n][0], pfh[n][1]);
          mma_bf16_16816(o[n][dt], va, pfl[n][0], pfl[n][1]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(EMPTY0 + 8u * s);
    }
    // the unit's end: o / l of each of this lane's columns
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int hc = 0; hc < 2; ++hc) {
        float l = lrow[n][hc];
        l += __shfl_xor_sync(0xffffffffu, l, 4);
        l += __shfl_xor_sync(0xffffffffu, l, 8);
        l += __shfl_xor_sync(0xffffffffu, l, 16);
        if (!cv[n][hc]) continue;
        const int col = (warp * NT + n) * 8 + 2 * tig + hc, t = col / g, h = col - t * g;
        float* ob = a.out + (size_t)(U.e0 + t) * a.out_stride + (size_t)(U.j * g + h) * HD;
        const float rl = 1.0f / l;
#pragma unroll
        for (int dt = 0; dt < DT; ++dt) {
          ob[dt * 16 + gid] = o[n][dt][hc] * rl;
          ob[dt * 16 + gid + 8] = o[n][dt][2 + hc] * rl;
        }
      }
  }
}

bool attn_prefill_supported(int kt, int hd, int g) { return kt == 1 && (hd == 64 || hd == 128) && g >= 1 && g <= 8; }

cudaError_t attn_prefill_prepare(int max_smem_optin) {
  for (auto fn : {attn_prefill_kernel<64>, attn_prefill_kernel<128>}) {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, fn);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem_optin - (int)fa.sharedSizeBytes);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_attn_prefill(const CUtensorMap& kmap, const CUtensorMap& vmap, const AttnPrefillArgs& a, int grid,
                                cudaStream_t s, bool pdl) {
  if (!attn_prefill_supported(1, a.hd, a.g)) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3((kPfWarps + 1) * 32);
  cfg.dynamicSmemBytes = a.hd == 64 ? attn_prefill_smem<64>() : attn_prefill_smem<128>();
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (a.hd == 64) return cudaLaunchKernelEx(&cfg, attn_prefill_kernel<64>, kmap, vmap, a);
  return cudaLaunchKernelEx(&cfg, attn_prefill_kernel<128>, kmap, vmap, a);
}

}  // namespace llm
