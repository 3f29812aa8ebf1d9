// Greedy and temperature / top-k / top-p sampling of one decode step.
//
// bend-ml-llama "The model", argmax: the first index of the largest logit.
// bend-ml-llama "Sampling", sample(xs, temp, k, p, u):
//   the k largest logits, largest first, equal values by lower id first; the weight of a
//   candidate v is exp(v/temp - top/temp); Z is the weights summed in candidate order; top-p
//   keeps each candidate whose cumulative weight before it is below p*Z (the first always);
//   Zp is the kept weights summed in order; u*Zp picks the first kept candidate whose
//   cumulative weight (itself included) is above it, else the last kept one.
//
// Every arithmetic step is a single IEEE operation in a fixed order, so a CPU that follows the
// same definition draws the same id bit for bit:
//   - candidates: a stable least-significant-digit radix sort (4-bit digits, 8 passes) of all
//     logits on an order-preserving 32-bit key (largest first); stability keeps equal values in
//     id order.  Each pass runs over up to 64 CTAs per row (count, scan, stable scatter).
//   - weights: exp_s, a fixed sequence of IEEE operations (Cody-Waite reduction, degree-8 Taylor
//     polynomial with fused multiply-adds, scaling by 2^n), never the hardware exp.
//   - the cumulative weights are one sequential f32 running sum; Z is its last value.  Adding
//     non-negative numbers never decreases a rounded sum, so the kept count and the draw are
//     binary searches over that running sum.
#include "sampler.cuh"

namespace llm {

constexpr int kSampThreads = 1024;
constexpr int kSortMaxSlices = kSortMaxSlicesPerRow;

LLM_D float exp_s(float x) {
  if (x != x) return x;
  if (x > 88.5f) return INFINITY;
  if (x < -104.0f) return 0.0f;
  const float LOG2E = 1.44269504088896340736f;
  const float LN2_HI = 0.693145751953125f;  // ln 2 to 16 significant bits: n * LN2_HI is exact
  const float LN2_LO = (float)(0.69314718055994530942 - 0.693145751953125);
  const float nf = rintf(__fmul_rn(x, LOG2E));
  const int n = (int)nf;
  float r = __fmaf_rn(-nf, LN2_HI, x);
  r = __fmaf_rn(-nf, LN2_LO, r);
  float p = (float)(1.0 / 40320.0);
  p = __fmaf_rn(p, r, (float)(1.0 / 5040.0));
  p = __fmaf_rn(p, r, (float)(1.0 / 720.0));
  p = __fmaf_rn(p, r, (float)(1.0 / 120.0));
  p = __fmaf_rn(p, r, (float)(1.0 / 24.0));
  p = __fmaf_rn(p, r, (float)(1.0 / 6.0));
  p = __fmaf_rn(p, r, 0.5f);
  p = __fmaf_rn(p, r, 1.0f);
  p = __fmaf_rn(p, r, 1.0f);
  if (n >= -126) return __fmul_rn(p, __uint_as_float((uint32_t)(n + 127) << 23));
  return __fmul_rn(__fmul_rn(p, __uint_as_float((uint32_t)(n + 64 + 127) << 23)),
                   __uint_as_float((uint32_t)(-64 + 127) << 23));
}

// order-preserving key, largest value first (ascending key); -0 and +0 equal
LLM_D uint32_t desc_key(float v) {
  uint32_t u = __float_as_uint(v);
  if (u == 0x80000000u) u = 0u;
  const uint32_t asc = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ~asc;
}

// first index of the largest value (ties: lower index)
LLM_D void argmax_merge(float& bv, int& bi, float v, int i) {
  if (v > bv || (v == bv && i < bi)) {
    bv = v;
    bi = i;
  }
}

__global__ void __launch_bounds__(kSampThreads) sample_kernel(const SampleArgs a) {
  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int V = a.V;
  const float* lg = a.logits + (size_t)b * a.logits_stride;
  __shared__ float s_v[32];
  __shared__ int s_i[32];

  grid_dep_wait();
  grid_dep_launch();

  // greedy: the first index of the largest logit
  {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    if ((a.logits_stride & 3) == 0) {
      // 16-byte loads, several in flight; each thread keeps the first index of its maximum
      const float4* l4 = reinterpret_cast<const float4*>(lg);
      const int n4 = V >> 2;
#pragma unroll 8
      for (int i = tid; i < n4; i += kSampThreads) {
        const float4 v = l4[i];
        argmax_merge(bv, bi, v.x, 4 * i);
        argmax_merge(bv, bi, v.y, 4 * i + 1);
        argmax_merge(bv, bi, v.z, 4 * i + 2);
        argmax_merge(bv, bi, v.w, 4 * i + 3);
      }
      for (int i = 4 * n4 + tid; i < V; i += kSampThreads) argmax_merge(bv, bi, lg[i], i);
    } else {
      for (int i = tid; i < V; i += kSampThreads) argmax_merge(bv, bi, lg[i], i);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      argmax_merge(bv, bi, ov, oi);
    }
    if (lane == 0) {
      s_v[warp] = bv;
      s_i[warp] = bi;
    }
    __syncthreads();
    if (warp == 0) {
      bv = s_v[lane];
      bi = s_i[lane];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        argmax_merge(bv, bi, ov, oi);
      }
      if (lane == 0) a.ids[b] = (bi == 0x7fffffff) ? 0 : bi;
    }
  }
}

// ---------------------------------------------------------------------------------------
// temperature / top-k / top-p: a stable radix sort of each row, then the in-order sums
// ---------------------------------------------------------------------------------------
// Sort: least-significant-digit radix on the 32-bit order key, 8-bit digits and 4 passes (4-bit
// and 8 where the digit-count scratch is small, as in the fixed-array sampler); every
// pass is count (per CTA slice) -> exclusive scan (per row, digit-major) -> stable scatter (each
// CTA writes its slice in index order).  Stability keeps equal values in id order, so the sorted
// row is exactly "largest value first, ties by lower id".

constexpr int kSortThreads = 256;

LLM_HD int sort_slice(int V) {  // elements per CTA: 2048, more when the row needs over 64 CTAs
  int s = (V + kSortMaxSlices - 1) / kSortMaxSlices;
  s = (s + kSortThreads - 1) / kSortThreads * kSortThreads;
  return s < 2048 ? 2048 : s;
}

__global__ void __launch_bounds__(kSortThreads) sort_init_kernel(const SampleArgs a) {
  grid_dep_wait();
  grid_dep_launch();
  const int b = blockIdx.y, S = sort_slice(a.V);
  const int s0 = blockIdx.x * S, s1 = min(a.V, s0 + S);
  const float* lg = a.logits + (size_t)b * a.logits_stride;
  uint32_t* k0 = a.keys + (size_t)b * 2 * a.V_pad;
  int32_t* i0 = a.idx + (size_t)b * 2 * a.V_pad;
  for (int i = s0 + threadIdx.x; i < s1; i += kSortThreads) {
    k0[i] = desc_key(lg[i]);
    i0[i] = i;
  }
}

// DB-bit digits (4 or 8): 32 / DB passes of 2^DB bins
template <int DB>
__global__ void __launch_bounds__(kSortThreads) sort_count_kernel(const SampleArgs a, int pass) {
  constexpr int ND = 1 << DB;
  constexpr uint32_t MASK = ND - 1;
  grid_dep_wait();
  grid_dep_launch();
  const int b = blockIdx.y, c = blockIdx.x, NB = gridDim.x, S = sort_slice(a.V), sh = DB * pass;
  const int s0 = c * S, s1 = min(a.V, s0 + S);
  const uint32_t* ks = a.keys + (size_t)b * 2 * a.V_pad + (pass & 1) * a.V_pad;
  __shared__ uint32_t cnt[ND];
  for (int i = threadIdx.x; i < ND; i += kSortThreads) cnt[i] = 0u;
  __syncthreads();
  const int lane = threadIdx.x & 31;
  for (int i0 = s0; i0 < s1; i0 += kSortThreads) {
    const int i = i0 + threadIdx.x;
    const uint32_t d = i < s1 ? (ks[i] >> sh) & MASK : (uint32_t)ND;
    const uint32_t peers = __match_any_sync(0xffffffffu, d);
    if (d < (uint32_t)ND && lane == __ffs(peers) - 1) atomicAdd(&cnt[d], (uint32_t)__popc(peers));
  }
  __syncthreads();
  for (int i = threadIdx.x; i < ND; i += kSortThreads) a.hist[((size_t)b * ND + i) * NB + c] = cnt[i];
}

// exclusive scan of one row's ND * NB digit counts, digit-major (thread t scans a contiguous run)
template <int DB>
__global__ void __launch_bounds__(kSortThreads) sort_scan_kernel(const SampleArgs a, int NB) {
  constexpr int ND = 1 << DB;
  grid_dep_wait();
  grid_dep_launch();
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t* h = a.hist + (size_t)b * ND * NB;
  const int n = ND * NB;                         // at most 256 * 64 = 16384 entries
  const int per = (n + kSortThreads - 1) / kSortThreads;
  const int i0 = tid * per, i1 = min(n, i0 + per);
  uint32_t sum = 0u;
  for (int i = i0; i < i1; ++i) sum += h[i];
  uint32_t incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  __shared__ uint32_t wt[kSortThreads / 32];
  if (lane == 31) wt[warp] = incl;
  __syncthreads();
  uint32_t before = 0u;
  for (int w = 0; w < warp; ++w) before += wt[w];
  uint32_t run = before + incl - sum;
  for (int i = i0; i < i1; ++i) {
    const uint32_t v = h[i];
    h[i] = run;
    run += v;
  }
}

template <int DB>
__global__ void __launch_bounds__(kSortThreads) sort_scatter_kernel(const SampleArgs a, int pass) {
  constexpr int ND = 1 << DB;
  constexpr uint32_t MASK = ND - 1;
  grid_dep_wait();
  grid_dep_launch();
  const int b = blockIdx.y, c = blockIdx.x, NB = gridDim.x, S = sort_slice(a.V), sh = DB * pass;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int NW = kSortThreads / 32;
  const int s0 = c * S, s1 = min(a.V, s0 + S);
  const size_t rowk = (size_t)b * 2 * a.V_pad;
  const uint32_t* ks = a.keys + rowk + (pass & 1) * a.V_pad;
  uint32_t* kd = a.keys + rowk + ((pass + 1) & 1) * a.V_pad;
  const int32_t* is = a.idx + rowk + (pass & 1) * a.V_pad;
  int32_t* id = a.idx + rowk + ((pass + 1) & 1) * a.V_pad;
  __shared__ uint32_t base[ND], tot[ND], wcnt[NW][ND], wpre[NW][ND];
  for (int i = tid; i < ND; i += kSortThreads) base[i] = a.hist[((size_t)b * ND + i) * NB + c];
  for (int i0 = s0; i0 < s1; i0 += kSortThreads) {
    for (int i = tid; i < NW * ND; i += kSortThreads) wcnt[i / ND][i % ND] = 0u;
    __syncthreads();
    const int i = i0 + tid;
    const bool valid = i < s1;
    const uint32_t key = valid ? ks[i] : 0u;
    const int32_t idv = valid ? is[i] : 0;
    const uint32_t d = valid ? (key >> sh) & MASK : (uint32_t)ND;
    const uint32_t peers = __match_any_sync(0xffffffffu, d);
    const uint32_t rank = __popc(peers & ((1u << lane) - 1u));
    if (valid && lane == __ffs(peers) - 1) wcnt[warp][d] = __popc(peers);
    __syncthreads();
    for (int dd = tid; dd < ND; dd += kSortThreads) {
      uint32_t r = 0u;
      for (int w = 0; w < NW; ++w) {
        wpre[w][dd] = r;
        r += wcnt[w][dd];
      }
      tot[dd] = r;
    }
    __syncthreads();
    if (valid) {
      const uint32_t dst = base[d] + wpre[warp][d] + rank;
      kd[dst] = key;
      id[dst] = idv;
    }
    __syncthreads();
    for (int dd = tid; dd < ND; dd += kSortThreads) base[dd] += tot[dd];
  }
}

// weights of the top k candidates, their in-order running sum, the kept count and the draw.
// cand[j] is the j-th candidate's id (largest logit first, ties by lower id); pre is [k] scratch
// in global memory.  Every thread of the CTA calls this; thread 0 writes ids[b].
constexpr int kFinalThreads = 1024;
constexpr int kRunChunk = 8192;

LLM_D void draw_from_candidates(const SampleArgs& a, int b, const int32_t* cand, int k, float* pre, float* chunk) {
  const int tid = threadIdx.x, nt = blockDim.x;
  const float* lg = a.logits + (size_t)b * a.logits_stride;
  const float temp = a.step->temp;
  const float top = lg[cand[0]];
  const float ttop = __fdiv_rn(top, temp);
  for (int j = tid; j < k; j += nt) pre[j] = exp_s(__fsub_rn(__fdiv_rn(lg[cand[j]], temp), ttop));
  __syncthreads();
  // the running sum is sequential by definition: one thread adds, in order, chunk by chunk
  float run = 0.0f;
  for (int c0 = 0; c0 < k; c0 += kRunChunk) {
    const int n = min(kRunChunk, k - c0);
    for (int j = tid; j < n; j += nt) chunk[j] = pre[c0 + j];
    __syncthreads();
    if (tid == 0) {
      // 16 values at a time in registers, the next 16 loaded while these are added, so the
      // dependent additions are the only latency left
      float4* c4 = reinterpret_cast<float4*>(chunk);
      const int n32 = n & ~15;
      float4 cur[4], nxt[4];
      if (n32 > 0)
#pragma unroll
        for (int q = 0; q < 4; ++q) cur[q] = c4[q];
      for (int j = 0; j < n32; j += 16) {
        if (j + 16 < n32)
#pragma unroll
          for (int q = 0; q < 4; ++q) nxt[q] = c4[(j >> 2) + 4 + q];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          run = __fadd_rn(run, cur[q].x); cur[q].x = run;
          run = __fadd_rn(run, cur[q].y); cur[q].y = run;
          run = __fadd_rn(run, cur[q].z); cur[q].z = run;
          run = __fadd_rn(run, cur[q].w); cur[q].w = run;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) c4[(j >> 2) + q] = cur[q];
#pragma unroll
        for (int q = 0; q < 4; ++q) cur[q] = nxt[q];
      }
      for (int j = n32; j < n; ++j) {
        run = __fadd_rn(run, chunk[j]);
        chunk[j] = run;
      }
    }
    __syncthreads();
    for (int j = tid; j < n; j += nt) pre[c0 + j] = chunk[j];
    __syncthreads();
  }
  if (tid == 0) {
    const float Z = pre[k - 1];
    const float lim = __fmul_rn(a.step->p, Z);
    // kept = 1 + number of leading running sums below lim, at most k
    int lo = 0, hi = k;  // first j with pre[j] >= lim
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (pre[mid] < lim) lo = mid + 1;
      else hi = mid;
    }
    const int kept = min(k, lo + 1);
    const float zp = pre[kept - 1];
    const float target = __fmul_rn(a.u[b], zp);
    lo = 0;
    hi = kept - 1;  // first j < kept-1 with target < pre[j], else kept-1
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (target < pre[mid]) hi = mid;
      else lo = mid + 1;
    }
    a.ids[b] = cand[lo];
  }
}

__global__ void __launch_bounds__(kFinalThreads) sample_final_kernel(const SampleArgs a) {
  grid_dep_wait();
  grid_dep_launch();
  const int b = blockIdx.x;
  __shared__ __align__(16) float chunk[kRunChunk];
  const int32_t* is = a.idx + (size_t)b * 2 * a.V_pad;  // after an even number of passes the sorted row is in buffer 0
  draw_from_candidates(a, b, is, min(a.step->k, a.V), a.pre + (size_t)b * a.V_pad, chunk);
}

// ---------------------------------------------------------------------------------------
// top-k for k <= kSelectMax: the k candidates by a radix select, not a sort of the whole row
// ---------------------------------------------------------------------------------------
// One CTA per row.  The k-th smallest order key T (the k-th largest logit) is found most
// significant byte first: four passes, each a 256-bin histogram of the keys that share the
// prefix found so far.  The candidates are then every id whose key is below T and the first
// k - (their number) ids whose key equals T, taken in ascending id order (threads own contiguous
// id ranges and a block scan orders them), and a bitonic sort of (key, id) pairs puts them in
// the sorted order of the full sort's first k: the same candidates in the same order, so the
// draw is bit for bit the same.

constexpr int kSelectMax = 1024;
constexpr int kSelectThreads = 1024;

__global__ void __launch_bounds__(kSelectThreads) sample_topk_kernel(const SampleArgs a) {
  grid_dep_wait();
  grid_dep_launch();
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int V = a.V;
  const int k = min(min(a.step->k, V), kSelectMax);  // (the host sends larger k to the sort)
  const float* lg = a.logits + (size_t)b * a.logits_stride;
  __shared__ uint32_t hist[256];
  __shared__ uint32_t s_prefix, s_rank, s_lt;
  __shared__ uint32_t wsum[kSelectThreads / 32];
  __shared__ unsigned long long cand[kSelectMax];
  __shared__ int32_t cand_id[kSelectMax];
  __shared__ __align__(16) float chunk[kSelectMax];

  // ---- radix select: T = the key of rank k - 1 (0-based) in ascending key order ----
  uint32_t prefix = 0u, rank = (uint32_t)(k - 1);
  for (int pass = 0; pass < 4; ++pass) {
    const int sh = 24 - 8 * pass;
    const uint32_t mask = pass == 0 ? 0u : 0xffffffffu << (sh + 8);
    if (tid < 256) hist[tid] = 0u;
    __syncthreads();
    for (int i = tid; i < V; i += kSelectThreads) {
      const uint32_t key = desc_key(lg[i]);
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> sh) & 255u], 1u);
    }
    __syncthreads();
    if (tid == 0) {
      uint32_t r = rank, d = 0;
      while (hist[d] <= r) r -= hist[d++];
      s_prefix = prefix | (d << sh);
      s_rank = r;
    }
    __syncthreads();
    prefix = s_prefix;
    rank = s_rank;
  }
  const uint32_t T = prefix;
  const uint32_t need_eq = rank + 1;  // ties at T to take (the k - count below T lowest ids)

  // ---- candidates, in ascending id order within each class ----
  const int per = (V + kSelectThreads - 1) / kSelectThreads;
  const int i0 = tid * per, i1 = min(V, i0 + per);
  uint32_t nlt = 0u, neq = 0u;
  for (int i = i0; i < i1; ++i) {
    const uint32_t key = desc_key(lg[i]);
    nlt += key < T;
    neq += key == T;
  }
  // exclusive block scans of nlt and neq (packed: below-T count in the high half)
  auto scan = [&](uint32_t v) {
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t x = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += x;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      uint32_t w = lane < kSelectThreads / 32 ? wsum[lane] : 0u;
      uint32_t wi = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t x = __shfl_up_sync(0xffffffffu, wi, o);
        if (lane >= o) wi += x;
      }
      if (lane < kSelectThreads / 32) wsum[lane] = wi - w;
    }
    __syncthreads();
    const uint32_t r = wsum[warp] + incl - v;
    __syncthreads();
    return r;
  };
  uint32_t olt = scan(nlt);
  uint32_t oeq = scan(neq);
  if (tid == kSelectThreads - 1) s_lt = olt + nlt;
  __syncthreads();
  const uint32_t total_lt = s_lt;  // = k - need_eq
  for (int i = i0; i < i1; ++i) {
    const uint32_t key = desc_key(lg[i]);
    if (key < T) {
      cand[olt++] = ((unsigned long long)key << 32) | (uint32_t)i;
    } else if (key == T) {
      if (oeq < need_eq) cand[total_lt + oeq] = ((unsigned long long)key << 32) | (uint32_t)i;
      ++oeq;
    }
  }
  // pad to a power of two and sort ascending (key, then id)
  int n2 = 1;
  while (n2 < k) n2 <<= 1;
  for (int j = k + tid; j < n2; j += kSelectThreads) cand[j] = ~0ull;
  __syncthreads();
  for (int size = 2; size <= n2; size <<= 1)
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int j = tid; j < n2; j += kSelectThreads) {
        const int p = j ^ stride;
        if (p > j) {
          const bool up = (j & size) == 0;
          const unsigned long long x = cand[j], y = cand[p];
          if ((x > y) == up) {
            cand[j] = y;
            cand[p] = x;
          }
        }
      }
      __syncthreads();
    }
  for (int j = tid; j < k; j += kSelectThreads) cand_id[j] = (int32_t)(cand[j] & 0xffffffffull);
  __syncthreads();
  draw_from_candidates(a, b, cand_id, k, a.pre + (size_t)b * a.V_pad, chunk);
}

static cudaError_t launch(void (*fn)(const SampleArgs), dim3 grid, int threads, const SampleArgs& a,
                          cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fn, a);
}

template <class Arg>
static cudaError_t launch2(void (*fn)(const SampleArgs, Arg), dim3 grid, int threads, const SampleArgs& a,
                           Arg x, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fn, a, x);
}

int sample_slices(int V) { return (V + sort_slice(V) - 1) / sort_slice(V); }

int sample_select_max() { return kSelectMax; }

cudaError_t launch_sample(const SampleArgs& a, int B, bool greedy, cudaStream_t s, bool pdl, bool select) {
  if (greedy) return launch(sample_kernel, dim3(B), kSampThreads, a, s, pdl);
  if (select) return launch(sample_topk_kernel, dim3(B), kSelectThreads, a, s, pdl);
  const int NB = sample_slices(a.V);
  cudaError_t e = launch(sort_init_kernel, dim3(NB, B), kSortThreads, a, s, pdl);
  // 8-bit digits (four passes) where the caller's digit counts have room, else 4-bit (eight)
  const bool wide = a.hist_per_row >= (size_t)256 * NB;
  const int npass = wide ? 4 : 8;
  for (int pass = 0; pass < npass && e == cudaSuccess; ++pass) {
    e = launch2(wide ? sort_count_kernel<8> : sort_count_kernel<4>, dim3(NB, B), kSortThreads, a, pass, s, true);
    if (e == cudaSuccess)
      e = launch2(wide ? sort_scan_kernel<8> : sort_scan_kernel<4>, dim3(B), kSortThreads, a, NB, s, true);
    if (e == cudaSuccess)
      e = launch2(wide ? sort_scatter_kernel<8> : sort_scatter_kernel<4>, dim3(NB, B), kSortThreads, a, pass, s, true);
  }
  if (e == cudaSuccess) e = launch(sample_final_kernel, dim3(B), kFinalThreads, a, s, true);
  return e;
}

}  // namespace llm
