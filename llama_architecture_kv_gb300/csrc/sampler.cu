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
//     id order.  One CTA per row; each thread owns a contiguous run, so the scatter is stable.
//   - weights: exp_s, a fixed sequence of IEEE operations (Cody-Waite reduction, degree-8 Taylor
//     polynomial with fused multiply-adds, scaling by 2^n), never the hardware exp.
//   - the cumulative weights are one sequential f32 running sum; Z is its last value.  Adding
//     non-negative numbers never decreases a rounded sum, so the kept count and the draw are
//     binary searches over that running sum.
#include "sampler.cuh"

namespace llm {

constexpr int kSampThreads = 1024;
constexpr int kDigits = 16;

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
  __shared__ int s_id;

  grid_dep_wait();
  grid_dep_launch();

  const float temp = a.step->temp;
  if (!(temp > 0.0f)) {
    // ---- greedy ----
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
    return;
  }

  // ---- top-k / top-p ----
  extern __shared__ __align__(16) uint32_t cnt[];  // [kDigits][kSampThreads]
  uint32_t* k0 = a.keys + (size_t)b * 2 * a.V_pad;
  uint32_t* k1 = k0 + a.V_pad;
  int32_t* i0 = a.idx + (size_t)b * 2 * a.V_pad;
  int32_t* i1 = i0 + a.V_pad;
  float* pre = a.pre + (size_t)b * a.V_pad;
  const int run = (V + kSampThreads - 1) / kSampThreads;
  const int lo = min(V, tid * run), hi = min(V, lo + run);
  for (int i = lo; i < hi; ++i) {
    k0[i] = desc_key(lg[i]);
    i0[i] = i;
  }
  __syncthreads();
  uint32_t *ks = k0, *kd = k1;
  int32_t *is = i0, *id = i1;
  for (int pass = 0; pass < 8; ++pass) {
    const int sh = 4 * pass;
#pragma unroll
    for (int d = 0; d < kDigits; ++d) cnt[d * kSampThreads + tid] = 0u;
    for (int i = lo; i < hi; ++i) cnt[((ks[i] >> sh) & 15u) * kSampThreads + tid] += 1u;
    __syncthreads();
    // exclusive scan over [digit][thread]: thread t owns entries 16t .. 16t+15
    uint32_t loc[16], sum = 0u;
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      loc[e] = cnt[tid * 16 + e];
      sum += loc[e];
    }
    uint32_t incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    __shared__ uint32_t wtot[32];
    if (lane == 31) wtot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      uint32_t w = wtot[lane], wi = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, wi, o);
        if (lane >= o) wi += v;
      }
      wtot[lane] = wi - w;
    }
    __syncthreads();
    uint32_t run_off = wtot[warp] + incl - sum;
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const uint32_t c = loc[e];
      cnt[tid * 16 + e] = run_off;
      run_off += c;
    }
    __syncthreads();
    for (int i = lo; i < hi; ++i) {
      const uint32_t key = ks[i];
      uint32_t& slot = cnt[((key >> sh) & 15u) * kSampThreads + tid];
      const uint32_t dst = slot++;
      kd[dst] = key;
      id[dst] = is[i];
    }
    __syncthreads();
    uint32_t* tk = ks; ks = kd; kd = tk;
    int32_t* ti = is; is = id; id = ti;
  }
  // ks / is: all ids, largest logit first, ties by id
  const int k = min(a.step->k, V);
  const float top = lg[is[0]];
  const float ttop = __fdiv_rn(top, temp);
  for (int j = tid; j < k; j += kSampThreads) pre[j] = exp_s(__fsub_rn(__fdiv_rn(lg[is[j]], temp), ttop));
  __syncthreads();
  if (tid == 0) {
    float s = 0.0f;
    int j = 0;
    for (; j + 8 <= k; j += 8) {
      float w[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) w[q] = pre[j + q];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        s = __fadd_rn(s, w[q]);
        pre[j + q] = s;
      }
    }
    for (; j < k; ++j) {
      s = __fadd_rn(s, pre[j]);
      pre[j] = s;
    }
    const float Z = s;
    const float lim = __fmul_rn(a.step->p, Z);
    // kept = 1 + number of leading running sums below lim, at most k
    int lo_ = 0, hi_ = k;  // first j with pre[j] >= lim
    while (lo_ < hi_) {
      const int mid = (lo_ + hi_) >> 1;
      if (pre[mid] < lim) lo_ = mid + 1;
      else hi_ = mid;
    }
    const int kept = min(k, lo_ + 1);
    const float zp = pre[kept - 1];
    const float target = __fmul_rn(a.u[b], zp);
    lo_ = 0;
    hi_ = kept - 1;  // first j < kept-1 with target < pre[j], else kept-1
    while (lo_ < hi_) {
      const int mid = (lo_ + hi_) >> 1;
      if (target < pre[mid]) hi_ = mid;
      else lo_ = mid + 1;
    }
    s_id = is[lo_];
  }
  __syncthreads();
  if (tid == 0) a.ids[b] = s_id;
}

size_t sample_smem() { return (size_t)kDigits * kSampThreads * 4; }

cudaError_t sample_prepare() {
  return cudaFuncSetAttribute(sample_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)sample_smem());
}

cudaError_t launch_sample(const SampleArgs& a, int B, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(B);
  cfg.blockDim = dim3(kSampThreads);
  cfg.dynamicSmemBytes = sample_smem();
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, sample_kernel, a);
}

}  // namespace llm
