// All layers of a batch-1 decode step in one persistent kernel (bf16 weights and cache).
//
// The step is the same arithmetic as the per-kernel path (bend-ml-llama "A layer", block;
// "The model", forward): per layer RMSNorm + Q/K/V with RoPE and the cache write, grouped-query
// attention over positions 0..t, o_proj + residual, RMSNorm + gate/up + SwiGLU, down +
// residual; then the final norm, the LM head and (optionally) the greedy argmax.
//
// Design: one CTA of 8 warps per SM, launched cooperatively so that every CTA is resident.  The
// phases of the step (five per layer, then the head) are separated by grid barriers (an atomic
// counter that thread 0 of every CTA bumps and polls, with a bounded wait) only where
// activations flow.  The weights do not depend on the activations, so each warp streams its
// whole sequence of weight pieces -- phase after phase, layer after layer -- through one private
// ring of shared-memory slots (two cp.async.bulk copies of 4 KB on one mbarrier per slot), two
// steps ahead of its computation: when a warp reaches a barrier its first pieces of the next
// phase are already in flight, so HBM does not idle across phase boundaries.  In the attention
// phase the same ring carries 16-position chunks of keys and values; a chunk holding position t
// (written by this step's Q/K/V phase) is copied only after that phase's barrier.
//   GEMV phases: rows in pairs ("groups": a RoPE pair, a gate/up pair, two neighbouring rows); a
//     CTA owns a balanced range of groups; a step is the same 4 KB piece of both rows, dealt to
//     the CTA's warps in turn; the (normalized) input sits in shared memory as f32 in two planes
//     (elements 0-3 and 4-7 of each 8-element chunk); each step's two warp sums go to shared
//     memory and the epilogue adds each row's pieces in order (as gemv_tma_kernel).
//   Attention phase: kv head j gets S = grid / kv CTAs, each a contiguous range of 16-position
//     chunks; lanes 0-15 / 16-31 score the chunk's positions for the group's even / odd heads,
//     an online softmax per head, then every lane accumulates its hd/32 dimensions of every
//     head; the warps' partials merge with one factor per (warp, head), the CTAs' partials of a
//     head are merged in split order by the last of them to finish (atomic ticket).
#include "mega.cuh"
#include "tc.cuh"

namespace llm {

constexpr int kMW = 8;                  // warps per CTA
constexpr int kMPiece = 4096;           // bytes of one row (or of 16 cache rows) per step
constexpr int kMStep = 2 * kMPiece;     // a step: two rows, or the keys and values of a chunk
constexpr int kMNS = 2;                 // steps in flight per warp
constexpr int kMChunk = 16;             // positions per attention step
constexpr int kMMaxG = 8;               // query heads per kv head
constexpr uint64_t kMWait = 4000000000ull;  // SM cycles: about 2 s at 2 GHz

enum { PH_QKV = 0, PH_ATTN = 1, PH_O = 2, PH_GU = 3, PH_DOWN = 4, PH_PER_LAYER = 5, PH_HEAD = 5 };

// the front of shared memory: the input planes of a GEMV phase, or the attention scratch
static LLM_HD size_t mega_x_bytes(int d, int f) {
  const int w = d > f ? d : f;
  size_t b = (size_t)w * 4;
  const size_t att = ((size_t)kMMaxG * 128 + (size_t)(kMW + 1) * kMMaxG * 130) * 4;
  if (att > b) b = att;
  return (b + 1023) & ~(size_t)1023;
}
static LLM_HD size_t mega_part_floats(int d, int f, int V, int grid) {
  // the largest per-CTA step count of any GEMV phase, two sums per step
  auto steps = [&](int rows, int cols) {
    const int groups = (rows + 1) / 2;
    const int per = (groups + grid - 1) / grid;
    return (size_t)per * (size_t)(((size_t)cols * 2 + kMPiece - 1) / kMPiece);
  };
  size_t s = steps(2 * f, d);
  const size_t s2 = steps(d, f), s3 = steps(V, d), s4 = steps(3 * d, d);
  if (s2 > s) s = s2;
  if (s3 > s) s = s3;
  if (s4 > s) s = s4;
  return 2 * s;
}

LLM_D uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// the position of the step and this CTA's share of phase ph
struct MPhase {
  int kind, layer;
  const char* W;     // GEMV weights
  int rows, cols, ppr, g0, g1;
  int j, split, c0, c1;  // attention: kv head, split, chunk range
  int nsteps;        // this CTA's steps
};

template <int HD>
__global__ void __launch_bounds__(kMW * 32, 1) mega_kernel(const MegaArgs a) {
  extern __shared__ __align__(1024) uint8_t msm[];
  constexpr int NW = kMW;
  constexpr int ROWB = HD * 2;
  constexpr int DPL = HD / 32;  // value dimensions per lane
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x, G = gridDim.x;
  const int d = a.d, f = a.f, g = a.g, kv = a.kv, H = a.H, cap = a.cap;
  const int t = a.step->pos;
  const int nph = a.L * PH_PER_LAYER + (a.head_mode ? 1 : 0);
  const int S = (G / kv) < kMegaMaxSplits ? G / kv : kMegaMaxSplits;  // attention splits per kv head

  const size_t xbytes = mega_x_bytes(d, f);
  float* xlo = reinterpret_cast<float*>(msm);  // input planes (GEMV phases)
  uint8_t* ring = msm + xbytes;
  const uint32_t ring_s = smem_u32(ring);
  const uint32_t bars = ring_s + (uint32_t)(NW * kMNS * kMStep);
  float* part = reinterpret_cast<float*>(ring + (size_t)NW * kMNS * (kMStep + 8));
  // attention scratch (aliases the input planes, unused in that phase)
  float* qsm = xlo;                                  // [g][HD]
  float* wpart = qsm + kMMaxG * HD;                  // [NW][g][HD + 2]
  float* mypart = wpart + NW * kMMaxG * (HD + 2);    // [g][HD + 2]
  __shared__ float red[NW];
  __shared__ float s_inv;
  __shared__ float wfac[NW * kMMaxG];
  __shared__ float fac[kMegaMaxSplits * kMMaxG];
  __shared__ int s_last;
  __shared__ float s_bv[NW];
  __shared__ int s_bi[NW];

  // ---- phase descriptors -------------------------------------------------------------------
  auto phase = [&](int ph) {
    MPhase P;
    P.kind = ph >= a.L * PH_PER_LAYER ? PH_HEAD : ph % PH_PER_LAYER;
    P.layer = ph >= a.L * PH_PER_LAYER ? 0 : ph / PH_PER_LAYER;
    P.W = nullptr;
    P.rows = P.cols = P.ppr = P.g0 = P.g1 = 0;
    P.j = P.split = P.c0 = P.c1 = 0;
    if (P.kind == PH_ATTN) {
      const int nchk = (t + 1 + kMChunk - 1) / kMChunk;
      if (c < kv * S) {
        P.j = c / S;
        P.split = c - P.j * S;
        P.c0 = (int)(((long long)nchk * P.split) / S);
        P.c1 = (int)(((long long)nchk * (P.split + 1)) / S);
      }
      P.nsteps = P.c1 - P.c0;
      return P;
    }
    const MegaLayer& Lw = a.layers[P.layer];
    switch (P.kind) {
      case PH_QKV: P.W = (const char*)Lw.qkv; P.rows = (H + 2 * kv) * HD; P.cols = d; break;
      case PH_O: P.W = (const char*)Lw.o; P.rows = d; P.cols = d; break;
      case PH_GU: P.W = (const char*)Lw.gu; P.rows = 2 * f; P.cols = d; break;
      case PH_DOWN: P.W = (const char*)Lw.down; P.rows = d; P.cols = f; break;
      default: P.W = (const char*)a.head; P.rows = a.V; P.cols = d; break;
    }
    const int groups = (P.rows + 1) >> 1;
    P.g0 = (int)(((long long)groups * c) / G);
    P.g1 = (int)(((long long)groups * (c + 1)) / G);
    P.ppr = (int)(((size_t)P.cols * 2 + kMPiece - 1) / kMPiece);
    P.nsteps = (P.g1 - P.g0) * P.ppr;
    return P;
  };
  auto warp_steps = [&](const MPhase& P) { return P.nsteps > warp ? (P.nsteps - warp + NW - 1) / NW : 0; };

  if (tid == 0) {
    for (int i = 0; i < NW * kMNS; ++i) mbar_init(bars + 8u * i, 1);
    mbar_fence_init();
  }
  __syncthreads();

  // ---- the issuing side of this warp (lane 0): a cursor over (phase, step) ------------------
  int iph = 0, it = 0, issued = 0, consumed = 0;
  MPhase IP = phase(0);
  auto settle = [&]() {
    while (iph < nph && it >= warp_steps(IP)) {
      ++iph;
      it = 0;
      if (iph < nph) IP = phase(iph);
    }
  };
  settle();
  int cur = 0;  // the phase this CTA is in (the number of barriers it has passed)
  // the cursor's step may be copied now: a chunk holding position t only once the Q/K/V phase
  // of its layer is over
  auto allowed = [&]() {
    if (IP.kind != PH_ATTN) return true;
    const int p = (IP.c0 + warp + it * NW) * kMChunk;
    return p + kMChunk <= t || cur >= iph;
  };
  auto issue = [&]() {
    const int slot = issued % kMNS;
    const uint32_t bar = bars + 8u * (warp * kMNS + slot);
    const uint32_t dst = ring_s + (uint32_t)((warp * kMNS + slot) * kMStep);
    const int q = warp + it * NW;
    const char* s0;
    const char* s1;
    uint32_t bytes;
    if (IP.kind == PH_ATTN) {
      const int p = (IP.c0 + q) * kMChunk;
      const int n = (t + 1 - p) < kMChunk ? t + 1 - p : kMChunk;
      int r, pp;  // the cache row and position holding position p of row 0 (paged steps: its page)
      cache_slot(a.step, cap, 0, p, r, pp);
      const size_t row = (((size_t)IP.layer * a.max_batch + r) * kv + IP.j) * cap + pp;
      s0 = (const char*)a.kc + row * ROWB;
      s1 = (const char*)a.vc + row * ROWB;
      bytes = (uint32_t)(n * ROWB);
    } else {
      const int gi = q / IP.ppr, pc = q - gi * IP.ppr;
      const size_t rb = (size_t)IP.cols * 2;
      const size_t r0 = 2 * (size_t)(IP.g0 + gi);
      const size_t r1 = r0 + 1 < (size_t)IP.rows ? r0 + 1 : r0;
      const size_t off = (size_t)pc * kMPiece;
      bytes = (uint32_t)(rb - off < (size_t)kMPiece ? rb - off : (size_t)kMPiece);
      s0 = IP.W + r0 * rb + off;
      s1 = IP.W + r1 * rb + off;
    }
    fence_proxy_async_smem();
    mbar_expect_tx(bar, 2 * bytes);
    bulk_load(dst, s0, bytes, bar);
    bulk_load(dst + kMPiece, s1, bytes, bar);
    ++issued;
    ++it;
    settle();
  };
  auto pump = [&]() {
    if (lane == 0)
      while (issued - consumed < kMNS && iph < nph && allowed()) issue();
    __syncwarp();
  };
  pump();

  bool ok = true;
  // grid barrier: every CTA's writes of this phase happen before any CTA's reads of the next
  auto grid_barrier = [&](uint32_t target) {
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      atomicAdd(a.bar, 1u);
      const uint64_t t0 = clock64();
      for (uint32_t i = 0; i < (1u << 30); ++i) {
        if (ld_acquire_u32(a.bar) >= target) break;
        // after a wait that ran out anywhere in the grid, later barriers do not wait (bounded total)
        if (ld_acquire_u32(reinterpret_cast<const uint32_t*>(a.status)) == (uint32_t)kErrDeviceTimeout) break;
        if ((uint64_t)clock64() - t0 > kMWait) {
          atomicCAS(a.status, 0, kErrDeviceTimeout);
          break;
        }
      }
      __threadfence();
    }
    __syncthreads();
  };

  // stage x' = norm ? g * x * inv_rms(x) : x into the two planes
  auto stage = [&](const float* x, const float* gain, int cols) {
    const int c4 = cols >> 2;
    const float4* xr = reinterpret_cast<const float4*>(x);
    float inv = 1.f;
    if (gain) {
      float ss = 0.f;
      for (int i = tid; i < c4; i += NW * 32) {
        const float4 v = __ldcg(xr + i);
        ss = fmaf(v.x, v.x, ss);
        ss = fmaf(v.y, v.y, ss);
        ss = fmaf(v.z, v.z, ss);
        ss = fmaf(v.w, v.w, ss);
      }
      ss = warp_sum(ss);
      if (lane == 0) red[warp] = ss;
      __syncthreads();
      if (tid == 0) {
        float s2 = 0.f;
        for (int w = 0; w < NW; ++w) s2 += red[w];
        s_inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(s2, (float)cols), a.eps)));
      }
      __syncthreads();
      inv = s_inv;
    }
    float* xhi = xlo + (cols >> 1);
    for (int i = tid; i < c4; i += NW * 32) {
      float4 v = __ldcg(xr + i);
      if (gain) {
        const float4 gv = __ldg(reinterpret_cast<const float4*>(gain) + i);
        v.x = __fmul_rn(gv.x, __fmul_rn(inv, v.x));
        v.y = __fmul_rn(gv.y, __fmul_rn(inv, v.y));
        v.z = __fmul_rn(gv.z, __fmul_rn(inv, v.z));
        v.w = __fmul_rn(gv.w, __fmul_rn(inv, v.w));
      }
      reinterpret_cast<float4*>((i & 1) ? xhi : xlo)[i >> 1] = v;
    }
    __syncthreads();
  };

  // wait for step number `consumed` of this warp
  auto wait_step = [&]() {
    const int slot = consumed % kMNS;
    const bool w = mbar_wait(bars + 8u * (warp * kMNS + slot), (uint32_t)(consumed / kMNS) & 1u, kMWait);
    return __all_sync(0xffffffffu, w);
  };

  for (int ph = 0; ph < nph; ++ph) {
    cur = ph;
    if (ph > 0) grid_barrier((uint32_t)G * (uint32_t)ph);
    pump();  // a chunk held back for this phase may go now
    const MPhase P = phase(ph);
    const int ns = warp_steps(P);

    if (P.kind == PH_ATTN) {
      // ---------------------------------------------------------------- attention
      const bool active = c < kv * S;
      if (active)
        for (int i = tid; i < g * HD; i += NW * 32) qsm[i] = __ldcg(a.q + (size_t)P.j * g * HD + i);
      __syncthreads();
      const int pl = lane & 15, par = lane >> 4;  // score lane: position, head parity
      float mrun[kMMaxG], lrun[kMMaxG], o[kMMaxG][DPL];
#pragma unroll
      for (int h = 0; h < kMMaxG; ++h) {
        mrun[h] = -INFINITY;
        lrun[h] = 0.f;
#pragma unroll
        for (int e = 0; e < DPL; ++e) o[h][e] = 0.f;
      }
      for (int k = 0; k < ns; ++k) {
        if (!(ok = ok && wait_step())) break;
        const uint8_t* kr = ring + (size_t)(warp * kMNS + consumed % kMNS) * kMStep;
        const uint8_t* vr = kr + kMPiece;
        const int p0 = (P.c0 + warp + k * NW) * kMChunk;
        const int n = (t + 1 - p0) < kMChunk ? t + 1 - p0 : kMChunk;
        const bool valid = pl < n;
        // scores of this lane's position for the heads of its parity (16-byte units of the key
        // row rotated by the position, so that the half-warp's reads spread over the banks)
        float sc[kMMaxG / 2];
#pragma unroll
        for (int hh = 0; hh < kMMaxG / 2; ++hh) sc[hh] = 0.f;
#pragma unroll 4
        for (int u0 = 0; u0 < HD / 8; ++u0) {
          const int u = (u0 + pl) & (HD / 8 - 1);
          float kf[8];
          unpack16<1>(*reinterpret_cast<const uint4*>(kr + pl * ROWB + u * 16), kf);
#pragma unroll
          for (int hh = 0; hh < kMMaxG / 2; ++hh) {
            const int h = 2 * hh + par;
            if (h < g) {
              const float4 q0 = *reinterpret_cast<const float4*>(qsm + h * HD + u * 8);
              const float4 q1 = *reinterpret_cast<const float4*>(qsm + h * HD + u * 8 + 4);
              float s = sc[hh];
              s = fmaf(q0.x, kf[0], s);
              s = fmaf(q0.y, kf[1], s);
              s = fmaf(q0.z, kf[2], s);
              s = fmaf(q0.w, kf[3], s);
              s = fmaf(q1.x, kf[4], s);
              s = fmaf(q1.y, kf[5], s);
              s = fmaf(q1.z, kf[6], s);
              s = fmaf(q1.w, kf[7], s);
              sc[hh] = s;
            }
          }
        }
        // online softmax per head: max and sum over the 16 lanes of its parity
        float wl[kMMaxG / 2];
#pragma unroll
        for (int hh = 0; hh < kMMaxG / 2; ++hh) {
          const float s = valid ? sc[hh] * a.scale : -INFINITY;
          float mx = s;
#pragma unroll
          for (int off = 8; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
          sc[hh] = s;
          wl[hh] = mx;  // (the chunk maximum, for now)
        }
#pragma unroll
        for (int h = 0; h < kMMaxG; ++h) {
          if (h < g) {
            const float mx = __shfl_sync(0xffffffffu, wl[h >> 1], (h & 1) * 16);
            const float mnew = fmaxf(mrun[h], mx);  // finite: position p0 is in the range
            const float corr = mrun[h] == -INFINITY ? 0.f : expf(mrun[h] - mnew);
            mrun[h] = mnew;
            lrun[h] *= corr;
#pragma unroll
            for (int e = 0; e < DPL; ++e) o[h][e] *= corr;
          }
        }
#pragma unroll
        for (int hh = 0; hh < kMMaxG / 2; ++hh) {
          const int h = 2 * hh + par;
          const float mine = par ? mrun[2 * hh + 1] : mrun[2 * hh];  // (static indices: no spill)
          wl[hh] = (h < g && sc[hh] != -INFINITY) ? expf(sc[hh] - mine) : 0.f;
          float sum = wl[hh];
#pragma unroll
          for (int off = 8; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
          sc[hh] = sum;  // the chunk's weight sum of head h (on the lanes of its parity)
        }
#pragma unroll
        for (int h = 0; h < kMMaxG; ++h)
          if (h < g) lrun[h] += __shfl_sync(0xffffffffu, sc[h >> 1], (h & 1) * 16);
        // values: this lane's DPL dimensions of every head
#pragma unroll 2
        for (int p = 0; p < n; ++p) {
          float vf[DPL];
          if constexpr (DPL == 4) {
            const uint2 u = *reinterpret_cast<const uint2*>(vr + p * ROWB + lane * 8);
            vf[0] = bf16_lo(u.x); vf[1] = bf16_hi(u.x); vf[2] = bf16_lo(u.y); vf[3] = bf16_hi(u.y);
          } else {
            const uint32_t u = *reinterpret_cast<const uint32_t*>(vr + p * ROWB + lane * 4);
            vf[0] = bf16_lo(u); vf[1] = bf16_hi(u);
          }
#pragma unroll
          for (int h = 0; h < kMMaxG; ++h) {
            if (h < g) {
              const float w = __shfl_sync(0xffffffffu, wl[h >> 1], p + (h & 1) * 16);
#pragma unroll
              for (int e = 0; e < DPL; ++e) o[h][e] = fmaf(w, vf[e], o[h][e]);
            }
          }
        }
        __syncwarp();
        ++consumed;
        pump();
      }
      // warp partials, then the CTA's, then the split merge
#pragma unroll
      for (int h = 0; h < kMMaxG; ++h) {
        if (h < g) {
          float* wp = wpart + (warp * kMMaxG + h) * (HD + 2);
#pragma unroll
          for (int e = 0; e < DPL; ++e) wp[lane * DPL + e] = o[h][e];
          if (lane == 0) {
            wp[HD] = mrun[h];
            wp[HD + 1] = lrun[h];
          }
        }
      }
      __syncthreads();
      for (int i = tid; i < g * NW; i += NW * 32) {
        const int h = i / NW, w = i - h * NW;
        float Mx = -INFINITY;
        for (int w2 = 0; w2 < NW; ++w2) Mx = fmaxf(Mx, wpart[(w2 * kMMaxG + h) * (HD + 2) + HD]);
        const float mw = wpart[(w * kMMaxG + h) * (HD + 2) + HD];
        wfac[i] = mw == -INFINITY ? 0.f : expf(mw - Mx);
        if (w == 0) mypart[h * (HD + 2) + HD] = Mx;
      }
      __syncthreads();
      for (int idx = tid; idx < g * (HD + 2); idx += NW * 32) {
        const int h = idx / (HD + 2), e = idx - h * (HD + 2);
        if (e == HD) continue;
        float r = 0.f;
        for (int w = 0; w < NW; ++w) r = fmaf(wfac[h * NW + w], wpart[(w * kMMaxG + h) * (HD + 2) + e], r);
        mypart[idx] = r;
      }
      __syncthreads();
      if (active) {
        float* pg = a.apart + ((size_t)P.j * g * kMegaMaxSplits) * (HD + 2);  // [g][splits][HD + 2]
        for (int idx = tid; idx < g * (HD + 2); idx += NW * 32) {
          const int h = idx / (HD + 2), e = idx - h * (HD + 2);
          pg[((size_t)h * kMegaMaxSplits + P.split) * (HD + 2) + e] = mypart[idx];
        }
        __threadfence();
        __syncthreads();
        if (tid == 0) s_last = atomicAdd(a.ticket + P.j, 1u) == (unsigned)(S - 1);
        __syncthreads();
        if (s_last) {
          __threadfence();
          for (int h = tid; h < g; h += NW * 32) {
            float Mx = -INFINITY;
            for (int s2 = 0; s2 < S; ++s2) Mx = fmaxf(Mx, __ldcg(pg + ((size_t)h * kMegaMaxSplits + s2) * (HD + 2) + HD));
            float L = 0.f;
            for (int s2 = 0; s2 < S; ++s2) {
              const float* pp = pg + ((size_t)h * kMegaMaxSplits + s2) * (HD + 2);
              const float ms = __ldcg(pp + HD);
              const float fct = ms == -INFINITY ? 0.f : expf(ms - Mx);
              fac[h * kMegaMaxSplits + s2] = fct;
              L += __ldcg(pp + HD + 1) * fct;
            }
            const float rl = 1.0f / L;
            for (int s2 = 0; s2 < S; ++s2) fac[h * kMegaMaxSplits + s2] *= rl;
          }
          __syncthreads();
          for (int idx = tid; idx < g * HD; idx += NW * 32) {
            const int h = idx / HD, e = idx - h * HD;
            float O = 0.f;
            for (int s2 = 0; s2 < S; ++s2)
              O = fmaf(fac[h * kMegaMaxSplits + s2], __ldcg(pg + ((size_t)h * kMegaMaxSplits + s2) * (HD + 2) + e), O);
            a.attn[(size_t)P.j * g * HD + idx] = O;
          }
          if (tid == 0) a.ticket[P.j] = 0u;
        }
      }
      continue;
    }

    // -------------------------------------------------------------------- GEMV phases
    {
      const MegaLayer& Lw = a.layers[P.layer];
      if (P.kind == PH_QKV) stage(a.x, Lw.ln1, d);
      else if (P.kind == PH_O) stage(a.attn, nullptr, d);
      else if (P.kind == PH_GU) stage(a.x1, Lw.ln2, d);
      else if (P.kind == PH_DOWN) stage(a.m, nullptr, f);
      else stage(a.x, a.lnf, d);
    }
    const size_t rb = (size_t)P.cols * 2;
    const float* xl0 = xlo;
    const float* xh0 = xlo + (P.cols >> 1);
    float a0[2], a1[2];
    for (int k = 0; k < ns; ++k) {
      if (!(ok = ok && wait_step())) break;
      const int q = warp + k * NW;
      const int pc = q - (q / P.ppr) * P.ppr;
      const size_t off = (size_t)pc * kMPiece;
      const int nch = (int)((rb - off < (size_t)kMPiece ? rb - off : (size_t)kMPiece) >> 4);
      const uint8_t* w0 = ring + (size_t)(warp * kMNS + consumed % kMNS) * kMStep;
      const float* xl = xl0 + (size_t)pc * (kMPiece / 4);
      const float* xh = xh0 + (size_t)pc * (kMPiece / 4);
      a0[0] = a0[1] = a1[0] = a1[1] = 0.f;
      auto chunk = [&](int jj, int pr) {
        float f0[8], f1[8];
        unpack16<1>(*reinterpret_cast<const uint4*>(w0 + jj * 16), f0);
        unpack16<1>(*reinterpret_cast<const uint4*>(w0 + kMPiece + jj * 16), f1);
        const float4 lo = *reinterpret_cast<const float4*>(xl + jj * 4);
        const float4 hi = *reinterpret_cast<const float4*>(xh + jj * 4);
        const float xv[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          a0[pr] = fmaf(f0[e], xv[e], a0[pr]);
          a1[pr] = fmaf(f1[e], xv[e], a1[pr]);
        }
      };
      if (nch == kMPiece / 16) {
#pragma unroll
        for (int i = 0; i < kMPiece / 16 / 32; ++i) chunk(lane + 32 * i, i & 1);
      } else {
        for (int jj = lane; jj < nch; jj += 32) chunk(jj, 0);
      }
      const float v0 = warp_sum(a0[0] + a0[1]);
      const float v1 = warp_sum(a1[0] + a1[1]);
      if (lane == 0) {
        part[2 * q] = v0;
        part[2 * q + 1] = v1;
      }
      __syncwarp();
      ++consumed;
      pump();
    }
    __syncthreads();
    // epilogue: each group's two rows, pieces added in order
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int i = tid; i < P.g1 - P.g0; i += NW * 32) {
      float v0 = 0.f, v1 = 0.f;
      for (int pc = 0; pc < P.ppr; ++pc) {
        v0 += part[2 * (i * P.ppr + pc)];
        v1 += part[2 * (i * P.ppr + pc) + 1];
      }
      const int gg = P.g0 + i;
      const int r0 = 2 * gg;
      if (P.kind == PH_QKV) {
        const int half = HD >> 1;
        const int head = r0 / HD, e = (r0 - head * HD) >> 1;
        int cr, cp;  // the cache row and position of position t of row 0
        cache_slot(a.step, cap, 0, t, cr, cp);
        const size_t cbase = (((size_t)P.layer * a.max_batch + cr) * kv) * cap;
        if (head < H + kv) {
          const float cs = a.rope_cos[(size_t)t * half + e], sn = a.rope_sin[(size_t)t * half + e];
          const float lo = __fadd_rn(__fmul_rn(v0, cs), __fmul_rn(-v1, sn));
          const float hi = __fadd_rn(__fmul_rn(v1, cs), __fmul_rn(v0, sn));
          if (head < H) {
            a.q[(size_t)head * HD + e] = lo;
            a.q[(size_t)head * HD + e + half] = hi;
          } else {
            const size_t ci = ((cbase + (size_t)(head - H) * cap) + cp) * HD;
            store_elem<1>(a.kc, ci + e, lo);
            store_elem<1>(a.kc, ci + e + half, hi);
          }
        } else {
          const size_t ci = ((cbase + (size_t)(head - H - kv) * cap) + cp) * HD;
          store_elem<1>(a.vc, ci + e, v0);
          store_elem<1>(a.vc, ci + e + half, v1);
        }
      } else if (P.kind == PH_O) {
        a.x1[r0] = __fadd_rn(__ldcg(a.x + r0), v0);
        if (r0 + 1 < P.rows) a.x1[r0 + 1] = __fadd_rn(__ldcg(a.x + r0 + 1), v1);
      } else if (P.kind == PH_GU) {
        const float si = __fdiv_rn(v0, __fadd_rn(1.0f, expf(-v0)));
        a.m[gg] = __fmul_rn(si, v1);
      } else if (P.kind == PH_DOWN) {
        a.x[r0] = __fadd_rn(__ldcg(a.x1 + r0), v0);
        if (r0 + 1 < P.rows) a.x[r0 + 1] = __fadd_rn(__ldcg(a.x1 + r0 + 1), v1);
      } else {
        a.logits[r0] = v0;
        if (v0 > bv || (v0 == bv && r0 < bi)) { bv = v0; bi = r0; }
        if (r0 + 1 < P.rows) {
          a.logits[r0 + 1] = v1;
          if (v1 > bv || (v1 == bv && r0 + 1 < bi)) { bv = v1; bi = r0 + 1; }
        }
      }
    }
    if (P.kind == PH_HEAD && a.head_mode == 2) {
      // the first index of the largest logit: this CTA's candidate, then the last CTA's reduction
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
      }
      if (lane == 0) {
        s_bv[warp] = bv;
        s_bi[warp] = bi;
      }
      __syncthreads();
      if (tid == 0) {
        bv = s_bv[0];
        bi = s_bi[0];
        for (int w = 1; w < NW; ++w)
          if (s_bv[w] > bv || (s_bv[w] == bv && s_bi[w] < bi)) { bv = s_bv[w]; bi = s_bi[w]; }
        a.cand_v[c] = bv;
        a.cand_i[c] = bi;
        __threadfence();
        s_last = atomicAdd(a.ticket + kv, 1u) == (unsigned)(G - 1);
        if (s_last) {
          __threadfence();
          float fv = -INFINITY;
          int fi = 0x7fffffff;
          for (int cc = 0; cc < G; ++cc) {
            const float cv = __ldcg(a.cand_v + cc);
            const int ci = __ldcg(a.cand_i + cc);
            if (cv > fv || (cv == fv && ci < fi)) { fv = cv; fi = ci; }
          }
          a.ids[0] = fi == 0x7fffffff ? 0 : fi;
          a.ticket[kv] = 0u;
        }
      }
    }
  }
  if (!ok && lane == 0) atomicCAS(a.status, 0, kErrDeviceTimeout);
  // no copy may still be writing shared memory when the CTA exits
  if (lane == 0)
    for (int k = consumed; k < issued; ++k)
      mbar_wait(bars + 8u * (warp * kMNS + k % kMNS), (uint32_t)(k / kMNS) & 1u, kMWait);
}

// ---------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------



bool mega_supported(int wt, int hd, int g, int d, int f) {
  return wt == 1 && (hd == 64 || hd == 128) && g >= 1 && g <= kMMaxG && d % 8 == 0 && f % 8 == 0;
}

size_t mega_smem(int d, int f) {
  // the input planes (or the attention scratch, the larger), the rings and their barriers, and the
  // partial sums (sized for the largest phase of a 152-CTA grid at the widest shapes here)
  return mega_x_bytes(d, f) + (size_t)kMW * kMNS * (kMStep + 8) + 8192 * 4;
}

cudaError_t mega_prepare(int max_smem_optin) {
  for (auto fn : {mega_kernel<64>, mega_kernel<128>}) {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, fn);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem_optin - (int)fa.sharedSizeBytes);
    if (e != cudaSuccess) return e;
  }

  return cudaSuccess;
}

cudaError_t launch_mega(const MegaArgs& a, int grid, cudaStream_t s) {
  if (mega_part_floats(a.d, a.f, a.V, grid) > 8192) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kMW * 32);
  cfg.dynamicSmemBytes = mega_smem(a.d, a.f);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (a.hd == 64) return cudaLaunchKernelEx(&cfg, mega_kernel<64>, a);
  return cudaLaunchKernelEx(&cfg, mega_kernel<128>, a);
}

}  // namespace llm
