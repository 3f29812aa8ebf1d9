// Device helpers shared by the kernels of libllm (sm_103a).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#define LLM_HD __host__ __device__ __forceinline__
#define LLM_D __device__ __forceinline__

namespace llm {

// ---- element types ----------------------------------------------------------------------
// Weights and cache are stored as f32 or as bf16 bit patterns (uint16).  Widening bf16 to
// f32 is exact (the bf16 bits are the upper half of the f32).

LLM_D float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
LLM_D float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }
LLM_D float bf16_to_f32(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

// f32 -> bf16 bits, round to nearest even (NaN stays NaN)
LLM_D uint16_t f32_to_bf16(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7f800000u) == 0x7f800000u) return (uint16_t)((u >> 16) | ((u & 0xffffu) ? 0x40u : 0u));
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

template <int WT> struct Elem;  // WT: 0 = f32, 1 = bf16
template <> struct Elem<0> {
  using T = float;
  static constexpr int per16 = 4;  // elements per 16-byte chunk
  static constexpr int bytes = 4;
};
template <> struct Elem<1> {
  using T = uint16_t;
  static constexpr int per16 = 8;
  static constexpr int bytes = 2;
};

// unpack a 16-byte chunk into f32 values
template <int WT> LLM_D void unpack16(const uint4& w, float* f);
template <> LLM_D void unpack16<0>(const uint4& w, float* f) {
  f[0] = __uint_as_float(w.x);
  f[1] = __uint_as_float(w.y);
  f[2] = __uint_as_float(w.z);
  f[3] = __uint_as_float(w.w);
}
template <> LLM_D void unpack16<1>(const uint4& w, float* f) {
  f[0] = bf16_lo(w.x); f[1] = bf16_hi(w.x);
  f[2] = bf16_lo(w.y); f[3] = bf16_hi(w.y);
  f[4] = bf16_lo(w.z); f[5] = bf16_hi(w.z);
  f[6] = bf16_lo(w.w); f[7] = bf16_hi(w.w);
}

template <int WT> LLM_D float load_elem(const void* p, uint64_t i) {
  if constexpr (WT == 0) return ((const float*)p)[i];
  else return bf16_to_f32(((const uint16_t*)p)[i]);
}
template <int WT> LLM_D void store_elem(void* p, uint64_t i, float v) {
  if constexpr (WT == 0) ((float*)p)[i] = v;
  else ((uint16_t*)p)[i] = f32_to_bf16(v);
}

// ---- memory -----------------------------------------------------------------------------

// streaming read of data read once (weights): no L1 allocation
LLM_D uint4 ld_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// hint: bring [p, p+bytes) into L2 (p 16-byte aligned, bytes a multiple of 16)
LLM_D void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// ---- programmatic dependent launch ----------------------------------------------------
// Kernels of one decode step are launched with programmatic stream serialization: a kernel
// may start while its predecessor drains; it must not touch memory the predecessor writes
// (or reads and it writes) before grid_dep_wait(), which returns once the predecessor grid
// has completed and its writes are visible.
LLM_D void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
LLM_D void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---- reductions -------------------------------------------------------------------------
LLM_D float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
LLM_D float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// ---- step parameters written by the step prologue --------------------------------------
// The state is followed in memory by the position of every row ([B] int32): rows may sit at
// different positions (a decode of rows at their own positions); pos is their maximum.  A prefill
// pass (its rows are prompt tokens, "entries") adds each entry's attention start, the first
// position the pass writes in the entry's cache row, and that cache row ([B] each) after them.
struct StepState {
  int32_t pos;     // the largest position of this step's rows
  int32_t B;       // rows in this step
  float temp;      // sampling: temperature (0: greedy)
  int32_t k;       // sampling: top-k
  float p;         // sampling: top-p
  int32_t table_stride;  // paged steps: entries per row of table
  const int32_t* table;  // paged steps: [B][table_stride] pool pages of each row's positions, or null
  int32_t ranges;        // 1: the rows' attention ranges follow their positions (prefill passes)
  int32_t pad;
  const int32_t* rowmap; // prefill passes: [B] cache row of each entry (no table), or null
};
// position of row b in this step
LLM_D int32_t row_pos(const StepState* s, int b) { return reinterpret_cast<const int32_t*>(s + 1)[b]; }
// Row b attends to positions row_start .. row_pos (0 .. row_pos unless ranges are given); this
// step writes its row's positions from row_wfirst on (row_pos itself unless ranges are given),
// so only cache positions below it may be read before the previous kernel finishes.
LLM_D int32_t row_start(const StepState* s, int b) {
  return s->ranges ? reinterpret_cast<const int32_t*>(s + 1)[s->B + b] : 0;
}
LLM_D int32_t row_wfirst(const StepState* s, int b) {
  return s->ranges ? reinterpret_cast<const int32_t*>(s + 1)[2 * s->B + b] : row_pos(s, b);
}

// Paged caches (Llama 3.1 8B Instruct card, "Entries": decode_paged): the cache of a layer is a
// pool of pages of kPage positions; page q is positions [(q % (cap / kPage)) * kPage, + kPage) of
// cache row q / (cap / kPage).  Position pos of row b lies in page table[b][pos / kPage]; without
// a table it lies in row b itself, or, in a prefill pass, in the entry's cache row rowmap[b].
// (r, pp): the cache row and position that hold it.
constexpr int kPage = 64;
LLM_D void cache_slot(const StepState* s, int cap, int b, int pos, int& r, int& pp) {
  if (!s->table) {
    r = s->rowmap ? s->rowmap[b] : b;
    pp = pos;
    return;
  }
  const int per_row = cap / kPage;
  const int page = s->table[(size_t)b * s->table_stride + pos / kPage];
  r = page / per_row;
  pp = (page - r * per_row) * kPage + (pos & (kPage - 1));
}
LLM_HD size_t step_state_bytes(int max_rows) { return sizeof(StepState) + (size_t)max_rows * 4 * 4; }

// device error codes (same values as llm.h)

constexpr int32_t kErrTokenRange = 5;
constexpr int32_t kErrDeviceTimeout = 9;

}  // namespace llm
