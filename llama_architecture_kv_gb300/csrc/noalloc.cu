// llm_sample_noalloc: the sampler without a handle and without any device allocation.
//
// Who needs it: code that must not call cudaMalloc — a caller running inside an allocator
// callback or a memory-pool hook, a plugin whose host application owns every device allocation
// and forbids others, or a process that has reserved all device memory up front.  llm_create
// allocates the sampler's sort buffers inside a handle; this entry point instead keeps them in
// one file-scope device array, so it needs neither a handle nor an allocation.
//
// The scratch array: kScratchBytes of device memory in this library's image, present on every
// GPU that loads the library until the process exits.  Layout: a 256-byte slot for the sampling
// parameters, then keys [B][2][V_pad] (uint32), ids [B][2][V_pad] (int32), running sums
// [B][V_pad] (f32) and the sort's digit counts [B][16][slices] (uint32, slices = the CTAs that
// share one row, at most V / 2048 + 1), V_pad = V rounded up to 32.  B * V_pad may be at most
// LLM_SAMPLE_NOALLOC_MAX_ELEMS (262144, e.g. 2 rows of a 128256-token vocabulary or 5 rows of
// 49152).  Every call writes every element it later reads, so nothing has to start at zero.
// All calls share the array: two calls whose kernels overlap on the GPU (other streams, other
// threads) race on it and their results are undefined.
//
// Host code may not use the array's name as a device pointer (on the host it names a stand-in,
// not device memory).  The set-up (scratch_for_current_device) looks the real address up with
// cudaGetSymbolAddress, with the device current, and records it per device together with the
// device's current context; a later call reuses it while that context is still current, and
// looks it up again after the context changed (cudaDeviceReset, another driver context).
//
// The array belongs to this file's CUDA module.  The runtime loads modules lazily, so the
// module -- and with it the array's device memory -- is created by the set-up, not at library
// load: that first set-up on a device does reserve memory.  llm_create runs it for its device;
// a caller without a handle makes one call on each device from a context that may allocate and
// before any stream capture there.  Calls after that allocate nothing.
#include <cudaTypedefs.h>

#include <mutex>

#include "llm.h"
#include "sampler.cuh"

using namespace llm;

namespace {

constexpr size_t kParamBytes = 256;
constexpr size_t kMaxRows = LLM_SAMPLE_NOALLOC_MAX_ELEMS / 32;
constexpr size_t kHistBytes = 16 * 4 * (LLM_SAMPLE_NOALLOC_MAX_ELEMS / 2048 + kMaxRows);
constexpr size_t kScratchBytes = kParamBytes + (size_t)LLM_SAMPLE_NOALLOC_MAX_ELEMS * (8 + 8 + 4) + kHistBytes;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_sample_scratch[kScratchBytes];

std::mutex g_setup_mu;
unsigned char* g_scratch_ptr[kMaxDevices] = {};
CUcontext g_scratch_ctx[kMaxDevices] = {};  // the context each recorded address belongs to
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
bool g_ctx_queried = false;

// the calling thread's current driver context, or null where the driver entry is unavailable
CUcontext current_context() {
  if (!g_ctx_queried) {
    g_ctx_queried = true;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess && fn)
      g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
  }
  CUcontext c = nullptr;
  if (g_ctx_current && g_ctx_current(&c) != CUDA_SUCCESS) c = nullptr;
  return c;
}

__global__ void noalloc_params_kernel(StepState* st, float temp, int32_t k, float p) {
  st->pos = 0;
  st->B = 0;
  st->temp = temp;
  st->k = k;
  st->p = p;
  st->table = nullptr;
  st->ranges = 0;
  st->rowmap = nullptr;
}

// the scratch address on the current device (looked up again when the device's context changed)
llm_status scratch_for_current_device(unsigned char** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return LLM_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (!g_scratch_ptr[dev]) {
    // (the first runtime call on the device makes its primary context current)
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_sample_scratch) != cudaSuccess || !p) return LLM_ERR_CUDA;
    g_scratch_ptr[dev] = static_cast<unsigned char*>(p);
    g_scratch_ctx[dev] = current_context();
  } else {
    CUcontext c = current_context();
    if (c != g_scratch_ctx[dev]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_sample_scratch) != cudaSuccess || !p) return LLM_ERR_CUDA;
      g_scratch_ptr[dev] = static_cast<unsigned char*>(p);
      g_scratch_ctx[dev] = c;
    }
  }
  *out = g_scratch_ptr[dev];
  return LLM_OK;
}

}  // namespace

namespace llm {
// the set-up of the allocation-free sampler's array on the current device (llm_create runs it)
cudaError_t noalloc_prepare() {
  unsigned char* base = nullptr;
  return scratch_for_current_device(&base) == LLM_OK ? cudaSuccess : cudaErrorInvalidSymbol;
}
}  // namespace llm

extern "C" llm_status llm_sample_noalloc(const float* logits_dev, int32_t B, int32_t V, float temp,
                                         int32_t k, float p, const float* u_dev, int32_t* ids_dev,
                                         void* cuda_stream) {
  if (!logits_dev || !ids_dev || B < 1 || V < 1) return LLM_ERR_ARG;
  const int64_t v_pad = ((int64_t)V + 31) & ~(int64_t)31;
  if ((int64_t)B * v_pad > LLM_SAMPLE_NOALLOC_MAX_ELEMS) return LLM_ERR_ARG;
  if (!(temp >= 0.0f) || temp == INFINITY) return LLM_ERR_ARG;
  if (temp > 0.0f && (k < 1 || !(p > 0.0f && p <= 1.0f) || !u_dev)) return LLM_ERR_ARG;
  unsigned char* base = nullptr;
  if (llm_status s = scratch_for_current_device(&base)) return s;
  cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
  StepState* st = reinterpret_cast<StepState*>(base);
  const size_t n = (size_t)B * (size_t)v_pad;
  uint32_t* keys = reinterpret_cast<uint32_t*>(base + kParamBytes);
  int32_t* idx = reinterpret_cast<int32_t*>(base + kParamBytes + n * 8);
  float* pre = reinterpret_cast<float*>(base + kParamBytes + n * 16);
  uint32_t* hist = reinterpret_cast<uint32_t*>(base + kParamBytes + n * 20);
  // B rows of sample_slices(V) CTAs each; sample_slices(V) <= V / 2048 + 1 and B * V <= the limit
  if ((size_t)B * (size_t)sample_slices(V) * 16 * 4 > kHistBytes) return LLM_ERR_ARG;
  noalloc_params_kernel<<<1, 1, 0, stream>>>(st, temp, k, p);
  if (cudaGetLastError() != cudaSuccess) return LLM_ERR_CUDA;
  SampleArgs a = {};
  a.logits = logits_dev;
  a.logits_stride = V;
  a.V = V;
  a.V_pad = (int32_t)v_pad;
  a.keys = keys;
  a.idx = idx;
  a.pre = pre;
  a.hist = hist;
  a.u = u_dev;
  a.ids = ids_dev;
  a.step = st;
  if (launch_sample(a, B, !(temp > 0.0f), stream, false) != cudaSuccess) return LLM_ERR_CUDA;
  return LLM_OK;
}
