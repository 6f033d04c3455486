// Bias-gradient column sum whose scratch is a static device array, for callers
// that cannot allocate device memory (declared in oases_debug.h).
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "oases_debug.h"

namespace oases {
void api_begin();
void api_set_error(const char* what);
oases_status api_end(cudaError_t e);
}  // namespace oases

namespace {

// Partial rows of the two-stage column sum; one copy per device, kept for the
// life of the process.  Host code must not use this name as a device address.
static __device__ __align__(256) float g_noalloc_scratch[OASES_NOALLOC_SCRATCH_FLOATS];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
struct Scratch {
  uint64_t ctx = 0;  // context the address was looked up in
  float* p = nullptr;
};
Scratch g_dev_scratch[kMaxDevices];

// Device address of g_noalloc_scratch on the current device, looked up once per
// device and context (with that device current): a context created after a
// cudaDeviceReset gets a new lookup, never the old address.  Returns nullptr
// and sets *err on failure.
float* scratch_for_current_device(cudaError_t* err) {
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= kMaxDevices) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  const uint64_t id = oases::current_ctx_id();
  std::lock_guard<std::mutex> lock(g_mu);
  Scratch& s = g_dev_scratch[dev];
  if (!s.p || s.ctx != id || id == 0) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (*err != cudaSuccess) return nullptr;
    s.p = static_cast<float*>(p);
    s.ctx = id;
  }
  return s.p;
}

}  // namespace

namespace oases {
void noalloc_release_host_caches() {
  std::lock_guard<std::mutex> lock(g_mu);
  for (Scratch& s : g_dev_scratch) s = Scratch{};
}
}  // namespace oases

extern "C" oases_status oases_bias_grad_noalloc(const void* in, int64_t ld, int M, int N,
                                                int dtype, float* out, void* stream) {
  using namespace oases;
  api_begin();
  if (M < 0 || N < 0 || dtype < 0 || dtype > 1 || ld < N) return OASES_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return OASES_OK;
  if (!in || !out) return OASES_ERR_INVALID_ARG;
  const size_t need = (size_t)colsum_blocks(M) * (size_t)N;
  if (need > OASES_NOALLOC_SCRATCH_FLOATS) {
    char msg[160];
    std::snprintf(msg, sizeof(msg),
                  "oases_bias_grad_noalloc: needs %zu scratch floats, the static array holds %u",
                  need, (unsigned)OASES_NOALLOC_SCRATCH_FLOATS);
    api_set_error(msg);
    return OASES_ERR_UNSUPPORTED;
  }
  cudaError_t e = cudaSuccess;
  float* scratch = scratch_for_current_device(&e);
  if (!scratch) return api_end(e);
  e = colsum_accum(in, ld, M, N, static_cast<DType>(dtype), scratch, out,
                   static_cast<cudaStream_t>(stream));
  return api_end(e);
}
