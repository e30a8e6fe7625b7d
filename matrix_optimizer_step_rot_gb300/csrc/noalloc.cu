// rot_step_noalloc: rot_step for callers that cannot allocate device memory.
//
// The step's temporaries live in one file-scope device array of
// ROT_NOALLOC_MAX_BYTES instead of a caller-provided workspace blob.  Every
// GPU that loads the library holds this array until the process exits.
#include <mutex>

#include "plan.h"
#include "rot.h"

static __device__ __align__(256) unsigned char g_noalloc_scratch[ROT_NOALLOC_MAX_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device.  Host code only
// sees a host-side stand-in under that name, so the address is looked up once
// per device, with that device current, and cached.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ROT_ECUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return ROT_ECUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return ROT_OK;
}

}  // namespace

extern "C" int rot_step_noalloc(const rot_plan* plan, float* const* W, const float* const* G,
                                void* state, float beta1, float beta2, float eps, float lr,
                                int32_t refresh, int32_t precision, float rank_rtol,
                                void* stream) {
  if (!plan) return ROT_EINVAL;
  if (plan->work_bytes > (uint64_t)ROT_NOALLOC_MAX_BYTES) return ROT_ETOOLARGE;
  void* scratch = nullptr;
  const int e = scratch_address(&scratch);
  if (e != ROT_OK) return e;
  return rot_step(plan, W, G, state, scratch, beta1, beta2, eps, lr, refresh, precision,
                  rank_rtol, stream);
}
