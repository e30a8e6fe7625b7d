// rot_step_noalloc: rot_step for callers that cannot allocate device memory.
//
// The step's temporaries live in one file-scope device array of
// ROT_NOALLOC_MAX_BYTES instead of a caller-provided workspace blob.  Every
// GPU that loads the library holds this array until the process exits.
#include <mutex>

#include "plan.h"
#include "rot.h"
#include "rot_internal.h"

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
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return ROT_ECUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return ROT_ENOTSUP;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return ROT_ECUDA;
    }
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
  // rot_step's own checks and early-outs first (an empty plan touches no
  // device), with a stand-in for the workspace pointer, which is not an
  // argument here; then the size limit, the device, and only then the
  // array's address
  const int args = rot::check_step_args(plan, W, G, state, reinterpret_cast<const void*>(256),
                                        refresh, precision, rank_rtol);
  if (args != ROT_OK || plan->count == 0) return args;
  if (plan->work_bytes > (uint64_t)ROT_NOALLOC_MAX_BYTES) return ROT_ETOOLARGE;
  const int dev = rot::check_device();
  if (dev != ROT_OK) return dev;
  void* scratch = nullptr;
  const int e = scratch_address(&scratch);
  if (e != ROT_OK) return e;
  return rot_step(plan, W, G, state, scratch, beta1, beta2, eps, lr, refresh, precision,
                  rank_rtol, stream);
}
