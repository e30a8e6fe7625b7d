// Launch instrumentation used by every kernel launch site of the library.
#pragma once

#include <cuda_runtime.h>

#include "rot.h"

namespace rot {

// Put one of these immediately around each kernel launch: it counts the
// launch and, while profiling is enabled, records events on `s` before and
// after it.  `work` is the launch's algorithmic work in the unit of its class
// (flops for GEMMs, bytes for memory-bound kernels, 0 if not modelled).
class ProfScope {
 public:
  ProfScope(int cls, double work, cudaStream_t s);
  ~ProfScope();
  ProfScope(const ProfScope&) = delete;
  ProfScope& operator=(const ProfScope&) = delete;

 private:
  int cls_;
  double work_;
  cudaStream_t s_;
  cudaEvent_t a_ = nullptr;
};

}  // namespace rot
