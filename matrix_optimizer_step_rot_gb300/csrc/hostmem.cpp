// Host allocations of the library (see HostAlloc in rot_internal.h), with a
// failure hook for tests: the allocation after a chosen number of successful
// ones throws std::bad_alloc, which the entry points report as ROT_ENOMEM.
#include <atomic>
#include <cstdlib>
#include <new>

#include "rot_internal.h"

namespace rot {
namespace {
// allocations still allowed before the injected failure; -1: none planned
std::atomic<int64_t> g_fail_after{-1};
}  // namespace

void set_host_alloc_failure(int64_t after) { g_fail_after.store(after < 0 ? -1 : after); }

void* host_alloc(std::size_t bytes) {
  int64_t left = g_fail_after.load(std::memory_order_relaxed);
  while (left >= 0) {
    const int64_t next = left == 0 ? -1 : left - 1;
    if (g_fail_after.compare_exchange_weak(left, next)) {
      if (left == 0) throw std::bad_alloc();
      break;
    }
  }
  void* p = std::malloc(bytes ? bytes : 1);
  if (!p) throw std::bad_alloc();
  return p;
}

void host_free(void* p) noexcept { std::free(p); }

}  // namespace rot
