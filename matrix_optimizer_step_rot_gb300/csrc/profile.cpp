// Launch instrumentation: a count of every kernel launch, and (when enabled)
// a CUDA event pair recorded on the launch stream around each launch, tagged
// with the launch's kernel class and its algorithmic work (flops or bytes).
#include "profile.h"

#include <mutex>
#include <vector>

namespace rot {
namespace {

struct Rec {
  int cls;
  cudaEvent_t a, b;
  double work;
};

std::mutex g_mu;
bool g_on = false;
std::vector<Rec> g_recs;
std::vector<cudaEvent_t> g_pool;
unsigned long long g_launches = 0;

cudaEvent_t take_event() {
  if (!g_pool.empty()) {
    cudaEvent_t e = g_pool.back();
    g_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

}  // namespace

ProfScope::ProfScope(int cls, double work, cudaStream_t s) : cls_(cls), work_(work), s_(s) {
  std::lock_guard<std::mutex> lk(g_mu);
  ++g_launches;
  if (g_on) {
    a_ = take_event();
    cudaEventRecord(a_, s_);
  }
}

ProfScope::~ProfScope() {
  if (!a_) return;
  std::lock_guard<std::mutex> lk(g_mu);
  cudaEvent_t b = take_event();
  cudaEventRecord(b, s_);
  g_recs.push_back({cls_, a_, b, work_});
}

}  // namespace rot

using namespace rot;

extern "C" {

int rot_profile_enable(int32_t on) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_on = on != 0;
  return ROT_OK;
}

int rot_profile_reset(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  for (Rec& r : g_recs) {
    g_pool.push_back(r.a);
    g_pool.push_back(r.b);
  }
  g_recs.clear();
  g_launches = 0;
  return ROT_OK;
}

uint64_t rot_launch_count(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  return g_launches;
}

int rot_profile_read(int32_t cls, uint64_t* launches, double* total_ms, double* max_ms,
                     double* work) {
  if (cls < 0 || cls >= ROT_PROF_CLASSES || !launches || !total_ms || !max_ms || !work)
    return ROT_EINVAL;
  std::lock_guard<std::mutex> lk(g_mu);
  uint64_t n = 0;
  double t = 0, mx = 0, w = 0;
  for (const Rec& r : g_recs) {
    if (r.cls != cls) continue;
    if (cudaEventSynchronize(r.b) != cudaSuccess) return ROT_ECUDA;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) return ROT_ECUDA;
    ++n;
    t += ms;
    mx = ms > mx ? ms : mx;
    w += r.work;
  }
  *launches = n;
  *total_ms = t;
  *max_ms = mx;
  *work = w;
  return ROT_OK;
}

}  // extern "C"
