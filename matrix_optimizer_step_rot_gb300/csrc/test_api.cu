// Test entry points (include/rot_testing.h) and the wait-limit setter.
#include "rot_internal.h"
#include "rot_testing.h"

using namespace rot;

namespace rot {
int launch_wait_timeout(uint64_t limit_ns, int* status, cudaStream_t stream);
}

namespace {
uint64_t split_bytes(int64_t rows, int64_t ld) { return align256(4ull * rows * ld); }
}  // namespace

extern "C" {

uint64_t rot_test_gemm_work_bytes(int32_t M, int32_t N, int32_t K) {
  if (M < 1 || N < 1 || K < 1) return 0;
  const int64_t ldk = pad_ld(K);
  return 2 * split_bytes(M, ldk) + 2 * split_bytes(N, ldk);
}

int rot_test_gemm(int32_t M, int32_t N, int32_t K, const float* A, int32_t lda, const float* B,
                  int32_t ldb, float* C, int32_t ldc, int32_t epi, float alpha,
                  int32_t precision, void* work, uint64_t work_bytes, int32_t* status,
                  void* stream) {
  if (M < 1 || N < 1 || K < 1 || !A || !B || !C || !work) return ROT_EINVAL;
  if (lda < K || ldb < K || epi < kEpiStoreSplit || epi > kEpiApplySplit) return ROT_EINVAL;
  if (precision != ROT_PREC_TF32 && precision != ROT_PREC_3XTF32 &&
      precision != ROT_PREC_3XTF32_PRECISE)
    return ROT_EINVAL;
  const bool transposed = epi == kEpiStoreSplitT || epi == kEpiStoreF32T;
  if (ldc < (transposed ? M : N)) return ROT_EINVAL;
  if (work_bytes < rot_test_gemm_work_bytes(M, N, K)) return ROT_EINVAL;
  if (reinterpret_cast<uintptr_t>(work) & 255) return ROT_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int ldk = (int)pad_ld(K);
  char* w = static_cast<char*>(work);
  float* a_hi = reinterpret_cast<float*>(w);
  float* a_lo = reinterpret_cast<float*>(w + split_bytes(M, ldk));
  float* b_hi = reinterpret_cast<float*>(w + 2 * split_bytes(M, ldk));
  float* b_lo = reinterpret_cast<float*>(w + 2 * split_bytes(M, ldk) + split_bytes(N, ldk));
  std::vector<SplitSeg> segs = {{A, lda, a_hi, a_lo, ldk, M, K}, {B, ldb, b_hi, b_lo, ldk, N, K}};
  int e = launch_split(segs, s);
  if (e != ROT_OK) return e;
  GemmProblem P;
  P.M = M;
  P.N = N;
  P.K = K;
  P.a_hi = a_hi;
  P.a_lo = a_lo;
  P.lda = ldk;
  P.b_hi = b_hi;
  P.b_lo = b_lo;
  P.ldb = ldk;
  P.c_hi = C;
  // split outputs keep lo right after hi: M x ldc rows, or N x ldc for C^T
  P.c_lo = (epi == kEpiStoreSplit || epi == kEpiApplySplit) ? C + (int64_t)M * ldc
           : (epi == kEpiStoreSplitT)                       ? C + (int64_t)N * ldc
                                                            : nullptr;
  P.ldc = ldc;
  P.epi = epi;
  P.alpha = alpha;
  return gemm_grouped({P}, precision, reinterpret_cast<int*>(status), s);
}

int rot_test_wait_timeout(uint64_t limit_ns, int32_t* status, void* stream) {
  if (!status || limit_ns > 10000000000ull) return ROT_EINVAL;
  return launch_wait_timeout(limit_ns, reinterpret_cast<int*>(status),
                             static_cast<cudaStream_t>(stream));
}

uint64_t rot_set_wait_timeout_ns(uint64_t ns) {
  const uint64_t old = g_wait_limit_ns;
  g_wait_limit_ns = ns;
  return old;
}

}  // extern "C"
