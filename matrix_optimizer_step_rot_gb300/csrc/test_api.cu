// Test entry points (include/rot_testing.h) and the wait-limit setter.
#include "plan.h"
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
  // TF32 splits of A and B; the 3xF16 path's fp16 splits, row scales and
  // norm slot take less than that plus 1 KB
  return 2 * split_bytes(M, ldk) + 2 * split_bytes(N, ldk) + 1024;
}

}  // extern "C"

namespace {

static_assert(ROT_TEST_PREC_3XF16_PRECISE == kPrecPrecise16, "test code of the precise 3xF16 kernel");

int test_gemm(int32_t M, int32_t N, int32_t K, const float* A, int32_t lda, const float* B,
              int32_t ldb, float* C, int32_t ldc, int32_t epi, float alpha, int32_t precision,
              void* work, uint64_t work_bytes, int32_t* status, void* stream) {
  if (M < 1 || N < 1 || K < 1 || !A || !B || !C || !work) return ROT_EINVAL;
  if (lda < K || ldb < K || epi < kEpiStoreSplit || epi > kEpiApplySplit) return ROT_EINVAL;
  const bool f16 = precision == ROT_PREC_3XF16 || precision == ROT_TEST_PREC_3XF16_PRECISE;
  if (precision != ROT_PREC_TF32 && precision != ROT_PREC_3XTF32 &&
      precision != ROT_PREC_3XTF32_PRECISE && !f16)
    return ROT_EINVAL;
  if (f16 && (epi == kEpiStoreSplit || epi == kEpiApplySplit))
    return ROT_EINVAL;  // no fp16 form of the untransposed split outputs
  const bool transposed = epi == kEpiStoreSplitT || epi == kEpiStoreF32T;
  if (ldc < (transposed ? M : N)) return ROT_EINVAL;
  if (work_bytes < rot_test_gemm_work_bytes(M, N, K)) return ROT_EINVAL;
  if (reinterpret_cast<uintptr_t>(work) & 255) return ROT_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int ldk = (int)pad_ld(K);
  char* w = static_cast<char*>(work);
  if (f16) {
    // A: per-row scales; B: one scale below its largest row norm (the
    // epilogue undoes both).  Scaled fp16 splits, then the row scales of A and
    // B's norm bound in a small tail.
    const uint64_t ha = align256(2ull * M * ldk), hb = align256(2ull * N * ldk);
    unsigned short* a16h = reinterpret_cast<unsigned short*>(w);
    unsigned short* a16l = reinterpret_cast<unsigned short*>(w + ha);
    unsigned short* b16h = reinterpret_cast<unsigned short*>(w + 2 * ha);
    unsigned short* b16l = reinterpret_cast<unsigned short*>(w + 2 * ha + hb);
    float* rinv = reinterpret_cast<float*>(w + 2 * ha + 2 * hb);
    float* bnorm = reinterpret_cast<float*>(w + 2 * ha + 2 * hb + align256(4ull * M));
    if (cudaMemsetAsync(bnorm, 0, 4, s) != cudaSuccess) return ROT_ECUDA;
    hvec<Split16Seg> pass1 = {{A, lda, a16h, a16l, ldk, M, K, rinv, nullptr, nullptr},
                                     {B, ldb, nullptr, nullptr, ldk, N, K, nullptr, bnorm, nullptr}};
    int e = launch_split16(pass1, s);
    if (e != ROT_OK) return e;
    hvec<Split16Seg> pass2 = {{B, ldb, b16h, b16l, ldk, N, K, nullptr, nullptr, bnorm}};
    e = launch_split16(pass2, s);
    if (e != ROT_OK) return e;
    GemmProblem P;
    P.M = M;
    P.N = N;
    P.K = K;
    P.a_hi = reinterpret_cast<const float*>(a16h);
    P.a_lo = reinterpret_cast<const float*>(a16l);
    P.lda = ldk;
    P.b_hi = reinterpret_cast<const float*>(b16h);
    P.b_lo = reinterpret_cast<const float*>(b16l);
    P.ldb = ldk;
    P.c_hi = C;
    // kEpiStoreSplitT in this mode writes C^T as a fp16 split, unscaled: hi
    // in the first N x ldc halves of C, lo right after
    P.epi = epi == kEpiStoreSplitT ? (int)kEpiStoreF16SplitT : epi;
    P.c_lo = epi == kEpiStoreSplitT
                 ? reinterpret_cast<float*>(reinterpret_cast<unsigned short*>(C) + (int64_t)N * ldc)
                 : nullptr;
    P.ldc = ldc;
    P.alpha = alpha;
    P.f16 = 1;
    P.row_inv = rinv;
    if (precision == ROT_PREC_3XF16) {
      P.in_r = bnorm;
      return gemm_grouped({P}, precision, reinterpret_cast<int*>(status), s);
    }
    P.inb.r = bnorm;  // the same scale as B's split, as a Bound
    return gemm_grouped({P}, kPrecPrecise16, reinterpret_cast<int*>(status), s);
  }
  float* a_hi = reinterpret_cast<float*>(w);
  float* a_lo = reinterpret_cast<float*>(w + split_bytes(M, ldk));
  float* b_hi = reinterpret_cast<float*>(w + 2 * split_bytes(M, ldk));
  float* b_lo = reinterpret_cast<float*>(w + 2 * split_bytes(M, ldk) + split_bytes(N, ldk));
  hvec<SplitSeg> segs = {{A, lda, a_hi, a_lo, ldk, M, K}, {B, ldb, b_hi, b_lo, ldk, N, K}};
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

}  // namespace

extern "C" {

int rot_test_gemm(int32_t M, int32_t N, int32_t K, const float* A, int32_t lda, const float* B,
                  int32_t ldb, float* C, int32_t ldc, int32_t epi, float alpha,
                  int32_t precision, void* work, uint64_t work_bytes, int32_t* status,
                  void* stream) {
  try {
    return test_gemm(M, N, K, A, lda, B, ldb, C, ldc, epi, alpha, precision, work, work_bytes,
                     status, stream);
  } catch (const std::bad_alloc&) {
    return ROT_ENOMEM;
  }
}

int rot_test_fail_host_alloc(int64_t after) {
  set_host_alloc_failure(after < 0 ? -1 : after);
  return ROT_OK;
}

int rot_test_wait_timeout(uint64_t limit_ns, int32_t* status, void* stream) {
  if (!status || limit_ns > 10000000000ull) return ROT_EINVAL;
  return launch_wait_timeout(limit_ns, reinterpret_cast<int*>(status),
                             static_cast<cudaStream_t>(stream));
}

int rot_test_guard_offsets(const rot_plan* plan, int32_t group, uint64_t* offsets,
                           int32_t capacity, int32_t* count) {
  if (!plan || !count || group < 0 || (size_t)group >= plan->groups.size()) return ROT_EINVAL;
  if (!rot::kChecked) return ROT_ENOTSUP;
  const rot::hvec<uint64_t>& g = plan->guards[group];
  *count = (int32_t)g.size();
  for (int32_t i = 0; offsets && i < capacity && (size_t)i < g.size(); ++i) offsets[i] = g[i];
  return ROT_OK;
}

int rot_test_check_guards(const rot_plan* plan, int32_t group, void* state, void* work,
                          void* stream) {
  if (!plan || !state || !work || group < 0 || (size_t)group >= plan->groups.size())
    return ROT_EINVAL;
  if (!rot::kChecked) return ROT_ENOTSUP;
  try {
    return rot::launch_guards(plan->guards[group], work, static_cast<int*>(state), true,
                              static_cast<cudaStream_t>(stream));
  } catch (const std::bad_alloc&) {
    return ROT_ENOMEM;
  }
}

uint64_t rot_set_wait_timeout_ns(uint64_t ns) {
  const uint64_t old = g_wait_limit_ns;
  g_wait_limit_ns = ns;
  return old;
}

}  // extern "C"
