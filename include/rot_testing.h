/*
 * rot_testing.h - test entry points of librot: run one internal kernel on
 * its own so that it can be checked in isolation.  Same conventions as
 * rot.h (return codes, caller-owned device memory, asynchronous on `stream`).
 */
#ifndef ROT_TESTING_H_
#define ROT_TESTING_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* C = A * B^T on the tensor-core grouped GEMM used by rot_step, for one
 * problem.  A: M x K, B: N x K, both float32 row-major device buffers with
 * leading dimensions lda, ldb.  The operands are first split into TF32
 * hi/lo pairs inside `work` (work_bytes >= rot_test_gemm_work_bytes(M, N,
 * K)).  epi selects the output: 0 C = split(A B^T) into C (hi) and C + M*ldc
 * (lo); 1 the same for C^T (N x M, ldc >= M); 2 C = A B^T (float32); 3 C^T
 * = (A B^T)^T; 4 C -= alpha A B^T; 5 C (split) -= alpha A B^T.  precision:
 * ROT_PREC_TF32, ROT_PREC_3XTF32, ROT_PREC_3XTF32_PRECISE, ROT_PREC_3XF16
 * (rot.h) or ROT_TEST_PREC_3XF16_PRECISE (the precise kernel on the scaled
 * fp16 splits, which the basis refresh runs in ROT_PREC_3XF16 mode).  With
 * either fp16 code, A gets per-row power-of-two scales and B one scale below
 * its largest row norm (undone by the epilogue); epi 1 then writes C^T as a
 * fp16 split (hi: N x ldc halves at C, lo right after), and epi 0 and 5 are
 * rejected.  status: device int that receives ROT_ETIMEOUT
 * if a device-side wait gives up (may be NULL).
 * Errors: ROT_EINVAL (sizes < 1, null pointers, work too small), ROT_ECUDA. */
#define ROT_TEST_PREC_3XF16_PRECISE 16

int rot_test_gemm(int32_t M, int32_t N, int32_t K, const float* A, int32_t lda, const float* B,
                  int32_t ldb, float* C, int32_t ldc, int32_t epi, float alpha,
                  int32_t precision, void* work, uint64_t work_bytes, int32_t* status,
                  void* stream);

/* Failure detection check: one thread waits, with the same bounded wait the
 * GEMM kernels use, on an mbarrier that nothing ever arrives on.  After
 * limit_ns (<= 10 s) the wait gives up and *status (device int) becomes
 * ROT_ETIMEOUT; the context stays usable.  Errors: ROT_EINVAL, ROT_ECUDA. */
int rot_test_wait_timeout(uint64_t limit_ns, int32_t* status, void* stream);

/* Host allocation failure injection.  The library's host containers (plan,
 * partitions, the step's launch descriptors) allocate through one allocator;
 * with after >= 0, the allocation that follows `after` more successful ones
 * fails once, and the entry point that made it returns ROT_ENOMEM (rot_step
 * then has stepped the micro-groups before the failing one, and none after
 * it).  after < 0 cancels a planned failure.  Host-side, no device work;
 * returns ROT_OK. */
int rot_test_fail_host_alloc(int64_t after);

/* Workspace bytes rot_test_gemm needs for these sizes. */
uint64_t rot_test_gemm_work_bytes(int32_t M, int32_t N, int32_t K);

/* Bounds-checked builds (the library compiled with ROT_CHECK; the survey's
 * canary words).  The plan then leaves a 256-byte guard region after every
 * slice of the workspace; rot_step fills each micro-group's guards with a
 * fixed pattern before the group's work and checks them after it, setting the
 * status word to ROT_ECORRUPT (rot_status) if any was overwritten.
 *
 * rot_test_guard_offsets: byte offsets (into the workspace) of micro-group
 * `group`'s guards, up to `capacity` of them into `offsets` (host array),
 * their number into *count.  Host-side.  Errors: ROT_EINVAL (null plan or
 * count, group out of range), ROT_ENOTSUP (a build without ROT_CHECK).
 *
 * rot_test_check_guards: runs only the check of micro-group `group`'s guards
 * on `stream` (device pointers `state`, `work` as for rot_step), so that a
 * test can overwrite a guard and see it reported.  Errors: ROT_EINVAL,
 * ROT_ENOTSUP, ROT_ECUDA. */
int rot_test_guard_offsets(const rot_plan* plan, int32_t group, uint64_t* offsets,
                           int32_t capacity, int32_t* count);
int rot_test_check_guards(const rot_plan* plan, int32_t group, void* state, void* work,
                          void* stream);

#ifdef __cplusplus
}
#endif

#endif /* ROT_TESTING_H_ */
