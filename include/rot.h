/*
 * rot.h - C ABI of the GB300 rotated-Adam matrix-optimizer step.
 *
 * The library runs one optimizer step over many independent 2-D float32
 * parameter matrices W (m x n, row-major) on one GPU.  Per matrix it keeps
 * momentum M (m x n), a second moment v (m x n) and two orthogonal bases
 * U (m x m) and V (n x n), and performs
 *
 *   (1) M <- beta1 M + (1 - beta1) G
 *   (2) on refresh steps: U <- QR+(M M^T U), V <- QR+(M^T M V)
 *   (3) G~ = U^T G V, M~ = U^T M V, v <- beta2 v + (1 - beta2) G~^2,
 *       D = M~ / (sqrt(v) + eps)
 *   (4) W <- W - lr U D V^T
 *
 * Sources: the momentum matrix, "power iteration + QR every K iterations" and
 * the two-sided rotation U^T W V are section 2.2 of the page
 * "分布式训练中的流水线并行与梯度陈旧性优化"; the per-coordinate update
 * m / (sqrt(v) + eps) is section 2.1 of that page; the second-moment update is
 * section 2.1 of "大模型分布式优化：通信、内存、计算三层解耦实战"; the
 * micro-group planner (global LPT sort, greedy grouping with rollback, min-heap
 * load simulation, byte cap) is section 3.2.2 of the Canzona page.
 * QR+ is Householder QR with R's diagonal made positive, stopped at the
 * numerical rank (first column whose remaining norm is <= rank_rtol times the
 * largest column norm of the input) and completed by the reflectors found so
 * far.  The power iteration is taken to a full basis (one subspace-iteration
 * step per refresh, starting from U = I, V = I).
 *
 * Conventions for every entry point
 * ---------------------------------
 * - Return 0 (ROT_OK) on success or a negative ROT_E* code.  No C++ exception
 *   crosses this boundary.  rot_strerror() names a code.
 * - "device pointer" means memory of the current CUDA device; the caller owns
 *   all device memory (W, G, the state blob and the workspace blob).  The
 *   library allocates no device memory.  The plan is host memory owned by the
 *   library between rot_plan_create() and rot_plan_destroy().
 * - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *   Device work is enqueued on it and the call returns without waiting, except
 *   where stated.
 * - Matrix dimensions: 1 <= m, n <= ROT_MAX_DIM.
 * - One CUDA device per process: the kernels' launch configuration (shared-
 *   memory limits, the SM count) is set up once, for the device current at
 *   the first step.  Data-parallel use runs one process per GPU.
 */
#ifndef ROT_H_
#define ROT_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ROT_OK 0
#define ROT_EINVAL (-1)      /* bad argument (null pointer, size, plan/state mismatch) */
#define ROT_ENOMEM (-2)      /* host allocation failed */
#define ROT_ECUDA (-3)       /* a CUDA call or kernel launch failed */
#define ROT_ETIMEOUT (-4)    /* a device-side wait gave up (see rot_status) */
#define ROT_ENONFINITE (-5)  /* a non-finite gradient or update was seen (reported by
                                rot_status while rot_set_nonfinite_check is on) */
#define ROT_ENOTSUP (-6)     /* GPU is not sm_103 or the feature is not built */
#define ROT_ETOOLARGE (-7)   /* plan needs more scratch than rot_step_noalloc holds */
#define ROT_ECORRUPT (-8)    /* bounds-checked builds (compiled with ROT_CHECK) only: a
                                guard region around a workspace slice was overwritten
                                during a step (reported by rot_status) */

#define ROT_PREC_TF32 1      /* one TF32 tensor-core product per GEMM */
#define ROT_PREC_3XTF32 3    /* hi*hi + hi*lo + lo*hi TF32 split, ~fp32 accuracy */
#define ROT_PREC_3XTF32_PRECISE 4 /* 3xTF32 with each K block of 32 summed in float32
                                     registers: float32-level accuracy at any K */
#define ROT_PREC_3XF16 5     /* the three split products on power-of-two-scaled fp16
                                splits (11 + 11 significant bits, as 3XTF32) at twice
                                the TF32 tensor-core rate; the basis refresh's products
                                run on the precise kernel's fp16 form, the QR's on
                                3XTF32_PRECISE */

#define ROT_MAX_DIM 65536

#define ROT_WHICH_M 0        /* momentum, m x n */
#define ROT_WHICH_V2 1       /* second moment v, m x n */
#define ROT_WHICH_U 2        /* left basis U, m x m */
#define ROT_WHICH_V 3        /* right basis V, n x n */

typedef struct rot_shape {
  int32_t m; /* rows (output features) */
  int32_t n; /* columns (input features) */
} rot_shape;

typedef struct rot_plan rot_plan;

/* Build the micro-group plan (host only, no device work).
 * Items are sorted by cost m^2 n + m n^2 + m^3 + n^3 descending (ties: input
 * order), then packed greedily into groups whose bytes (4 m n per item) stay
 * <= c_max_bytes; an item that does not fit rolls the group back and opens a
 * new one, and an item larger than c_max_bytes forms a group of its own
 * (Canzona page, section 3.2.2).  count == 0 gives a plan with no groups.
 * Errors: ROT_EINVAL for a null `out`, count < 0, shapes == NULL with
 * count > 0, a dimension outside [1, ROT_MAX_DIM] or c_max_bytes == 0;
 * ROT_ENOMEM.  On error *out is set to NULL. */
int rot_plan_create(const rot_shape* shapes, int32_t count, uint64_t c_max_bytes,
                    rot_plan** out);

/* Same as rot_plan_create with `ranks` simulated ranks in the min-heap load
 * simulation (each item goes to the rank with the least accumulated cost in
 * its group, ties to the lowest id; the byte cap applies per rank).  ranks = 1
 * is rot_plan_create.  Used to check the planner; the step runs on one GPU
 * whatever `ranks` was.  Errors as rot_plan_create, plus ranks < 1. */
int rot_plan_create_ex(const rot_shape* shapes, int32_t count, uint64_t c_max_bytes,
                       int32_t ranks, rot_plan** out);

/* ---- data-parallel partition (host only, no device work) -----------------
 *
 * Where the matrices of a model are split across data-parallel ranks (each
 * rank updates the matrices it owns; the rest are gathered afterwards), these
 * entry points give the owner of every matrix.  Items are given in physical
 * order and grouped into consecutive buckets (bucket b = the next
 * bucket_sizes[b] items); a bucket is cut into `ranks` consecutive pieces,
 * rank r taking piece r, with every cut on an item boundary (an item is never
 * split).  The sizes must be >= 0 and add up to `count`.
 */

/* Work (processing-time proxy) of each item: m^2 n + m n^2 + m^3 + n^3, the
 * micro-group planner's cost.  Errors: ROT_EINVAL for null pointers with
 * count > 0, count < 0 or a dimension outside [1, ROT_MAX_DIM]. */
int rot_item_work(const rot_shape* shapes, int32_t count, uint64_t* work);

/* Static ownership by parameter start (Canzona page, section 3.1.1), bucket by
 * bucket as a ZeRO-1 flat buffer is sharded: bucket b's items lie back to back
 * in E_b elements (elems[i] each), cut into shards of ceil(E_b / ranks)
 * elements; an item belongs to the shard holding its first element.
 * owners: `count` entries written.  Errors: ROT_EINVAL for null pointers with
 * count > 0 (or n_buckets > 0), ranks < 1, a negative size, sizes not adding
 * up to `count`, or a bucket total above 2^64 - 1. */
int rot_partition_static(const uint64_t* elems, int32_t count, const int32_t* bucket_sizes,
                         int32_t n_buckets, int32_t ranks, int32_t* owners);

/* alpha-balanced greedy LPT partition (Canzona page, section 3.2.1).  Buckets
 * are visited by total work W_b, largest first (ties: lower index first).  For
 * each, with per-rank loads L so far: ideal A = sum L / ranks, the mean load
 * before the bucket, as the page's code prints it; deficit
 * d_r = max(0, A - L_r); fill share d_r / sum d (1/ranks if every d_r is 0);
 * share s_r = (1 - alpha) / ranks + alpha * fill_r; cut r goes to the item
 * boundary whose prefix work is nearest to W_b (s_0 + ... + s_r) (ties: the
 * earlier boundary); L grows by each piece's work.  alpha = 0 splits every
 * bucket evenly, alpha = 1 fills the ranks furthest below the ideal.  The
 * floating-point steps are float64, in this order, with no contraction, so
 * every host gets the same cuts.
 * owners: `count` entries; loads (may be NULL): `ranks` entries, each rank's
 * total work.  Errors: ROT_EINVAL as rot_partition_static, plus alpha outside
 * [0, 1] (or NaN) and total work >= 2^53 (loads must stay exact in a double);
 * ROT_ENOMEM. */
int rot_partition_alpha(const uint64_t* work, int32_t count, const int32_t* bucket_sizes,
                        int32_t n_buckets, int32_t ranks, double alpha, int32_t* owners,
                        uint64_t* loads);

/* rot_partition_alpha with a choice of ideal load.  ROT_ALPHA_IDEAL_BEFORE is
 * rot_partition_alpha (A = sum L / ranks).  ROT_ALPHA_IDEAL_AFTER takes the
 * even share once the bucket is placed, A = (sum L + W_b) / ranks: with it,
 * alpha = 1 levels the loads whenever the bucket covers the deficits, where
 * the printed rule hands the whole bucket to the ranks below the old mean
 * (loads (100, 98) and a bucket of 50 unit items end at (100, 148) under it,
 * at (124, 124) under this one).  Errors as rot_partition_alpha, plus an
 * unknown `ideal`. */
#define ROT_ALPHA_IDEAL_BEFORE 0
#define ROT_ALPHA_IDEAL_AFTER 1
int rot_partition_alpha_ex(const uint64_t* work, int32_t count, const int32_t* bucket_sizes,
                           int32_t n_buckets, int32_t ranks, double alpha, int32_t ideal,
                           int32_t* owners, uint64_t* loads);

/* Free a plan (NULL is accepted). */
void rot_plan_destroy(rot_plan* plan);

/* Number of micro-groups.  Errors: ROT_EINVAL for null arguments. */
int rot_plan_groups(const rot_plan* plan, int32_t* n_groups);

/* Group g: its items (input indices in LPT order; the pointer is borrowed and
 * valid until rot_plan_destroy), item count, total bytes and total cost.
 * Any output pointer may be NULL.  Errors: ROT_EINVAL for g out of range. */
int rot_plan_group(const rot_plan* plan, int32_t g, const int32_t** items,
                   int32_t* n_items, uint64_t* bytes, uint64_t* cost);

/* Owner rank of every input index (borrowed array of `count` entries). */
int rot_plan_owners(const rot_plan* plan, const int32_t** owners);

/* State format of a plan (set before rot_state_bytes / rot_state_init; the
 * layout of the state blob depends on it).
 * ROT_STATE_FULL (default): M, v and M~ in float32; each basis, in the two
 *   orientations the products read, as a 2^14-scaled fp16 split (22
 *   significant bits).
 * ROT_STATE_COMPACT: the reduced-precision state of the pages -- the first
 *   moments M and M~ in bf16, v in float32 (the ZeRO essay, section 3.3:
 *   m in BF16, v in FP32) and each basis orientation a single fp16 (the
 *   rotation page, section 3.1: rotation matrices stored in float16).  About
 *   half the bytes of the full format; bases orthogonal to about 2^-11 sqrt(p)
 *   and W changed by about the method's own spread at these precisions (its
 *   parity is checked against that, not against the float32 bars).
 * Errors: ROT_EINVAL (null plan, unknown format), ROT_ENOMEM. */
#define ROT_STATE_FULL 0
#define ROT_STATE_COMPACT 1
int rot_plan_set_state_format(rot_plan* plan, int32_t format);

/* Bytes of the caller-allocated state blob (M, v, U, V of every matrix plus a
 * status word; persists across steps) and of the workspace blob (temporaries
 * of one step, sized for the largest micro-group; contents need not persist).
 * Both blobs must be 256-byte aligned device memory.  Either output may be
 * NULL. */
int rot_state_bytes(const rot_plan* plan, uint64_t* state_bytes, uint64_t* work_bytes);

/* Initialise the state: M = 0, v = 0, U = I, V = I, status word cleared.
 * Errors: ROT_EINVAL (null plan/state), ROT_ECUDA. */
int rot_state_init(const rot_plan* plan, void* state, void* stream);

/* One optimizer step for every matrix of the plan, micro-group by micro-group.
 * W, G: host arrays of `count` device pointers, in input order; W[i] (m x n,
 * row-major, float32) is updated in place, G[i] is read only.  state: the
 * initialised state blob; work: the workspace blob.  refresh != 0 runs the
 * basis refresh (2) before the rotated update.  precision of the rotation
 * products: ROT_PREC_TF32, ROT_PREC_3XTF32, ROT_PREC_3XTF32_PRECISE or
 * ROT_PREC_3XF16 (the basis refresh always runs with float32-level accuracy:
 * its products on the precise kernel, K blocks summed with compensation, in
 * the TF32 split or, with ROT_PREC_3XF16, the scaled fp16 split; the QR in
 * ROT_PREC_3XTF32_PRECISE).
 * The mode may change from step to step.  rank_rtol in
 * [1e-6, 1): the QR's numerical-rank threshold relative to the largest
 * column norm.  Non-finite inputs propagate (IEEE).
 * Errors: ROT_EINVAL (null pointers, unknown precision, rank_rtol out of
 * range), ROT_ENOTSUP (device is not sm_103, or refresh != 0 for a matrix with
 * m or n above 24576: the QR holds a panel slice of at most 1536 rows in each
 * of at most 16 CTAs of a cluster), ROT_ECUDA (launch failure).  An empty plan
 * returns ROT_OK without touching the device.
 * Device-side problems are reported by rot_status. */
int rot_step(const rot_plan* plan, float* const* W, const float* const* G, void* state,
             void* work, float beta1, float beta2, float eps, float lr, int32_t refresh,
             int32_t precision, float rank_rtol, void* stream);

/* rot_step without a workspace argument, for callers that cannot allocate
 * device memory themselves (for example code running inside a host framework
 * that owns every device allocation, or a fixed-budget embedding that may not
 * call cudaMalloc).  The paper has no counterpart: it is an addition of this
 * library.  The step's temporaries live in one static device array of
 * ROT_NOALLOC_MAX_BYTES that every GPU loading the library holds until the
 * process exits; the caller still passes W, G and the state blob.  Plans whose
 * workspace (rot_state_bytes' work_bytes) exceeds that size are rejected with
 * ROT_ETOOLARGE before any device work.  The first call on a device looks up
 * the array's device address (cudaGetSymbolAddress) with that device current;
 * make that first call before any stream capture.  Nothing is allocated.  All
 * calls share the one array and leave their temporaries in it: calls whose
 * device work overlaps (other streams, other host threads) race on it, so
 * order them on one stream.  Other arguments, results and errors as
 * rot_step. */
#define ROT_NOALLOC_MAX_BYTES (64u << 20)
int rot_step_noalloc(const rot_plan* plan, float* const* W, const float* const* G, void* state,
                     float beta1, float beta2, float eps, float lr, int32_t refresh,
                     int32_t precision, float rank_rtol, void* stream);

/* Synchronise `stream`, then read and clear the device status word of
 * `state`: *status = ROT_OK; ROT_ETIMEOUT if a device-side wait exceeded its
 * spin limit since the last call; ROT_ENONFINITE if, while the non-finite
 * check was on, a gradient element or an element of an update D was NaN or
 * infinite (the first problem seen is kept).  Returns ROT_ECUDA if the
 * synchronisation fails. */
int rot_status(const rot_plan* plan, void* state, int32_t* status, void* stream);

/* Copy one state matrix of input item `item` as float32 row-major into the
 * device buffer dst (M or v: m x n; U: m x m; V: n x n).  Asynchronous.
 * Errors: ROT_EINVAL (item or which out of range, null pointers). */
int rot_state_export(const rot_plan* plan, const void* state, int32_t item, int32_t which,
                     float* dst, void* stream);

/* Numerical ranks of U's and V's inputs at the last refresh of `item`
 * (device memory is read after synchronising `stream`; -1 before any
 * refresh).  Errors: ROT_EINVAL, ROT_ECUDA. */
int rot_state_ranks(const rot_plan* plan, const void* state, int32_t item, int32_t* rank_u,
                    int32_t* rank_v, void* stream);

/* Non-finite check (a diagnostic in the spirit of the ZeRO essay's section
 * 4.4 checks on gradients and the second moment): with on != 0, later steps'
 * element-wise kernels test every gradient element and every element of the
 * rotated update D = M~ / (sqrt(v) + eps), and rot_status then reports
 * ROT_ENONFINITE if one was not finite.  The values themselves still
 * propagate (IEEE) into their own matrix's results.  Off by default; the test
 * costs no extra memory traffic.  Returns the previous setting.  Host-side
 * setting shared by all plans. */
int32_t rot_set_nonfinite_check(int32_t on);

/* Set the upper bound, in nanoseconds, on every device-side wait of later
 * launches (default 2 000 000 000 = 2 s); returns the previous bound.  A wait
 * that reaches it abandons its kernel's remaining work, and rot_status()
 * then reports ROT_ETIMEOUT.  Host-side setting, not thread-safe against
 * concurrent rot_step calls. */
uint64_t rot_set_wait_timeout_ns(uint64_t ns);

/* Instrumentation.  Every kernel launch of the library is counted; while
 * profiling is enabled, a CUDA event pair is also recorded on the launch
 * stream around each launch, tagged with its kernel class and algorithmic
 * work.  Host-side state shared by all plans; thread-safe. */
#define ROT_PROF_GEMM 0        /* tensor-core GEMM (TF32 / 3xTF32); work = 2 M N K flops */
#define ROT_PROF_ELEMENTWISE 1 /* momentum, Adam, transposes, splits; work = bytes moved */
#define ROT_PROF_QR_PANEL 2    /* QR panel factorisation; work = 0 (latency bound) */
#define ROT_PROF_QR_APPLY 3    /* QR block-reflector updates; work = flops (32-wide panels) */
#define ROT_PROF_QR_OTHER 4    /* QR set-up, column norms, identity, sign fix; work = 0 */
#define ROT_PROF_GEMM_PRECISE 5 /* precise 3xTF32 GEMM (refresh products, QR blocks) */
#define ROT_PROF_GEMM_F16 6    /* 3xF16 tensor-core GEMM; work = 2 M N K flops */
#define ROT_PROF_GEMM_PRECISE_F16 7 /* the precise GEMM on scaled fp16 splits (the
                                       refresh products in ROT_PREC_3XF16 mode) */
#define ROT_PROF_CLASSES 8

/* Turn event recording on (on != 0) or off.  Returns ROT_OK. */
int rot_profile_enable(int32_t on);

/* Drop every record and zero the launch counter.  Returns ROT_OK. */
int rot_profile_reset(void);

/* Kernel launches since the last reset. */
uint64_t rot_launch_count(void);

/* Summary of the records of class `cls`: number of launches, total and
 * largest event-measured duration (ms) and summed work.  Waits for the
 * recorded events.  Errors: ROT_EINVAL (class out of range, null outputs),
 * ROT_ECUDA. */
int rot_profile_read(int32_t cls, uint64_t* launches, double* total_ms, double* max_ms,
                     double* work);

/* Static description of an error code. */
const char* rot_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* ROT_H_ */
