// Internal declarations shared by the CUDA translation units of librot.
// Not part of the public ABI (include/rot.h is).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <cstddef>
#include <new>
#include <vector>

#include "rot.h"

namespace rot {

// ---------------------------------------------------------------------------
// Host allocations.  The library's host containers (plan, partition, launch
// descriptors) allocate through host_alloc, which throws std::bad_alloc on
// failure; every entry point turns that into ROT_ENOMEM.  A test can make the
// n-th later allocation fail (rot_test_fail_host_alloc).
// ---------------------------------------------------------------------------

void* host_alloc(std::size_t bytes);
void host_free(void* p) noexcept;
// after >= 0: the allocation after `after` more successful ones fails (once);
// after < 0: no failure.
void set_host_alloc_failure(int64_t after);

template <class T>
struct HostAlloc {
  using value_type = T;
  HostAlloc() noexcept = default;
  template <class U>
  HostAlloc(const HostAlloc<U>&) noexcept {}
  T* allocate(std::size_t n) {
    if (n > static_cast<std::size_t>(-1) / sizeof(T)) throw std::bad_alloc();
    return static_cast<T*>(host_alloc(n * sizeof(T)));
  }
  void deallocate(T* p, std::size_t) noexcept { host_free(p); }
};
template <class T, class U>
bool operator==(const HostAlloc<T>&, const HostAlloc<U>&) noexcept { return true; }
template <class T, class U>
bool operator!=(const HostAlloc<T>&, const HostAlloc<U>&) noexcept { return false; }

template <class T>
using hvec = std::vector<T, HostAlloc<T>>;

// ---------------------------------------------------------------------------
// Layout helpers
// ---------------------------------------------------------------------------

// Leading dimensions of every buffer the library owns are padded to 32 floats
// (128 bytes): rows start 128-byte aligned, which tensor-map (TMA) loads need.
constexpr int kLdAlign = 32;
inline int64_t pad_ld(int64_t x) { return (x + kLdAlign - 1) / kLdAlign * kLdAlign; }
inline uint64_t align256(uint64_t x) { return (x + 255) & ~uint64_t(255); }

// Bounds-checked builds (compiled with ROT_CHECK): a guard region of
// kGuardBytes follows every workspace slice (plan.cpp), filled with
// kGuardWord before a micro-group's work and checked after it.
#ifdef ROT_CHECK
constexpr bool kChecked = true;
#else
constexpr bool kChecked = false;
#endif
constexpr uint64_t kGuardBytes = 256;
constexpr uint32_t kGuardWord = 0xA5C3E1F7u;
// fill (check = false) or check (true) the guards at `offsets` in `work`;
// a changed word sets *status to ROT_ECORRUPT (if it held ROT_OK)
int launch_guards(const hvec<uint64_t>& offsets, void* work, int* status, bool check,
                  cudaStream_t stream);

// A float32 matrix stored as an exact split x = hi + lo, hi = x rounded to
// TF32 (10 explicit mantissa bits), lo = x - hi.  Tensor-core operands are
// always held in this form; the float32 value is hi + lo.
struct Split {
  float* hi;
  float* lo;
};

// ---------------------------------------------------------------------------
// Grouped GEMM: C[M x N] = A[M x K] * B^T, with A (M x K) and B (N x K) both
// row-major with K contiguous ("K-major"), given as splits.
// ---------------------------------------------------------------------------

enum GemmEpi : int {
  kEpiStoreSplit = 0,   // C (row-major, ldc) <- split(acc)
  kEpiStoreSplitT = 1,  // C^T (row-major N x M, ldc) <- split(acc)
  kEpiStoreF32 = 2,     // C (row-major) <- acc, float32 into c.hi
  kEpiStoreF32T = 3,    // C^T <- acc, float32 into c.hi
  kEpiApply = 4,        // C (row-major, float32 in c.hi) -= alpha * acc
  kEpiApplySplit = 5,   // C (row-major split) <- split(hi + lo - alpha * acc)
                        // (with mma_only: the TF32-rounded split of arrays only MMAs read)
  kEpiStoreF16SplitT = 6,  // C^T (row-major N x M fp16 arrays) <- scaled fp16 split (3xF16)
  kEpiStoreBF16 = 7,    // C (row-major) <- acc rounded to bf16, into c.hi (compact state)
};

// A power-of-two operand or output scale of the precise 3xF16 products,
// taken from a bound on the magnitudes it scales: bound = (*r)^(sq ? 2 : 1) *
// mul, scale = pow2_below(bound) (split.cuh).  The producer of a scaled
// array and its consumer evaluate the same expression, so the two scales
// cancel exactly.  r == nullptr: no scale.
struct Bound {
  const float* r = nullptr;
  float mul = 1.f;
  int sq = 0;
};

struct GemmProblem {
  int M, N, K;
  const float* a_hi;
  const float* a_lo;
  int lda;
  const float* b_hi;
  const float* b_lo;
  int ldb;
  float* c_hi;
  float* c_lo;
  int ldc;
  int epi;
  float alpha;
  int mma_only = 0;  // split outputs feed only tensor cores: round lo to TF32
  // ROT_PREC_3XF16 problems: a_* and b_* (and c_* for kEpiStoreF16SplitT) are
  // fp16 arrays (cast), lda/ldb/ldc in elements.  The accumulator is scaled
  // by c0 * row_inv[row] / pow2_below(*in_r); a fp16 split output is scaled by
  // pow2_below(*out_r) (see split.cuh).  Null pointers mean 1.
  int f16 = 0;
  const float* row_inv = nullptr;
  const float* in_r = nullptr;
  const float* out_r = nullptr;
  float c0 = 1.f;
  // kPrecPrecise16 problems: the accumulator is scaled by c0 * row_inv[row] *
  // col_inv[col] / scale(ina) / scale(inb) (A's rows, B's rows and uniform
  // operand scales), and a fp16 split output by scale(outb).  in_r / out_r
  // are not read.
  const float* col_inv = nullptr;
  Bound ina, inb, outb;
};

// 3xTF32 with each K block of 32 accumulated afresh in TMEM (cross terms
// first, hi*hi last) and summed in float32 registers (ROT_PREC_3XTF32_PRECISE);
// used for products whose results cancel.
constexpr int kPrecPrecise = ROT_PREC_3XTF32_PRECISE;

// The same K-blocked, compensated kernel on scaled fp16 splits (kind::f16,
// K blocks of 64, twice the TF32 rate; problems marked f16): the basis
// refresh's products in ROT_PREC_3XF16 mode.  Not a rot_step mode.
constexpr int kPrecPrecise16 = 16;

// Upper bound on every device-side wait, in nanoseconds.
extern uint64_t g_wait_limit_ns;

// Whether the element-wise kernels report non-finite gradients and updates
// (rot_set_nonfinite_check).
extern std::atomic<int> g_nonfinite_check;

// Runs every problem of `probs` (any count; launched in chunks).  precision is
// ROT_PREC_TF32, ROT_PREC_3XTF32, ROT_PREC_3XF16 (problems marked f16) or
// kPrecPrecise.  status: device status word (may be
// nullptr) set to ROT_ETIMEOUT if a bounded wait gives up.
int gemm_grouped(const hvec<GemmProblem>& probs, int precision, int* status,
                 cudaStream_t stream);

// ---------------------------------------------------------------------------
// Element-wise kernels (one entry per matrix)
// ---------------------------------------------------------------------------

struct MomentumSeg {
  const float* g;  // caller's gradient, row-major, ld = cols
  float* m;        // state momentum (float32, or bf16 when m_bf16), ld = ldm
  float* g_hi;     // workspace gradient split (tensor-core operand), ld = ldm
  float* g_lo;
  int rows, cols, ldm;
  float* m_hi;     // refresh steps: M's exact TF32 split (workspace), else null
  float* m_lo;
  int m_bf16 = 0;  // compact state: M is stored as bf16
};
// flag: the status word when the non-finite check is on (non-finite G or D
// sets it to ROT_ENONFINITE), else null.
int launch_momentum(const hvec<MomentumSeg>& segs, float beta1, int* flag, cudaStream_t stream);

struct AdamSeg {
  const float* gt;  // G~ float32, ld
  float* mt;        // state M~ float32 (bf16 when mt_bf16), ld (updated in place when incremental)
  float* v;         // state second moment, ld
  float* d_hi;      // D split out, ld
  float* d_lo;
  int rows, cols, ld;
  int mt_bf16 = 0;
};
// incremental != 0: M~ <- beta1 M~ + (1 - beta1) G~ first (bases unchanged
// since the last step); else M~ was just recomputed as U^T M V.
int launch_adam(const hvec<AdamSeg>& segs, float beta1, float beta2, float eps,
                int incremental, int* flag, cudaStream_t stream);

// 3xF16 variants, one block per row.  Momentum as above, and G's scaled fp16
// split: row r gets the power-of-two scale s_r with max|G_r| s_r < 2^14,
// g_rinv[r] = 1 / s_r, and *g_rmax grows to the largest row 2-norm (it must
// be 0 or smaller beforehand).  g_hi / g_lo are fp16 arrays (ld = ldm).
struct Momentum16Seg {
  const float* g;
  float* m;  // state momentum (float32)
  unsigned short* g_hi;
  unsigned short* g_lo;
  float* g_rinv;
  float* g_rmax;
  int rows, cols, ldm;
  // refresh steps: M's row-scaled fp16 split (m16_hi == nullptr: none), and
  // its exact TF32 split where m_hi is set
  unsigned short* m16_hi;
  unsigned short* m16_lo;
  float* m_rinv;
  float* m_rmax;
  float* m_hi;
  float* m_lo;
  int m_bf16 = 0;  // compact state: M is stored as bf16
  float* m_amax = nullptr;  // refresh steps: grows to the largest |M_ij| (if set)
};
int launch_momentum16(const hvec<Momentum16Seg>& segs, float beta1, int* flag,
                      cudaStream_t stream);

// Adam as above with D written as a scaled fp16 split (per-row scales into
// d_rinv, largest row 2-norm into *d_rmax).
struct Adam16Seg {
  const float* gt;
  float* mt;
  float* v;
  unsigned short* d_hi;
  unsigned short* d_lo;
  float* d_rinv;
  float* d_rmax;
  int rows, cols, ld;
  int mt_bf16 = 0;  // compact state: M~ is stored as bf16
};
int launch_adam16(const hvec<Adam16Seg>& segs, float beta1, float beta2, float eps,
                  int incremental, int* flag, cudaStream_t stream);

// hi/lo (fp16, rows x cols, ld_dst) = fp16 split of 2^14 (s_hi + s_lo), for
// the bases (|entries| <= 1).
struct ToF16Seg {
  const float* s_hi;
  const float* s_lo;
  int ld_src;
  unsigned short* hi;
  unsigned short* lo;
  int ld_dst;
  int rows, cols;
};
int launch_to_f16(const hvec<ToF16Seg>& segs, cudaStream_t stream);

// Scaled fp16 split of a float32 matrix (test entry point): per-row scales
// (rinv != nullptr) or one scale from *bound; rmax (if set) grows to the
// largest row 2-norm; hi == nullptr computes the norms only.
struct Split16Seg {
  const float* src;
  int ld_src;
  unsigned short* hi;
  unsigned short* lo;
  int ld_dst;
  int rows, cols;
  float* rinv;
  float* rmax;
  const float* bound;
};
int launch_split16(const hvec<Split16Seg>& segs, cudaStream_t stream);

// dst (cols x rows, ld_dst) = src^T, where src (rows x cols, ld_src) is a split;
// dst is written as a split.  src_is_split = 0 reads float32 from src.hi.
struct TransposeSeg {
  const float* s_hi;
  const float* s_lo;
  int ld_src;
  float* d_hi;
  float* d_lo;
  int ld_dst;
  int rows, cols;
  int src_is_split;
  int dst_is_split;
  int dst_mma_only = 0;  // the split output feeds only tensor cores
};
int launch_transpose(const hvec<TransposeSeg>& segs, cudaStream_t stream);

// M^T as a fp16 split with one power-of-two scale for the whole matrix:
// d = split(M^T * pow2_below(*rmax)), *rmax a bound on every |M_ij| (the
// largest |M_ij| that the momentum kernel leaves).  m: the state's momentum
// (rows x cols, float32 or bf16 when m_bf16, ld_src elements); d_hi / d_lo:
// fp16 arrays, cols x rows, ld_dst elements.
struct TransposeF16Seg {
  const float* m;
  int ld_src;
  unsigned short* d_hi;
  unsigned short* d_lo;
  int ld_dst;
  int rows, cols;
  const float* rmax;
  int m_bf16;
};
int launch_transpose16(const hvec<TransposeF16Seg>& segs, cudaStream_t stream);

// TF32 split (hi, lo: float32 arrays, lo rounded to TF32 as well) of a basis
// held as a 2^14-scaled fp16 split; dst is src (transpose == 0) or src^T.
struct ToTf32Seg {
  const unsigned short* s_hi;
  const unsigned short* s_lo;
  int ld_src;
  float* d_hi;
  float* d_lo;
  int ld_dst;
  int rows, cols;  // of src
};
int launch_to_tf32(const hvec<ToTf32Seg>& segs, cudaStream_t stream);    // dst = src
int launch_to_tf32_t(const hvec<ToTf32Seg>& segs, cudaStream_t stream);  // dst = src^T

// dst (float32, rows x cols, ld_dst) = (hi + lo) / 2^14 of a 2^14-scaled fp16
// split (basis export).
int launch_combine16(const unsigned short* hi, const unsigned short* lo, int ld_src, float* dst,
                     int ld_dst, int rows, int cols, cudaStream_t stream);

// Fill a p x p split with the identity (lo = 0), or a rows x cols split with 0.
struct FillSeg {
  float* hi;
  float* lo;
  int rows, cols, ld;
  int identity;
  int f16 = 0;  // hi, lo are fp16 arrays; the identity is written as 2^14
};
int launch_fill(const hvec<FillSeg>& segs, cudaStream_t stream);

// hi/lo (rows x cols, ld_dst) = TF32 split of src (float32, ld_src).
struct SplitSeg {
  const float* src;
  int ld_src;
  float* hi;
  float* lo;
  int ld_dst;
  int rows, cols;
};
int launch_split(const hvec<SplitSeg>& segs, cudaStream_t stream);

// dst (rows x cols, ld_dst, float32) = hi + lo (or hi alone when lo == nullptr;
// src_bf16: hi is a bf16 array and lo is ignored).
int launch_combine(const float* hi, const float* lo, int ld_src, float* dst, int ld_dst,
                   int rows, int cols, cudaStream_t stream, int src_bf16 = 0);

// ---------------------------------------------------------------------------
// Batched blocked Householder QR+ (Q factor only)
// ---------------------------------------------------------------------------

constexpr int kQrPanel = 32;   // panel width b
constexpr int kQrBlock = 256;  // block-reflector width

struct QrProblem {
  Split at;     // p x ld: row j holds column j of A; overwritten by reflectors
  Split qt;     // p x ld: Q^T accumulates here
  Split yt;     // p x kQrBlock: the current block's reflectors, transposed
  Split w1t;    // kQrBlock x ld: (Y T)^T or (Y T^T)^T of the current block
  Split z;      // p x kQrBlock: X (Y T) of the current block
  float* s;     // kQrBlock x kQrBlock: Gram Y^T Y of the current block
  float* tmp;   // kQrBlock x kQrBlock: T of the current block, float32
  Split tb;     // per block: T (kQrBlock x kQrBlock)
  Split tbt;    // per block: T^T
  // Q formation in pairs of blocks (rank-512 updates): the pair's factor
  // T (2 kQrBlock x 2 kQrBlock) and its parts S01 = Y_b^T Y_{b+1} and
  // X^T = (S01 T_{b+1})^T (kQrBlock x kQrBlock each)
  Split tpair;
  Split s01;
  Split xt;
  float* tf;    // per panel: 32 x 32 triangular factor
  float* part;  // within-block update: per element chunk and row tile, Y^T a partials
  float* beta;  // rmax: R diagonal before the sign fix
  int* ctrl;    // [0] rank, [1] stopped flag, [2..] per-panel active counts
  float* tau;   // largest column norm of A
  int p, ld, rmax;
  // outputs (state): U (row-major) and U^T as fp16 splits scaled by 2^14
  // (ld_out elements per row; a null lo keeps hi alone, rounded to fp16),
  // and the rank
  int ld_out;
  int* rank_out;
  unsigned short* u16_hi;
  unsigned short* u16_lo;
  unsigned short* ut16_hi;
  unsigned short* ut16_lo;
};
int qr_batched(const hvec<QrProblem>& probs, float rank_rtol, int* status,
               cudaStream_t stream);

// Bytes of QR scratch besides `at` and `qt` for one problem (256-aligned
// pieces), and the binding of those pieces to a problem's pointers.
uint64_t qr_aux_bytes(int p, int rmax);
void qr_bind_aux(QrProblem& q, char* aux, int p, int rmax);

// Largest p the QR accepts (panel slices must fit a 16-CTA cluster).
constexpr int kQrMaxDim = 16 * 1536;

// ROT_OK if the current device is sm_103, ROT_ENOTSUP if it is another GPU,
// ROT_ECUDA if no device can be queried (CUDA's last error is then cleared).
int check_device();

// rot_step's host-side argument checks, in its order (no device access).
int check_step_args(const rot_plan* plan, float* const* W, const float* const* G,
                    const void* state, const void* work, int32_t refresh, int32_t precision,
                    float rank_rtol);

}  // namespace rot
