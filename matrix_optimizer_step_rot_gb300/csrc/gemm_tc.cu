// Grouped GEMM on the sm_103a tensor cores (tcgen05, TMEM accumulators,
// TMA-fed shared-memory ring), C = A * B^T with A (M x K) and B (N x K) both
// K-major float32 matrices held as TF32 splits.
//
// ROT_PREC_3XTF32 issues three kind::tf32 MMAs per K step (hi*lo, lo*hi,
// hi*hi) and recovers about float32 accuracy; ROT_PREC_TF32 issues one
// (hi*hi).  ROT_PREC_3XF16 issues the same three products on power-of-two
// scaled fp16 splits (kind::f16, twice the TF32 rate, 22 significant bits as
// well); its operands are fp16 arrays and its epilogue undoes the scaling.
// Accumulation is float32 in TMEM in every mode.
//
// Structure: a persistent kernel, one CTA per SM, walks the flattened tile
// list of every problem in the launch.  Per CTA:
//   warp 0     one thread issues TMA loads into a STAGES-deep ring
//   warp 1     allocates TMEM; one thread issues the MMAs of a 128 x BN tile
//              into one of two TMEM accumulators
//   warps 2-5  epilogue: tcgen05.ld the accumulator (each warp its 32-lane
//              quarter), apply the output mode, store to global memory
// mbarriers link the roles; every wait is bounded in time, and a timeout
// raises a CTA-wide abort flag, drains in-flight copies and MMAs, frees TMEM
// and reports ROT_ETIMEOUT through the status word.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cstring>

#include "profile.h"
#include "rot_internal.h"
#include "split.cuh"
#include "tc_ptx.cuh"

namespace rot {

uint64_t g_wait_limit_ns = 2000000000ull;  // 2 s; see rot_set_wait_timeout_ns

namespace {

constexpr int BM = 128;  // UMMA M (cta_group::1): one TMEM lane per row
constexpr int BK = 32;   // 32 float32 = 128 bytes = one swizzle-atom row
constexpr int kMaxP = 40;
constexpr int kThreads = 192;

struct TcProblem {
  CUtensorMap a_hi, a_lo, b_hi, b_lo;
  int M, N, K;
  int tiles_n;
  int tile_start;
  int epi;
  int ldc;
  float alpha;
  int mma_only;
  float* c_hi;
  float* c_lo;
  // 3xF16 scaling (powers of two): the accumulator is multiplied by
  // c0 * row_inv[row] (if set) / pow2_below(*in_r) (if set); fp16 split
  // outputs are then multiplied by pow2_below(*out_r) (if set).
  const float* row_inv;
  const float* in_r;
  const float* out_r;
  float c0;
  // the precise 3xF16 kernel's scales (GemmProblem): per column of C and
  // uniform for A, B and the fp16 split output
  const float* col_inv;
  Bound ina, inb, outb;
};

struct TcBatch {
  TcProblem p[kMaxP];
  int count;
  int total_tiles;
  int* status;
  unsigned long long limit_ns;
};
static_assert(sizeof(TcBatch) <= 32764, "kernel parameter block above 32764 bytes");

// The bound of a Bound (see rot_internal.h); evaluated the same way wherever
// a scale is applied or undone.
__device__ __forceinline__ float bound_value(const Bound& b) {
  const float r = *b.r;
  return (b.sq ? r * r : r) * b.mul;
}

template <int BN, int STAGES, bool SPLIT3>
struct Cfg {
  static constexpr int kABytes = BM * BK * 4;
  static constexpr int kBBytes = BN * BK * 4;
  static constexpr int kStageBytes = (kABytes + kBBytes) * (SPLIT3 ? 2 : 1);
  static constexpr int kSmem = STAGES * kStageBytes + 1024 /*align*/ + 256 /*barriers*/;
  static constexpr int kTmemCols = 2 * BN;
  static_assert(kTmemCols == 256 || kTmemCols == 512, "TMEM allocation must be a power of 2");
};

// Tile order within a problem: groups of kGroupM row blocks, column-major
// inside a group.  The persistent CTAs work on consecutive tiles at the same
// time, so a wave touches ~kGroupM row blocks of A and ~(CTAs / kGroupM)
// column blocks of B, which L2 keeps, instead of a few rows of A against every
// column block of B (re-read from DRAM by every wave).  The order does not
// change any result: tiles are independent.
constexpr int kGroupM = 8;

__device__ __forceinline__ void decode(const TcBatch& b, int tile, int& pi, int& m0, int& nt) {
  pi = 0;
  while (pi + 1 < b.count && tile >= b.p[pi + 1].tile_start) ++pi;
  const TcProblem& P = b.p[pi];
  const int local = tile - P.tile_start;
  const int tn = P.tiles_n, tm = (P.M + BM - 1) / BM;
  const int per_group = kGroupM * tn;
  const int g = local / per_group, r = local - g * per_group;
  const int h = min(kGroupM, tm - g * kGroupM);  // the last group may be shorter
  m0 = (g * kGroupM + r % h) * BM;
  nt = r / h;
}

// Waits without regard to the abort flag (used only to drain at exit).  The
// drain keeps waiting at least 100 ms whatever the wait limit, so that copies
// and MMAs in flight land before the CTA's shared memory and TMEM are freed.
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  limit_ns = limit_ns > 100000000ull ? limit_ns : 100000000ull;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    if (ptx::mbar_try_wait(bar, parity)) return;
    if ((it & 63u) == 0u && (ptx::globaltimer_ns() - t0 > limit_ns || it > (1u << 30))) return;
  }
}

__device__ __forceinline__ void store_chunk(const TcProblem& P, int row, int col0,
                                            const uint32_t (&r)[32]) {
  const int M = P.M, N = P.N;
  const int ncol = min(32, N - col0);
  switch (P.epi) {
    case kEpiStoreSplitT:
    case kEpiStoreF32T: {
      // column j of C is row j of C^T: the warp's 32 lanes (32 consecutive
      // rows i) write 32 consecutive floats
      if (row >= M) return;
      const bool split = P.epi == kEpiStoreSplitT;
#pragma unroll
      for (int t = 0; t < 32; ++t) {
        if (t < ncol) {
          const float v = __uint_as_float(r[t]);
          const int64_t o = (int64_t)(col0 + t) * P.ldc + row;
          if (split) {
            float h, l;
            if (P.mma_only) {
              split_tf32_mma(v, h, l);
            } else {
              split_tf32(v, h, l);
            }
            P.c_hi[o] = h;
            P.c_lo[o] = l;
          } else {
            P.c_hi[o] = v;
          }
        }
      }
      return;
    }
    case kEpiStoreSplit:
    case kEpiStoreF32: {
      if (row >= M) return;
      const bool split = P.epi == kEpiStoreSplit;
      float* hi = P.c_hi + (int64_t)row * P.ldc + col0;
      float* lo = split ? P.c_lo + (int64_t)row * P.ldc + col0 : nullptr;
      if (ncol == 32 && (P.ldc & 3) == 0 && ((reinterpret_cast<uintptr_t>(hi) & 15) == 0) &&
          (!split || (reinterpret_cast<uintptr_t>(lo) & 15) == 0)) {
#pragma unroll
        for (int t = 0; t < 32; t += 4) {
          float4 h4, l4;
          float* hp = &h4.x;
          float* lp = &l4.x;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const float v = __uint_as_float(r[t + u]);
            if (split) {
              if (P.mma_only) {
                split_tf32_mma(v, hp[u], lp[u]);
              } else {
                split_tf32(v, hp[u], lp[u]);
              }
            } else {
              hp[u] = v;
            }
          }
          *reinterpret_cast<float4*>(hi + t) = h4;
          if (split) *reinterpret_cast<float4*>(lo + t) = l4;
        }
      } else {
#pragma unroll
        for (int t = 0; t < 32; ++t) {
          if (t < ncol) {
            const float v = __uint_as_float(r[t]);
            if (split) {
              float h, l;
              if (P.mma_only) {
                split_tf32_mma(v, h, l);
              } else {
                split_tf32(v, h, l);
              }
              hi[t] = h;
              lo[t] = l;
            } else {
              hi[t] = v;
            }
          }
        }
      }
      return;
    }
    case kEpiStoreBF16: {
      if (row >= M) return;
      __nv_bfloat16* c = reinterpret_cast<__nv_bfloat16*>(P.c_hi) + (int64_t)row * P.ldc + col0;
#pragma unroll
      for (int t = 0; t < 32; ++t)
        if (t < ncol) c[t] = __float2bfloat16_rn(__uint_as_float(r[t]));
      return;
    }
    case kEpiApply: {
      // every load is issued before the first store: a store may alias a
      // later load as far as the compiler knows, which would otherwise put
      // one memory latency between consecutive loads
      if (row >= M) return;
      float* w = P.c_hi + (int64_t)row * P.ldc + col0;
      if (ncol == 32 && (P.ldc & 3) == 0 && (reinterpret_cast<uintptr_t>(w) & 15) == 0) {
        float4 x[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] = reinterpret_cast<const float4*>(w)[i];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          x[i].x -= P.alpha * __uint_as_float(r[4 * i]);
          x[i].y -= P.alpha * __uint_as_float(r[4 * i + 1]);
          x[i].z -= P.alpha * __uint_as_float(r[4 * i + 2]);
          x[i].w -= P.alpha * __uint_as_float(r[4 * i + 3]);
          reinterpret_cast<float4*>(w)[i] = x[i];
        }
      } else {
        float x[32];
#pragma unroll
        for (int t = 0; t < 32; ++t)
          if (t < ncol) x[t] = w[t];
#pragma unroll
        for (int t = 0; t < 32; ++t)
          if (t < ncol) w[t] = x[t] - P.alpha * __uint_as_float(r[t]);
      }
      return;
    }
    case kEpiApplySplit: {
      if (row >= M) return;
      float* hi = P.c_hi + (int64_t)row * P.ldc + col0;
      float* lo = P.c_lo + (int64_t)row * P.ldc + col0;
      if (ncol == 32 && (P.ldc & 3) == 0 && ((reinterpret_cast<uintptr_t>(hi) & 15) == 0) &&
          ((reinterpret_cast<uintptr_t>(lo) & 15) == 0)) {
        // per half row-chunk, all eight loads in flight before the first
        // store (see kEpiApply); halves keep the registers within budget
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float4 h4[4], l4[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            h4[i] = reinterpret_cast<const float4*>(hi)[4 * half + i];
            l4[i] = reinterpret_cast<const float4*>(lo)[4 * half + i];
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float* hp = &h4[i].x;
            float* lp = &l4[i].x;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const float v =
                  (hp[u] + lp[u]) - P.alpha * __uint_as_float(r[16 * half + 4 * i + u]);
              if (P.mma_only) {
                split_tf32_mma(v, hp[u], lp[u]);
              } else {
                split_tf32(v, hp[u], lp[u]);
              }
            }
            reinterpret_cast<float4*>(hi)[4 * half + i] = h4[i];
            reinterpret_cast<float4*>(lo)[4 * half + i] = l4[i];
          }
        }
      } else {
#pragma unroll
        for (int t = 0; t < 32; ++t) {
          if (t < ncol) {
            const float v = (hi[t] + lo[t]) - P.alpha * __uint_as_float(r[t]);
            float h, l;
            if (P.mma_only) {
              split_tf32_mma(v, h, l);
            } else {
              split_tf32(v, h, l);
            }
            hi[t] = h;
            lo[t] = l;
          }
        }
      }
      return;
    }
  }
}

// kEpiStoreF16SplitT: C^T (N x M fp16 rows, ldc elements) <- fp16 split of
// acc * f; the warp's 32 lanes (32 consecutive rows i) write 64 contiguous
// bytes per column.
__device__ __forceinline__ void store_chunk_f16t(const TcProblem& P, int row, int col0,
                                                 const uint32_t (&r)[32], float f) {
  if (row >= P.M) return;
  const int ncol = min(32, P.N - col0);
  unsigned short* hi = reinterpret_cast<unsigned short*>(P.c_hi);
  unsigned short* lo = reinterpret_cast<unsigned short*>(P.c_lo);
#pragma unroll
  for (int t = 0; t < 32; ++t) {
    if (t < ncol) {
      unsigned short h, l;
      split_f16(__uint_as_float(r[t]) * f, h, l);
      const int64_t o = (int64_t)(col0 + t) * P.ldc + row;
      hi[o] = h;
      lo[o] = l;
    }
  }
}

template <int BN, int STAGES, bool SPLIT3, bool F16 = false>
__global__ void __launch_bounds__(kThreads, 1) gemm_tc_kernel(const __grid_constant__ TcBatch b) {
  using C = Cfg<BN, STAGES, SPLIT3>;
  constexpr int BKE = F16 ? 2 * BK : BK;  // elements per 128-byte K block
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * C::kStageBytes);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t limit = b.limit_ns;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&tfull[a], 1);
      ptx::mbar_init(&tempty[a], 4);
    }
    ptx::mbar_init(drain, 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, C::kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    for (int i = 0; i < b.count; ++i) {
      ptx::tma_prefetch_desc(&b.p[i].a_hi);
      ptx::tma_prefetch_desc(&b.p[i].b_hi);
    }
    int stage = 0;
    uint32_t phase = 0;
    uint32_t armed_mask = 0, armed_parity = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < b.total_tiles; tile += gridDim.x) {
      int pi, m0, nt;
      decode(b, tile, pi, m0, nt);
      const TcProblem& P = b.p[pi];
      const int n0 = nt * BN;
      const int kblocks = (P.K + BKE - 1) / BKE;
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!ptx::mbar_wait(&empty[stage], phase ^ 1u, abort_flag, limit)) {
          ok = false;
          break;
        }
        uint8_t* st = smem + stage * C::kStageBytes;
        ptx::mbar_arrive_expect_tx(&full[stage], C::kStageBytes);
        armed_mask |= 1u << stage;
        armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
        const int x = kb * BKE;
        ptx::tma_load_2d(st, &P.a_hi, &full[stage], x, m0);
        if (SPLIT3) {
          ptx::tma_load_2d(st + C::kABytes, &P.a_lo, &full[stage], x, m0);
          ptx::tma_load_2d(st + 2 * C::kABytes, &P.b_hi, &full[stage], x, n0);
          ptx::tma_load_2d(st + 2 * C::kABytes + C::kBBytes, &P.b_lo, &full[stage], x, n0);
        } else {
          ptx::tma_load_2d(st + C::kABytes, &P.b_hi, &full[stage], x, n0);
        }
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    // wait for this thread's copies still in flight before the CTA exits
    for (int s = 0; s < STAGES; ++s)
      if (armed_mask & (1u << s)) mbar_drain(&full[s], (armed_parity >> s) & 1u, limit);
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issue
    constexpr uint32_t idesc = F16 ? ptx::idesc_f16(BM, BN) : ptx::idesc_tf32(BM, BN);
    auto mma = [&](uint32_t d, uint64_t a, uint64_t bb, uint32_t accum) {
      if (F16) {
        ptx::umma_f16(d, a, bb, idesc, accum);
      } else {
        ptx::umma_tf32(d, a, bb, idesc, accum);
      }
    };
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < b.total_tiles; tile += gridDim.x) {
      int pi, m0, nt;
      decode(b, tile, pi, m0, nt);
      const int kblocks = (b.p[pi].K + BKE - 1) / BKE;
      if (!ptx::mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, limit)) break;
      ptx::tc_fence_after();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!ptx::mbar_wait(&full[stage], phase, abort_flag, limit)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t s = ptx::smem_u32(smem + stage * C::kStageBytes);
        const uint64_t ah = ptx::sw128_kmajor_desc(s);
        const uint64_t al = ptx::sw128_kmajor_desc(s + C::kABytes);
        const uint64_t bh = ptx::sw128_kmajor_desc(s + (SPLIT3 ? 2 : 1) * C::kABytes);
        const uint64_t bl = ptx::sw128_kmajor_desc(s + 2 * C::kABytes + C::kBBytes);
#pragma unroll
        for (int kk = 0; kk < BK / 8; ++kk) {  // 32 bytes per step: 8 tf32 or 16 fp16
          const uint64_t off = static_cast<uint64_t>(kk * 32 >> 4);
          const uint32_t accum = (kb > 0 || kk > 0) ? 1u : 0u;
          if (SPLIT3) {
            mma(d_tmem, ah + off, bl + off, accum);
            mma(d_tmem, al + off, bh + off, 1u);
            mma(d_tmem, ah + off, bh + off, 1u);
          } else {
            mma(d_tmem, ah + off, bh + off, accum);
          }
        }
        ptx::umma_commit(&empty[stage]);  // frees the stage once these MMAs finish
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      ptx::umma_commit(&tfull[acc]);  // accumulator ready for the epilogue
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    // every MMA this thread issued has completed before TMEM is freed
    ptx::umma_commit(drain);
    mbar_drain(drain, 0, limit);
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31 belong to this warp
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < b.total_tiles; tile += gridDim.x) {
      int pi, m0, nt;
      decode(b, tile, pi, m0, nt);
      const TcProblem& P = b.p[pi];
      const int n0 = nt * BN;
      if (!ptx::mbar_wait(&tfull[acc], acc_phase, abort_flag, limit)) break;
      ptx::tc_fence_after();
      const int row = m0 + quarter * 32 + lane;
      const uint32_t taddr =
          tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(acc * BN);
      float f = 1.f, fout = 1.f;
      if (F16) {  // undo the operands' power-of-two scales (exact)
        f = P.c0;
        if (P.row_inv && row < P.M) f *= P.row_inv[row];
        if (P.in_r) f *= pow2_below_inv(*P.in_r, kF16ScaleExp);
        if (P.out_r) fout = pow2_below(*P.out_r, kF16ScaleExp);
      }
      for (int c = 0; c < BN && n0 + c < P.N; c += 32) {
        uint32_t r[32];
        ptx::tmem_ld_32x32b_x32(taddr + static_cast<uint32_t>(c), r);
        ptx::tmem_wait_ld();
        if (F16 && P.epi == kEpiStoreF16SplitT) {
          store_chunk_f16t(P, row, n0 + c, r, f * fout);
        } else {
          if (F16) {
#pragma unroll
            for (int t = 0; t < 32; ++t) r[t] = __float_as_uint(__uint_as_float(r[t]) * f);
          }
          store_chunk(P, row, n0 + c, r);
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&tempty[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, C::kTmemCols);
  }
  if (threadIdx.x == 0 && *abort_flag && b.status) atomicExch(b.status, ROT_ETIMEOUT);
}

// ---------------------------------------------------------------------------
// Row-major output through shared memory.  In store_chunk lane l of a warp
// holds row row0 + l, so each of the warp's accesses touches 32 rows (16
// bytes of each).  Here the warp's 32 x 32 chunk goes through a padded
// staging area (row stride 33 floats: both the write and the read are free of
// bank conflicts) and comes back one row at a time, lane l holding column
// col0 + l: every global access of the warp is 32 consecutive elements.  The
// apply modes issue the loads of eight rows (sixteen for the split) before
// their stores.  Row-major
// modes only (the transposed ones are already row-contiguous per warp).
// ---------------------------------------------------------------------------

constexpr int kStageStride = 33;  // floats per staged row
constexpr int kStageFloats = 32 * kStageStride;

__device__ __forceinline__ bool rows_path(int epi) {
  return epi == kEpiStoreSplit || epi == kEpiStoreF32 || epi == kEpiApply ||
         epi == kEpiApplySplit || epi == kEpiStoreBF16;
}

__device__ __forceinline__ void store_chunk_rows(const TcProblem& P, int row0, int col0,
                                                 const uint32_t (&r)[32], float* stage) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int c = 0; c < 32; ++c) stage[lane * kStageStride + c] = __uint_as_float(r[c]);
  __syncwarp();
  const int col = col0 + lane;
  const bool cok = col < P.N;
  const int nrow = min(32, P.M - row0);
  const float alpha = P.alpha;
  switch (P.epi) {
    case kEpiStoreSplit:
    case kEpiStoreF32: {
      const bool split = P.epi == kEpiStoreSplit;
      for (int i = 0; i < nrow; ++i) {
        const float v = stage[i * kStageStride + lane];
        if (!cok) continue;
        const int64_t o = (int64_t)(row0 + i) * P.ldc + col;
        if (split) {
          float h, l;
          if (P.mma_only) {
            split_tf32_mma(v, h, l);
          } else {
            split_tf32(v, h, l);
          }
          P.c_hi[o] = h;
          P.c_lo[o] = l;
        } else {
          P.c_hi[o] = v;
        }
      }
      break;
    }
    case kEpiStoreBF16: {
      __nv_bfloat16* c = reinterpret_cast<__nv_bfloat16*>(P.c_hi);
      for (int i = 0; i < nrow; ++i)
        if (cok)
          c[(int64_t)(row0 + i) * P.ldc + col] = __float2bfloat16_rn(stage[i * kStageStride + lane]);
      break;
    }
    case kEpiApply: {
      for (int i0 = 0; i0 < nrow; i0 += 8) {
        float x[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int i = i0 + u;
          x[u] = (cok && i < nrow) ? P.c_hi[(int64_t)(row0 + i) * P.ldc + col] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int i = i0 + u;
          if (cok && i < nrow)
            P.c_hi[(int64_t)(row0 + i) * P.ldc + col] =
                x[u] - alpha * stage[i * kStageStride + lane];
        }
      }
      break;
    }
    case kEpiApplySplit: {
      for (int i0 = 0; i0 < nrow; i0 += 16) {
        float h[16], l[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const int i = i0 + u;
          const int64_t o = (int64_t)(row0 + i) * P.ldc + col;
          const bool ok = cok && i < nrow;
          h[u] = ok ? P.c_hi[o] : 0.f;
          l[u] = ok ? P.c_lo[o] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const int i = i0 + u;
          if (cok && i < nrow) {
            const int64_t o = (int64_t)(row0 + i) * P.ldc + col;
            float hh, ll;
            const float v = (h[u] + l[u]) - alpha * stage[i * kStageStride + lane];
            if (P.mma_only) {
              split_tf32_mma(v, hh, ll);
            } else {
              split_tf32(v, hh, ll);
            }
            P.c_hi[o] = hh;
            P.c_lo[o] = ll;
          }
        }
      }
      break;
    }
    default:
      break;
  }
  __syncwarp();  // the staging area is read before the next chunk rewrites it
}

// ---------------------------------------------------------------------------
// Precise 3xTF32 variant (BN = 128).  The tensor cores truncate every partial
// sum they add into a TMEM accumulator, an error that grows with K and that
// cancellation (a - Y T Y^T a with a small result) then magnifies.  Here each
// K block of 32 is accumulated afresh in TMEM and the epilogue warps add it to
// a float32 running sum.  Within a block the cross terms hi*lo + lo*hi (2^-11
// of the result) are issued first and the four hi*hi MMAs last, so only those
// four adds truncate at the result's magnitude.  (Accumulating two or four
// K blocks per buffer instead measured 2.8x / 6x the error.)
// The sum over the K/32 blocks is taken in two levels.  Each epilogue thread
// adds the block partials of each 16-column piece in registers (a plain
// float32 sum of up to four terms) and every four blocks adds that group sum
// into a running sum held in TMEM with compensation (Kahan, "Further remarks
// on reducing truncation errors", CACM 1965): the group sum's rounding error
// is carried into the next fold, so the running sum's error stays at a few
// units in the last place whatever K is, instead of growing like sqrt(K/32).
// Measured relative error of a product with K = 6144 / 12288: 1.25e-7 with
// this sum, 2.8e-7 / 3.8e-7 with a plain float32 sum of the blocks.
// The four pieces are folded in turn (piece q after blocks q, q + 4, ...),
// so each block costs one TMEM load and one add per element plus at most one
// piece's fold, and no block stalls the MMAs behind a long fold.
// TMEM: 2 K-block buffers x 128 columns, then the tile's 128 x 128 running
// sums (columns 256..383) and their compensations (384..511).  Eight
// epilogue warps: warp w owns TMEM lanes 32 (w % 4) .. +31 and columns
// 64 ((w - 2) / 4) .. +63 of each region.
// Short products (SHORT: every K <= kPreciseShortK, at most 16 blocks, the
// QR's rank-256 and rank-512 updates and their factors) keep the whole sum in registers,
// a plain float32 sum of the blocks, and use the four TMEM buffers so that
// the MMAs run three blocks ahead while the epilogue finishes a tile.
// F16: the same kernel on power-of-two scaled fp16 splits (kind::f16, 11 + 11
// significant bits like the TF32 split).  A 128-byte TMA stage then holds 64
// elements of K for the twelve MMA slots of a TF32 stage, twice the work.  It
// is accumulated as two TMEM blocks of 32 (six MMAs each; one block of 64
// measured about 1.2x the error on Gram products), and the pieces are folded
// once per stage, so the sums in registers still cover up to 256 elements of
// K between folds.  The epilogue undoes the operands' scales on the
// compensated sum and may write a scaled fp16 split (kEpiStoreF16SplitT).
// ---------------------------------------------------------------------------

constexpr int kThreadsPrecise = 320;
constexpr int kPreciseBufs = 2;
constexpr int kPreciseEpiWarps = 8;
constexpr int kPreciseCols = 64;           // columns per epilogue warp
constexpr int kPreciseGroup = kPreciseCols / 16;  // K blocks summed in registers between folds
constexpr uint32_t kPreciseSumCol = 256;   // first TMEM column of the running sums
constexpr uint32_t kPreciseCompCol = 384;  // first TMEM column of their compensations
constexpr int kPreciseShortK = 512;        // the SHORT variant's largest K

// s + x with the rounding error carried in c (Kahan): returns the new s.
__device__ __forceinline__ float kahan_add(float s, float x, float& c) {
  const float y = x - c;
  const float t = s + y;
  c = (t - s) - y;
  return t;
}

template <int STAGES, bool SHORT, bool F16>
__global__ void __launch_bounds__(kThreadsPrecise, 1)
    gemm_tc_precise_kernel(const __grid_constant__ TcBatch b) {
  constexpr int BN = 128;
  constexpr int BKE = F16 ? 2 * BK : BK;  // elements per 128-byte K stage
  // TMEM K blocks per stage: 32 elements each in both forms (two per fp16
  // stage), kMmaPerBlock 32-byte MMA steps per block and term
  constexpr int kSub = F16 ? 2 : 1;
  constexpr int kMmaPerBlock = BK / 8 / kSub;
  constexpr int kBufs = SHORT ? 4 : kPreciseBufs;
  using C = Cfg<BN, STAGES, true>;
  constexpr uint32_t kCols = 512;
  static_assert((2 * STAGES + 2 * kBufs + 1) * 8 + 8 <= 256, "barrier area");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * C::kStageBytes);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + kBufs;
  uint64_t* drain = tempty + kBufs;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // row-major output staging, one area per epilogue warp, after the barriers
  float* stage_area = reinterpret_cast<float*>(smem + STAGES * C::kStageBytes + 256);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t limit = b.limit_ns;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < kBufs; ++a) {
      ptx::mbar_init(&tfull[a], 1);
      ptx::mbar_init(&tempty[a], kPreciseEpiWarps);
    }
    ptx::mbar_init(drain, 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, kCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    for (int i = 0; i < b.count; ++i) {
      ptx::tma_prefetch_desc(&b.p[i].a_hi);
      ptx::tma_prefetch_desc(&b.p[i].b_hi);
    }
    int stage = 0;
    uint32_t phase = 0;
    uint32_t armed_mask = 0, armed_parity = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < b.total_tiles; tile += gridDim.x) {
      int pi, m0, nt;
      decode(b, tile, pi, m0, nt);
      const TcProblem& P = b.p[pi];
      const int n0 = nt * BN;
      const int kblocks = (P.K + BKE - 1) / BKE;
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!ptx::mbar_wait(&empty[stage], phase ^ 1u, abort_flag, limit)) {
          ok = false;
          break;
        }
        uint8_t* st = smem + stage * C::kStageBytes;
        ptx::mbar_arrive_expect_tx(&full[stage], C::kStageBytes);
        armed_mask |= 1u << stage;
        armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
        const int x = kb * BKE;
        ptx::tma_load_2d(st, &P.a_hi, &full[stage], x, m0);
        ptx::tma_load_2d(st + C::kABytes, &P.a_lo, &full[stage], x, m0);
        ptx::tma_load_2d(st + 2 * C::kABytes, &P.b_hi, &full[stage], x, n0);
        ptx::tma_load_2d(st + 2 * C::kABytes + C::kBBytes, &P.b_lo, &full[stage], x, n0);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    for (int s = 0; s < STAGES; ++s)
      if (armed_mask & (1u << s)) mbar_drain(&full[s], (armed_parity >> s) & 1u, limit);
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issue
    constexpr uint32_t idesc = F16 ? ptx::idesc_f16(BM, BN) : ptx::idesc_tf32(BM, BN);
    auto mma = [&](uint32_t d, uint64_t a, uint64_t bb, uint32_t accum) {
      if (F16) {
        ptx::umma_f16(d, a, bb, idesc, accum);
      } else {
        ptx::umma_tf32(d, a, bb, idesc, accum);
      }
    };
    int stage = 0;
    uint32_t phase = 0;
    uint32_t chunk = 0;  // K blocks issued so far by this CTA
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < b.total_tiles; tile += gridDim.x) {
      int pi, m0, nt;
      decode(b, tile, pi, m0, nt);
      const int kstages = (b.p[pi].K + BKE - 1) / BKE;
      for (int ks = 0; ok && ks < kstages; ++ks) {
        if (!ptx::mbar_wait(&full[stage], phase, abort_flag, limit)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t s = ptx::smem_u32(smem + stage * C::kStageBytes);
        const uint64_t ah = ptx::sw128_kmajor_desc(s);
        const uint64_t al = ptx::sw128_kmajor_desc(s + C::kABytes);
        const uint64_t bh = ptx::sw128_kmajor_desc(s + 2 * C::kABytes);
        const uint64_t bl = ptx::sw128_kmajor_desc(s + 2 * C::kABytes + C::kBBytes);
#pragma unroll
        for (int sb = 0; sb < kSub; ++sb, ++chunk) {  // the stage's K blocks
          const uint32_t buf = chunk % kBufs, use = chunk / kBufs;
          if (!ptx::mbar_wait(&tempty[buf], (use & 1u) ^ 1u, abort_flag, limit)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t d = tmem_base + buf * BN;
          // 32 bytes per MMA (8 tf32 or 16 fp16 elements of K)
#pragma unroll
          for (int kk = 0; kk < kMmaPerBlock; ++kk) {  // cross terms first ...
            const uint64_t off = static_cast<uint64_t>((sb * kMmaPerBlock + kk) * 32 >> 4);
            mma(d, ah + off, bl + off, kk > 0 ? 1u : 0u);
            mma(d, al + off, bh + off, 1u);
          }
#pragma unroll
          for (int kk = 0; kk < kMmaPerBlock; ++kk) {  // ... then hi*hi
            const uint64_t off = static_cast<uint64_t>((sb * kMmaPerBlock + kk) * 32 >> 4);
            mma(d, ah + off, bh + off, 1u);
          }
          ptx::umma_commit(&tfull[buf]);
        }
        if (!ok) break;
        ptx::umma_commit(&empty[stage]);  // frees the stage once its MMAs finish
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    ptx::umma_commit(drain);
    mbar_drain(drain, 0, limit);
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;
    const int colgrp = (warp - 2) >> 2;  // columns 64 colgrp .. +63 of the tile
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t sums = tmem_base + lane_off + kPreciseSumCol + colgrp * kPreciseCols;
    const uint32_t comps = tmem_base + lane_off + kPreciseCompCol + colgrp * kPreciseCols;
    uint32_t chunk = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < b.total_tiles; tile += gridDim.x) {
      int pi, m0, nt;
      decode(b, tile, pi, m0, nt);
      const TcProblem& P = b.p[pi];
      const int n0 = nt * BN;
      const int kblocks = kSub * ((P.K + BKE - 1) / BKE);
      // grp: per 16-column piece, the sum of the blocks since the piece's
      // last fold.  Folds come one per block (TF32 form) or one per stage of
      // two blocks (fp16 form), piece q at folds q, q + 4, q + 8, ..., so that
      // no block carries more than one piece's fold.
      float grp[kPreciseCols];
#pragma unroll
      for (int c = 0; c < kPreciseCols; ++c) grp[c] = 0.f;
      {  // the apply modes read C after the last block: bring it into L2 now
        const int prow = m0 + quarter * 32 + lane, pcol = n0 + colgrp * kPreciseCols;
        if ((P.epi == kEpiApply || P.epi == kEpiApplySplit) && prow < P.M && pcol < P.N) {
          const int last = min(P.N - 1, pcol + kPreciseCols - 1) - pcol;
          const int64_t o = (int64_t)prow * P.ldc + pcol;
#pragma unroll
          for (int c = 0; c < kPreciseCols; c += 32) {
            ptx::prefetch_l2(P.c_hi + o + min(c, last));
            if (P.epi == kEpiApplySplit) ptx::prefetch_l2(P.c_lo + o + min(c, last));
          }
          ptx::prefetch_l2(P.c_hi + o + last);
          if (P.epi == kEpiApplySplit) ptx::prefetch_l2(P.c_lo + o + last);
        }
      }
      for (int kb = 0; kb < kblocks; ++kb, ++chunk) {
        const uint32_t buf = chunk % kBufs, use = chunk / kBufs;
        if (!ptx::mbar_wait(&tfull[buf], use & 1u, abort_flag, limit)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t t = tmem_base + lane_off + buf * BN + colgrp * kPreciseCols;
        // the block partial (one TMEM round trip) into the group sums
        {
          uint32_t xa[32], xb[32];
          ptx::tmem_ld_32x32b_x32(t, xa);
          ptx::tmem_ld_32x32b_x32(t + 32, xb);
          ptx::tmem_wait_ld();
          ptx::tc_fence_before();  // the block buffer is read: release it
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&tempty[buf]);
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            grp[c] += __uint_as_float(xa[c]);
            grp[32 + c] += __uint_as_float(xb[c]);
          }
        }
        if (SHORT) continue;  // the whole sum stays in registers
        // after every kSub-th block, fold piece (kb / kSub) % 4 into the
        // compensated running sum (fp16 stages: one fold per stage)
        if (kb % kSub != kSub - 1) continue;
        const int fi = kb / kSub;
        const int fq = fi % kPreciseGroup;
#pragma unroll
        for (int q = 0; q < kPreciseCols / 16; ++q) {
          if (q != fq) continue;
          uint32_t sv[16], cv[16];
          if (fi >= kPreciseGroup) {  // the piece has been folded before
            ptx::tmem_wait_st();      // (its stores, four folds ago, are done)
            ptx::tmem_ld_32x32b_x16(sums + 16 * q, sv);
            ptx::tmem_ld_32x32b_x16(comps + 16 * q, cv);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              float comp = __uint_as_float(cv[c]);
              sv[c] = __float_as_uint(kahan_add(__uint_as_float(sv[c]), grp[16 * q + c], comp));
              cv[c] = __float_as_uint(comp);
            }
          } else {  // first fold: sum = group sum, compensation 0
            // (written 0 x group sum: a literal zero here makes the compiler
            // hold sixteen zero registers across the whole K loop)
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              sv[c] = __float_as_uint(grp[16 * q + c]);
              cv[c] = __float_as_uint(0.f * grp[16 * q + c]);
            }
          }
          ptx::tmem_st_32x32b_x16(sums + 16 * q, sv);
          ptx::tmem_st_32x32b_x16(comps + 16 * q, cv);
#pragma unroll
          for (int c = 0; c < 16; ++c) grp[16 * q + c] = 0.f;
        }
      }
      if (!ok) break;
      // the blocks since each piece's last fold complete its sum, in place
      if (!SHORT) ptx::tmem_wait_st();
#pragma unroll
      for (int q = 0; q < kPreciseCols / 16; ++q) {
        // never folded (its first fold comes after block kSub (q + 1) - 1):
        // grp holds the whole sum
        if (SHORT || kblocks <= kSub * (q + 1) - 1) continue;
        uint32_t sv[16], cv[16];
        ptx::tmem_ld_32x32b_x16(sums + 16 * q, sv);
        ptx::tmem_ld_32x32b_x16(comps + 16 * q, cv);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          float comp = __uint_as_float(cv[c]);
          const float sum = kahan_add(__uint_as_float(sv[c]), grp[16 * q + c], comp);
          grp[16 * q + c] = sum - comp;  // the compensated sum
        }
      }
      const int row = m0 + quarter * 32 + lane;
      float fout = 1.f;
      if (F16) {  // undo the operands' power-of-two scales (exact)
        float f = P.c0;
        if (P.row_inv && row < P.M) f *= P.row_inv[row];
        if (P.ina.r) f *= pow2_below_inv(bound_value(P.ina), kF16ScaleExp);
        if (P.inb.r) f *= pow2_below_inv(bound_value(P.inb), kF16ScaleExp);
        if (P.outb.r) fout = pow2_below(bound_value(P.outb), kF16ScaleExp);
        // B's row scales: lane l loads those of columns l and 32 + l, and
        // the warp passes them round (64 loads per thread spilled registers)
        const int cbase = n0 + colgrp * kPreciseCols;
        float ci0 = 1.f, ci1 = 1.f;
        if (P.col_inv) {
          ci0 = P.col_inv[min(cbase + lane, P.N - 1)];
          ci1 = P.col_inv[min(cbase + 32 + lane, P.N - 1)];
        }
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          grp[c] *= f * __shfl_sync(0xffffffffu, ci0, c);
          grp[32 + c] *= f * __shfl_sync(0xffffffffu, ci1, c);
        }
      }
      float* stage = stage_area + (warp - 2) * kStageFloats;
#pragma unroll
      for (int q = 0; q < kPreciseCols / 32; ++q) {
        const int col0 = n0 + colgrp * kPreciseCols + q * 32;
        uint32_t r[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) r[c] = __float_as_uint(grp[32 * q + c]);
        if (col0 < P.N) {
          if (F16) {  // (the refresh's outputs are transposed: no staging)
            if (P.epi == kEpiStoreF16SplitT) {
              store_chunk_f16t(P, row, col0, r, fout);
            } else {
              store_chunk(P, row, col0, r);
            }
          } else if (rows_path(P.epi)) {
            store_chunk_rows(P, m0 + quarter * 32, col0, r, stage);
          } else {
            store_chunk(P, row, col0, r);
          }
        }
      }
    }
  }

  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, kCols);
  }
  if (threadIdx.x == 0 && *abort_flag && b.status) atomicExch(b.status, ROT_ETIMEOUT);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int get_encoder() {
  if (g_encode) return ROT_OK;
  cudaDriverEntryPointQueryResult q;
  void* fn = nullptr;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn)
    return ROT_ECUDA;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return ROT_OK;
}

// Row-major rows x K matrix (leading dimension ld elements) of float32 or
// fp16, boxes of box_rows x 128 bytes with 128-byte swizzle; out-of-range
// elements read as 0.
int encode(CUtensorMap* map, const float* base, int rows, int K, int ld, int box_rows,
           bool f16 = false) {
  const int esize = f16 ? 2 : 4;
  if ((reinterpret_cast<uintptr_t>(base) & 15) || ((int64_t)ld * esize) % 16) return ROT_EINVAL;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * esize};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / esize), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                        2, const_cast<float*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ROT_OK : ROT_EINVAL;
}

int num_sms() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  }
  return n;
}

using TcKernel = void (*)(TcBatch);

// The kernel of a launch configuration (the precise variants only where asked
// for, so that no unused configuration is compiled).
template <int BN, int STAGES, bool SPLIT3, bool PRECISE, bool F16, bool SHORT>
TcKernel pick_kernel() {
  if constexpr (PRECISE)
    return gemm_tc_precise_kernel<STAGES, SHORT, F16>;
  else
    return gemm_tc_kernel<BN, STAGES, SPLIT3, F16>;
}

template <int BN, int STAGES, bool SPLIT3, bool PRECISE = false, bool F16 = false>
int launch(const hvec<GemmProblem>& probs, int* status, cudaStream_t stream) {
  using C = Cfg<BN, STAGES, SPLIT3>;
  // the precise kernel also stages its row-major output (one area per epilogue warp)
  constexpr int kSmem =
      C::kSmem + (PRECISE ? kPreciseEpiWarps * kStageFloats * (int)sizeof(float) : 0);
  static_assert(kSmem <= 232448, "dynamic shared memory above 227 KB");
  static_assert(!PRECISE || (BN == 128 && SPLIT3), "precise variants are split, BN = 128");
  const TcKernel kernel = pick_kernel<BN, STAGES, SPLIT3, PRECISE, F16, false>();
  const TcKernel kernel_short = pick_kernel<BN, STAGES, SPLIT3, PRECISE, F16, true>();
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) !=
            cudaSuccess ||
        cudaFuncSetAttribute(kernel_short, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmem) != cudaSuccess)
      return ROT_ECUDA;
    attr = true;
  }
  if (get_encoder() != ROT_OK) return ROT_ECUDA;
  thread_local static TcBatch b;  // ~23 KB parameter block: keep off the stack
  size_t i = 0;
  while (i < probs.size()) {
    std::memset(&b, 0, sizeof(b));
    int total = 0, kmax = 0;
    double flops = 0.0;
    while (i < probs.size() && b.count < kMaxP) {
      const GemmProblem& G = probs[i++];
      if (G.M <= 0 || G.N <= 0) continue;
      if (G.K <= 0 || (G.f16 != 0) != F16) return ROT_EINVAL;
      if (G.epi == kEpiStoreF16SplitT && !F16) return ROT_EINVAL;
      TcProblem& P = b.p[b.count];
      if (encode(&P.a_hi, G.a_hi, G.M, G.K, G.lda, BM, F16) != ROT_OK ||
          encode(&P.b_hi, G.b_hi, G.N, G.K, G.ldb, BN, F16) != ROT_OK)
        return ROT_EINVAL;
      if (SPLIT3 && (encode(&P.a_lo, G.a_lo, G.M, G.K, G.lda, BM, F16) != ROT_OK ||
                     encode(&P.b_lo, G.b_lo, G.N, G.K, G.ldb, BN, F16) != ROT_OK))
        return ROT_EINVAL;
      P.M = G.M;
      P.N = G.N;
      P.K = G.K;
      P.tiles_n = (G.N + BN - 1) / BN;
      P.tile_start = total;
      P.epi = G.epi;
      P.ldc = G.ldc;
      P.alpha = G.alpha;
      P.mma_only = G.mma_only;
      P.c_hi = G.c_hi;
      P.c_lo = G.c_lo;
      P.row_inv = G.row_inv;
      P.in_r = G.in_r;
      P.out_r = G.out_r;
      P.c0 = G.c0;
      P.col_inv = G.col_inv;
      P.ina = G.ina;
      P.inb = G.inb;
      P.outb = G.outb;
      total += ((G.M + BM - 1) / BM) * P.tiles_n;
      kmax = std::max(kmax, G.K);
      flops += 2.0 * G.M * (double)G.N * G.K;
      ++b.count;
    }
    if (total == 0) continue;
    b.total_tiles = total;
    b.status = status;
    b.limit_ns = g_wait_limit_ns;
    const int grid = std::min(total, num_sms());
    {
      ProfScope prof(PRECISE ? (F16 ? ROT_PROF_GEMM_PRECISE_F16 : ROT_PROF_GEMM_PRECISE)
                             : (F16 ? ROT_PROF_GEMM_F16 : ROT_PROF_GEMM),
                     flops, stream);
      const TcKernel k = (PRECISE && kmax <= kPreciseShortK) ? kernel_short : kernel;
      k<<<grid, PRECISE ? kThreadsPrecise : kThreads, kSmem, stream>>>(b);
    }
    if (cudaGetLastError() != cudaSuccess) return ROT_ECUDA;
  }
  return ROT_OK;
}

__global__ void wait_timeout_kernel(unsigned long long limit_ns, int* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    abort_flag = 0;
    ptx::fence_barrier_init();
  }
  __syncthreads();
  // nothing ever arrives on `bar`: the bounded wait must give up
  if (threadIdx.x == 0) {
    const bool ok = ptx::mbar_wait(&bar, 0, &abort_flag, limit_ns);
    if (!ok && abort_flag) atomicExch(status, ROT_ETIMEOUT);
  }
}

}  // namespace

int launch_wait_timeout(uint64_t limit_ns, int* status, cudaStream_t stream) {
  ProfScope prof(ROT_PROF_GEMM, 0.0, stream);
  wait_timeout_kernel<<<1, 32, 0, stream>>>(limit_ns, status);
  return cudaGetLastError() == cudaSuccess ? ROT_OK : ROT_ECUDA;
}

int gemm_tc(const hvec<GemmProblem>& probs, int precision, int* status,
            cudaStream_t stream) {
  if (precision == kPrecPrecise) return launch<128, 3, true, true>(probs, status, stream);
  if (precision == kPrecPrecise16) return launch<128, 3, true, true, true>(probs, status, stream);
  if (precision == ROT_PREC_3XF16) {
    bool narrow16 = true;
    for (const GemmProblem& P : probs) narrow16 = narrow16 && P.N <= 128;
    return narrow16 ? launch<128, 3, true, false, true>(probs, status, stream)
                    : launch<256, 2, true, false, true>(probs, status, stream);
  }
  // narrow products (every N <= 128) use 128-wide tiles so no MMA column is wasted
  bool narrow = true;
  for (const GemmProblem& P : probs) narrow = narrow && P.N <= 128;
  if (precision == ROT_PREC_3XTF32) {
    return narrow ? launch<128, 3, true>(probs, status, stream)
                  : launch<256, 2, true>(probs, status, stream);
  }
  return narrow ? launch<128, 6, false>(probs, status, stream)
                : launch<256, 4, false>(probs, status, stream);
}

}  // namespace rot
