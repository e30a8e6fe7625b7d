// Batched blocked Householder QR+ (Q factor only) for the basis refresh.
//
// Definition (page "分布式训练中的流水线并行与梯度陈旧性优化", section 2.2:
// the refresh orthonormalises the power-iteration product with a QR): for a
// square A, tau = rank_rtol * max_j ||a_j||; for k = 0, 1, ...: x =
// (H_{k-1}..H_0 A)[k:, k], stop when ||x|| <= tau, else beta_k = -sgn(x_0)||x||
// (sgn(0) = +1), w = x - beta_k e_0, H_k = I - 2 w w^T / (w^T w).  Q = H_0 ...
// H_{r-1} I, and column k < r is multiplied by sgn(beta_k) so that R's diagonal
// is positive.  The input's rank is at most rmax (= min(m, n) for the bases of
// an m x n momentum), so only the first rmax columns are ever factored.
//
// Storage: the input arrives transposed and split (row j of `at` = column j
// of A, as hi + lo), so a column and a reflector are contiguous.  Reflector k
// overwrites row k from element k on, normalised to unit length (v = w/||w||,
// H_k = I - 2 v v^T); the R entries the factorisation leaves in front of it
// are zeroed, so rows of `at` serve directly as the reflector matrix Y^T.
//
// Blocking (compact WY: Schreiber & Van Loan, "A storage-efficient WY
// representation for products of Householder transformations", 1989; Golub &
// Van Loan, "Matrix Computations", section 5.1.7):
//   * panels of b = 32 columns are factored by one thread-block cluster per
//     matrix with the panel resident in distributed shared memory;
//   * the rest of the panel's 256-column block is updated on CUDA cores with
//     the panel's 32 x 32 triangular factor;
//   * each 256-column block's reflectors form H_k..H_{k+255} = I - Y T Y^T;
//     the columns after the block (up to rmax) receive a <- (I - Y T^T Y^T) a,
//     and Q is accumulated backwards a pair of blocks at a time (the pair's
//     factor joined from the two blocks'), q <- (I - Y T Y^T) q, both as
//     three tensor-core GEMMs (T^T Y^T or T Y^T, then X (Y T), X -= Z Y^T),
//     on the precise kernel (K-blocks summed in float32): Q's orthogonality
//     error adds up over all p^2 entries.
// A range guard (qr_colnorm_kernel, qr_scale_kernel) rescales inputs whose
// squared column norms would leave float32's range.
#include <cooperative_groups.h>

#include <algorithm>
#include <cstring>

#include "profile.h"
#include "rot_internal.h"
#include "split.cuh"
#include "tc_ptx.cuh"

namespace cg = cooperative_groups;

namespace rot {
namespace {

constexpr int B = kQrPanel;   // panel width (32)
constexpr int NB = kQrBlock;  // block width (256)
constexpr int kMaxQ = 64;
constexpr unsigned kFull = 0xffffffffu;

struct QrBatch {
  int count;
  int* status;                  // ROT_ETIMEOUT when a bounded wait runs out
  unsigned long long limit_ns;  // the bound
  QrProblem p[kMaxQ];
};
static_assert(sizeof(QrBatch) <= 32764, "kernel parameter block above the 32764-byte limit");

// Remote store into a peer CTA's shared memory (the address of `local` in the
// CTA of cluster rank `rank`) that completes as 4 transaction bytes on the
// barrier at `bar`'s offset in that CTA.
__device__ __forceinline__ void push_b32(const void* local, float v, const uint64_t* bar,
                                         uint32_t rank) {
  uint32_t ra, rb;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
               : "=r"(ra)
               : "r"(ptx::smem_u32(local)), "r"(rank));
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
               : "=r"(rb)
               : "r"(ptx::smem_u32(bar)), "r"(rank));
  asm volatile("st.async.weak.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::
                   "r"(ra),
               "r"(__float_as_uint(v)), "r"(rb)
               : "memory");
}

__host__ __device__ inline int npanels(int rmax) { return (rmax + B - 1) / B; }
__host__ __device__ inline int nblocks(int rmax) { return (rmax + NB - 1) / NB; }

// ---------------------------------------------------------------------------
// reductions
// ---------------------------------------------------------------------------

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// 32 values per thread -> lane L of each warp holds the warp's total of v[L]
// (31 shuffles: each step halves the values a lane keeps).
__device__ __forceinline__ float warp_transpose_sum(float (&v)[B]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < off; ++i) {
      const float send = upper ? v[i] : v[i + off];
      const float keep = upper ? v[i + off] : v[i];
      v[i] = keep + __shfl_xor_sync(kFull, send, off);
    }
  }
  return v[0];
}

__device__ __forceinline__ int rank_now(const QrProblem& q) {
  return q.ctrl[1] ? q.ctrl[0] : q.rmax;
}

// ---------------------------------------------------------------------------
// set-up: scratch reset and the threshold's column norms
// ---------------------------------------------------------------------------

__global__ void qr_init_kernel(const __grid_constant__ QrBatch b) {
  const QrProblem& q = b.p[blockIdx.x];
  const int np = npanels(q.rmax);
  for (int i = threadIdx.x; i < np + 2; i += blockDim.x) q.ctrl[i] = (i == 0) ? -1 : 0;
  if (threadIdx.x == 0) {
    q.tau[0] = 0.f;
    q.tau[1] = 0.f;
  }
}

// Range guard.  Q+ of s A is Q+ of A for s > 0 (the reflectors are scale-free
// and the rank threshold is relative).  When max |a_ij| lies outside
// [2^-50, 2^50] -- where squared column norms of a p <= 2^15 input could under-
// or overflow float32 -- the rows the factorisation reads are multiplied by a
// power of two s with max |a_ij| s < 1 (exact), and the rank threshold with
// them; inside that range s = 1 and nothing is touched.
__device__ __forceinline__ float qr_range_scale(float amax) {
  return (amax >= 8.8817842e-16f && amax <= 1.1258999e15f) ? 1.f : pow2_below(amax, 0);
}

// max_j ||a_j|| (rows of `at`) into tau[0] and max |a_ij| into tau[1], by
// atomicMax on the float's bits (values >= 0).  Each column's sum of squares
// is taken on the column times a power of two c with max |x| c < 1 and then
// divided by c: the same bits as the plain sum where that does not under- or
// overflow, the right value where it would.
__global__ void qr_colnorm_kernel(const __grid_constant__ QrBatch b) {
  const QrProblem& q = b.p[blockIdx.y];
  const int lane = threadIdx.x & 31;
  const int warps = blockDim.x >> 5;
  float best = 0.f, amax = 0.f;
  for (int j = blockIdx.x * warps + (threadIdx.x >> 5); j < q.p; j += gridDim.x * warps) {
    const int64_t o = (int64_t)j * q.ld;
    float cm = 0.f;
    for (int e = lane; e < q.p; e += 32) cm = fmaxf(cm, fabsf(q.at.hi[o + e] + q.at.lo[o + e]));
    cm = warp_max(cm);
    const float c = pow2_below(cm, 0);
    float s = 0.f;
    for (int e = lane; e < q.p; e += 32) {
      const float x = (q.at.hi[o + e] + q.at.lo[o + e]) * c;
      s = fmaf(x, x, s);
    }
    s = warp_sum(s);
    best = fmaxf(best, sqrtf(s) * pow2_below_inv(cm, 0));
    amax = fmaxf(amax, cm);
  }
  if (lane == 0 && best > 0.f) atomicMax(reinterpret_cast<int*>(q.tau), __float_as_int(best));
  if (lane == 0 && amax > 0.f) atomicMax(reinterpret_cast<int*>(q.tau + 1), __float_as_int(amax));
}

// s A on the rows the factorisation reads (the first rmax columns of A), when
// the range guard asks for it.
__global__ void qr_scale_kernel(const __grid_constant__ QrBatch b) {
  const QrProblem& q = b.p[blockIdx.y];
  const float sc = qr_range_scale(q.tau[1]);
  if (sc == 1.f) return;
  for (int j = blockIdx.x; j < q.rmax; j += gridDim.x) {
    const int64_t o = (int64_t)j * q.ld;
    for (int e = threadIdx.x; e < q.p; e += blockDim.x) {
      q.at.hi[o + e] *= sc;
      q.at.lo[o + e] *= sc;
    }
  }
}

// ---------------------------------------------------------------------------
// panel factorisation: one cluster of `cs` CTAs per matrix, columns
// k0 .. k0+bw-1; CTA c of the cluster holds elements [k0 + c R, k0 + (c+1) R)
// of the panel's rows in shared memory.
//
// One pass and one cluster-wide reduction per column: the pass that applies
// H_j to the later columns also accumulates, for column j+1, the dot products
// x_{j+1} . a_c with every panel row (c = j+1 gives ||x_{j+1}||^2), and the
// thread holding element k+1 records the pivot row a_c[k+1].  Since
// w = x - beta e_k, w . a_c = x . a_c - beta a_c[k] follows from those sums,
// and so do the Gram entries w_i . w_j of the panel's triangular factor.
// The 64 partial values of every CTA go to every CTA through distributed
// shared memory; every warp of every CTA adds them in the same order, so all
// of them take the same decisions, and each warp derives the reflector's
// coefficients itself.  A column therefore costs one block barrier (the
// warps' partial sums) and one cluster barrier (the exchange).
// ---------------------------------------------------------------------------

constexpr int kPanelThreads = 256;
constexpr int kMaxCluster = 16;  // 16 needs the non-portable cluster size

__global__ void __launch_bounds__(kPanelThreads)
    qr_panel_kernel(const __grid_constant__ QrBatch b, int k0, float rtol, int R) {
  cg::cluster_group cl = cg::this_cluster();
  const int cs = (int)cl.num_blocks();
  const int crank = (int)cl.block_rank();
  const QrProblem& q = b.p[blockIdx.x / cs];
  extern __shared__ float panel[];  // [B][R]
  __shared__ float slot[2][kMaxCluster][2 * B];
  __shared__ float red[B][kPanelThreads / 32 + 1];
  __shared__ float s_piv[2][B];  // pivot row a_c[k] of the column being reduced, by parity
  __shared__ float s_coef[B];
  __shared__ float w_coef[kPanelThreads / 32][B];  // each warp's copy of the coefficients
  __shared__ float s_ww[B], s_beta[B];
  __shared__ float gram[B][B + 1];
  __shared__ float tmat[B][B + 1];
  __shared__ uint64_t xbar[2];  // the exchange of each parity completes here

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nthr = blockDim.x, nwarp = nthr >> 5;
  const int p = q.p, ld = q.ld;
  const int panel_id = k0 / B;
  const bool in_range = k0 < q.rmax;
  const int bw = in_range ? min(B, q.rmax - k0) : 0;
  const int e0 = k0 + crank * R, e1 = min(p, e0 + R);
  float* at_hi = q.at.hi;
  float* at_lo = q.at.lo;

  if (!in_range) {  // the same for every CTA of the cluster
    cl.sync();
    return;
  }
  if (q.ctrl[1] != 0) {
    // stopped in an earlier panel: these rows are identities; clear them so
    // that the block GEMMs read zeros there
    for (int j = 0; j < bw; ++j)
      for (int e = crank * nthr + tid; e < p; e += cs * nthr) {
        const int64_t o = (int64_t)(k0 + j) * ld + e;
        at_hi[o] = 0.f;
        at_lo[o] = 0.f;
      }
    if (crank == 0 && tid == 0) q.ctrl[2 + panel_id] = 0;
    cl.sync();
    return;
  }

  // load my slice of the panel; clear the R entries in front of it
  // (elements 0 .. k0-1 of the panel's rows, so that a row of `at` is its
  // reflector from element 0: Q formation reads pairs of blocks from the
  // first block's start)
  for (int i = tid; i < bw * R; i += nthr) {
    const int j = i / R, e = e0 + i % R;
    float x = 0.f;
    if (e < e1) {
      const int64_t o = (int64_t)(k0 + j) * ld + e;
      x = at_hi[o] + at_lo[o];
    }
    panel[i] = x;
  }
  for (int j = 0; j < bw; ++j)
    for (int e = crank * nthr + tid; e < k0; e += cs * nthr) {
      const int64_t o = (int64_t)(k0 + j) * ld + e;
      at_hi[o] = 0.f;
      at_lo[o] = 0.f;
    }
  if (tid < 2 * B) (&s_piv[0][0])[tid] = 0.f;
  if (tid == 0) {
    ptx::mbar_init(&xbar[0], 1);
    ptx::mbar_init(&xbar[1], 1);
    ptx::fence_barrier_init();
  }
  cl.sync();  // every CTA's barriers exist before any CTA pushes to them

  // Block-reduce acc[] (and the pivot row) for the next column, exchange with
  // the cluster through slot[par], and leave the cluster totals in every
  // warp's registers: lane c gets tot_dot = x . a_c and tot_piv = a_c[k].
  // Hazards: red and s_piv[par] are read after the block barrier and written
  // again only after the next column's cluster barrier (s_piv alternates by
  // parity, and its reader clears it for the column after next); slot[par]
  // is rewritten by other CTAs only after they pass the next cluster barrier,
  // which this CTA reaches after its reads.
  // The exchange completes on this CTA's barrier xbar[par] (armed for the
  // cs x 64 values of the column; a peer's values may land before the
  // arming, which the barrier's transaction count allows) instead of a
  // cluster barrier.  A slot and barrier of parity par are written again only
  // two columns later, by a peer that has by then received this CTA's values
  // of the column in between, which this CTA sends only after reading them.
  uint32_t xphase = 0;  // bit p: parity of xbar[p]'s current phase
  bool xfailed = false;  // a wait ran out: stop waiting (the status says so)
  auto reduce_and_share = [&](float (&acc)[B], int par, float& tot_dot, float& tot_piv) {
    const float part = warp_transpose_sum(acc);
    red[lane][warp] = part;
    __syncthreads();
    if (tid == 0) ptx::mbar_arrive_expect_tx(&xbar[par], (uint32_t)(cs * 2 * B * 4));
    if (tid < 2 * B) {
      float t;
      if (tid < B) {
        t = 0.f;
        for (int w = 0; w < nwarp; ++w) t += red[tid][w];
      } else {
        t = s_piv[par][tid - B];
        s_piv[par][tid - B] = 0.f;
      }
      for (int c = 0; c < cs; ++c) push_b32(&slot[par][crank][tid], t, &xbar[par], (uint32_t)c);
    }
    const uint32_t ph = (xphase >> par) & 1u;
    xphase ^= 1u << par;
    if (!xfailed && !ptx::mbar_try_wait(&xbar[par], ph)) {
      const uint64_t t0 = ptx::globaltimer_ns();
      for (uint32_t it = 1;; ++it) {
        if (ptx::mbar_try_wait(&xbar[par], ph)) break;
        if ((it & 63u) == 0u && (ptx::globaltimer_ns() - t0 > b.limit_ns || it > (1u << 30))) {
          xfailed = true;
          if (b.status) atomicExch(b.status, ROT_ETIMEOUT);
          break;
        }
      }
    }
    tot_dot = 0.f;
    tot_piv = 0.f;
    for (int c = 0; c < cs; ++c) {
      tot_dot += slot[par][c][lane];
      tot_piv += slot[par][c][B + lane];
    }
  };

  // sums for column 0: x_0 . a_c over my elements >= k0, pivot row a_c[k0]
  float tot_dot, tot_piv;
  {
    float acc[B];
#pragma unroll
    for (int c = 0; c < B; ++c) acc[c] = 0.f;
    for (int e = e0 + tid; e < e1; e += nthr) {
      const float xn = panel[e - e0];
#pragma unroll
      for (int c = 0; c < B; ++c)
        if (c < bw) acc[c] = fmaf(xn, panel[c * R + (e - e0)], acc[c]);
      if (e == k0)
        for (int c = 0; c < bw; ++c) s_piv[0][c] = panel[c * R + (e - e0)];
    }
    reduce_and_share(acc, 0, tot_dot, tot_piv);
  }

  const float thr = rtol * (q.tau[0] * qr_range_scale(q.tau[1]));
  int active = bw;
  for (int j = 0; j < bw; ++j) {
    const int k = k0 + j;
    const float sn = __shfl_sync(kFull, tot_dot, j);  // ||x_j||^2
    const float x0 = __shfl_sync(kFull, tot_piv, j);  // x_j[0] = a_j[k]
    const float nx = sqrtf(sn);
    if (nx <= thr) {  // numerical rank reached: H_k .. are identities
      active = j;
      break;
    }
    const float beta = x0 >= 0.f ? -nx : nx;
    const float w0 = x0 - beta;
    const float ww = 2.f * fmaf(fabsf(x0), nx, sn);  // ||x - beta e0||^2, no cancellation
    const float d = tot_dot - beta * tot_piv;         // lane c: w_j . a_c
    if (warp == 0) {
      if (lane < j) gram[lane][j] = d;
      if (lane == 0) {
        s_ww[j] = ww;
        s_beta[j] = beta;
      }
    }
    // the thread that handles element k in the pass below is thread 0
    if (tid == 0 && k >= e0 && k < e1) panel[j * R + (k - e0)] = w0;
    if (j + 1 == bw) break;  // nothing after the last column
    w_coef[warp][lane] = 2.f * d / ww;  // lane c > j: column c's coefficient
    __syncwarp();

    // apply H_k to columns j+1.. (my elements >= k) and accumulate column
    // j+1's sums over my elements >= k+1
    float acc[B];
#pragma unroll
    for (int c = 0; c < B; ++c) acc[c] = 0.f;
    const float* wr = panel + j * R;
    const float* coef = w_coef[warp];
    const int par = (j + 1) & 1;
    for (int e = max(k, e0) + tid; e < e1; e += nthr) {
      const int o = e - e0;
      const float we = wr[o];
      for (int c = j + 1; c < bw; ++c) panel[c * R + o] -= coef[c] * we;
      if (e > k) {
        const float xn = panel[(j + 1) * R + o];
#pragma unroll
        for (int c = 0; c < B; ++c)
          if (c < bw) acc[c] = fmaf(xn, panel[c * R + o], acc[c]);
        if (e == k + 1)
          for (int c = 0; c < bw; ++c) s_piv[par][c] = panel[c * R + o];
      }
    }
    __syncwarp();  // this warp's coefficients are read: free for the next column
    reduce_and_share(acc, par, tot_dot, tot_piv);
  }
  __syncthreads();  // every reflector, gram entry and norm of the panel is written

  // Reflectors are stored normalised, v = w / ||w|| (H = I - 2 v v^T), so the
  // triangular factors and Gram matrices built from them are well scaled
  // whatever the column norms were.  Zero the R entries inside the panel
  // (elements < k of reflector row k) and the rows past the rank; write my
  // slice back as a split.
  if (tid < B) s_coef[tid] = tid < active ? 1.f / sqrtf(s_ww[tid]) : 0.f;
  __syncthreads();
  for (int i = tid; i < bw * R; i += nthr) {
    const int j = i / R, e = e0 + i % R;
    if (e >= e1) continue;
    float x = panel[i] * s_coef[j];
    if (j >= active || e < k0 + j) x = 0.f;
    float h, l;
    split_tf32(x, h, l);
    const int64_t o = (int64_t)(k0 + j) * ld + e;
    at_hi[o] = h;
    at_lo[o] = l;
  }

  if (crank == 0) {
    // panel factor T of the normalised reflectors: T_jj = 2,
    // T[0:j, j] = -2 T[0:j, 0:j] (v_{0:j}^T v_j), v_l . v_j = gram[l][j] / (||w_l|| ||w_j||)
    if (warp == 0) {
      for (int i = lane; i < B * (B + 1); i += 32) (&tmat[0][0])[i] = 0.f;
      __syncwarp();
      for (int j = 0; j < active; ++j) {
        const float tjj = 2.f;
        float t = 0.f;
        if (lane < j)
          for (int l = lane; l < j; ++l)
            t = fmaf(tmat[lane][l], gram[l][j] * s_coef[l] * s_coef[j], t);
        __syncwarp();
        if (lane < j) tmat[lane][j] = -tjj * t;
        if (lane == j) tmat[j][j] = tjj;
        __syncwarp();
      }
    }
    __syncthreads();
    float* tf = q.tf + (int64_t)panel_id * B * B;
    for (int i = tid; i < B * B; i += nthr) tf[i] = tmat[i / B][i % B];
    if (tid < active) q.beta[k0 + tid] = s_beta[tid];
    if (tid == 0) {
      q.ctrl[2 + panel_id] = active;
      if (active < bw) {
        q.ctrl[1] = 1;
        q.ctrl[0] = k0 + active;
      }
    }
  }
  cl.sync();  // no CTA leaves while its shared memory may still be written
}

// ---------------------------------------------------------------------------
// within-block update: rows k0+b .. (block end)-1 of `at` get the panel's
// reflectors, a <- a - Y (T^T (Y^T a)), elements k0..p-1 (CUDA cores).
// Split along the elements so that every launch fills the GPU: the first
// kernel writes, per 256-element chunk and 32-row tile, the partial products
// Y^T a; the second adds the chunks' partials in a fixed order (so results
// do not depend on scheduling), applies T^T and updates its chunk.
// ---------------------------------------------------------------------------

constexpr int kRows = 32;
constexpr int kChunk = 256;
constexpr int kRowTiles = (NB - B) / kRows;  // rows after the first panel of a block

__device__ __forceinline__ bool apply_tile(const QrProblem& q, int k0, int& active, int& r0,
                                           int& row_end, int& e_begin, int& e_end) {
  if (k0 >= q.rmax) return false;
  active = q.ctrl[2 + k0 / B];
  if (active == 0) return false;
  row_end = min(q.rmax, (k0 / NB) * NB + NB);
  r0 = k0 + B + blockIdx.y * kRows;
  if (r0 >= row_end) return false;
  e_begin = k0 + blockIdx.x * kChunk;
  if (e_begin >= q.p) return false;
  e_end = min(q.p, e_begin + kChunk);
  return true;
}

__global__ void __launch_bounds__(256) qr_apply_partial_kernel(const __grid_constant__ QrBatch b,
                                                               int k0) {
  const QrProblem& q = b.p[blockIdx.z];
  int active, r0, row_end, e_begin, e_end;
  if (!apply_tile(q, k0, active, r0, row_end, e_begin, e_end)) return;
  const int ld = q.ld;
  const float* xh = q.at.hi;
  const float* xl = q.at.lo;
  __shared__ float xs[kRows][33];
  __shared__ float ys[B][33];
  const int tid = threadIdx.x, r = tid >> 3, i4 = (tid & 7) * 4;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  // each thread's four elements of a 32 x 32 sub-chunk, loaded one sub-chunk
  // ahead (the loads are in flight while the previous one is multiplied)
  float xv[4], yv[4];
  auto load = [&](int c0) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int t = tid + 256 * u, rr = t >> 5, ee = t & 31, e = c0 + ee;
      const int row = r0 + rr;
      xv[u] = 0.f;
      yv[u] = 0.f;
      if (row < row_end && e < e_end) {
        const int64_t o = (int64_t)row * ld + e;
        xv[u] = xh[o] + xl[o];
      }
      if (rr < active && e < e_end && e >= k0 + rr) {
        const int64_t o = (int64_t)(k0 + rr) * ld + e;
        yv[u] = xh[o] + xl[o];
      }
    }
  };
  load(e_begin);
  for (int c0 = e_begin; c0 < e_end; c0 += 32) {
    __syncthreads();
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int t = tid + 256 * u;
      xs[t >> 5][t & 31] = xv[u];
      ys[t >> 5][t & 31] = yv[u];
    }
    __syncthreads();
    if (c0 + 32 < e_end) load(c0 + 32);
#pragma unroll 8
    for (int ee = 0; ee < 32; ++ee) {
      const float xe = xs[r][ee];
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[c] = fmaf(xe, ys[i4 + c][ee], acc[c]);
    }
  }
  float* part = q.part + ((int64_t)blockIdx.x * kRowTiles + blockIdx.y) * (kRows * B);
#pragma unroll
  for (int c = 0; c < 4; ++c) part[r * B + i4 + c] = acc[c];
}

__global__ void __launch_bounds__(256) qr_apply_update_kernel(const __grid_constant__ QrBatch b,
                                                              int k0) {
  const QrProblem& q = b.p[blockIdx.z];
  int active, r0, row_end, e_begin, e_end;
  if (!apply_tile(q, k0, active, r0, row_end, e_begin, e_end)) return;
  const int ld = q.ld;
  float* xh = q.at.hi;
  float* xl = q.at.lo;
  __shared__ float ys[B][33];
  __shared__ float z[kRows][B + 1];
  __shared__ float zt[kRows][B + 1];
  __shared__ float tm[B][B + 1];
  const int tid = threadIdx.x;
  const float* tf = q.tf + (int64_t)(k0 / B) * B * B;
  for (int i = tid; i < B * B; i += 256) tm[i / B][i % B] = tf[i];
  // z = sum of the chunks' partials, in chunk order
  const int nchunks = (q.p - k0 + kChunk - 1) / kChunk;
  for (int i = tid; i < kRows * B; i += 256) {
    float t = 0.f;
    for (int c = 0; c < nchunks; ++c)
      t += q.part[((int64_t)c * kRowTiles + blockIdx.y) * (kRows * B) + i];
    z[i / B][i % B] = t;
  }
  __syncthreads();
  const int r = tid >> 3, i4 = (tid & 7) * 4;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int i = i4 + c;
    float t = 0.f;
    for (int jj = 0; jj < B; ++jj) t = fmaf(z[r][jj], tm[jj][i], t);  // (T^T z)_i
    zt[r][i] = t;
  }
  const int e4 = (tid & 7) * 4;
  const int row = r0 + r;
  // the next sub-chunk's reflector elements (four per thread) and this
  // thread's four elements of its row, loaded one sub-chunk ahead; all of a
  // sub-chunk's loads go out before its stores (a store could alias a later
  // load as far as the compiler knows)
  float yv[4], hv[4], lv[4];
  auto load = [&](int c0) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int t = tid + 256 * u, yi = t >> 5, ee = t & 31, e = c0 + ee;
      yv[u] = 0.f;
      if (yi < active && e < e_end && e >= k0 + yi) {
        const int64_t o = (int64_t)(k0 + yi) * ld + e;
        yv[u] = xh[o] + xl[o];
      }
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int e = c0 + e4 + c;
      hv[c] = 0.f;
      lv[c] = 0.f;
      if (row < row_end && e < e_end) {
        const int64_t o = (int64_t)row * ld + e;
        hv[c] = xh[o];
        lv[c] = xl[o];
      }
    }
  };
  load(e_begin);
  for (int c0 = e_begin; c0 < e_end; c0 += 32) {
    __syncthreads();
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int t = tid + 256 * u;
      ys[t >> 5][t & 31] = yv[u];
    }
    __syncthreads();
    float hc[4], lc[4];  // this sub-chunk's row elements
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      hc[c] = hv[c];
      lc[c] = lv[c];
    }
    if (c0 + 32 < e_end) load(c0 + 32);
    if (row < row_end) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int e = c0 + e4 + c;
        if (e < e_end) {
          float t = 0.f;
#pragma unroll 8
          for (int i = 0; i < B; ++i) t = fmaf(zt[r][i], ys[i][e4 + c], t);
          const int64_t o = (int64_t)row * ld + e;
          float h, l;
          split_tf32((hc[c] + lc[c]) - t, h, l);
          xh[o] = h;
          xl[o] = l;
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// block factor T (nb x nb, upper triangular, nb <= NB = 256) from the Gram
// S = Y^T Y of the block's reflectors.  The compact-WY product of two
// consecutive runs of reflectors joins their factors as
// T = [[T0, -T0 S01 T1], [0, T1]]; applied recursively down to runs of 32,
// where the column recurrence T_ii = 2 / S_ii, T[0:i, i] = -T_ii T[0:i, 0:i]
// S[0:i, i] takes over (one warp per run of 32, warp barriers only).  The
// joins at widths 32, 64 and 128 are small register-blocked products.
// Reflectors past the numerical rank get zero rows and columns.  T is
// assembled in float32 scratch and written as T and T^T splits (ld NB).  One
// CTA per matrix, 256 threads, three 128 x 129 shared tiles.
// ---------------------------------------------------------------------------

constexpr int TH = NB / 2;  // 128
constexpr int kTThreads = 256;
constexpr int kLeaf = 32;   // run of reflectors the column recurrence handles

// C (n x n, ld TH + 1) = A B for n x n shared tiles, all 256 threads: thread t
// computes row t / (256 / n), n^2 / 256 consecutive columns.
template <int n>
__device__ __forceinline__ void tile_mul(const float* A, const float* Bt, float* C) {
  constexpr int LD = TH + 1;
  constexpr int tpr = kTThreads / n, cpt = n * n / kTThreads;
  const int r = threadIdx.x / tpr, c0 = (threadIdx.x % tpr) * cpt;
  float acc[cpt];
#pragma unroll
  for (int c = 0; c < cpt; ++c) acc[c] = 0.f;
  for (int k = 0; k < n; ++k) {
    const float av = A[r * LD + k];
#pragma unroll
    for (int c = 0; c < cpt; ++c) acc[c] = fmaf(av, Bt[k * LD + c0 + c], acc[c]);
  }
#pragma unroll
  for (int c = 0; c < cpt; ++c) C[r * LD + c0 + c] = acc[c];
}

// T[o:o+n, o+n:o+2n] = -T0 (S01 T1) with T0, T1 the diagonal blocks at o and
// o + n (already in T), S01 = S[o:o+n, o+n:o+2n].
template <int n>
__device__ void join_block(const QrProblem& q, float* T, int o, int nb, float* tA, float* tB,
                           float* tC) {
  constexpr int LD = TH + 1;
  const int tid = threadIdx.x;
  for (int i = tid; i < n * n; i += kTThreads) {
    const int r = i / n, c = i % n;
    tA[r * LD + c] = o + n + c < nb ? q.s[(int64_t)(o + r) * NB + o + n + c] : 0.f;  // S01
    tB[r * LD + c] = T[(int64_t)(o + n + r) * NB + o + n + c];                      // T1
  }
  __syncthreads();
  tile_mul<n>(tA, tB, tC);  // X = S01 T1
  __syncthreads();
  for (int i = tid; i < n * n; i += kTThreads)
    tA[(i / n) * LD + i % n] = T[(int64_t)(o + i / n) * NB + o + i % n];  // T0
  __syncthreads();
  tile_mul<n>(tA, tC, tB);  // T0 X
  __syncthreads();
  for (int i = tid; i < n * n; i += kTThreads)
    T[(int64_t)(o + i / n) * NB + o + n + i % n] = -tB[(i / n) * LD + i % n];
  __syncthreads();
}

__global__ void __launch_bounds__(kTThreads) qr_tblock_kernel(const __grid_constant__ QrBatch b,
                                                              int kb0) {
  const QrProblem& q = b.p[blockIdx.x];
  if (kb0 >= q.rmax) return;
  extern __shared__ float sm[];
  constexpr int LD = TH + 1;
  float* tA = sm;
  float* tB = sm + TH * LD;
  float* tC = sm + 2 * TH * LD;
  const int nb = min(NB, q.rmax - kb0);
  const int act = max(0, min(nb, rank_now(q) - kb0));
  const int blk = kb0 / NB;
  const int tid = threadIdx.x, nt = blockDim.x;
  float* T = q.tmp;  // NB x NB float32
  for (int i = tid; i < NB * NB; i += nt) T[i] = 0.f;
  __syncthreads();

  // runs of 32 by the column recurrence: warp w takes reflectors 32w .. 32w+31
  // (its S block and T block in 32 x 33 shared tiles carved from tA .. tC)
  {
    const int w = tid >> 5, lane = tid & 31, o = w * kLeaf;
    constexpr int LL = kLeaf + 1;
    float* ls = sm + w * 2 * kLeaf * LL;  // 8 warps x 2 x 32 x 33 floats < 3 tiles
    float* lt = ls + kLeaf * LL;
    for (int i = lane; i < kLeaf * kLeaf; i += 32) {
      const int r = o + i / kLeaf, c = o + i % kLeaf;
      ls[(i / kLeaf) * LL + i % kLeaf] = (r < nb && c < nb) ? q.s[(int64_t)r * NB + c] : 0.f;
      lt[(i / kLeaf) * LL + i % kLeaf] = 0.f;
    }
    __syncwarp();
    const int a = max(0, min(kLeaf, act - o));
    for (int i = 0; i < a; ++i) {
      const float tii = 2.f / ls[i * LL + i];
      float t = 0.f;
      if (lane < i)
        for (int l = lane; l < i; ++l) t = fmaf(lt[lane * LL + l], ls[l * LL + i], t);
      __syncwarp();
      if (lane < i) lt[lane * LL + i] = -tii * t;
      if (lane == i) lt[i * LL + i] = tii;
      __syncwarp();
    }
    for (int i = lane; i < kLeaf * kLeaf; i += 32)
      T[(int64_t)(o + i / kLeaf) * NB + o + i % kLeaf] = lt[(i / kLeaf) * LL + i % kLeaf];
  }
  __syncthreads();

  // joins: 32 -> 64 -> 128 -> 256 (only where the second run has active reflectors)
  for (int o = 0; o < NB; o += 64)
    if (act > o + 32) join_block<32>(q, T, o, nb, tA, tB, tC);
  for (int o = 0; o < NB; o += 128)
    if (act > o + 64) join_block<64>(q, T, o, nb, tA, tB, tC);
  if (act > TH) join_block<TH>(q, T, 0, nb, tA, tB, tC);
  __syncthreads();

  float* th = q.tb.hi + (int64_t)blk * NB * NB;
  float* tl = q.tb.lo + (int64_t)blk * NB * NB;
  float* uh = q.tbt.hi + (int64_t)blk * NB * NB;
  float* ul = q.tbt.lo + (int64_t)blk * NB * NB;
  for (int i = tid; i < NB * NB; i += nt) {
    float h, l;
    split_tf32_mma(T[i], h, l);
    th[i] = h;
    tl[i] = l;
  }
  // T^T through 32 x 33 shared tiles (one per warp), so that both the reads
  // of T and the writes of T^T are row-contiguous
  {
    const int w = tid >> 5, lane = tid & 31;
    float* tile = sm + w * 32 * 33;
    for (int tt = w; tt < (NB / 32) * (NB / 32); tt += nt >> 5) {
      const int r0 = (tt / (NB / 32)) * 32, c0 = (tt % (NB / 32)) * 32;
      for (int i = 0; i < 32; ++i) tile[i * 33 + lane] = T[(int64_t)(r0 + i) * NB + c0 + lane];
      __syncwarp();
      for (int i = 0; i < 32; ++i) {  // row c0 + i of T^T = column c0 + i of T
        float h, l;
        split_tf32_mma(tile[lane * 33 + i], h, l);
        const int64_t o = (int64_t)(c0 + i) * NB + r0 + lane;
        uh[o] = h;
        ul[o] = l;
      }
      __syncwarp();
    }
  }
}

// ---------------------------------------------------------------------------
// Q^T = I (split), then the sign fix and the outputs U^T and U, as the
// 2^14-scaled fp16 splits the state keeps (22 significant bits, the
// precision of the TF32 splits the tensor cores read)
// ---------------------------------------------------------------------------

__global__ void qr_eye_kernel(const __grid_constant__ QrBatch b) {
  const QrProblem& q = b.p[blockIdx.y];
  const int64_t total = (int64_t)q.p * q.p;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int r = (int)(e / q.p), c = (int)(e % q.p);
    const int64_t o = (int64_t)r * q.ld + c;
    q.qt.hi[o] = r == c ? 1.f : 0.f;
    q.qt.lo[o] = 0.f;
  }
}

// The factor of a pair of consecutive blocks b, b+1 (compact WY):
// T = [[T_b, -T_b S01 T_{b+1}], [0, T_{b+1}]], 2 NB x 2 NB (ld 2 NB).  This
// kernel places T_b and T_{b+1} and zeroes the rest; the upper-right block is
// then added by a product.  Problems whose pair has one block are skipped.
__global__ void qr_pair_assemble_kernel(const __grid_constant__ QrBatch b, int kb0) {
  const QrProblem& q = b.p[blockIdx.y];
  if (kb0 + NB >= q.rmax) return;
  const int64_t blk = kb0 / NB;
  const float* t0h = q.tb.hi + blk * NB * NB;
  const float* t0l = q.tb.lo + blk * NB * NB;
  const float* t1h = q.tb.hi + (blk + 1) * NB * NB;
  const float* t1l = q.tb.lo + (blk + 1) * NB * NB;
  for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < 4 * NB * NB;
       e += gridDim.x * blockDim.x) {
    const int r = e / (2 * NB), c = e % (2 * NB);
    float h = 0.f, l = 0.f;
    if (r < NB && c < NB) {
      h = t0h[r * NB + c];
      l = t0l[r * NB + c];
    } else if (r >= NB && c >= NB) {
      h = t1h[(r - NB) * NB + c - NB];
      l = t1l[(r - NB) * NB + c - NB];
    }
    q.tpair.hi[e] = h;
    q.tpair.lo[e] = l;
  }
}

__global__ void qr_finalize_kernel(const __grid_constant__ QrBatch b) {
  __shared__ float tile[32][33];
  const QrProblem& q = b.p[blockIdx.y];
  const int rank = rank_now(q);
  const int tiles = (q.p + 31) / 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  for (int t = blockIdx.x; t < tiles * tiles; t += gridDim.x) {
    const int r0 = (t / tiles) * 32, c0 = (t % tiles) * 32;
    for (int i = ty; i < 32; i += 8) {
      const int r = r0 + i, c = c0 + tx;
      float v = 0.f;
      if (r < q.p && c < q.p) {
        const int64_t oi = (int64_t)r * q.ld + c;
        v = q.qt.hi[oi] + q.qt.lo[oi];
        if (r < rank && q.beta[r] < 0.f) v = -v;  // row r of Q^T = column r of Q
        const int64_t o = (int64_t)r * q.ld_out + c;
        if (q.ut16_lo) {
          split_f16(v * kF16UnitScale, q.ut16_hi[o], q.ut16_lo[o]);
        } else {
          q.ut16_hi[o] = __half_as_ushort(__float2half_rn(v * kF16UnitScale));
        }
      }
      tile[i][tx] = v;
    }
    __syncthreads();
    for (int i = ty; i < 32; i += 8) {
      const int r = c0 + i, c = r0 + tx;  // U[r][c] = Q^T[c][r]
      if (r < q.p && c < q.p) {
        const int64_t o = (int64_t)r * q.ld_out + c;
        if (q.u16_lo) {
          split_f16(tile[tx][i] * kF16UnitScale, q.u16_hi[o], q.u16_lo[o]);
        } else {
          q.u16_hi[o] = __half_as_ushort(__float2half_rn(tile[tx][i] * kF16UnitScale));
        }
      }
    }
    __syncthreads();
  }
  if (blockIdx.x == 0 && threadIdx.x == 0 && q.rank_out) *q.rank_out = rank;
}

// ---------------------------------------------------------------------------
// host helpers
// ---------------------------------------------------------------------------

GemmProblem gp(int M, int N, int K, const float* ah, const float* al, int lda, const float* bh,
               const float* bl, int ldb, float* ch, float* cl, int ldc, int epi,
               float alpha = 0.f, int mma_only = 0) {
  GemmProblem P;
  P.mma_only = mma_only;
  P.M = M;
  P.N = N;
  P.K = K;
  P.a_hi = ah;
  P.a_lo = al;
  P.lda = lda;
  P.b_hi = bh;
  P.b_lo = bl;
  P.ldb = ldb;
  P.c_hi = ch;
  P.c_lo = cl;
  P.ldc = ldc;
  P.epi = epi;
  P.alpha = alpha;
  return P;
}

int panel_slice(int pmax, int cs) { return ((pmax + cs - 1) / cs + 3) / 4 * 4; }

int configure_panel(size_t smem) {
  static size_t configured = 0;
  if (smem > configured) {
    if (cudaFuncSetAttribute(qr_panel_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess ||
        cudaFuncSetAttribute(qr_panel_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed,
                             1) != cudaSuccess)
      return ROT_ECUDA;
    configured = smem;
  }
  return ROT_OK;
}

// Cluster size for the panel kernel: at least enough CTAs that a slice of
// the panel fits in shared memory (<= 1536 elements x 32 rows = 192 KB); then
// the largest size (up to 16, each CTA keeping >= 640 elements) at which
// every cluster of the batch can be resident at once (two CTAs to an SM
// where their slices fit: a column's pass over a CTA's slice is bound by
// shared-memory traffic, so smaller slices shorten every column).
int pick_cluster(int count, int pmax, int sms) {
  const int lo = std::max(1, (pmax + 1535) / 1536);
  int best = std::min(lo, kMaxCluster);
  for (int cs = best; cs <= kMaxCluster; ++cs) {
    if (cs > lo && pmax / cs < 640) break;  // small slices: cluster barriers dominate
    if (cs * count > 2 * sms) break;
    const size_t smem = sizeof(float) * (size_t)B * panel_slice(pmax, cs);
    if (configure_panel(smem) != ROT_OK) break;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(count * cs));
    cfg.blockDim = dim3(kPanelThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, qr_panel_kernel, &cfg) != cudaSuccess) {
      cudaGetLastError();
      break;
    }
    if (clusters >= count) best = cs;
  }
  return best;
}

int launch_panel(const QrBatch& b, int k0, float rtol, int cs, int R, cudaStream_t stream) {
  const size_t smem = sizeof(float) * (size_t)B * R;
  if (configure_panel(smem) != ROT_OK) return ROT_ECUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(b.count * cs));
  cfg.blockDim = dim3(kPanelThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  ProfScope prof(ROT_PROF_QR_PANEL, 0.0, stream);
  return cudaLaunchKernelEx(&cfg, qr_panel_kernel, b, k0, rtol, R) == cudaSuccess ? ROT_OK
                                                                                   : ROT_ECUDA;
}

}  // namespace

uint64_t qr_aux_bytes(int p, int rmax) {
  const uint64_t np = (uint64_t)npanels(rmax), nbk = (uint64_t)nblocks(rmax);
  const uint64_t ld = (uint64_t)pad_ld(p);
  return align256(np * B * B * 4)                   // panel T factors
         + align256((uint64_t)rmax * 4 + 4)         // beta
         + align256((np + 2) * 4) + 256             // ctrl, tau
         + 2 * align256((uint64_t)p * 2 * NB * 4)   // yt split (up to a pair of blocks)
         + 2 * align256((uint64_t)2 * NB * ld * 4)  // w1t split
         + 2 * align256((uint64_t)p * 2 * NB * 4)   // z split
         + align256((uint64_t)NB * NB * 4)          // Gram S
         + align256((uint64_t)NB * NB * 4)          // T assembly scratch
         + 4 * align256(nbk * NB * NB * 4)          // T and T^T splits per block
         + 2 * align256((uint64_t)4 * NB * NB * 4)  // a pair's T split
         + 4 * align256((uint64_t)NB * NB * 4)      // S01 and X^T splits
         + align256(((uint64_t)p / kChunk + 1) * kRowTiles * kRows * B * 4);  // partials
}

void qr_bind_aux(QrProblem& q, char* aux, int p, int rmax) {
  const uint64_t np = (uint64_t)npanels(rmax), nbk = (uint64_t)nblocks(rmax);
  const uint64_t ld = (uint64_t)pad_ld(p);
  uint64_t o = 0;
  auto take = [&](uint64_t bytes) {
    char* ptr = aux + o;
    o += align256(bytes);
    return ptr;
  };
  q.tf = reinterpret_cast<float*>(take(np * B * B * 4));
  q.beta = reinterpret_cast<float*>(take((uint64_t)rmax * 4 + 4));
  q.ctrl = reinterpret_cast<int*>(take((np + 2) * 4));
  q.tau = reinterpret_cast<float*>(take(256));
  q.yt.hi = reinterpret_cast<float*>(take((uint64_t)p * 2 * NB * 4));
  q.yt.lo = reinterpret_cast<float*>(take((uint64_t)p * 2 * NB * 4));
  q.w1t.hi = reinterpret_cast<float*>(take((uint64_t)2 * NB * ld * 4));
  q.w1t.lo = reinterpret_cast<float*>(take((uint64_t)2 * NB * ld * 4));
  q.z.hi = reinterpret_cast<float*>(take((uint64_t)p * 2 * NB * 4));
  q.z.lo = reinterpret_cast<float*>(take((uint64_t)p * 2 * NB * 4));
  q.s = reinterpret_cast<float*>(take((uint64_t)NB * NB * 4));
  q.tmp = reinterpret_cast<float*>(take((uint64_t)NB * NB * 4));
  q.tb.hi = reinterpret_cast<float*>(take(nbk * NB * NB * 4));
  q.tb.lo = reinterpret_cast<float*>(take(nbk * NB * NB * 4));
  q.tbt.hi = reinterpret_cast<float*>(take(nbk * NB * NB * 4));
  q.tbt.lo = reinterpret_cast<float*>(take(nbk * NB * NB * 4));
  q.tpair.hi = reinterpret_cast<float*>(take((uint64_t)4 * NB * NB * 4));
  q.tpair.lo = reinterpret_cast<float*>(take((uint64_t)4 * NB * NB * 4));
  q.s01.hi = reinterpret_cast<float*>(take((uint64_t)NB * NB * 4));
  q.s01.lo = reinterpret_cast<float*>(take((uint64_t)NB * NB * 4));
  q.xt.hi = reinterpret_cast<float*>(take((uint64_t)NB * NB * 4));
  q.xt.lo = reinterpret_cast<float*>(take((uint64_t)NB * NB * 4));
  q.part = reinterpret_cast<float*>(take(((uint64_t)p / kChunk + 1) * kRowTiles * kRows * B * 4));
}

int qr_batched(const hvec<QrProblem>& probs, float rank_rtol, int* status,
               cudaStream_t stream) {
  int sms = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (sms <= 0) sms = 1;
  static bool tattr = false;
  if (!tattr) {
    if (cudaFuncSetAttribute(qr_tblock_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)(3 * TH * (TH + 1) * sizeof(float))) != cudaSuccess)
      return ROT_ECUDA;
    tattr = true;
  }
  for (size_t base = 0; base < probs.size(); base += kMaxQ) {
    QrBatch b;
    std::memset(&b, 0, sizeof(b));
    b.count = (int)std::min<size_t>(kMaxQ, probs.size() - base);
    b.status = status;
    b.limit_ns = g_wait_limit_ns;
    int rmax = 0, pmax = 0;
    for (int i = 0; i < b.count; ++i) {
      b.p[i] = probs[base + i];
      rmax = std::max(rmax, b.p[i].rmax);
      pmax = std::max(pmax, b.p[i].p);
    }
    const unsigned n = (unsigned)b.count;
    const int cs = pick_cluster(b.count, pmax, sms);
    const int R = panel_slice(pmax, cs);
    {
      ProfScope prof(ROT_PROF_QR_OTHER, 0.0, stream);
      qr_init_kernel<<<n, 64, 0, stream>>>(b);
    }
    {
      ProfScope prof(ROT_PROF_QR_OTHER, 0.0, stream);
      qr_colnorm_kernel<<<dim3(std::max(1, std::min(64, pmax / 64)), n), 256, 0, stream>>>(b);
    }
    {
      ProfScope prof(ROT_PROF_QR_OTHER, 0.0, stream);
      qr_scale_kernel<<<dim3(std::max(1, std::min(512, rmax / 4)), n), 256, 0, stream>>>(b);
    }
    if (cudaGetLastError() != cudaSuccess) return ROT_ECUDA;

    // ---- factorisation, block by block
    for (int kb0 = 0; kb0 < rmax; kb0 += NB) {
      for (int k0 = kb0; k0 < std::min(rmax, kb0 + NB); k0 += B) {
        if (launch_panel(b, k0, rank_rtol, cs, R, stream) != ROT_OK) return ROT_ECUDA;
        const int rows = std::min(rmax, kb0 + NB) - k0 - B;
        if (rows > 0) {
          double f = 0.0;
          for (int i = 0; i < b.count; ++i) {
            const QrProblem& q = b.p[i];
            const int re = std::min(q.rmax, kb0 + NB);
            if (k0 < q.rmax && re > k0 + B) f += 4.0 * B * (double)(re - k0 - B) * (q.p - k0);
          }
          const dim3 grid((unsigned)((pmax - k0 + kChunk - 1) / kChunk),
                          (unsigned)((rows + kRows - 1) / kRows), n);
          {
            ProfScope prof(ROT_PROF_QR_APPLY, f * 0.5, stream);
            qr_apply_partial_kernel<<<grid, 256, 0, stream>>>(b, k0);
          }
          {
            ProfScope prof(ROT_PROF_QR_APPLY, f * 0.5, stream);
            qr_apply_update_kernel<<<grid, 256, 0, stream>>>(b, k0);
          }
        }
      }
      // block factor T from the Gram of the block's reflectors
      hvec<GemmProblem> gram;
      for (int i = 0; i < b.count; ++i) {
        const QrProblem& q = b.p[i];
        if (kb0 >= q.rmax) continue;
        const int nb = std::min(NB, q.rmax - kb0);
        const int64_t o = (int64_t)kb0 * q.ld + kb0;
        gram.push_back(gp(nb, nb, q.p - kb0, q.at.hi + o, q.at.lo + o, q.ld, q.at.hi + o,
                          q.at.lo + o, q.ld, q.s, nullptr, NB, kEpiStoreF32));
      }
      if (gemm_grouped(gram, kPrecPrecise, status, stream) != ROT_OK) return ROT_ECUDA;
      {
        ProfScope prof(ROT_PROF_QR_OTHER, 0.0, stream);
        qr_tblock_kernel<<<n, kTThreads, 3 * TH * (TH + 1) * sizeof(float), stream>>>(b, kb0);
      }
      // trailing columns kb0+NB .. rmax-1: a <- a - Y (T^T (Y^T a))
      hvec<TransposeSeg> tr;
      hvec<GemmProblem> f1, f2, f3;
      for (int i = 0; i < b.count; ++i) {
        const QrProblem& q = b.p[i];
        const int kend = kb0 + NB;
        if (kend >= q.rmax) continue;
        const int nb = NB, L = q.p - kb0, nr = q.rmax - kend;
        const int blk = kb0 / NB;
        const int64_t oy = (int64_t)kb0 * q.ld + kb0, ox = (int64_t)kend * q.ld + kb0;
        tr.push_back({q.at.hi + oy, q.at.lo + oy, q.ld, q.yt.hi, q.yt.lo, NB, nb, L, 1, 1, 1});
        f1.push_back(gp(nb, L, nb, q.tbt.hi + (int64_t)blk * NB * NB,
                        q.tbt.lo + (int64_t)blk * NB * NB, NB, q.yt.hi, q.yt.lo, NB, q.w1t.hi,
                        q.w1t.lo, q.ld, kEpiStoreSplit, 0.f, 1));
        f2.push_back(gp(nr, nb, L, q.at.hi + ox, q.at.lo + ox, q.ld, q.w1t.hi, q.w1t.lo, q.ld,
                        q.z.hi, q.z.lo, NB, kEpiStoreSplit, 0.f, 1));
        f3.push_back(gp(nr, L, nb, q.z.hi, q.z.lo, NB, q.yt.hi, q.yt.lo, NB, q.at.hi + ox,
                        q.at.lo + ox, q.ld, kEpiApplySplit, 1.f));
      }
      if (!tr.empty()) {
        if (launch_transpose(tr, stream) != ROT_OK) return ROT_ECUDA;
        if (gemm_grouped(f1, kPrecPrecise, status, stream) != ROT_OK) return ROT_ECUDA;
        if (gemm_grouped(f2, kPrecPrecise, status, stream) != ROT_OK) return ROT_ECUDA;
        if (gemm_grouped(f3, kPrecPrecise, status, stream) != ROT_OK) return ROT_ECUDA;
      }
    }

    // ---- Q = H_0 ... H_{r-1} I, accumulated backwards block by block
    {
      const int64_t most = (int64_t)pmax * pmax;
      ProfScope prof(ROT_PROF_QR_OTHER, 0.0, stream);
      qr_eye_kernel<<<dim3((unsigned)std::min<int64_t>(4096, (most + 1023) / 1024), n), 256, 0,
                      stream>>>(b);
    }
    // Pairs of blocks (b, b+1) are applied together as one rank-(up to 512)
    // update, with the pair's factor joined from the two blocks' factors: half
    // the passes over Q, and twice the K of each update.  A last block without
    // a partner is applied alone.
    const int npairs = (nblocks(rmax) + 1) / 2;
    for (int pp = npairs - 1; pp >= 0; --pp) {
      const int kb0 = pp * 2 * NB;
      hvec<GemmProblem> gs, gx, gt;
      for (int i = 0; i < b.count; ++i) {
        const QrProblem& q = b.p[i];
        const int e1 = kb0 + NB;  // the second block's first reflector
        if (e1 >= q.rmax) continue;
        const int nb1 = std::min(NB, q.rmax - e1);
        const int64_t blk = kb0 / NB;
        // S01 = Y_b^T Y_{b+1} (NB x nb1), over elements >= e1 (Y_{b+1} is 0 before)
        gs.push_back(gp(NB, nb1, q.p - e1, q.at.hi + (int64_t)kb0 * q.ld + e1,
                        q.at.lo + (int64_t)kb0 * q.ld + e1, q.ld,
                        q.at.hi + (int64_t)e1 * q.ld + e1, q.at.lo + (int64_t)e1 * q.ld + e1,
                        q.ld, q.s01.hi, q.s01.lo, NB, kEpiStoreSplit, 0.f, 1));
        // X^T = T_{b+1}^T S01^T (nb1 x NB)
        gx.push_back(gp(nb1, NB, nb1, q.tbt.hi + (blk + 1) * NB * NB,
                        q.tbt.lo + (blk + 1) * NB * NB, NB, q.s01.hi, q.s01.lo, NB, q.xt.hi,
                        q.xt.lo, NB, kEpiStoreSplit, 0.f, 1));
        // upper-right block of the pair's factor: 0 - T_b X
        gt.push_back(gp(NB, nb1, NB, q.tb.hi + blk * NB * NB, q.tb.lo + blk * NB * NB, NB,
                        q.xt.hi, q.xt.lo, NB, q.tpair.hi + NB, q.tpair.lo + NB, 2 * NB,
                        kEpiApplySplit, 1.f, 1));
      }
      if (!gs.empty()) {
        if (gemm_grouped(gs, kPrecPrecise, status, stream) != ROT_OK) return ROT_ECUDA;
        if (gemm_grouped(gx, kPrecPrecise, status, stream) != ROT_OK) return ROT_ECUDA;
        {
          ProfScope prof(ROT_PROF_QR_OTHER, 0.0, stream);
          qr_pair_assemble_kernel<<<dim3(64, n), 256, 0, stream>>>(b, kb0);
        }
        if (gemm_grouped(gt, kPrecPrecise, status, stream) != ROT_OK) return ROT_ECUDA;
      }
      hvec<TransposeSeg> tr;
      hvec<GemmProblem> q1, q2, q3;
      for (int i = 0; i < b.count; ++i) {
        const QrProblem& q = b.p[i];
        if (kb0 >= q.rmax) continue;
        const int nb = std::min(2 * NB, q.rmax - kb0), L = q.p - kb0;
        const bool pair = nb > NB;
        const int64_t oy = (int64_t)kb0 * q.ld + kb0;
        const float* th = pair ? q.tpair.hi : q.tb.hi + (int64_t)(kb0 / NB) * NB * NB;
        const float* tl = pair ? q.tpair.lo : q.tb.lo + (int64_t)(kb0 / NB) * NB * NB;
        tr.push_back({q.at.hi + oy, q.at.lo + oy, q.ld, q.yt.hi, q.yt.lo, 2 * NB, nb, L, 1, 1, 1});
        q1.push_back(gp(nb, L, nb, th, tl, pair ? 2 * NB : NB, q.yt.hi, q.yt.lo, 2 * NB,
                        q.w1t.hi, q.w1t.lo, q.ld, kEpiStoreSplit, 0.f, 1));
        q2.push_back(gp(L, nb, L, q.qt.hi + oy, q.qt.lo + oy, q.ld, q.w1t.hi, q.w1t.lo, q.ld,
                        q.z.hi, q.z.lo, 2 * NB, kEpiStoreSplit, 0.f, 1));
        q3.push_back(gp(L, L, nb, q.z.hi, q.z.lo, 2 * NB, q.yt.hi, q.yt.lo, 2 * NB,
                        q.qt.hi + oy, q.qt.lo + oy, q.ld, kEpiApplySplit, 1.f));
      }
      if (tr.empty()) continue;
      if (launch_transpose(tr, stream) != ROT_OK) return ROT_ECUDA;
      // precise: Q's orthogonality error adds up over all p^2 entries (the
      // rank-256/512 updates too: accumulated in TMEM, in 3xTF32 or 3xF16, they
      // moved the bases' orthogonality and the W parity measurably)
      if (gemm_grouped(q1, kPrecPrecise, status, stream) != ROT_OK) return ROT_ECUDA;
      if (gemm_grouped(q2, kPrecPrecise, status, stream) != ROT_OK) return ROT_ECUDA;
      if (gemm_grouped(q3, kPrecPrecise, status, stream) != ROT_OK) return ROT_ECUDA;
    }
    const int tiles = (pmax + 31) / 32;
    {
      ProfScope prof(ROT_PROF_QR_OTHER, 0.0, stream);
      qr_finalize_kernel<<<dim3((unsigned)std::min(tiles * tiles, 4096), n), 256, 0, stream>>>(b);
    }
    if (cudaGetLastError() != cudaSuccess) return ROT_ECUDA;
  }
  return ROT_OK;
}

}  // namespace rot
