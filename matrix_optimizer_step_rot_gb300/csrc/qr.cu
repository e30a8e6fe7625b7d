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
// Storage: the input arrives transposed (row j of `at` = column j of A), so a
// column and a reflector are contiguous.  Reflector k overwrites row k from
// element k on (w_0 at the diagonal, the tail of x after it).
//
// Blocking (Golub & Van Loan, "Matrix Computations", section 5.1.7, compact
// WY): a panel of b = 32 columns is factored by one CTA per matrix; its
// reflectors form H_{k0}..H_{k0+b-1} = I - Y T Y^T with T upper triangular
// (T_jj = 2 / w_j^T w_j, T[0:j, j] = -T_jj T[0:j, 0:j] Y[:, 0:j]^T w_j).  The
// trailing columns then receive a <- (I - Y T^T Y^T) a, and Q is accumulated
// backwards panel by panel with q <- (I - Y T Y^T) q.
#include <algorithm>
#include <cstring>

#include "profile.h"
#include "rot_internal.h"
#include "split.cuh"

namespace rot {
namespace {

constexpr int B = kQrPanel;
constexpr int kMaxQ = 64;
constexpr unsigned kFull = 0xffffffffu;

struct QrBatch {
  int count;
  QrProblem p[kMaxQ];
};

// scratch layout inside QrProblem pointers (set on the host): see qr_aux_bytes
__host__ __device__ inline int npanels(int rmax) { return (rmax + B - 1) / B; }

// ---------------------------------------------------------------------------
// reductions
// ---------------------------------------------------------------------------

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

// Sum of v over the block, returned to every thread.  `red` has >= 32 floats.
__device__ float block_sum(float v, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = lane < nw ? red[lane] : 0.f;
  return warp_sum(t);
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

// ---------------------------------------------------------------------------
// set-up: scratch reset and the threshold's column norms
// ---------------------------------------------------------------------------

__global__ void qr_init_kernel(const __grid_constant__ QrBatch b) {
  const QrProblem& q = b.p[blockIdx.x];
  const int np = npanels(q.rmax);
  for (int i = threadIdx.x; i < np + 2; i += blockDim.x) q.ctrl[i] = (i == 0) ? -1 : 0;
  if (threadIdx.x == 0) q.tau[0] = 0.f;
}

// max_j ||a_j|| (rows of `at`), by atomicMax on the float's bits (values >= 0).
__global__ void qr_colnorm_kernel(const __grid_constant__ QrBatch b) {
  const QrProblem& q = b.p[blockIdx.y];
  const int lane = threadIdx.x & 31;
  const int warps = blockDim.x >> 5;
  float best = 0.f;
  for (int j = blockIdx.x * warps + (threadIdx.x >> 5); j < q.p; j += gridDim.x * warps) {
    const float* row = q.at + (int64_t)j * q.ld;
    float s = 0.f;
    for (int e = lane; e < q.p; e += 32) s = fmaf(row[e], row[e], s);
    s = warp_sum(s);
    best = fmaxf(best, sqrtf(s));
  }
  if (lane == 0 && best > 0.f) atomicMax(reinterpret_cast<int*>(q.tau), __float_as_int(best));
}

// ---------------------------------------------------------------------------
// panel factorisation: one CTA per matrix, columns k0 .. k0+bw-1
// ---------------------------------------------------------------------------

constexpr int kPanelThreads = 512;

__global__ void __launch_bounds__(kPanelThreads)
    qr_panel_kernel(const __grid_constant__ QrBatch b, int k0, float rtol) {
  const QrProblem& q = b.p[blockIdx.x];
  if (k0 >= q.rmax) return;
  const int panel = k0 / B;
  if (q.ctrl[1]) {  // stopped in an earlier panel
    if (threadIdx.x == 0) q.ctrl[2 + panel] = 0;
    return;
  }
  __shared__ float red[B][33];
  __shared__ float s_red[32];
  __shared__ float s_dot[B];
  __shared__ float s_ww[B];
  __shared__ float s_beta[B];
  __shared__ float gram[B][B + 1];  // gram[i][j] = w_i . w_j, i < j
  __shared__ float tmat[B][B + 1];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nthr = blockDim.x, nwarp = nthr >> 5;
  const int p = q.p, ld = q.ld;
  float* at = q.at;
  const float thr = rtol * q.tau[0];
  const int bw = min(B, q.rmax - k0);
  int active = bw;

  for (int j = 0; j < bw; ++j) {
    const int k = k0 + j;
    float* xr = at + (int64_t)k * ld;
    float s = 0.f;
    for (int e = k + tid; e < p; e += nthr) s = fmaf(xr[e], xr[e], s);
    s = block_sum(s, s_red);
    const float nx = sqrtf(s);
    if (nx <= thr) {  // numerical rank reached: H_k .. are identities
      active = j;
      break;
    }
    const float x0 = xr[k];
    const float beta = x0 >= 0.f ? -nx : nx;
    const float w0 = x0 - beta;
    const float ww = 2.f * fmaf(fabsf(x0), nx, s);  // ||x - beta e0||^2, no cancellation
    __syncthreads();  // every thread has read xr[k]
    if (tid == 0) {
      xr[k] = w0;
      s_ww[j] = ww;
      s_beta[j] = beta;
    }
    __syncthreads();

    // dots of w with the other panel rows over elements k..p-1: for c < j the
    // row holds reflector c (its support starts at k0+c < k), for c > j the
    // not yet reduced column c.
    float acc[B];
#pragma unroll
    for (int c = 0; c < B; ++c) acc[c] = 0.f;
    for (int e = k + tid; e < p; e += nthr) {
      const float we = xr[e];
#pragma unroll
      for (int c = 0; c < B; ++c)
        if (c < bw && c != j) acc[c] = fmaf(we, at[(int64_t)(k0 + c) * ld + e], acc[c]);
    }
    const float part = warp_transpose_sum(acc);  // lane c: this warp's sum for c
    red[lane][warp] = part;
    __syncthreads();
    if (tid < B) {
      float t = 0.f;
      for (int w = 0; w < nwarp; ++w) t += red[tid][w];
      s_dot[tid] = t;
      if (tid < j) gram[tid][j] = t;
    }
    __syncthreads();

    // apply H_k to the remaining panel columns
    for (int e = k + tid; e < p; e += nthr) {
      const float we = xr[e];
      for (int c = j + 1; c < bw; ++c) {
        const float coef = 2.f * s_dot[c] / ww;
        at[(int64_t)(k0 + c) * ld + e] -= coef * we;
      }
    }
    __syncthreads();
  }

  // T: T_jj = 2 / ww_j ; T[0:j, j] = -T_jj * T[0:j, 0:j] * gram[0:j, j]
  if (warp == 0) {
    for (int i = lane; i < B * (B + 1); i += 32) (&tmat[0][0])[i] = 0.f;
    __syncwarp();
    for (int j = 0; j < active; ++j) {
      const float tjj = 2.f / s_ww[j];
      float t = 0.f;
      if (lane < j) {
        for (int l = lane; l < j; ++l) t = fmaf(tmat[lane][l], gram[l][j], t);
      }
      __syncwarp();
      if (lane < j) tmat[lane][j] = -tjj * t;
      if (lane == j) tmat[j][j] = tjj;
      __syncwarp();
    }
  }
  __syncthreads();
  float* tf = q.tf + (int64_t)panel * B * B;
  for (int i = tid; i < B * B; i += nthr) tf[i] = tmat[i / B][i % B];
  if (tid < active) q.beta[k0 + tid] = s_beta[tid];
  if (tid == 0) {
    q.ctrl[2 + panel] = active;
    if (active < bw) {
      q.ctrl[1] = 1;
      q.ctrl[0] = k0 + active;
    }
  }
}

// ---------------------------------------------------------------------------
// apply one panel's block reflector to 32 rows of a row-stored matrix:
//   mode 0 (factorisation, rows k0+b .. rmax-1 of `at`): a <- a - Y (T^T (Y^T a))
//   mode 1 (Q formation, rows k0 .. p-1 of `qt`):        q <- q - Y (T (Y^T q))
// Only elements k0..p-1 of each row are touched.
// ---------------------------------------------------------------------------

constexpr int kRows = 32;

__global__ void __launch_bounds__(256)
    qr_apply_kernel(const __grid_constant__ QrBatch b, int k0, int mode) {
  const QrProblem& q = b.p[blockIdx.y];
  if (k0 >= q.rmax) return;
  const int panel = k0 / B;
  const int active = q.ctrl[2 + panel];
  if (active == 0) return;
  const int p = q.p, ld = q.ld;
  const int row_begin = mode == 0 ? k0 + B : k0;
  const int row_end = mode == 0 ? q.rmax : p;
  const int r0 = row_begin + blockIdx.x * kRows;
  if (r0 >= row_end) return;
  float* X = mode == 0 ? q.at : q.qt;
  const float* Y = q.at;  // reflector i: row k0+i, elements >= k0+i

  __shared__ float xs[kRows][33];
  __shared__ float ys[B][33];
  __shared__ float z[kRows][B + 1];
  __shared__ float zt[kRows][B + 1];
  __shared__ float tm[B][B + 1];
  const int tid = threadIdx.x;
  const float* tf = q.tf + (int64_t)panel * B * B;
  for (int i = tid; i < B * B; i += 256) tm[i / B][i % B] = tf[i];

  // phase 1: z[r][i] = sum_e X[r][e] Y_i[e]
  const int r = tid >> 3, i4 = (tid & 7) * 4;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int e0 = k0; e0 < p; e0 += 32) {
    __syncthreads();
    for (int t = tid; t < kRows * 32; t += 256) {
      const int rr = t >> 5, ee = t & 31, e = e0 + ee;
      const int row = r0 + rr;
      xs[rr][ee] = (row < row_end && e < p) ? X[(int64_t)row * ld + e] : 0.f;
      const int yi = rr;  // reflector index (B == kRows == 32)
      ys[yi][ee] = (yi < active && e < p && e >= k0 + yi) ? Y[(int64_t)(k0 + yi) * ld + e] : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int ee = 0; ee < 32; ++ee) {
      const float xv = xs[r][ee];
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[c] = fmaf(xv, ys[i4 + c][ee], acc[c]);
    }
  }
#pragma unroll
  for (int c = 0; c < 4; ++c) z[r][i4 + c] = acc[c];
  __syncthreads();

  // phase 2: zt = z T (mode 0: rows of T^T z) or z T^T (mode 1: rows of T z)
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int i = i4 + c;
    float t = 0.f;
    for (int jj = 0; jj < B; ++jj) t = fmaf(z[r][jj], mode == 0 ? tm[jj][i] : tm[i][jj], t);
    zt[r][i] = t;
  }
  __syncthreads();

  // phase 3: X[r][e] -= sum_i zt[r][i] Y_i[e]
  const int e4 = (tid & 7) * 4;
  for (int e0 = k0; e0 < p; e0 += 32) {
    __syncthreads();
    for (int t = tid; t < B * 32; t += 256) {
      const int yi = t >> 5, ee = t & 31, e = e0 + ee;
      ys[yi][ee] = (yi < active && e < p && e >= k0 + yi) ? Y[(int64_t)(k0 + yi) * ld + e] : 0.f;
    }
    __syncthreads();
    const int row = r0 + r;
    if (row < row_end) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int e = e0 + e4 + c;
        if (e < p) {
          float t = 0.f;
#pragma unroll 8
          for (int i = 0; i < B; ++i) t = fmaf(zt[r][i], ys[i][e4 + c], t);
          X[(int64_t)row * ld + e] -= t;
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Q^T = I, then the sign fix and the split outputs U^T (= Q^T) and U (= Q)
// ---------------------------------------------------------------------------

__global__ void qr_eye_kernel(const __grid_constant__ QrBatch b) {
  const QrProblem& q = b.p[blockIdx.y];
  const int64_t total = (int64_t)q.p * q.p;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int r = (int)(e / q.p), c = (int)(e % q.p);
    q.qt[(int64_t)r * q.ld + c] = r == c ? 1.f : 0.f;
  }
}

__global__ void qr_finalize_kernel(const __grid_constant__ QrBatch b) {
  __shared__ float tile[32][33];
  const QrProblem& q = b.p[blockIdx.y];
  const int rank = q.ctrl[1] ? q.ctrl[0] : q.rmax;
  const int tiles = (q.p + 31) / 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  for (int t = blockIdx.x; t < tiles * tiles; t += gridDim.x) {
    const int r0 = (t / tiles) * 32, c0 = (t % tiles) * 32;
    for (int i = ty; i < 32; i += 8) {
      const int r = r0 + i, c = c0 + tx;
      float v = 0.f;
      if (r < q.p && c < q.p) {
        v = q.qt[(int64_t)r * q.ld + c];
        if (r < rank && q.beta[r] < 0.f) v = -v;  // row r of Q^T = column r of Q
        float h, l;
        split_tf32(v, h, l);
        const int64_t o = (int64_t)r * q.ld_out + c;
        q.ut.hi[o] = h;
        q.ut.lo[o] = l;
      }
      tile[i][tx] = v;
    }
    __syncthreads();
    for (int i = ty; i < 32; i += 8) {
      const int r = c0 + i, c = r0 + tx;  // U[r][c] = Q^T[c][r]
      if (r < q.p && c < q.p) {
        float h, l;
        split_tf32(tile[tx][i], h, l);
        const int64_t o = (int64_t)r * q.ld_out + c;
        q.u.hi[o] = h;
        q.u.lo[o] = l;
      }
    }
    __syncthreads();
  }
  if (blockIdx.x == 0 && threadIdx.x == 0 && q.rank_out) *q.rank_out = rank;
}

}  // namespace

uint64_t qr_aux_bytes(int p, int rmax) {
  (void)p;
  const uint64_t np = (uint64_t)npanels(rmax);
  return align256(np * B * B * 4) + align256((uint64_t)rmax * 4 + 4) + align256((np + 2) * 4) +
         256;
}

int qr_batched(const std::vector<QrProblem>& probs, float rank_rtol, int* status,
               cudaStream_t stream) {
  (void)status;
  for (size_t base = 0; base < probs.size(); base += kMaxQ) {
    QrBatch b;
    std::memset(&b, 0, sizeof(b));
    b.count = (int)std::min<size_t>(kMaxQ, probs.size() - base);
    int rmax = 0, pmax = 0;
    for (int i = 0; i < b.count; ++i) {
      b.p[i] = probs[base + i];
      rmax = std::max(rmax, b.p[i].rmax);
      pmax = std::max(pmax, b.p[i].p);
    }
    const unsigned n = (unsigned)b.count;
    // algorithmic flops of one block-reflector application to `rows` rows of
    // length len: z = Y^T x and x -= Y z', 2 * 2 * b flops per element
    auto apply_flops = [&](int k0, int mode) {
      double f = 0.0;
      for (int i = 0; i < b.count; ++i) {
        const QrProblem& q = b.p[i];
        if (k0 >= q.rmax) continue;
        const int rows = mode == 0 ? std::max(0, q.rmax - k0 - B) : q.p - k0;
        f += 4.0 * B * (double)rows * (q.p - k0);
      }
      return f;
    };
    {
      ProfScope prof(ROT_PROF_QR_OTHER, 0.0, stream);
      qr_init_kernel<<<n, 64, 0, stream>>>(b);
    }
    {
      ProfScope prof(ROT_PROF_QR_OTHER, 0.0, stream);
      qr_colnorm_kernel<<<dim3(std::max(1, std::min(64, pmax / 64)), n), 256, 0, stream>>>(b);
    }
    for (int k0 = 0; k0 < rmax; k0 += B) {
      {
        ProfScope prof(ROT_PROF_QR_PANEL, 0.0, stream);
        qr_panel_kernel<<<n, kPanelThreads, 0, stream>>>(b, k0, rank_rtol);
      }
      const int rows = std::max(0, rmax - k0 - B);
      if (rows > 0) {
        ProfScope prof(ROT_PROF_QR_APPLY, apply_flops(k0, 0), stream);
        qr_apply_kernel<<<dim3((rows + kRows - 1) / kRows, n), 256, 0, stream>>>(b, k0, 0);
      }
    }
    {
      const int64_t most = (int64_t)pmax * pmax;
      ProfScope prof(ROT_PROF_QR_OTHER, 0.0, stream);
      qr_eye_kernel<<<dim3((unsigned)std::min<int64_t>(4096, (most + 1023) / 1024), n), 256, 0,
                      stream>>>(b);
    }
    for (int k0 = ((rmax - 1) / B) * B; k0 >= 0; k0 -= B) {
      const int rows = pmax - k0;
      ProfScope prof(ROT_PROF_QR_APPLY, apply_flops(k0, 1), stream);
      qr_apply_kernel<<<dim3((rows + kRows - 1) / kRows, n), 256, 0, stream>>>(b, k0, 1);
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
