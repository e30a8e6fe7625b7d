// Grouped GEMM on CUDA cores (float32 FFMA), C = A * B^T with K-major A and B.
// Operands arrive as TF32 splits; this kernel recombines hi + lo (the exact
// float32 value) for ROT_PREC_3XTF32 and uses hi alone for ROT_PREC_TF32.
#include <algorithm>
#include <cstring>

#include "rot_internal.h"
#include "split.cuh"

namespace rot {
namespace {

constexpr int kBM = 64, kBN = 64, kBK = 16;
constexpr int kMaxProb = 48;

struct SimtBatch {
  int count;
  int use_lo;
  int tile_start[kMaxProb + 1];
  int tiles_n[kMaxProb];
  GemmProblem p[kMaxProb];
};

__device__ __forceinline__ void store_out(const GemmProblem& P, int i, int j, float acc) {
  if (i >= P.M || j >= P.N) return;
  switch (P.epi) {
    case kEpiStoreSplit: {
      float h, l;
      split_tf32(acc, h, l);
      const int64_t o = (int64_t)i * P.ldc + j;
      P.c_hi[o] = h;
      P.c_lo[o] = l;
      break;
    }
    case kEpiStoreSplitT: {
      float h, l;
      split_tf32(acc, h, l);
      const int64_t o = (int64_t)j * P.ldc + i;
      P.c_hi[o] = h;
      P.c_lo[o] = l;
      break;
    }
    case kEpiStoreF32:
      P.c_hi[(int64_t)i * P.ldc + j] = acc;
      break;
    case kEpiStoreF32T:
      P.c_hi[(int64_t)j * P.ldc + i] = acc;
      break;
    case kEpiApply: {
      const int64_t o = (int64_t)i * P.ldc + j;
      P.c_hi[o] = P.c_hi[o] - P.alpha * acc;
      break;
    }
  }
}

__global__ void __launch_bounds__(256) gemm_simt_kernel(const __grid_constant__ SimtBatch b) {
  __shared__ float As[kBK][kBM + 4];
  __shared__ float Bs[kBK][kBN + 4];
  const int tile = blockIdx.x;
  int pi = 0;
  while (pi + 1 < b.count && tile >= b.tile_start[pi + 1]) ++pi;
  const GemmProblem& P = b.p[pi];
  const int local = tile - b.tile_start[pi];
  const int m0 = (local / b.tiles_n[pi]) * kBM, n0 = (local % b.tiles_n[pi]) * kBN;
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < P.K; k0 += kBK) {
    for (int e = tid; e < kBM * kBK; e += 256) {
      const int r = e / kBK, k = e % kBK;
      float a = 0.f, bb = 0.f;
      if (m0 + r < P.M && k0 + k < P.K) {
        const int64_t o = (int64_t)(m0 + r) * P.lda + k0 + k;
        a = P.a_hi[o] + (b.use_lo ? P.a_lo[o] : 0.f);
      }
      if (n0 + r < P.N && k0 + k < P.K) {
        const int64_t o = (int64_t)(n0 + r) * P.ldb + k0 + k;
        bb = P.b_hi[o] + (b.use_lo ? P.b_lo[o] : 0.f);
      }
      As[k][r] = a;
      Bs[k][r] = bb;
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kBK; ++k) {
      float av[4], bv[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        av[q] = As[k][ty * 4 + q];
        bv[q] = Bs[k][tx * 4 + q];
      }
#pragma unroll
      for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) acc[x][y] = fmaf(av[x], bv[y], acc[x][y]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int x = 0; x < 4; ++x)
#pragma unroll
    for (int y = 0; y < 4; ++y) store_out(P, m0 + ty * 4 + x, n0 + tx * 4 + y, acc[x][y]);
}

}  // namespace

int gemm_simt(const std::vector<GemmProblem>& probs, int precision, cudaStream_t stream) {
  for (size_t base = 0; base < probs.size(); base += kMaxProb) {
    SimtBatch b;
    std::memset(&b, 0, sizeof(b));
    b.use_lo = precision == ROT_PREC_3XTF32 ? 1 : 0;
    int total = 0;
    const int count = (int)std::min<size_t>(kMaxProb, probs.size() - base);
    for (int i = 0; i < count; ++i) {
      const GemmProblem& P = probs[base + i];
      if (P.M <= 0 || P.N <= 0) continue;
      b.p[b.count] = P;
      b.tile_start[b.count] = total;
      b.tiles_n[b.count] = (P.N + kBN - 1) / kBN;
      total += ((P.M + kBM - 1) / kBM) * b.tiles_n[b.count];
      ++b.count;
    }
    b.tile_start[b.count] = total;
    if (total == 0) continue;
    gemm_simt_kernel<<<total, 256, 0, stream>>>(b);
    if (cudaGetLastError() != cudaSuccess) return ROT_ECUDA;
  }
  return ROT_OK;
}

}  // namespace rot
