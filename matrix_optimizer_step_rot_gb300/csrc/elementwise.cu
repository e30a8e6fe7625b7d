// Element-wise kernels of the step: momentum (+ the split of G the rotation
// reads), the Adam update in rotated coordinates, transposes, fills, fp16
// copies and exports.
//
// All of them are HBM-bound.  Each launch covers many matrices: blockIdx.y
// selects the matrix, blockIdx.x strides over its elements (or, for the 3xF16
// row kernels, over its rows: one block per row, since a row's power-of-two
// scale needs the row's max first); the per-matrix descriptors travel in the
// kernel's parameter block.
#include <algorithm>
#include <cstring>

#include "profile.h"
#include "rot_internal.h"
#include <cuda_bf16.h>

#include "split.cuh"

namespace rot {
namespace {

constexpr int kMaxSegs = 64;
constexpr int kThreads = 256;

template <class Seg>
struct SegBatch {
  int count;
  Seg seg[kMaxSegs];
};

inline unsigned grid_x_for(int64_t elems) {
  int64_t blocks = (elems + kThreads * 4 - 1) / (kThreads * 4);
  return (unsigned)std::max<int64_t>(1, std::min<int64_t>(blocks, 4096));
}

// bytes_per_elem: algorithmic bytes each element moves (for instrumentation)
template <class Seg, class Kernel, class... Args>
int launch_segs(const hvec<Seg>& segs, double bytes_per_elem, Kernel kernel,
                cudaStream_t stream, Args... args) {
  for (size_t base = 0; base < segs.size(); base += kMaxSegs) {
    SegBatch<Seg> b;
    std::memset(&b, 0, sizeof(b));
    b.count = (int)std::min<size_t>(kMaxSegs, segs.size() - base);
    int64_t most = 0;
    double elems = 0.0;
    for (int i = 0; i < b.count; ++i) {
      b.seg[i] = segs[base + i];
      most = std::max<int64_t>(most, (int64_t)b.seg[i].rows * b.seg[i].cols);
      elems += (double)b.seg[i].rows * b.seg[i].cols;
    }
    if (most == 0) continue;
    dim3 grid(grid_x_for(most), b.count);
    ProfScope prof(ROT_PROF_ELEMENTWISE, elems * bytes_per_elem, stream);
    kernel<<<grid, kThreads, 0, stream>>>(b, args...);
    if (cudaGetLastError() != cudaSuccess) return ROT_ECUDA;
  }
  return ROT_OK;
}

// State values held as float32, or as bf16 in the compact state format.
__device__ __forceinline__ float ld_state(const float* p, int64_t o, bool bf16) {
  return bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[o]) : p[o];
}
__device__ __forceinline__ void st_state(float* p, int64_t o, float x, bool bf16) {
  if (bf16) {
    reinterpret_cast<__nv_bfloat16*>(p)[o] = __float2bfloat16_rn(x);
  } else {
    p[o] = x;
  }
}
// x as the state keeps it (rounded to bf16 in the compact format)
__device__ __forceinline__ float as_state(float x, bool bf16) {
  return bf16 ? __bfloat162float(__float2bfloat16_rn(x)) : x;
}

// Optional non-finite check (rot_set_nonfinite_check): `flag` is the status
// word or null.  A thread that saw a non-finite value sets it to
// ROT_ENONFINITE once (unless another status is already there); the values
// themselves propagate untouched.
__device__ __forceinline__ void report_nonfinite(int* flag, bool seen) {
  if (flag && seen) atomicCAS(flag, 0, ROT_ENONFINITE);
}

// M <- beta1 M + (1 - beta1) G (float32); also writes G's split and, on
// refresh steps, M's exact TF32 split.
__global__ void momentum_kernel(const __grid_constant__ SegBatch<MomentumSeg> b, float beta1,
                                int* flag) {
  const MomentumSeg& s = b.seg[blockIdx.y];
  const int64_t total = (int64_t)s.rows * s.cols;
  const float one_minus = 1.0f - beta1;
  const bool check = flag != nullptr;
  bool bad = false;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int r = (int)(e / s.cols), c = (int)(e - (int64_t)r * s.cols);
    const int64_t o = (int64_t)r * s.ldm + c;
    const float g = s.g[e];
    bad |= check && !isfinite(g);
    const float m = as_state(beta1 * ld_state(s.m, o, s.m_bf16) + one_minus * g, s.m_bf16);
    st_state(s.m, o, m, s.m_bf16);
    float h, l;
    if (s.m_hi) {
      split_tf32(m, h, l);
      s.m_hi[o] = h;
      s.m_lo[o] = l;
    }
    split_tf32_mma(g, h, l);
    s.g_hi[o] = h;
    s.g_lo[o] = l;
  }
  report_nonfinite(flag, bad);
}

// [M~ <- beta1 M~ + (1 - beta1) G~;]  v <- beta2 v + (1 - beta2) G~^2 ;
// D = M~ / (sqrt(v) + eps)  (D as a split)
__global__ void adam_kernel(const __grid_constant__ SegBatch<AdamSeg> b, float beta1, float beta2,
                            float eps, int incremental, int* flag) {
  const AdamSeg& s = b.seg[blockIdx.y];
  const bool check = flag != nullptr;
  bool bad = false;
  const int64_t total = (int64_t)s.rows * s.cols;
  const float one_minus1 = 1.0f - beta1;
  const float one_minus = 1.0f - beta2;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int r = (int)(e / s.cols), c = (int)(e - (int64_t)r * s.cols);
    const int64_t o = (int64_t)r * s.ld + c;
    const float g = s.gt[o];
    float m = ld_state(s.mt, o, s.mt_bf16);
    if (incremental) {
      m = as_state(beta1 * m + one_minus1 * g, s.mt_bf16);
      st_state(s.mt, o, m, s.mt_bf16);
    }
    const float v = beta2 * s.v[o] + one_minus * (g * g);
    s.v[o] = v;
    const float d = m / (sqrtf(v) + eps);
    bad |= check && !isfinite(d);
    float h, l;
    split_tf32_mma(d, h, l);
    s.d_hi[o] = h;
    s.d_lo[o] = l;
  }
  report_nonfinite(flag, bad);
}

// Sum and max over the block (256 threads); every thread gets both.
__device__ __forceinline__ void block_sum_max(float& sum, float& mx) {
  __shared__ float ssum[kThreads / 32], smax[kThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    sum += __shfl_xor_sync(0xffffffffu, sum, o);
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  __syncthreads();  // the previous row's readers are done with ssum / smax
  if (lane == 0) {
    ssum[warp] = sum;
    smax[warp] = mx;
  }
  __syncthreads();
  sum = 0.f;
  mx = 0.f;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) {
    sum += ssum[w];
    mx = fmaxf(mx, smax[w]);
  }
}

// Upper bound on a row's 2-norm from its sum of squares and max |x|: the sum
// may overflow float32 for finite rows, then sqrt(cols) max|x| bounds it.
__device__ __forceinline__ float row_norm_bound(float sum, float mx, int cols) {
  const float rn = sqrtf(sum);
  return (rn <= 3.402823466e38f || !(mx <= 3.402823466e38f)) ? rn : mx * sqrtf((float)cols);
}

// Non-negative float maximum through its bit pattern (monotone for x >= 0;
// a NaN wins, so that non-finite values reach the scale logic).
__device__ __forceinline__ void atomic_max_nonneg(float* slot, float x) {
  atomicMax(reinterpret_cast<int*>(slot), __float_as_int(x));
}

// 3xF16 momentum: one block per row (blockIdx.x strides over rows).  First
// pass: M's update and the row's max |g| and sum g^2; second pass (G re-read,
// from L2): the scaled fp16 split of G.  Four columns per thread and access
// (16-byte loads) where the row allows, single columns for the rest.
__device__ __forceinline__ void momentum_elem(float x, float& m, float beta1, float one_minus,
                                              float& sum, float& mx) {
  m = beta1 * m + one_minus * x;
  sum = fmaf(x, x, sum);
  mx = fmaxf(mx, fabsf(x));
}

__global__ void momentum16_kernel(const __grid_constant__ SegBatch<Momentum16Seg> b,
                                  float beta1, int* flag) {
  const Momentum16Seg& s = b.seg[blockIdx.y];
  const float one_minus = 1.0f - beta1;
  const bool bf = s.m_bf16 != 0;
  const int nv = (!bf && (s.cols & 3) == 0 && (reinterpret_cast<uintptr_t>(s.g) & 15) == 0)
                     ? s.cols / 4 : 0;
  for (int r = blockIdx.x; r < s.rows; r += gridDim.x) {
    const float* g = s.g + (int64_t)r * s.cols;
    float* mr = bf ? reinterpret_cast<float*>(reinterpret_cast<__nv_bfloat16*>(s.m) +
                                              (int64_t)r * s.ldm)
                   : s.m + (int64_t)r * s.ldm;
    unsigned short* gh = s.g_hi + (int64_t)r * s.ldm;
    unsigned short* gl = s.g_lo + (int64_t)r * s.ldm;
    float sum = 0.f, mx = 0.f;
    for (int q = threadIdx.x; q < nv; q += blockDim.x) {
      const float4 x = reinterpret_cast<const float4*>(g)[q];
      float4 mm = reinterpret_cast<float4*>(mr)[q];
      momentum_elem(x.x, mm.x, beta1, one_minus, sum, mx);
      momentum_elem(x.y, mm.y, beta1, one_minus, sum, mx);
      momentum_elem(x.z, mm.z, beta1, one_minus, sum, mx);
      momentum_elem(x.w, mm.w, beta1, one_minus, sum, mx);
      reinterpret_cast<float4*>(mr)[q] = mm;
    }
    for (int c = 4 * nv + threadIdx.x; c < s.cols; c += blockDim.x) {
      float m = ld_state(mr, c, bf);
      momentum_elem(g[c], m, beta1, one_minus, sum, mx);
      st_state(mr, c, m, bf);
    }
    block_sum_max(sum, mx);
    const float scale = pow2_below(mx, kF16ScaleExp);
    if (threadIdx.x == 0) {
      s.g_rinv[r] = pow2_below_inv(mx, kF16ScaleExp);
      atomic_max_nonneg(s.g_rmax, row_norm_bound(sum, mx, s.cols));
      // the row's sum of squares is finite iff every g of the row is
      report_nonfinite(flag, !isfinite(sum) && !(sum > 3.402823466e38f && isfinite(mx)));
    }
    if (s.m16_hi) {
      // M's new row (this thread's own writes above), its scale and splits
      float msum = 0.f, mmx = 0.f;
      for (int c = threadIdx.x; c < s.cols; c += blockDim.x) {
        const float m = ld_state(mr, c, bf);
        msum = fmaf(m, m, msum);
        mmx = fmaxf(mmx, fabsf(m));
      }
      block_sum_max(msum, mmx);
      const float mscale = pow2_below(mmx, kF16ScaleExp);
      if (threadIdx.x == 0) {
        s.m_rinv[r] = pow2_below_inv(mmx, kF16ScaleExp);
        atomic_max_nonneg(s.m_rmax, row_norm_bound(msum, mmx, s.cols));
        if (s.m_amax) atomic_max_nonneg(s.m_amax, mmx);
      }
      unsigned short* m16h = s.m16_hi + (int64_t)r * s.ldm;
      unsigned short* m16l = s.m16_lo + (int64_t)r * s.ldm;
      if (s.m_hi) {
        float* mth = s.m_hi + (int64_t)r * s.ldm;
        float* mtl = s.m_lo + (int64_t)r * s.ldm;
        for (int c = threadIdx.x; c < s.cols; c += blockDim.x) {
          const float m = ld_state(mr, c, bf);
          split_f16(m * mscale, m16h[c], m16l[c]);
          split_tf32(m, mth[c], mtl[c]);
        }
      } else {
        for (int c = threadIdx.x; c < s.cols; c += blockDim.x)
          split_f16(ld_state(mr, c, bf) * mscale, m16h[c], m16l[c]);
      }
    }
    for (int q = threadIdx.x; q < nv; q += blockDim.x) {
      const float4 x = reinterpret_cast<const float4*>(g)[q];
      ushort4 h, l;
      split_f16(x.x * scale, h.x, l.x);
      split_f16(x.y * scale, h.y, l.y);
      split_f16(x.z * scale, h.z, l.z);
      split_f16(x.w * scale, h.w, l.w);
      reinterpret_cast<ushort4*>(gh)[q] = h;
      reinterpret_cast<ushort4*>(gl)[q] = l;
    }
    for (int c = 4 * nv + threadIdx.x; c < s.cols; c += blockDim.x)
      split_f16(g[c] * scale, gh[c], gl[c]);
  }
}

// 3xF16 Adam: one block per row.  First pass as adam_kernel (M~, v; D's row
// max and sum of squares); second pass recomputes D from the M~ and v this
// thread just wrote (bitwise the same values) and stores its scaled split.
// The rows (library buffers, ld a multiple of 32) take 16-byte accesses.
__device__ __forceinline__ float adam_elem(float g, float& m, float& v, float beta1,
                                           float one_minus1, float beta2, float one_minus,
                                           float eps, int incremental, float& sum, float& mx) {
  if (incremental) m = beta1 * m + one_minus1 * g;
  v = beta2 * v + one_minus * (g * g);
  const float d = m / (sqrtf(v) + eps);
  sum = fmaf(d, d, sum);
  mx = fmaxf(mx, fabsf(d));
  return d;
}

__global__ void adam16_kernel(const __grid_constant__ SegBatch<Adam16Seg> b, float beta1,
                              float beta2, float eps, int incremental, int* flag) {
  const Adam16Seg& s = b.seg[blockIdx.y];
  const float one_minus1 = 1.0f - beta1;
  const float one_minus = 1.0f - beta2;
  const bool bf = s.mt_bf16 != 0;
  const int nv = bf ? 0 : s.cols / 4;
  for (int r = blockIdx.x; r < s.rows; r += gridDim.x) {
    const float* gt = s.gt + (int64_t)r * s.ld;
    float* mt = bf ? reinterpret_cast<float*>(reinterpret_cast<__nv_bfloat16*>(s.mt) +
                                              (int64_t)r * s.ld)
                   : s.mt + (int64_t)r * s.ld;
    float* v = s.v + (int64_t)r * s.ld;
    unsigned short* dh = s.d_hi + (int64_t)r * s.ld;
    unsigned short* dl = s.d_lo + (int64_t)r * s.ld;
    float sum = 0.f, mx = 0.f;
    for (int q = threadIdx.x; q < nv; q += blockDim.x) {
      const float4 g = reinterpret_cast<const float4*>(gt)[q];
      float4 m = reinterpret_cast<float4*>(mt)[q];
      float4 w = reinterpret_cast<float4*>(v)[q];
      adam_elem(g.x, m.x, w.x, beta1, one_minus1, beta2, one_minus, eps, incremental, sum, mx);
      adam_elem(g.y, m.y, w.y, beta1, one_minus1, beta2, one_minus, eps, incremental, sum, mx);
      adam_elem(g.z, m.z, w.z, beta1, one_minus1, beta2, one_minus, eps, incremental, sum, mx);
      adam_elem(g.w, m.w, w.w, beta1, one_minus1, beta2, one_minus, eps, incremental, sum, mx);
      if (incremental) reinterpret_cast<float4*>(mt)[q] = m;
      reinterpret_cast<float4*>(v)[q] = w;
    }
    for (int c = 4 * nv + threadIdx.x; c < s.cols; c += blockDim.x) {
      float m = ld_state(mt, c, bf), w = v[c];
      if (incremental) {  // the stored (rounded) M~ is the one D uses
        m = as_state(beta1 * m + one_minus1 * gt[c], bf);
        st_state(mt, c, m, bf);
      }
      adam_elem(gt[c], m, w, beta1, one_minus1, beta2, one_minus, eps, 0, sum, mx);
      v[c] = w;
    }
    block_sum_max(sum, mx);
    const float scale = pow2_below(mx, kF16ScaleExp);
    if (threadIdx.x == 0) {
      s.d_rinv[r] = pow2_below_inv(mx, kF16ScaleExp);
      atomic_max_nonneg(s.d_rmax, row_norm_bound(sum, mx, s.cols));
      report_nonfinite(flag, !isfinite(sum) && !(sum > 3.402823466e38f && isfinite(mx)));
    }
    for (int q = threadIdx.x; q < nv; q += blockDim.x) {
      const float4 m = reinterpret_cast<const float4*>(mt)[q];
      const float4 w = reinterpret_cast<const float4*>(v)[q];
      ushort4 h, l;
      split_f16(m.x / (sqrtf(w.x) + eps) * scale, h.x, l.x);
      split_f16(m.y / (sqrtf(w.y) + eps) * scale, h.y, l.y);
      split_f16(m.z / (sqrtf(w.z) + eps) * scale, h.z, l.z);
      split_f16(m.w / (sqrtf(w.w) + eps) * scale, h.w, l.w);
      reinterpret_cast<ushort4*>(dh)[q] = h;
      reinterpret_cast<ushort4*>(dl)[q] = l;
    }
    for (int c = 4 * nv + threadIdx.x; c < s.cols; c += blockDim.x)
      split_f16(ld_state(mt, c, bf) / (sqrtf(v[c]) + eps) * scale, dh[c], dl[c]);
  }
}

// Scaled fp16 split of a float32 matrix, one block per row: per-row scales
// (rinv set) or one scale from *bound; rmax (if set) grows to the largest row
// 2-norm.  hi == nullptr: norms only.
__global__ void split16_kernel(const __grid_constant__ SegBatch<Split16Seg> b) {
  const Split16Seg& s = b.seg[blockIdx.y];
  for (int r = blockIdx.x; r < s.rows; r += gridDim.x) {
    const float* x = s.src + (int64_t)r * s.ld_src;
    float sum = 0.f, mx = 0.f;
    for (int c = threadIdx.x; c < s.cols; c += blockDim.x) {
      sum = fmaf(x[c], x[c], sum);
      mx = fmaxf(mx, fabsf(x[c]));
    }
    block_sum_max(sum, mx);
    const float scale = s.bound ? pow2_below(*s.bound, kF16ScaleExp) : pow2_below(mx, kF16ScaleExp);
    if (threadIdx.x == 0) {
      if (s.rinv) s.rinv[r] = pow2_below_inv(mx, kF16ScaleExp);
      if (s.rmax) atomic_max_nonneg(s.rmax, row_norm_bound(sum, mx, s.cols));
    }
    if (s.hi)
      for (int c = threadIdx.x; c < s.cols; c += blockDim.x) {
        const int64_t o = (int64_t)r * s.ld_dst + c;
        split_f16(x[c] * scale, s.hi[o], s.lo[o]);
      }
  }
}

// TF32 split (lo rounded to TF32: tensor-core operands only) of a basis held
// as a 2^14-scaled fp16 split, optionally transposed (32 x 32 tiles through
// shared memory).
template <bool TRANSPOSE>
__global__ void to_tf32_kernel(const __grid_constant__ SegBatch<ToTf32Seg> b) {
  __shared__ float tile[32][33];
  const ToTf32Seg& s = b.seg[blockIdx.y];
  const int tiles_r = (s.rows + 31) / 32, tiles_c = (s.cols + 31) / 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
  for (int t = blockIdx.x; t < tiles_r * tiles_c; t += gridDim.x) {
    const int r0 = (t / tiles_c) * 32, c0 = (t % tiles_c) * 32;
    for (int i = ty; i < 32; i += 8) {
      const int r = r0 + i, c = c0 + tx;
      float x = 0.f;
      if (r < s.rows && c < s.cols) {
        const int64_t o = (int64_t)r * s.ld_src + c;
        x = (__half2float(__ushort_as_half(s.s_hi[o])) +
             __half2float(__ushort_as_half(s.s_lo[o]))) * kF16UnitScaleInv;
      }
      if (TRANSPOSE) {
        tile[i][tx] = x;
      } else if (r < s.rows && c < s.cols) {
        float h, l;
        split_tf32_mma(x, h, l);
        const int64_t o = (int64_t)r * s.ld_dst + c;
        s.d_hi[o] = h;
        s.d_lo[o] = l;
      }
    }
    if (TRANSPOSE) {
      __syncthreads();
      for (int i = ty; i < 32; i += 8) {
        const int c = c0 + i, r = r0 + tx;  // output row c, column r
        if (r < s.rows && c < s.cols) {
          float h, l;
          split_tf32_mma(tile[tx][i], h, l);
          const int64_t o = (int64_t)c * s.ld_dst + r;
          s.d_hi[o] = h;
          s.d_lo[o] = l;
        }
      }
      __syncthreads();
    }
  }
}

// M^T as a fp16 split under one power-of-two scale (TransposeF16Seg), 32 x 32
// tiles through shared memory: rows of M are read and rows of M^T written
// 32 consecutive elements at a time.
__global__ void transpose16_kernel(const __grid_constant__ SegBatch<TransposeF16Seg> b) {
  __shared__ float tile[32][33];
  const TransposeF16Seg& s = b.seg[blockIdx.y];
  const bool bf = s.m_bf16 != 0;
  const float scale = pow2_below(*s.rmax, kF16ScaleExp);
  const int tiles_r = (s.rows + 31) / 32, tiles_c = (s.cols + 31) / 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
  for (int t = blockIdx.x; t < tiles_r * tiles_c; t += gridDim.x) {
    const int r0 = (t / tiles_c) * 32, c0 = (t % tiles_c) * 32;
    for (int i = ty; i < 32; i += 8) {
      const int r = r0 + i, c = c0 + tx;
      tile[i][tx] = (r < s.rows && c < s.cols) ? ld_state(s.m, (int64_t)r * s.ld_src + c, bf) : 0.f;
    }
    __syncthreads();
    for (int i = ty; i < 32; i += 8) {
      const int c = c0 + i, r = r0 + tx;  // output row c, column r
      if (r < s.rows && c < s.cols) {
        const int64_t o = (int64_t)c * s.ld_dst + r;
        split_f16(tile[tx][i] * scale, s.d_hi[o], s.d_lo[o]);
      }
    }
    __syncthreads();
  }
}

__global__ void combine16_kernel(const unsigned short* hi, const unsigned short* lo, int ld_src,
                                 float* dst, int ld_dst, int rows, int cols) {
  const int64_t total = (int64_t)rows * cols;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int r = (int)(e / cols), c = (int)(e - (int64_t)r * cols);
    const int64_t o = (int64_t)r * ld_src + c;
    dst[(int64_t)r * ld_dst + c] =
        (__half2float(__ushort_as_half(hi[o])) + __half2float(__ushort_as_half(lo[o]))) *
        kF16UnitScaleInv;
  }
}

__global__ void to_f16_kernel(const __grid_constant__ SegBatch<ToF16Seg> b) {
  const ToF16Seg& s = b.seg[blockIdx.y];
  const int64_t total = (int64_t)s.rows * s.cols;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int r = (int)(e / s.cols), c = (int)(e - (int64_t)r * s.cols);
    const int64_t i = (int64_t)r * s.ld_src + c;
    const int64_t o = (int64_t)r * s.ld_dst + c;
    split_f16((s.s_hi[i] + s.s_lo[i]) * kF16UnitScale, s.hi[o], s.lo[o]);
  }
}

// Tiled transpose through shared memory (32 x 32 tiles, padded against bank
// conflicts).  blockIdx.y = matrix, blockIdx.x strides over tiles.
__global__ void transpose_kernel(const __grid_constant__ SegBatch<TransposeSeg> b) {
  __shared__ float th[32][33];
  __shared__ float tl[32][33];
  const TransposeSeg& s = b.seg[blockIdx.y];
  const int tiles_r = (s.rows + 31) / 32, tiles_c = (s.cols + 31) / 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
  for (int t = blockIdx.x; t < tiles_r * tiles_c; t += gridDim.x) {
    const int r0 = (t / tiles_c) * 32, c0 = (t % tiles_c) * 32;
    for (int i = ty; i < 32; i += 8) {
      const int r = r0 + i, c = c0 + tx;
      float x = 0.f, y = 0.f;
      if (r < s.rows && c < s.cols) {
        const int64_t o = (int64_t)r * s.ld_src + c;
        x = s.s_hi[o];
        y = s.src_is_split ? s.s_lo[o] : 0.f;
      }
      th[i][tx] = x;
      tl[i][tx] = y;
    }
    __syncthreads();
    for (int i = ty; i < 32; i += 8) {
      const int c = c0 + i, r = r0 + tx;  // output row c, column r
      if (r < s.rows && c < s.cols) {
        const float v = th[tx][i] + tl[tx][i];
        const int64_t o = (int64_t)c * s.ld_dst + r;
        if (s.dst_is_split) {
          float h, l;
          if (s.dst_mma_only) {
            split_tf32_mma(v, h, l);
          } else {
            split_tf32(v, h, l);
          }
          s.d_hi[o] = h;
          s.d_lo[o] = l;
        } else {
          s.d_hi[o] = v;
        }
      }
    }
    __syncthreads();
  }
}

__global__ void fill_kernel(const __grid_constant__ SegBatch<FillSeg> b) {
  const FillSeg& s = b.seg[blockIdx.y];
  const int64_t total = (int64_t)s.rows * s.cols;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int r = (int)(e / s.cols), c = (int)(e - (int64_t)r * s.cols);
    const int64_t o = (int64_t)r * s.ld + c;
    if (s.f16) {  // fp16 split scaled by 2^14: the identity's 1 is 2^14, lo 0
      reinterpret_cast<unsigned short*>(s.hi)[o] =
          __half_as_ushort(__float2half_rn((s.identity && r == c) ? kF16UnitScale : 0.0f));
      if (s.lo) reinterpret_cast<unsigned short*>(s.lo)[o] = __half_as_ushort(__float2half_rn(0.f));
    } else {
      s.hi[o] = (s.identity && r == c) ? 1.0f : 0.0f;
      if (s.lo) s.lo[o] = 0.0f;
    }
  }
}

__global__ void split_kernel(const __grid_constant__ SegBatch<SplitSeg> b) {
  const SplitSeg& s = b.seg[blockIdx.y];
  const int64_t total = (int64_t)s.rows * s.cols;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int r = (int)(e / s.cols), c = (int)(e - (int64_t)r * s.cols);
    float h, l;
    split_tf32_mma(s.src[(int64_t)r * s.ld_src + c], h, l);
    const int64_t o = (int64_t)r * s.ld_dst + c;
    s.hi[o] = h;
    s.lo[o] = l;
  }
}

__global__ void combine_kernel(const float* hi, const float* lo, int ld_src, float* dst,
                               int ld_dst, int rows, int cols, int src_bf16) {
  const int64_t total = (int64_t)rows * cols;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int r = (int)(e / cols), c = (int)(e - (int64_t)r * cols);
    const int64_t o = (int64_t)r * ld_src + c;
    dst[(int64_t)r * ld_dst + c] =
        src_bf16 ? ld_state(hi, o, true) : (lo ? hi[o] + lo[o] : hi[o]);
  }
}

}  // namespace

int launch_momentum(const hvec<MomentumSeg>& segs, float beta1, int* flag,
                    cudaStream_t stream) {
  // read G (4) and M (4); write M (4) and G's split (8) (refresh steps: and
  // M's split, 8)
  const bool split_m = !segs.empty() && segs[0].m_hi;
  return launch_segs(segs, split_m ? 28.0 : 20.0, momentum_kernel, stream, beta1, flag);
}

int launch_adam(const hvec<AdamSeg>& segs, float beta1, float beta2, float eps,
                int incremental, int* flag, cudaStream_t stream) {
  // read G~, M~, v (12); write v (4) and D's split (8); incremental: write M~ (4)
  return launch_segs(segs, incremental ? 28.0 : 24.0, adam_kernel, stream, beta1, beta2, eps,
                     incremental, flag);
}

// One block per row: grid.x covers the rows (up to 1024 blocks per matrix).
template <class Seg, class Kernel, class... Args>
int launch_rows(const hvec<Seg>& segs, double bytes_per_elem, Kernel kernel,
                cudaStream_t stream, Args... args) {
  for (size_t base = 0; base < segs.size(); base += kMaxSegs) {
    SegBatch<Seg> b;
    std::memset(&b, 0, sizeof(b));
    b.count = (int)std::min<size_t>(kMaxSegs, segs.size() - base);
    int most = 0;
    double elems = 0.0;
    for (int i = 0; i < b.count; ++i) {
      b.seg[i] = segs[base + i];
      if (b.seg[i].cols > 0) most = std::max(most, b.seg[i].rows);
      elems += (double)b.seg[i].rows * b.seg[i].cols;
    }
    if (most == 0) continue;
    dim3 grid((unsigned)std::min(most, 1024), b.count);
    ProfScope prof(ROT_PROF_ELEMENTWISE, elems * bytes_per_elem, stream);
    kernel<<<grid, kThreads, 0, stream>>>(b, args...);
    if (cudaGetLastError() != cudaSuccess) return ROT_ECUDA;
  }
  return ROT_OK;
}

int launch_momentum16(const hvec<Momentum16Seg>& segs, float beta1, int* flag,
                      cudaStream_t stream) {
  // read G (4) and M (4); write M (4) and G's fp16 split (4) (refresh steps:
  // and M's fp16 split, 4, and TF32 split, 8)
  // read G, M (8); write M, G's fp16 split (8); refresh: M's fp16 split (4)
  // and, where asked for, its TF32 split (8)
  const bool split_m = !segs.empty() && segs[0].m16_hi;
  const bool tf32_m = split_m && segs[0].m_hi;
  return launch_rows(segs, tf32_m ? 28.0 : (split_m ? 20.0 : 16.0), momentum16_kernel, stream,
                     beta1, flag);
}

namespace {

int to_tf32_segs(const hvec<ToTf32Seg>& segs, bool transpose, cudaStream_t stream) {
  // read the fp16 split (4), write the TF32 split (8)
  for (size_t base = 0; base < segs.size(); base += kMaxSegs) {
    SegBatch<ToTf32Seg> b;
    std::memset(&b, 0, sizeof(b));
    b.count = (int)std::min<size_t>(kMaxSegs, segs.size() - base);
    int64_t most = 0;
    double elems = 0.0;
    for (int i = 0; i < b.count; ++i) {
      b.seg[i] = segs[base + i];
      most = std::max<int64_t>(most, (int64_t)((b.seg[i].rows + 31) / 32) * ((b.seg[i].cols + 31) / 32));
      elems += (double)b.seg[i].rows * b.seg[i].cols;
    }
    if (most == 0) continue;
    dim3 grid((unsigned)std::min<int64_t>(most, 4096), b.count);
    ProfScope prof(ROT_PROF_ELEMENTWISE, elems * 12.0, stream);
    if (transpose) {
      to_tf32_kernel<true><<<grid, kThreads, 0, stream>>>(b);
    } else {
      to_tf32_kernel<false><<<grid, kThreads, 0, stream>>>(b);
    }
    if (cudaGetLastError() != cudaSuccess) return ROT_ECUDA;
  }
  return ROT_OK;
}

}  // namespace

int launch_to_tf32(const hvec<ToTf32Seg>& segs, cudaStream_t stream) {
  return to_tf32_segs(segs, false, stream);
}

int launch_to_tf32_t(const hvec<ToTf32Seg>& segs, cudaStream_t stream) {
  return to_tf32_segs(segs, true, stream);
}

int launch_combine16(const unsigned short* hi, const unsigned short* lo, int ld_src, float* dst,
                     int ld_dst, int rows, int cols, cudaStream_t stream) {
  const int64_t total = (int64_t)rows * cols;
  if (total == 0) return ROT_OK;
  ProfScope prof(ROT_PROF_ELEMENTWISE, (double)total * 8, stream);
  combine16_kernel<<<grid_x_for(total), kThreads, 0, stream>>>(hi, lo, ld_src, dst, ld_dst,
                                                               rows, cols);
  return cudaGetLastError() == cudaSuccess ? ROT_OK : ROT_ECUDA;
}

int launch_adam16(const hvec<Adam16Seg>& segs, float beta1, float beta2, float eps,
                  int incremental, int* flag, cudaStream_t stream) {
  // read G~, M~, v (12); write v (4) and D's fp16 split (4); incremental: write M~ (4)
  return launch_rows(segs, incremental ? 24.0 : 20.0, adam16_kernel, stream, beta1, beta2, eps,
                     incremental, flag);
}

int launch_split16(const hvec<Split16Seg>& segs, cudaStream_t stream) {
  return launch_rows(segs, 8.0, split16_kernel, stream);
}

int launch_to_f16(const hvec<ToF16Seg>& segs, cudaStream_t stream) {
  return launch_segs(segs, 12.0, to_f16_kernel, stream);
}

int launch_transpose16(const hvec<TransposeF16Seg>& segs, cudaStream_t stream) {
  for (size_t base = 0; base < segs.size(); base += kMaxSegs) {
    SegBatch<TransposeF16Seg> b;
    std::memset(&b, 0, sizeof(b));
    b.count = (int)std::min<size_t>(kMaxSegs, segs.size() - base);
    int64_t most = 0;
    double bytes = 0.0;
    for (int i = 0; i < b.count; ++i) {
      b.seg[i] = segs[base + i];
      most = std::max<int64_t>(most, (int64_t)((b.seg[i].rows + 31) / 32) *
                                         ((b.seg[i].cols + 31) / 32));
      // read M (4, or 2 as bf16); write the fp16 split (4)
      bytes += (double)b.seg[i].rows * b.seg[i].cols * (b.seg[i].m_bf16 ? 6 : 8);
    }
    if (most == 0) continue;
    dim3 grid((unsigned)std::min<int64_t>(most, 2048), b.count);
    ProfScope prof(ROT_PROF_ELEMENTWISE, bytes, stream);
    transpose16_kernel<<<grid, 256, 0, stream>>>(b);
    if (cudaGetLastError() != cudaSuccess) return ROT_ECUDA;
  }
  return ROT_OK;
}

int launch_transpose(const hvec<TransposeSeg>& segs, cudaStream_t stream) {
  for (size_t base = 0; base < segs.size(); base += kMaxSegs) {
    SegBatch<TransposeSeg> b;
    std::memset(&b, 0, sizeof(b));
    b.count = (int)std::min<size_t>(kMaxSegs, segs.size() - base);
    int64_t most = 0;
    double bytes = 0.0;
    for (int i = 0; i < b.count; ++i) {
      b.seg[i] = segs[base + i];
      most = std::max<int64_t>(most, (int64_t)((b.seg[i].rows + 31) / 32) *
                                         ((b.seg[i].cols + 31) / 32));
      bytes += (double)b.seg[i].rows * b.seg[i].cols *
               ((b.seg[i].src_is_split ? 8 : 4) + (b.seg[i].dst_is_split ? 8 : 4));
    }
    if (most == 0) continue;
    dim3 grid((unsigned)std::min<int64_t>(most, 2048), b.count);
    ProfScope prof(ROT_PROF_ELEMENTWISE, bytes, stream);
    transpose_kernel<<<grid, 256, 0, stream>>>(b);
    if (cudaGetLastError() != cudaSuccess) return ROT_ECUDA;
  }
  return ROT_OK;
}

// ---------------------------------------------------------------------------
// Guard regions of bounds-checked builds: one CTA of 64 threads per region,
// one 32-bit word per thread.
// ---------------------------------------------------------------------------

constexpr int kMaxGuards = 1024;

struct GuardBatch {
  int count;
  uint64_t off[kMaxGuards];
};

__global__ void guard_kernel(const __grid_constant__ GuardBatch b, uint32_t* work, int* status,
                             int check) {
  if (blockIdx.x >= b.count) return;
  uint32_t* g = work + b.off[blockIdx.x] / 4;
  for (int i = threadIdx.x; i < (int)(kGuardBytes / 4); i += blockDim.x) {
    if (!check) {
      g[i] = kGuardWord;
    } else if (g[i] != kGuardWord && status) {
      atomicCAS(status, ROT_OK, ROT_ECORRUPT);
    }
  }
}

int launch_guards(const hvec<uint64_t>& offsets, void* work, int* status, bool check,
                  cudaStream_t stream) {
  thread_local static GuardBatch b;  // ~8 KB parameter block: keep off the stack
  for (size_t base = 0; base < offsets.size(); base += kMaxGuards) {
    b.count = (int)std::min<size_t>(kMaxGuards, offsets.size() - base);
    for (int i = 0; i < b.count; ++i) b.off[i] = offsets[base + i];
    guard_kernel<<<b.count, 64, 0, stream>>>(b, static_cast<uint32_t*>(work), status,
                                            check ? 1 : 0);
    if (cudaGetLastError() != cudaSuccess) return ROT_ECUDA;
  }
  return ROT_OK;
}

int launch_fill(const hvec<FillSeg>& segs, cudaStream_t stream) {
  return launch_segs(segs, 8.0, fill_kernel, stream);
}

int launch_split(const hvec<SplitSeg>& segs, cudaStream_t stream) {
  return launch_segs(segs, 12.0, split_kernel, stream);
}

int launch_combine(const float* hi, const float* lo, int ld_src, float* dst, int ld_dst,
                   int rows, int cols, cudaStream_t stream, int src_bf16) {
  const int64_t total = (int64_t)rows * cols;
  if (total == 0) return ROT_OK;
  ProfScope prof(ROT_PROF_ELEMENTWISE, (double)total * (lo ? 12 : 8), stream);
  combine_kernel<<<grid_x_for(total), kThreads, 0, stream>>>(hi, lo, ld_src, dst, ld_dst, rows,
                                                             cols, src_bf16);
  return cudaGetLastError() == cudaSuccess ? ROT_OK : ROT_ECUDA;
}

}  // namespace rot
