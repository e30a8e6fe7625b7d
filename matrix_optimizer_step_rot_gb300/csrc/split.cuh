// TF32 split of a float32 value: x = hi + lo exactly, with hi = x rounded to
// TF32 (round to nearest, ties away: PTX cvt.rna.tf32.f32) and lo = x - hi.
// Three TF32 products hi*hi + hi*lo + lo*hi then recover about float32
// accuracy (Markidis et al., "NVIDIA Tensor Core Programmability,
// Performance & Precision", 2018; Ootomo & Yokota, "Recovering single
// precision accuracy from Tensor Cores while surpassing the FP32 theoretical
// peak performance", 2022).
#pragma once

#include <cuda_fp16.h>

namespace rot {

__device__ __forceinline__ float tf32_round(float x) {
  unsigned u;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(u) : "f"(x));
  return __uint_as_float(u);
}

__device__ __forceinline__ void split_tf32(float x, float& hi, float& lo) {
  hi = tf32_round(x);
  lo = x - hi;
}

// Split for operands that only the tensor cores read: lo is rounded to TF32
// as well (round to nearest).  The tensor cores would otherwise truncate lo's
// low 13 bits (2^-21 relative to x); rounded, the pair carries x to within
// 2^-22 relative.  hi + lo is then not exactly x, so arrays that are also
// recombined into float32 keep the exact split above.
__device__ __forceinline__ void split_tf32_mma(float x, float& hi, float& lo) {
  hi = tf32_round(x);
  lo = tf32_round(x - hi);
}


// ---------------------------------------------------------------------------
// Scaled fp16 split (ROT_PREC_3XF16).  An operand x is multiplied by a power
// of two s chosen so that |x s| < 2^14, then hi = fp16(x s) and
// lo = fp16(x s - hi), both rounded to nearest: 11 + 11 significant bits, the
// same as the TF32 split, and the three fp16 products hi*hi + hi*lo + lo*hi
// recover the product to about float32 accuracy (the same argument as for
// 3xTF32; the fp16 tensor-core rate is twice the TF32 one).  Scaling by a
// power of two is exact, and the epilogue undoes it exactly.
// ---------------------------------------------------------------------------

// 2^k / 2^e, where 2^(e-1) <= r < 2^e: r times the result is < 2^k.  For r = 0,
// a non-finite r or an exponent out of range the result saturates (1 for
// r <= 0 or non-finite, so that infinities and NaNs propagate unscaled).
__device__ __forceinline__ float pow2_below(float r, int k) {
  if (!(r > 0.f) || !(r <= 3.402823466e38f)) return 1.f;
  const int biased = (__float_as_int(r) >> 23) & 255;  // 0 for subnormal r
  const int e = (biased == 0 ? 1 : biased) - 126;     // r < 2^e
  int s = k - e;
  s = s < -126 ? -126 : (s > 127 ? 127 : s);
  return __int_as_float((s + 127) << 23);
}

// 1 / pow2_below(r, k), exactly.
__device__ __forceinline__ float pow2_below_inv(float r, int k) {
  if (!(r > 0.f) || !(r <= 3.402823466e38f)) return 1.f;
  const int biased = (__float_as_int(r) >> 23) & 255;
  const int e = (biased == 0 ? 1 : biased) - 126;
  int s = e - k;
  s = s < -126 ? -126 : (s > 127 ? 127 : s);
  return __int_as_float((s + 127) << 23);
}

constexpr int kF16ScaleExp = 14;            // scaled operands stay below 2^14
constexpr float kF16UnitScale = 16384.f;    // fixed scale of U, V (|entries| <= 1)
constexpr float kF16UnitScaleInv = 1.f / 16384.f;

__device__ __forceinline__ void split_f16(float xs, unsigned short& hi, unsigned short& lo) {
  const __half h = __float2half_rn(xs);
  const __half l = __float2half_rn(xs - __half2float(h));
  hi = __half_as_ushort(h);
  lo = __half_as_ushort(l);
}

}  // namespace rot
