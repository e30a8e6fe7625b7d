// TF32 split of a float32 value: x = hi + lo exactly, with hi = x rounded to
// TF32 (round to nearest, ties away: PTX cvt.rna.tf32.f32) and lo = x - hi.
// Three TF32 products hi*hi + hi*lo + lo*hi then recover about float32
// accuracy (Markidis et al., "NVIDIA Tensor Core Programmability,
// Performance & Precision", 2018; Ootomo & Yokota, "Recovering single
// precision accuracy from Tensor Cores while surpassing the FP32 theoretical
// peak performance", 2022).
#pragma once

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

}  // namespace rot
