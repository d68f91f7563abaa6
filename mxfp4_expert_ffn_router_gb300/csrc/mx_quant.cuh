// mx_quant.cuh -- MXFP4 quantisation of activations (device functions).
//
// OCP Microscaling Formats (MX) v1.0, conversion to an MX format: per block of 32
// values the shared scale is X = 2^(floor(log2 amax) - 2) (2 = the largest
// exponent of E2M1), clamped to the E8M0 range 2^-127 .. 2^127, stored as the
// byte e + 127; an all-zero block gets the byte 0.  Each element is v / X rounded
// to the nearest E2M1 value {0, .5, 1, 1.5, 2, 3, 4, 6} (ties to the even code),
// saturating at 6; the code's sign bit is set iff v < 0.  v / X is exact in fp32
// (a power-of-two scaling of a bf16 value), so every rounding decision is the same
// as in exact arithmetic.
#pragma once
#include <stdint.h>

namespace k3moe {

// Shared exponent e of a block (X = 2^e) from its largest magnitude.
__device__ __forceinline__ int mx_shared_exp(float amax) {
  if (!(amax > 0.f)) return -127;  // all-zero (or NaN-only) block
  if (amax == INFINITY) return 127;
  int ex;
  frexpf(amax, &ex);  // amax = f * 2^ex, f in [0.5, 1): floor(log2 amax) = ex - 1
  return max(-127, min(127, ex - 3));
}

// 2^e for e in [-127, 127] as fp32 (2^-127 is a subnormal, exact).
__device__ __forceinline__ float mx_pow2(int e) {
  return e >= -126 ? __uint_as_float(static_cast<uint32_t>(e + 127) << 23) : __uint_as_float(0x00400000u);
}

// |v| / X onto the E2M1 grid: the 3-bit magnitude code.  The grid midpoints
// 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5 go to the even code (strict or non-strict
// comparison per midpoint); q >= 6 saturates; NaN gives 0.
__device__ __forceinline__ uint32_t e2m1_rne_code(float q) {
  return static_cast<uint32_t>(q > 0.25f) + static_cast<uint32_t>(q >= 0.75f) + static_cast<uint32_t>(q > 1.25f) +
         static_cast<uint32_t>(q >= 1.75f) + static_cast<uint32_t>(q > 2.5f) + static_cast<uint32_t>(q >= 3.5f) +
         static_cast<uint32_t>(q > 5.0f);
}

// Value of a 3-bit E2M1 magnitude code.
__device__ __forceinline__ float e2m1_mag_value(uint32_t c) {
  return c < 4u ? 0.5f * static_cast<float>(c) : static_cast<float>(1u << ((c >> 1) - 1u)) * (1.0f + 0.5f * (c & 1u));
}

// 4-bit code of v in a block with shared exponent e (X = 2^e): sign bit 3.
__device__ __forceinline__ uint32_t mx_code(float v, float inv_x) {
  const uint32_t c = e2m1_rne_code(fabsf(v) * inv_x);
  return v < 0.f ? (c | 8u) : c;
}

// Value of a 4-bit code in a block with scale X.
__device__ __forceinline__ float mx_value(uint32_t code, float x) {
  const float m = e2m1_mag_value(code & 7u) * x;
  return (code & 8u) ? -m : m;
}

}  // namespace k3moe
