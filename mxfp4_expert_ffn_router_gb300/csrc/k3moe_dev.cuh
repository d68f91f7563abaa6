// k3moe_dev.cuh -- device helpers shared by the k3moe CUDA kernels (sm_103a).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/k3moe.h"

namespace k3moe {

// ---- programmatic dependent launch (PDL) ----------------------------------
// wait: block until the preceding kernel in the stream has completed (or
// triggered) -- must come before the first read of its outputs.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// launch_dependents: allow the next kernel in the stream to start its prologue.
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void set_status(int32_t *st, int32_t bits) {
  if (st) atomicOr(st, bits);
}

// ---- small numeric helpers -------------------------------------------------
__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// fp32 -> bf16 bits, round to nearest even (NaN -> quiet NaN).
__device__ __forceinline__ uint16_t f32_to_bf16_rne(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return 0x7FC0u;
  u += 0x7FFFu + ((u >> 16) & 1u);
  return static_cast<uint16_t>(u >> 16);
}

// E8M0 byte -> 2^(b-127) as fp32 (b = 0 gives the subnormal 2^-127; 255 NaN).
__device__ __forceinline__ float e8m0_to_f32(uint32_t b) {
  if (b == 0u) return __uint_as_float(0x00400000u);
  if (b == 255u) return __uint_as_float(0x7FC00000u);
  return __uint_as_float(b << 23);
}

// 2^e as fp32 for an integer e in [-126, 127].
__device__ __forceinline__ float exp2i(int e) { return __uint_as_float(static_cast<uint32_t>(e + 127) << 23); }

// Four packed bytes of E2M1 pairs -> four f16x2 registers (element 2i in the low half).
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t (&h)[4]) {
  asm("{\n\t.reg .b8 q0, q1, q2, q3;\n\t"
      "mov.b32 {q0, q1, q2, q3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, q0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, q1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, q2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, q3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}

// acc += a.lo * b.lo + a.hi * b.hi with fp32 accumulation of exact f16 products.
__device__ __forceinline__ float fma2_f16_f32(uint32_t a, uint32_t b, float acc) {
  asm("{\n\t.reg .b16 alo, ahi, blo, bhi;\n\t"
      "mov.b32 {alo, ahi}, %1;\n\t"
      "mov.b32 {blo, bhi}, %2;\n\t"
      "fma.rn.f32.f16 %0, alo, blo, %0;\n\t"
      "fma.rn.f32.f16 %0, ahi, bhi, %0;\n\t}"
      : "+f"(acc)
      : "r"(a), "r"(b));
  return acc;
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void *p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

}  // namespace k3moe
