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

// ---- top-k selection within one warp (router logits, k <= 32) ----------------
// Order-preserving key of an fp32 value (larger value -> larger key; -0 and +0
// share a key).  Keys of finite and infinite values are >= 0x007FFFFF (the key of
// -inf), so 0 marks a slot that holds no element.
__device__ __forceinline__ uint32_t order_key(float v) {
  uint32_t u = __float_as_uint(v);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The largest of a lane's NK keys and the lowest slot holding it, by a pairwise
// tree whose ties keep the left (lower) slot: log2(NK) levels instead of a chain
// of NK dependent compares.
template <int NK>
__device__ __forceinline__ void lane_best_key(const uint32_t (&key)[NK], uint32_t &kb, int &ib) {
  if constexpr (NK == 1) {
    kb = key[0];
    ib = 0;
  } else {
    uint32_t v[NK / 2];
    int ix[NK / 2];
#pragma unroll
    for (int i = 0; i < NK / 2; ++i) {
      const bool r = key[2 * i + 1] > key[2 * i];
      v[i] = r ? key[2 * i + 1] : key[2 * i];
      ix[i] = r ? 2 * i + 1 : 2 * i;
    }
#pragma unroll
    for (int n = NK / 4; n >= 1; n >>= 1) {
#pragma unroll
      for (int i = 0; i < n; ++i) {  // in place: node i reads 2i and 2i + 1, both >= i
        const bool r = v[2 * i + 1] > v[2 * i];
        v[i] = r ? v[2 * i + 1] : v[2 * i];
        ix[i] = r ? ix[2 * i + 1] : ix[2 * i];
      }
    }
    kb = v[0];
    ib = ix[0];
  }
}

// The k (<= 32) largest keys of a warp in (key desc, element asc) order, slot i
// of lane l standing for element l + 32 i: lane j returns the element of pick j
// (lanes j >= k return 0).  One round per pick: the largest key by one warp
// reduction, then the smallest element holding it by another; the winning lane
// drops that key and finds its next best.  At least k slots must hold a key above
// 0 (every real element does).  The warp is converged; key[] is consumed.
template <int NK>
__device__ __forceinline__ int warp_top_k(uint32_t (&key)[NK], int k) {
  const int lane = threadIdx.x & 31;
  uint32_t kb;
  int ib;
  lane_best_key<NK>(key, kb, ib);
  int pick = 0;
  for (int j = 0; j < k; ++j) {
    const uint32_t bk = __reduce_max_sync(0xFFFFFFFFu, kb);
    const unsigned cand = kb == bk ? static_cast<unsigned>(lane + 32 * ib) : 0xFFFFFFFFu;
    const unsigned be = __reduce_min_sync(0xFFFFFFFFu, cand);
    if (lane == j) pick = static_cast<int>(be);
    if (static_cast<int>(be & 31u) == lane) {
      const int rm = static_cast<int>(be >> 5);
#pragma unroll
      for (int i = 0; i < NK; ++i)
        if (i == rm) key[i] = 0u;
      lane_best_key<NK>(key, kb, ib);
    }
  }
  return pick;
}

// Routing weights of the k picks held one per lane (lane j: the logit of pick j,
// the first pick holding the largest): exp(l - m) / sum exp(l - m) in double,
// summed by an xor butterfly, then rounded to float; a largest logit of +inf
// splits the weight among the +inf picks, one of -inf gives 1/k.  Lanes j >= k
// return 0.  The warp is converged.
__device__ __forceinline__ float warp_route_weight(float myv, int k) {
  const int lane = threadIdx.x & 31;
  const bool active = lane < k;
  const float mx = __shfl_sync(0xFFFFFFFFu, myv, 0);
  float wj;
  if (mx == -INFINITY) {
    wj = 1.0f / static_cast<float>(k);
  } else if (mx == INFINITY) {
    const int ninf = __popc(__ballot_sync(0xFFFFFFFFu, active && myv == INFINITY));
    wj = (myv == INFINITY) ? 1.0f / static_cast<float>(ninf) : 0.0f;
  } else {
    const double ex = active ? exp(static_cast<double>(myv) - static_cast<double>(mx)) : 0.0;
    double sum = ex;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, off);
    wj = static_cast<float>(ex / sum);
  }
  return active ? wj : 0.0f;
}

}  // namespace k3moe
