// combine.cu -- routing-weighted sum of each token's k expert outputs.
//
// out[t] = sum_{j=0..k-1} w[t][j] * Y[inv[t*k+j]], fp32 in increasing j (one
// fixed order, as the kimi-k3-in-c article's section "02" requires of every
// accumulation), then bf16 round-to-nearest-even.  An assignment that the
// bucketing dropped (inv < 0) contributes zero, never unread memory (the
// CHANGELOG walkthrough's "[Unreleased] Fixed").  HBM-bound: 128-bit loads of Y.
#include "k3moe_dev.cuh"
#include "k3moe_launch.h"

namespace k3moe {

// residual (bf16 [T][H] or NULL): the sum is added to it once, after the j loop
// (the residual stream of a stack of MoE layers: x_next = x + MoE(x)).
__global__ void __launch_bounds__(256, 4)
    combine_kernel(const float *__restrict__ Y, const float *__restrict__ w,
                   const int32_t *__restrict__ inv, int T, int H, int k, int A,
                   const uint16_t *residual, uint16_t *out, float *__restrict__ out_f32) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.y;
  const int c4 = blockIdx.x * 256 + threadIdx.x;  // group of 4 columns
  if (t >= T || 4 * c4 >= H) return;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j = 0; j < k; ++j) {
    const int p = inv[t * k + j];
    if (p < 0 || p >= A) continue;
    const float wj = w[t * k + j];
    const float4 y = *reinterpret_cast<const float4 *>(Y + static_cast<size_t>(p) * H + 4 * c4);
    acc.x = fmaf(wj, y.x, acc.x);
    acc.y = fmaf(wj, y.y, acc.y);
    acc.z = fmaf(wj, y.z, acc.z);
    acc.w = fmaf(wj, y.w, acc.w);
  }
  const size_t o = static_cast<size_t>(t) * H + 4 * c4;
  if (residual) {
    const uint2 r = *reinterpret_cast<const uint2 *>(residual + o);
    acc.x += bf16_bits_to_f32(static_cast<uint16_t>(r.x & 0xFFFFu));
    acc.y += bf16_bits_to_f32(static_cast<uint16_t>(r.x >> 16));
    acc.z += bf16_bits_to_f32(static_cast<uint16_t>(r.y & 0xFFFFu));
    acc.w += bf16_bits_to_f32(static_cast<uint16_t>(r.y >> 16));
  }
  if (out_f32) *reinterpret_cast<float4 *>(out_f32 + o) = acc;
  const uint32_t lo = f32_to_bf16_rne(acc.x) | (static_cast<uint32_t>(f32_to_bf16_rne(acc.y)) << 16);
  const uint32_t hi = f32_to_bf16_rne(acc.z) | (static_cast<uint32_t>(f32_to_bf16_rne(acc.w)) << 16);
  *reinterpret_cast<uint2 *>(out + o) = make_uint2(lo, hi);
}

int launch_combine(const k3moe_shape &s, const float *Y, const float *w, const int32_t *inv,
                   const uint16_t *residual, uint16_t *out, float *out_f32, cudaStream_t st) {
  if (s.T == 0) return 0;
  const dim3 grid((s.H / 4 + 255) / 256, s.T), block(256);
  return launch_pdl(combine_kernel, grid, block, 0, st, Y, w, inv, s.T, s.H, s.k, s.T * s.k, residual, out,
                    out_f32) == cudaSuccess
             ? 0
             : -1;
}

}  // namespace k3moe
