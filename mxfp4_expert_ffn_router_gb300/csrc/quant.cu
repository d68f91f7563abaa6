// quant.cu -- MXFP4 quantisation of bf16 activations (the W4A4 mode's input
// step), one thread per block of 32 values; the rule is in mx_quant.cuh (OCP
// Microscaling Formats v1.0, conversion to MXFP4).
#include "k3moe_dev.cuh"
#include "k3moe_launch.h"
#include "mx_quant.cuh"

namespace k3moe {

// codes: 16 bytes per block (low nibble = even element), scales: one E8M0 byte per block.
__global__ void __launch_bounds__(256)
    quant_mxfp4_kernel(const uint16_t *__restrict__ x, long long nblocks, uint8_t *__restrict__ codes,
                       uint8_t *__restrict__ scales) {
  pdl_wait();
  pdl_trigger();
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long b = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; b < nblocks; b += stride) {
    const uint4 *src = reinterpret_cast<const uint4 *>(x + b * 32);
    float v[32];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 u = src[q];
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        v[8 * q + 2 * m] = __uint_as_float(w[m] << 16);
        v[8 * q + 2 * m + 1] = __uint_as_float(w[m] & 0xFFFF0000u);
      }
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));  // fmaxf skips NaN
    const int e = mx_shared_exp(amax);
    const float inv_x = mx_pow2(-e);
    uint32_t o[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int i = 0; i < 32; ++i) o[i >> 3] |= mx_code(v[i], inv_x) << (4 * (i & 7));
    *reinterpret_cast<uint4 *>(codes + b * 16) = make_uint4(o[0], o[1], o[2], o[3]);
    scales[b] = static_cast<uint8_t>(e + 127);
  }
}

int launch_quantize_mxfp4(long long n, const uint16_t *x, uint8_t *codes, uint8_t *scales, cudaStream_t st) {
  const long long nblocks = n / 32;
  if (nblocks == 0) return 0;
  long long grid = (nblocks + 255) / 256;
  if (grid > 152LL * 16) grid = 152LL * 16;
  return launch_pdl(quant_mxfp4_kernel, dim3(static_cast<unsigned>(grid)), dim3(256), 0, st, x, nblocks, codes,
                    scales) == cudaSuccess
             ? 0
             : -1;
}

}  // namespace k3moe
