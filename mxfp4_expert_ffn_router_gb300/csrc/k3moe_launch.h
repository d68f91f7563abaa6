// k3moe_launch.h -- host-side launch helpers and the internal kernel entry points.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/k3moe.h"

namespace k3moe {

// Shared by every C-ABI entry point (defined in k3moe.cu).
int abi_check_shape(const k3moe_shape &s);  // K3MOE_OK or K3MOE_ERR_SHAPE
int abi_check_arch();                       // K3MOE_OK or K3MOE_ERR_ARCH (current device)
// Status of a launch sequence: rc != 0 or a pending CUDA error gives
// K3MOE_ERR_LAUNCH, with the error consumed and its text kept for
// k3moe_last_cuda_error().
int abi_launched(int rc);

// Launch with programmatic stream serialization, so a kernel's prologue may
// overlap the tail of its predecessor; every kernel calls pdl_wait() before it
// reads anything a predecessor wrote.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

int launch_route(const k3moe_shape &s, const float *logits, int32_t *idx, float *w,
                 int32_t *status, cudaStream_t st);
size_t bucket_workspace(const k3moe_shape &s);
int launch_bucket(const k3moe_shape &s, const int32_t *idx, int32_t *counts, int32_t *offsets,
                  int32_t *perm, int32_t *inv, void *ws, int32_t *status, cudaStream_t st);
size_t ffn_gemv_workspace(const k3moe_shape &s);
size_t ffn_gemv_h_offset(const k3moe_shape &s);
int launch_ffn_gemv(const k3moe_shape &s, const uint16_t *x, const k3moe_weights &w,
                    const int32_t *offsets, const int32_t *perm, float *Y, void *ws,
                    int32_t *status, cudaStream_t st);
// The GEMV mode's workspace pieces, and its front (active slots, x to prescaled
// f16) and middle (h to prescaled f16) kernels.
struct GemvBufs {
  int4 *slots;      // {expert, first bucket position, tokens, present} per active slot
  int32_t *meta;    // [0] = active slots
  int32_t *xexp;    // prescale exponent per token
  uint4 *x16;       // x as prescaled f16, piece-major [T][H/8]
  uint16_t *hrow;   // h, bf16 [A][I] (the rounding point)
  uint4 *h16;       // h as prescaled f16, piece-major [A][I/8]
  int32_t *hexp;    // prescale exponent per bucket position
};
GemvBufs gemv_bufs(const k3moe_shape &s, void *ws);
int launch_gemv_prep(const k3moe_shape &s, const uint16_t *x, const k3moe_weights &w, const int32_t *offsets,
                     const GemvBufs &b, int32_t *status, cudaStream_t st);
int launch_gemv_h16(const k3moe_shape &s, const GemvBufs &b, cudaStream_t st);
int sm_count();
bool layer_front_fits(const k3moe_shape &s);
int launch_layer_gemv_fast(const k3moe_shape &s, const float *logits, const uint16_t *x, const k3moe_weights &w,
                           int32_t *idx, float *wts, int32_t *counts, int32_t *offsets, int32_t *perm, int32_t *inv,
                           float *Y, uint16_t *out, float *out_f32, void *ws, int32_t *status, cudaStream_t st);
size_t ffn_gemm_workspace(const k3moe_shape &s);
size_t ffn_gemm_h_offset(const k3moe_shape &s);
bool ffn_gemm_supported(const k3moe_shape &s);
int launch_ffn_gemm(const k3moe_shape &s, const uint16_t *x, const k3moe_weights &w, const int32_t *offsets,
                    const int32_t *perm, float *Y, void *ws, int32_t *status, cudaStream_t st, bool a4);
// 2-D TMA map over rows x K 16-bit values (row stride 2K bytes, 16-byte aligned
// base): boxes of 64 values x 128 rows, 128-byte swizzle, rows and columns past
// the end read as zero.  False when the driver's encoder is unavailable or refuses.
bool make_row_map(CUtensorMap *m, void *base, int rows, int K);
int launch_router(const k3moe_shape &s, const uint16_t *x, const uint16_t *wr, float *logits, int32_t *idx,
                  float *w, int32_t *status, cudaStream_t st);
bool router_gemm_supported(const k3moe_shape &s);
size_t cache_arena_bytes(const k3moe_shape &s, int slots);
void cache_tables(const k3moe_shape &s, int slots, void *arena, k3moe_weights *out);
int launch_cache_init(const k3moe_shape &s, int slots, void *arena, cudaStream_t st);
int launch_cache_fetch(const k3moe_shape &s, int slots, void *arena, const k3moe_weights &host_w,
                       const int32_t *counts, int cbase, int cn, unsigned long long *stats, int32_t *status,
                       cudaStream_t st);
int launch_quantize_mxfp4(long long n, const uint16_t *x, uint8_t *codes, uint8_t *scales, cudaStream_t st);
int launch_combine(const k3moe_shape &s, const float *Y, const float *w, const int32_t *inv,
                   const uint16_t *residual, uint16_t *out, float *out_f32, cudaStream_t st);

}  // namespace k3moe
