// route.cu -- router top-k selection and softmax weights (one warp per token).
//
// Follows the kimi-k3-in-c CHANGELOG walkthrough, "[0.1.0] Added": each MoE
// layer routes a token to 16 of 896 experts; the score is the softmax of the
// router logits renormalised over the selected experts, selection is on the raw
// fp32 logits (exact comparisons), ties go to the lower expert index.
#include "k3moe_dev.cuh"
#include "k3moe_launch.h"

namespace k3moe {

// PER = logits held per lane (E <= 32 * PER).  Lane l holds experts l + 32 i.
template <int PER>
__global__ void __launch_bounds__(128) route_kernel(const float *__restrict__ logits, int T, int E,
                                                    int k, int32_t *__restrict__ idx,
                                                    float *__restrict__ w, int32_t *status) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 4 + (threadIdx.x >> 5);
  if (t >= T) return;
  const float *row = logits + static_cast<size_t>(t) * E;
  float v[PER];
  bool nan_here = false;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int e = lane + 32 * i;
    v[i] = (e < E) ? __ldg(row + e) : __uint_as_float(0x7FC00000u);  // NaN = not selectable
    if (e < E && v[i] != v[i]) nan_here = true;
  }
  int32_t *it = idx + static_cast<size_t>(t) * k;
  float *wt = w + static_cast<size_t>(t) * k;
  if (__any_sync(0xFFFFFFFFu, nan_here)) {
    if (lane < k) {
      it[lane] = lane;
      wt[lane] = 1.0f / static_cast<float>(k);
    }
    if (lane == 0) set_status(status, K3MOE_DEV_NONFINITE);
    return;
  }
  // k rounds of a warp-wide arg-max over (value desc, index asc).
  float my_v = 0.f;
  int my_e = 0;
  for (int j = 0; j < k; ++j) {
    float bv = 0.f;
    int be = 0x7FFFFFFF;  // "none"
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      // i ascending = expert index ascending, so a strict '>' keeps the lower index on ties
      if (v[i] == v[i] && (be == 0x7FFFFFFF || v[i] > bv)) {
        bv = v[i];
        be = lane + 32 * i;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, off);
      const int oe = __shfl_xor_sync(0xFFFFFFFFu, be, off);
      if (oe != 0x7FFFFFFF && (be == 0x7FFFFFFF || ov > bv || (ov == bv && oe < be))) {
        bv = ov;
        be = oe;
      }
    }
    if ((be & 31) == lane) {  // the owner retires the winner
#pragma unroll
      for (int i = 0; i < PER; ++i)
        if (lane + 32 * i == be) v[i] = __uint_as_float(0x7FC00000u);
    }
    if (lane == j) {
      my_v = bv;
      my_e = be;
    }
  }
  // weights over the k picks; exp and the normalisation in double (exact argument)
  const float m = __shfl_sync(0xFFFFFFFFu, my_v, 0);
  const bool active = lane < k;
  float wj;
  if (m == -INFINITY) {
    wj = 1.0f / static_cast<float>(k);
  } else if (m == INFINITY) {
    const int ninf = __popc(__ballot_sync(0xFFFFFFFFu, active && my_v == INFINITY));
    wj = (my_v == INFINITY) ? 1.0f / static_cast<float>(ninf) : 0.0f;
  } else {
    const double ex = active ? exp(static_cast<double>(my_v) - static_cast<double>(m)) : 0.0;
    double sum = ex;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, off);
    wj = static_cast<float>(ex / sum);
  }
  if (active) {
    it[lane] = my_e;
    wt[lane] = wj;
  }
}

int launch_route(const k3moe_shape &s, const float *logits, int32_t *idx, float *w,
                 int32_t *status, cudaStream_t st) {
  if (s.T == 0) return 0;
  const dim3 grid((s.T + 3) / 4), block(128);
  const int per = (s.E + 31) / 32;
  cudaError_t err;
#define K3_ROUTE_CASE(P)                                                                        \
  if (per <= P)                                                                                 \
    err = launch_pdl(route_kernel<P>, grid, block, 0, st, logits, s.T, s.E, s.k, idx, w, status); \
  else
  K3_ROUTE_CASE(1)
  K3_ROUTE_CASE(2)
  K3_ROUTE_CASE(4)
  K3_ROUTE_CASE(8)
  K3_ROUTE_CASE(16)
  K3_ROUTE_CASE(28)
  K3_ROUTE_CASE(32)
  K3_ROUTE_CASE(64)
  K3_ROUTE_CASE(128)
  return -1;
#undef K3_ROUTE_CASE
  return err == cudaSuccess ? 0 : -1;
}

}  // namespace k3moe
