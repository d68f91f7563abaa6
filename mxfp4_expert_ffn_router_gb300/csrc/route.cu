// route.cu -- router top-k selection and softmax weights.
//
// Follows the kimi-k3-in-c CHANGELOG walkthrough, "[0.1.0] Added": each MoE
// layer routes a token to 16 of 896 experts; the score is the softmax of the
// router logits renormalised over the selected experts, selection is on the raw
// fp32 logits (exact comparisons), ties go to the lower expert index.
//
// Per token: each logit becomes an order-preserving unsigned key (-0 and +0 the
// same key).  The k picks are ordered by (key descending, index ascending) and
// their weights are exp(l - m) / sum exp(l - m) over the picks, in double.
//  * E <= 1024: one warp per token holds the keys (lane l: experts l, l + 32, ...)
//    and takes the picks by k rounds of a warp arg-max (warp_top_k);
//  * larger E: one block per token; a 32-step bitwise search finds tau, the
//    largest key with at least k keys >= tau (the k-th largest key); every key
//    > tau is selected, and keys equal to tau are selected in index order until
//    k are taken.
// Both give the same picks and weights bit for bit.
#include "k3moe_dev.cuh"
#include "k3moe_launch.h"

namespace k3moe {

namespace {

// Sum of one int per thread over the block (all threads get it).  `buf` holds 32
// ints; consecutive calls must alternate buffers (the second barrier of a call
// is the next call's first).
__device__ __forceinline__ int block_sum(int v, int *buf) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarp = blockDim.x >> 5;
  v = __reduce_add_sync(0xFFFFFFFFu, v);
  if (lane == 0) buf[warp] = v;
  __syncthreads();
  return __reduce_add_sync(0xFFFFFFFFu, lane < nwarp ? buf[lane] : 0);
}

}  // namespace

// PER = logits per thread (E <= PER * blockDim.x); element e = i * blockDim.x + tid.
template <int PER>
__global__ void __launch_bounds__(1024) route_kernel(const float *__restrict__ logits, int T, int E, int k,
                                                     int32_t *__restrict__ idx, float *__restrict__ w,
                                                     int32_t *status) {
  pdl_wait();
  pdl_trigger();
  __shared__ int sbuf[2][32];
  __shared__ int s_n;
  __shared__ uint32_t s_key[32];
  __shared__ int s_e[32];
  __shared__ float s_v[32];
  __shared__ float s_sorted[32];
  const int t = blockIdx.x;
  if (t >= T) return;
  const int tid = threadIdx.x, nth = blockDim.x, lane = tid & 31;
  const float *row = logits + static_cast<size_t>(t) * E;
  int32_t *it = idx + static_cast<size_t>(t) * k;
  float *wt = w + static_cast<size_t>(t) * k;
  uint32_t key[PER];
  float val[PER];
  bool nan_here = false;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int e = i * nth + tid;
    val[i] = 0.f;
    key[i] = 0u;
    if (e < E) {
      val[i] = __ldg(row + e);
      if (val[i] != val[i]) nan_here = true;
      key[i] = order_key(val[i]);
    }
  }
  if (tid == 0) s_n = 0;
  if (__syncthreads_or(nan_here)) {
    if (tid < k) {
      it[tid] = tid;
      wt[tid] = 1.0f / static_cast<float>(k);
    }
    if (tid == 0) set_status(status, K3MOE_DEV_NONFINITE);
    return;
  }
  // tau = the k-th largest key: the largest value with count(key >= tau) >= k
  uint32_t tau = 0u;
  int par = 0;
  for (int b = 31; b >= 0; --b) {
    const uint32_t cand = tau | (1u << b);
    int c = 0;
#pragma unroll
    for (int i = 0; i < PER; ++i) c += key[i] >= cand;
    if (block_sum(c, sbuf[par]) >= k) tau = cand;
    par ^= 1;
  }
  int c_gt = 0;
#pragma unroll
  for (int i = 0; i < PER; ++i) c_gt += key[i] > tau;
  c_gt = block_sum(c_gt, sbuf[par]);
  par ^= 1;
  const int need = k - c_gt;  // ties at tau to take, lowest indices first
  int ties_before = 0;        // ties in earlier rounds (lower indices)
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const bool tie = key[i] == tau && key[i] != 0u;
    const unsigned m = __ballot_sync(0xFFFFFFFFu, tie);
    // exclusive prefix of the per-warp tie counts over the warps of this round
    const int warp = tid >> 5, nwarp = nth >> 5;
    int *buf = sbuf[par];
    par ^= 1;
    if (lane == 0) buf[warp] = __popc(m);
    __syncthreads();
    const int wc = lane < nwarp ? buf[lane] : 0;
    int incl = wc;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
      if (lane >= off) incl += o;
    }
    const int round_total = __shfl_sync(0xFFFFFFFFu, incl, 31);
    const int warp_excl = __shfl_sync(0xFFFFFFFFu, incl - wc, warp);
    const int rank = ties_before + warp_excl + __popc(m & ((1u << lane) - 1u));
    const bool sel = key[i] > tau || (tie && rank < need);
    if (sel) {
      const int slot = atomicAdd(&s_n, 1);
      if (slot < 32) {
        s_key[slot] = key[i];
        s_e[slot] = i * nth + tid;
        s_v[slot] = val[i];
      }
    }
    ties_before += round_total;
  }
  __syncthreads();
  if (tid < k) {  // k picks in shared memory: order by (key desc, index asc)
    const uint32_t mk = s_key[tid];
    const int me = s_e[tid];
    int r = 0;
    for (int j = 0; j < k; ++j) r += (s_key[j] > mk) || (s_key[j] == mk && s_e[j] < me);
    it[r] = me;
    s_sorted[r] = s_v[tid];
  }
  __syncthreads();
  if (tid < 32) {  // weights over the k picks; exp and the normalisation in double
    const float wj = warp_route_weight(lane < k ? s_sorted[lane] : 0.f, k);
    if (lane < k) wt[lane] = wj;
  }
}

// One warp per token, E <= 32 NK: lane l holds the keys of experts l, l + 32, ...
// (0 past E); a row holding a NaN takes experts 0..k-1 with weights 1/k and is
// reported, as in route_kernel.
template <int NK>
__global__ void __launch_bounds__(256) route_warp_kernel(const float *__restrict__ logits, int T, int E, int k,
                                                         int32_t *__restrict__ idx, float *__restrict__ w,
                                                         int32_t *status) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const long long t = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;  // the whole warp
  const float *row = logits + t * E;
  uint32_t key[NK];
  bool nan_here = false;
#pragma unroll
  for (int i = 0; i < NK; ++i) {
    const int e = lane + 32 * i;
    float v = 0.f;
    if (e < E) v = __ldg(row + e);
    nan_here |= e < E && v != v;
    key[i] = e < E ? order_key(v) : 0u;
  }
  int32_t *it = idx + t * k;
  float *wt = w + t * k;
  if (__any_sync(0xFFFFFFFFu, nan_here)) {
    if (lane < k) {
      it[lane] = lane;
      wt[lane] = 1.0f / static_cast<float>(k);
    }
    if (lane == 0) set_status(status, K3MOE_DEV_NONFINITE);
    return;
  }
  const int pick = warp_top_k<NK>(key, k);
  const float wj = warp_route_weight(lane < k ? __ldg(row + pick) : 0.f, k);
  if (lane < k) {
    it[lane] = pick;
    wt[lane] = wj;
  }
}

int launch_route(const k3moe_shape &s, const float *logits, int32_t *idx, float *w,
                 int32_t *status, cudaStream_t st) {
  if (s.T == 0) return 0;
  if (s.E <= 1024) {  // a warp per token, 8 tokens per block
    const dim3 grid(static_cast<unsigned>((s.T + 7) / 8)), block(256);
    const int nk = (s.E + 31) / 32;
    cudaError_t err;
    if (nk <= 1)
      err = launch_pdl(route_warp_kernel<1>, grid, block, 0, st, logits, s.T, s.E, s.k, idx, w, status);
    else if (nk <= 2)
      err = launch_pdl(route_warp_kernel<2>, grid, block, 0, st, logits, s.T, s.E, s.k, idx, w, status);
    else if (nk <= 4)
      err = launch_pdl(route_warp_kernel<4>, grid, block, 0, st, logits, s.T, s.E, s.k, idx, w, status);
    else if (nk <= 8)
      err = launch_pdl(route_warp_kernel<8>, grid, block, 0, st, logits, s.T, s.E, s.k, idx, w, status);
    else if (nk <= 16)
      err = launch_pdl(route_warp_kernel<16>, grid, block, 0, st, logits, s.T, s.E, s.k, idx, w, status);
    else
      err = launch_pdl(route_warp_kernel<32>, grid, block, 0, st, logits, s.T, s.E, s.k, idx, w, status);
    return err == cudaSuccess ? 0 : -1;
  }
  const int nth = s.E >= 1024 ? 1024 : ((s.E + 31) / 32) * 32;
  const int per = (s.E + nth - 1) / nth;  // <= 4 for E <= 4096
  const dim3 grid(s.T), block(nth);
  cudaError_t err;
  if (per == 1)
    err = launch_pdl(route_kernel<1>, grid, block, 0, st, logits, s.T, s.E, s.k, idx, w, status);
  else if (per == 2)
    err = launch_pdl(route_kernel<2>, grid, block, 0, st, logits, s.T, s.E, s.k, idx, w, status);
  else if (per <= 4)
    err = launch_pdl(route_kernel<4>, grid, block, 0, st, logits, s.T, s.E, s.k, idx, w, status);
  else
    return -1;
  return err == cudaSuccess ? 0 : -1;
}

}  // namespace k3moe
