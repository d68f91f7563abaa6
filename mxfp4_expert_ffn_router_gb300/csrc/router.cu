// router.cu -- the router scores of every expert for every token, the input of
// the top-16-of-896 selection (kimi-k3-in-c CHANGELOG walkthrough, "[0.1.0]
// Added"; article section "01": 16 of 896 experts woken per token).
//
// logits[t][e] = sum_h x[t][h] * wr[e][h] for bf16 x [T][H] and the bf16 router
// matrix wr [E][H], fp32 accumulation of exact products (a bf16 x bf16 product
// is exact in fp32).  The route kernel then selects on these fp32 scores.
//
// Two kernels, by batch size:
//  * router_gemv_kernel (few tokens): one warp per expert row, 16-byte loads of
//    the row (read once per group of up to 8 tokens), x through L1; every lane
//    keeps 8 partial sums per token (one per position in a 16-byte chunk) over
//    its chunks in increasing order, adds them in a fixed tree and the warp
//    reduces with an xor butterfly (every lane ends with the same bits).  The
//    longest chain of roundings is ceil(H / 256) - 1 + 3 + 5.
//  * router_gemm_kernel (token chunks): tcgen05.mma kind::f16 with both bf16
//    operands in shared memory, M = 128 experts, N = 256 tokens, K = 16 per
//    MMA (four per asm block); TMA loads a 128-row x 64-value box of wr and two
//    of x (128-byte swizzle) per stage into a 4-stage ring; the accumulator lives
//    in tensor memory and the epilogue warps write it to logits with one
//    coalesced 128-byte store per token and warp.  Warps 0-3 epilogue
//    (tensor-memory lane quadrant = warp), warp 4 TMA, warp 5 tensor-memory owner
//    and MMA issuer.  256 tokens per tile rather than 128 let each wr box serve
//    twice the tokens: the fills from L2 to shared memory, not the tensor core,
//    bound a tile.
#include <cuda.h>

#include "k3moe_dev.cuh"
#include "k3moe_launch.h"
#include "tc_sm103.cuh"

namespace k3moe {

namespace {

constexpr int kRgWarps = 4;        // warps per GEMV block (one expert row each)
constexpr int kRouterGemmMinT = 64;

// bf16 pairs of a 32-bit word -> fp32 (element 2i in the low half)
__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

}  // namespace

// NT tokens per pass over a row, NL 16-byte loads of the row in flight per lane.
template <int NT, int NL>
__global__ void __launch_bounds__(kRgWarps * 32)
    router_gemv_kernel(const uint16_t *__restrict__ x, const uint16_t *__restrict__ wr, int T, int H, int E,
                       float *__restrict__ logits) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int e = blockIdx.x * kRgWarps + (threadIdx.x >> 5);
  if (e >= E) return;
  const int nch = H / 8;  // 16-byte chunks per row
  const uint4 *row = reinterpret_cast<const uint4 *>(wr + static_cast<size_t>(e) * H);
  for (int t0 = 0; t0 < T; t0 += NT) {
    const int nt = min(NT, T - t0);
    float acc[NT][8];
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[t][q] = 0.f;
    // chunks lane, lane + 32, ... in increasing order, NL loads ahead
    for (int c0 = lane; c0 < nch; c0 += NL * 32) {
      uint4 wv[NL];
#pragma unroll
      for (int j = 0; j < NL; ++j) {
        const int c = c0 + 32 * j;
        wv[j] = c < nch ? ldg_nc_v4(row + c) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int j = 0; j < NL; ++j) {
        const int c = c0 + 32 * j;
        if (c < nch) {
          const uint32_t ww[4] = {wv[j].x, wv[j].y, wv[j].z, wv[j].w};
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            if (t < nt) {
              const uint4 xv = __ldg(reinterpret_cast<const uint4 *>(x + static_cast<size_t>(t0 + t) * H) + c);
              const uint32_t xx[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
              for (int m = 0; m < 4; ++m) {
                acc[t][2 * m] = fmaf(bf_lo(ww[m]), bf_lo(xx[m]), acc[t][2 * m]);
                acc[t][2 * m + 1] = fmaf(bf_hi(ww[m]), bf_hi(xx[m]), acc[t][2 * m + 1]);
              }
            }
          }
        }
      }
    }
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      float v = ((acc[t][0] + acc[t][1]) + (acc[t][2] + acc[t][3])) +
                ((acc[t][4] + acc[t][5]) + (acc[t][6] + acc[t][7]));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
      if (lane == t && t < nt) logits[static_cast<size_t>(t0 + t) * E + e] = v;
    }
  }
}

// ----------------------------------------------------------------------------
namespace {

constexpr int kRmM = 128;   // experts per tile (MMA M, tensor-memory lanes)
constexpr int kRmN = 256;   // tokens per tile (MMA N, accumulator columns)
constexpr int kRmK = 64;    // K per stage: one 128-byte swizzle atom of bf16
constexpr int kRmStages = 4;
constexpr int kRmTileB = 128 * kRmK * 2;    // 16 KiB: one 128-row operand box
constexpr int kRmStageB = 3 * kRmTileB;     // wr box + two x boxes (256 token rows, contiguous)
constexpr int kRmSmem = 1024 + kRmStages * kRmStageB;
constexpr int kRmThreads = 6 * 32;
constexpr int kRmTmaWarp = 4, kRmMmaWarp = 5;
constexpr int kRmTmemCols = kRmN;

// Instruction descriptor, kind::f16 with bf16 A and B, fp32 D, both K-major.
__device__ __forceinline__ uint32_t idesc_bf16(int M, int N) {
  return (1u << 4)                                 // D format: f32
         | (1u << 7)                               // A format: bf16
         | (1u << 10)                              // B format: bf16
         | (static_cast<uint32_t>(N >> 3) << 17)   // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);  // M / 16
}

// The four MMAs of a stage (K = 16 each): both descriptors advance 32 bytes (2 in
// the address field) per MMA; the first accumulates when `acc` is nonzero.
__device__ __forceinline__ void tc_mma4_bf16_ss(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc,
                                                uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t.reg .b64 a1, a2, a3, b1, b2, b3;\n\t"
      "setp.ne.b32 p, %4, 0;\n\tsetp.eq.b32 q, %3, %3;\n\t"
      "add.u64 a1, %1, 2;\n\tadd.u64 a2, %1, 4;\n\tadd.u64 a3, %1, 6;\n\t"
      "add.u64 b1, %2, 2;\n\tadd.u64 b2, %2, 4;\n\tadd.u64 b3, %2, 6;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, q;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a2, b2, %3, q;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], a3, b3, %3, q;\n\t}" ::"r"(tmem_d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

}  // namespace

__global__ void __launch_bounds__(kRmThreads, 1)
    router_gemm_kernel(const __grid_constant__ CUtensorMap amap, const __grid_constant__ CUtensorMap bmap, int T,
                       int H, int E, float *__restrict__ logits, int32_t *status) {
  extern __shared__ __align__(1024) uint8_t rsm_raw[];
  uint8_t *rsm = rsm_raw + ((1024u - (su32(rsm_raw) & 1023u)) & 1023u);
  __shared__ uint64_t full_bar[kRmStages], empty_bar[kRmStages], acc_bar;
  __shared__ uint32_t tmem_holder;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int e0 = blockIdx.x * kRmM, t0 = blockIdx.y * kRmN;
  const int ksteps = (H + kRmK - 1) / kRmK;
  pdl_wait();
  pdl_trigger();
  if (tid == 0) {
    for (int s = 0; s < kRmStages; ++s) {
      mb_init(&full_bar[s], 1);   // producer arrival + the two boxes' bytes
      mb_init(&empty_bar[s], 1);  // tcgen05.commit
    }
    mb_init(&acc_bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kRmMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(&tmem_holder)),
                 "r"(kRmTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_holder;
  bool timeout = false;

  if (warp == kRmTmaWarp) {
    if (lane == 0) {
      int issued = 0;
      for (int ks = 0; ks < ksteps; ++ks) {
        const int s = ks % kRmStages;
        const uint32_t lap = static_cast<uint32_t>(ks / kRmStages);
        if (!mb_wait(&empty_bar[s], (lap & 1u) ^ 1u)) {
          timeout = true;
          break;
        }
        uint8_t *a = rsm + s * kRmStageB;
        mb_arrive_tx(&full_bar[s], kRmStageB);
        tma_load_2d(a, &amap, ks * kRmK, e0, &full_bar[s]);
        tma_load_2d(a + kRmTileB, &bmap, ks * kRmK, t0, &full_bar[s]);
        tma_load_2d(a + 2 * kRmTileB, &bmap, ks * kRmK, t0 + 128, &full_bar[s]);
        issued = ks + 1;
      }
      // drain: every issued copy has landed before this CTA can leave
      for (int ks = issued - kRmStages < 0 ? 0 : issued - kRmStages; ks < issued; ++ks)
        if (!mb_wait(&full_bar[ks % kRmStages], static_cast<uint32_t>(ks / kRmStages) & 1u)) timeout = true;
    }
  } else if (warp == kRmMmaWarp) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(kRmM, kRmN);
      int done = 0;
      for (int ks = 0; ks < ksteps; ++ks) {
        const int s = ks % kRmStages;
        if (!mb_wait(&full_bar[s], static_cast<uint32_t>(ks / kRmStages) & 1u)) {
          timeout = true;
          break;
        }
        tc_fence_after();
        const uint32_t a0 = su32(rsm + s * kRmStageB), b0 = a0 + kRmTileB;
        // K = 16 per MMA: +32 bytes inside the swizzle atom; the 256 token rows of B
        // are the two x boxes, contiguous (8-row atoms of 1024 bytes throughout)
        static_assert(kRmK == 64, "one stage = four MMAs");
        tc_mma4_bf16_ss(tmem, smem_desc_sw128(a0), smem_desc_sw128(b0), idesc, ks > 0 ? 1u : 0u);
        tc_commit(&empty_bar[s]);
        done = ks + 1;
      }
      if (done == ksteps) tc_commit(&acc_bar);
    }
  } else {
    // epilogue: thread = expert row e0 + 32 warp + lane, 16 token columns per load
    const bool ok = mb_wait(&acc_bar, 0);
    if (!ok) timeout = true;
    tc_fence_after();
    const int e = e0 + 32 * warp + lane;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * warp) << 16);
    for (int c0 = 0; ok && c0 < kRmN; c0 += 16) {
      float v[16];
      tc_ld16(lane_addr + c0, v);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int t = t0 + c0 + j;
        if (t < T && e < E) logits[static_cast<size_t>(t) * E + e] = v[j];
      }
    }
  }
  if (timeout) set_status(status, K3MOE_DEV_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  if (warp == kRmMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kRmTmemCols) : "memory");
  }
}

bool router_gemm_supported(const k3moe_shape &s) {
  CUtensorMap probe;
  static int ok = -1;
  if (ok < 0) ok = make_row_map(&probe, reinterpret_cast<void *>(256), 128, 128) ? 1 : 0;
  return ok == 1 && s.H % 8 == 0;
}

int launch_router(const k3moe_shape &s, const uint16_t *x, const uint16_t *wr, float *logits, int32_t *idx,
                  float *w, int32_t *status, cudaStream_t st) {
  if (s.T == 0) return 0;
  if (s.T >= kRouterGemmMinT && router_gemm_supported(s)) {
    CUtensorMap amap, bmap;
    if (!make_row_map(&amap, const_cast<uint16_t *>(wr), s.E, s.H) ||
        !make_row_map(&bmap, const_cast<uint16_t *>(x), s.T, s.H))
      return -1;
    static bool attr = false;
    if (!attr) {
      if (cudaFuncSetAttribute(router_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kRmSmem) !=
          cudaSuccess)
        return -1;
      attr = true;
    }
    const dim3 grid((s.E + kRmM - 1) / kRmM, (s.T + kRmN - 1) / kRmN);
    if (launch_pdl(router_gemm_kernel, grid, dim3(kRmThreads), kRmSmem, st, amap, bmap, s.T, s.H, s.E, logits,
                   status) != cudaSuccess)
      return -1;
  } else {
    const dim3 grid((s.E + kRgWarps - 1) / kRgWarps), block(kRgWarps * 32);
    const cudaError_t err =
        s.T <= 2 ? launch_pdl(router_gemv_kernel<2, 8>, grid, block, 0, st, x, wr, s.T, s.H, s.E, logits)
                 : launch_pdl(router_gemv_kernel<8, 4>, grid, block, 0, st, x, wr, s.T, s.H, s.E, logits);
    if (err != cudaSuccess) return -1;
  }
  return launch_route(s, logits, idx, w, status, st);
}

}  // namespace k3moe
