// ffn_stream.cu -- STREAM mode: the GEMV mode's arithmetic with the weight rows
// delivered by TMA bulk copies into a shared-memory ring.
//
// The kimi-k3-in-c CHANGELOG walkthrough, "[0.1.0] Added": the matmul consumes
// the packed MXFP4 nibbles directly and never materialises a dequantised
// expert; "[1.0.0] Added": each unique routed expert is fetched once per token
// chunk.  Decoding in registers (cvt e2m1x2 -> f16x2, exact), f16 activations
// after an exact power-of-two prescale, exact products summed in fp32 in the
// GEMV kernels' order (lane c takes the 16-byte chunks c, c + 32, ... of a row;
// per chunk two partial sums over its four words, scaled by the chunk's e8m0
// factor; then an xor butterfly over the warp), so the two modes give bitwise
// the same h and Y.
//
// What differs is how the weight bytes reach the SM.  A register-pipelined warp
// can keep only a few KB in flight; here one producer thread per CTA keeps a
// ring of 17-30 KB stages in flight with cp.async.bulk (1-D TMA) into shared
// memory, completing on per-stage mbarriers, so each SM holds up to ~200 KB of
// weight reads in flight, and 16 consumer warps compute from shared memory.
//
// Kernels of one call (after the GEMV mode's prep kernel):
//   stream_rows<0> unit = (active slot, 4 row pairs): 4 gate rows and their 4 up
//                  rows (contiguous in memory: two bulk copies of codes, two of
//                  scales); warp w of the unit's group computes pair w (gate and
//                  up rows share every activation load) for every token of the
//                  slot and writes h = bf16(silu(g) u) with max |h| per row.
//   gemv_h16       h rows -> prescaled f16 (the GEMV mode's kernel)
//   stream_rows<1> unit = (active slot, 16 rows of W2); warp w of the group
//                  computes 4 rows sharing the activation loads; Y[p][row].
// One CTA per SM, persistent: CTA c takes units c, c + G, ...; its i-th unit goes
// to ring stage i mod S and to consumer group i mod 4 (4 warps), so four units
// are computed at once while the others load.  Every wait is bounded; after a
// timeout the CTA sets K3MOE_DEV_TIMEOUT, stops loading and computing, and waits
// (bounded) for its copies in flight before it exits.
#include <cuda_fp16.h>

#include "k3moe_dev.cuh"
#include "k3moe_launch.h"
#include "tc_sm103.cuh"

namespace k3moe {

namespace {

constexpr int kSCons = 16;                    // consumer warps
constexpr int kSGroups = 4;                   // consumer groups (4 warps each), one unit each
constexpr int kSWarpsPerGroup = kSCons / kSGroups;
constexpr int kSThreads = (kSCons + 1) * 32;  // + the producer warp
constexpr int kSPairs = kSWarpsPerGroup;      // gate/up row pairs per unit (one per warp)
constexpr int kSDnRowsPerWarp = 4;            // down rows per warp
constexpr int kSDnRows = kSWarpsPerGroup * kSDnRowsPerWarp;  // down rows per unit
constexpr int kSRingBudget = 200 * 1024;      // shared memory for the ring
constexpr int kSMaxStages = 12;

__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   su32(dst)),
               "l"(src), "r"(bytes), "r"(su32(bar))
               : "memory");
}

// Bounded wait that also gives up once another warp of the CTA has given up.
__device__ __forceinline__ bool wait_or_abort(uint64_t *b, uint32_t parity, volatile int *abort) {
  for (long long i = 0; i < kSpinTc; ++i) {
    if (mb_try(b, parity)) return true;
    if (*abort) return false;
    if (i > 32) __nanosleep(20);
  }
  *abort = 1;
  return false;
}

// e8m0 byte -> 2^(b-127) (b = 0: 2^-127; 255: NaN), as in the GEMV kernels.
__device__ __forceinline__ float st_e8m0(uint32_t b) { return e8m0_to_f32(b); }

// multiply by 2^p for |p| <= 200 (two exact steps)
__device__ __forceinline__ float st_pow2(float v, int p) {
  const int p1 = p / 2, p2 = p - p1;
  return v * exp2i(p1) * exp2i(p2);
}

// The lane's share of R rows . one activation row: chunks c = lane + 32 j
// (c < nch, increasing j), codes of row r at crow + r * cstride and its scale
// bytes at srow + r * sstride (shared or global memory); the activation row
// `arow` piece-major (uint4 q * nch + c holds values 32c + 8q .. + 7), each load
// shared by the R rows.  Per chunk two partial sums over its four words, then
// the chunk's e8m0 factor; the warp's xor butterfly sums the lanes.
template <int R, int NCH>
__device__ __forceinline__ void rows_dot(const uint8_t *crow, size_t cstride, const uint8_t *srow, size_t sstride,
                                         const uint4 *arow, int nch, int lane, float (&acc)[R]) {
  const int n = NCH > 0 ? NCH : nch;
#pragma unroll
  for (int r = 0; r < R; ++r) acc[r] = 0.f;
#pragma unroll(NCH > 0 ? NCH / 32 : 1)
  for (int c = lane; c < n; c += 32) {
    uint4 cw[R];
    uint32_t sb[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      cw[r] = *reinterpret_cast<const uint4 *>(crow + r * cstride + 16 * c);
      sb[r] = srow[r * sstride + c];
    }
    float d0[R], d1[R];
#pragma unroll
    for (int r = 0; r < R; ++r) d0[r] = d1[r] = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 xv = __ldg(arow + q * n + c);
#pragma unroll
      for (int r = 0; r < R; ++r) {
        uint32_t wh[4];
        const uint32_t word = q == 0 ? cw[r].x : q == 1 ? cw[r].y : q == 2 ? cw[r].z : cw[r].w;
        e2m1x8_to_f16x2(word, wh);
        d0[r] = fma2_f16_f32(wh[0], xv.x, d0[r]);
        d1[r] = fma2_f16_f32(wh[1], xv.y, d1[r]);
        d0[r] = fma2_f16_f32(wh[2], xv.z, d0[r]);
        d1[r] = fma2_f16_f32(wh[3], xv.w, d1[r]);
      }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) acc[r] = fmaf(d0[r] + d1[r], st_e8m0(sb[r]), acc[r]);
  }
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc[r] += __shfl_xor_sync(0xFFFFFFFFu, acc[r], off);
}

}  // namespace

struct StreamParams {
  k3moe_weights w;
  int H, I, k, A;
  const int32_t *perm;
  const int4 *slots;     // {expert, first bucket position, tokens, present}
  const int32_t *meta;   // [0] = active slots
  const int32_t *aexp;   // prescale exponent: per token (gate/up) or per bucket position (down)
  const uint4 *act;      // x16 [T][H/8] (gate/up) or h16 [A][I/8] (down), piece-major
  uint16_t *hrow;        // gate/up output, bf16 [A][I]
  int32_t *hmax;         // gate/up output, max |h| per bucket position
  float *Y;              // down output, [A][H]
  int32_t *status;
  int stages;
  int stage_bytes;       // codes of the unit's rows, then their scales
};

// KIND 0: gate/up (unit = kSPairs row pairs); KIND 1: down (unit = kSDnRows rows).
// NCH: chunks per row when it is a compile-time shape (224: K = 7168, 64:
// K = 2048), else 0 (guarded loop).
template <int KIND, int NCH>
__global__ void __launch_bounds__(kSThreads, 1) stream_rows_kernel(StreamParams P) {
  extern __shared__ __align__(128) uint8_t ssm[];
  __shared__ uint64_t full_bar[kSMaxStages], empty_bar[kSMaxStages];
  __shared__ int abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int K = KIND == 0 ? P.H : P.I;
  const int nch = K / 32;
  const int cbytes = K / 2, sbytes = K / 32;  // per row
  constexpr int R = KIND == 0 ? 2 * kSPairs : kSDnRows;  // weight rows per unit
  const int S = P.stages;
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mb_init(&full_bar[s], 1);
      mb_init(&empty_bar[s], kSWarpsPerGroup);
    }
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  const int per_slot = KIND == 0 ? P.I / kSPairs : P.H / kSDnRows;
  const long long nunits = static_cast<long long>(P.meta[0]) * per_slot;
  volatile int *abort = &abort_flag;
  bool timeout = false;

  if (warp == kSCons) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      long long issued = 0;
      for (long long u = blockIdx.x; u < nunits; u += gridDim.x, ++issued) {
        const int s = static_cast<int>(issued % S);
        const uint32_t lap = static_cast<uint32_t>(issued / S);
        if (!wait_or_abort(&empty_bar[s], (lap & 1u) ^ 1u, abort)) {
          timeout = true;
          break;
        }
        const int4 sl = __ldg(P.slots + static_cast<int>(u / per_slot));
        const int rb = static_cast<int>(u % per_slot);
        uint8_t *stage = ssm + static_cast<size_t>(s) * P.stage_bytes;
        if (!sl.w) {
          mb_arrive_tx(&full_bar[s], 0u);
          continue;
        }
        const uint8_t *cb = KIND == 0 ? P.w.w13_codes[sl.x] : P.w.w2_codes[sl.x];
        const uint8_t *sb = KIND == 0 ? P.w.w13_scales[sl.x] : P.w.w2_scales[sl.x];
        const bool sbulk = (reinterpret_cast<uintptr_t>(sb) & 15u) == 0;
        const uint32_t codes = static_cast<uint32_t>(R) * cbytes;
        const uint32_t scal = sbulk ? static_cast<uint32_t>(R) * sbytes : 0u;
        mb_arrive_tx(&full_bar[s], codes + scal);
        if (KIND == 0) {  // the unit's gate rows, then their up rows
          const size_t g0 = static_cast<size_t>(rb) * kSPairs, u0 = static_cast<size_t>(P.I) + g0;
          bulk_g2s(stage, cb + g0 * cbytes, codes / 2, &full_bar[s]);
          bulk_g2s(stage + codes / 2, cb + u0 * cbytes, codes / 2, &full_bar[s]);
          if (sbulk) {
            bulk_g2s(stage + codes, sb + g0 * sbytes, scal / 2, &full_bar[s]);
            bulk_g2s(stage + codes + scal / 2, sb + u0 * sbytes, scal / 2, &full_bar[s]);
          }
        } else {
          const size_t r0 = static_cast<size_t>(rb) * kSDnRows;
          bulk_g2s(stage, cb + r0 * cbytes, codes, &full_bar[s]);
          if (sbulk) bulk_g2s(stage + codes, sb + r0 * sbytes, scal, &full_bar[s]);
        }
      }
      // every copy issued has landed before the CTA may leave
      for (long long j = issued > S ? issued - S : 0; j < issued; ++j)
        if (!mb_wait(&full_bar[j % S], static_cast<uint32_t>(j / S) & 1u)) timeout = true;
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int grp = warp / kSWarpsPerGroup, wl = warp % kSWarpsPerGroup;
    long long i = grp;
    for (long long u = blockIdx.x + static_cast<long long>(grp) * gridDim.x; u < nunits;
         u += static_cast<long long>(kSGroups) * gridDim.x, i += kSGroups) {
      const int s = static_cast<int>(i % S);
      const bool ok = wait_or_abort(&full_bar[s], static_cast<uint32_t>(i / S) & 1u, abort);
      if (!ok) {
        timeout = true;
        break;
      }
      const int4 sl = __ldg(P.slots + static_cast<int>(u / per_slot));
      const int rb = static_cast<int>(u % per_slot);
      const bool present = sl.w != 0;
      const uint8_t *stage = ssm + static_cast<size_t>(s) * P.stage_bytes;
      const uint8_t *sbg = nullptr;
      if (present) sbg = KIND == 0 ? P.w.w13_scales[sl.x] : P.w.w2_scales[sl.x];
      const bool sbulk = (reinterpret_cast<uintptr_t>(sbg) & 15u) == 0;
      if (KIND == 0) {
        // pair wl: gate row rb*4 + wl (stage row wl) and its up row (stage row 4 + wl)
        const int gi = rb * kSPairs + wl;
        const uint8_t *crow = stage + static_cast<size_t>(wl) * cbytes;
        const size_t cstride = static_cast<size_t>(kSPairs) * cbytes;
        const uint8_t *srow = sbulk ? stage + static_cast<size_t>(R) * cbytes + static_cast<size_t>(wl) * sbytes
                                    : sbg + static_cast<size_t>(gi) * sbytes;
        const size_t sstride = sbulk ? static_cast<size_t>(kSPairs) * sbytes : static_cast<size_t>(P.I) * sbytes;
        for (int t = 0; t < sl.z; ++t) {
          const int p = sl.y + t;
          const int a = __ldg(P.perm + p);
          const bool aok = a >= 0 && a < P.A;
          if (!aok && lane == 0) set_status(P.status, K3MOE_DEV_BOUNDS);
          const int tok = aok ? a / P.k : 0;
          float hv = 0.f;
          if (present) {
            float acc[2];
            rows_dot<2, NCH>(crow, cstride, srow, sstride, P.act + static_cast<size_t>(tok) * (K / 8), nch, lane,
                             acc);
            const int ex = __ldg(P.aexp + tok);
            const float gg = st_pow2(acc[0], ex), uu = st_pow2(acc[1], ex);
            hv = (gg / (1.0f + expf(-gg))) * uu;
          }
          if (lane == 0) {
            const uint16_t hb = f32_to_bf16_rne(hv);
            P.hrow[static_cast<size_t>(p) * P.I + gi] = hb;
            atomicMax(P.hmax + p, static_cast<int>(__float_as_uint(fabsf(bf16_bits_to_f32(hb)))));
          }
        }
      } else {
        // rows wl*4 .. wl*4 + 3 of the unit
        const int r0 = rb * kSDnRows + wl * kSDnRowsPerWarp;
        const uint8_t *crow = stage + static_cast<size_t>(wl * kSDnRowsPerWarp) * cbytes;
        const uint8_t *srow = sbulk ? stage + static_cast<size_t>(R) * cbytes +
                                          static_cast<size_t>(wl * kSDnRowsPerWarp) * sbytes
                                    : sbg + static_cast<size_t>(r0) * sbytes;
        for (int t = 0; t < sl.z; ++t) {
          const int p = sl.y + t;
          float acc[kSDnRowsPerWarp];
          if (present) {
            rows_dot<kSDnRowsPerWarp, NCH>(crow, cbytes, srow, sbytes, P.act + static_cast<size_t>(p) * (K / 8), nch,
                                           lane, acc);
          }
          const int ex = __ldg(P.aexp + p);
#pragma unroll
          for (int r = 0; r < kSDnRowsPerWarp; ++r)
            if (lane == r) P.Y[static_cast<size_t>(p) * P.H + r0 + r] = present ? st_pow2(acc[r], ex) : 0.f;
        }
      }
      __syncwarp();
      if (lane == 0) mb_arrive(&empty_bar[s]);
    }
  }
  if (timeout) set_status(P.status, K3MOE_DEV_TIMEOUT);
}

// ----------------------------------------------------------------------------
namespace {

int stage_bytes(int rows, int K) { return ((rows * (K / 2 + K / 32)) + 127) & ~127; }

int ring_stages(int sb) {
  const int n = kSRingBudget / sb;
  return n < kSMaxStages ? n : kSMaxStages;
}

template <int KIND, int NCH>
cudaError_t launch_stream_rows(const StreamParams &P, cudaStream_t st) {
  static bool attr = false;
  const int smem = P.stages * P.stage_bytes;
  if (!attr) {
    const cudaError_t e =
        cudaFuncSetAttribute(stream_rows_kernel<KIND, NCH>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSRingBudget);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  return launch_pdl(stream_rows_kernel<KIND, NCH>, dim3(sm_count()), dim3(kSThreads), smem, st, P);
}

}  // namespace

size_t ffn_stream_workspace(const k3moe_shape &s) { return ffn_gemv_workspace(s); }
size_t ffn_stream_h_offset(const k3moe_shape &s) { return ffn_gemv_h_offset(s); }

bool ffn_stream_supported(const k3moe_shape &s) {
  // bulk copies of the scales of 4 rows need (H / 32) * 4 to be a multiple of 16;
  // a unit's rows must fit the ring at least kSGroups + 1 times
  if (s.H % 128 || s.H > 8192 || s.I > 8192) return false;
  return ring_stages(stage_bytes(2 * kSPairs, s.H)) > kSGroups &&
         ring_stages(stage_bytes(kSDnRows, s.I)) > kSGroups;
}

int launch_ffn_stream(const k3moe_shape &s, const uint16_t *x, const k3moe_weights &w,
                      const int32_t *offsets, const int32_t *perm, float *Y, void *ws,
                      int32_t *status, cudaStream_t st) {
  if (s.T == 0) return 0;
  const GemvBufs b = gemv_bufs(s, ws);
  if (launch_gemv_prep(s, x, w, offsets, b, status, st)) return -1;
  StreamParams P;
  P.w = w;
  P.H = s.H;
  P.I = s.I;
  P.k = s.k;
  P.A = s.T * s.k;
  P.perm = perm;
  P.slots = b.slots;
  P.meta = b.meta;
  P.aexp = b.xexp;
  P.act = b.x16;
  P.hrow = b.hrow;
  P.hmax = b.hmax;
  P.Y = Y;
  P.status = status;
  P.stage_bytes = stage_bytes(2 * kSPairs, s.H);
  P.stages = ring_stages(P.stage_bytes);
  const cudaError_t e0 = s.H == 7168 ? launch_stream_rows<0, 224>(P, st) : launch_stream_rows<0, 0>(P, st);
  if (e0 != cudaSuccess) return -1;
  if (launch_gemv_h16(s, b, st)) return -1;
  P.aexp = b.hexp;
  P.act = b.h16;
  P.stage_bytes = stage_bytes(kSDnRows, s.I);
  P.stages = ring_stages(P.stage_bytes);
  const cudaError_t e1 = s.I == 2048 ? launch_stream_rows<1, 64>(P, st) : launch_stream_rows<1, 0>(P, st);
  return e1 == cudaSuccess ? 0 : -1;
}

}  // namespace k3moe
