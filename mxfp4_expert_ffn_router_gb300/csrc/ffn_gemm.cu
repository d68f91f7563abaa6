// ffn_gemm.cu -- the MXFP4 expert FFN of token chunks as grouped GEMMs on the
// 5th-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// The kimi-k3-in-c CHANGELOG walkthrough, "[1.0.0] Added" (chunk-union prefill):
// the tokens of a chunk are grouped by routed expert, each unique expert's
// weights are fetched once per chunk, and the result equals the per-token path.
// Here each expert's tokens form the N dimension of two GEMMs:
//   gate/up:  D[2I x n] = W13 (MXFP4 -> bf16, exact) . X_e^T (bf16)   -> h = bf16(silu(g) u)
//   down:     D[H  x n] = W2  (MXFP4 -> bf16, exact) . h_e^T (bf16)   -> Y
// with fp32 accumulation in tensor memory (kind::f16, bf16 operands).  The
// dequantisation e2m1 * 2^(s-127) -> bf16 is exact for every finite scale, so
// the GEMMs compute the same products as the CUDA-core path, summed in another
// (fixed) order.
//
// One CTA (4 warps) per tile (active expert, 128 weight rows, <= 128 tokens).
// Per K step of 64: all threads dequantise the weight tile and gather the token
// tile into a 128B-swizzled K-major shared-memory stage; thread 0 issues four
// tcgen05.mma (K = 16 each) and commits them to the stage's mbarrier; the next
// stage is filled while the tensor core works (two stages).  The epilogue reads
// the accumulator with tcgen05.ld and writes h (bf16) or Y (fp32) rows through
// shared memory so the global stores are coalesced.
#include <cuda_fp16.h>
#include <cuda_bf16.h>

#include "k3moe_dev.cuh"
#include "k3moe_launch.h"

namespace k3moe {

namespace {

constexpr int kThreadsG = 128;  // 4 warps: all load/dequantise, thread 0 issues MMAs
constexpr int kTileM = 128;     // weight rows per tile
constexpr int kTileN = 128;     // tokens per tile (max)
constexpr int kTileK = 64;      // K per stage: one 128-byte swizzle atom of bf16
constexpr int kStagesG = 2;
constexpr int kStageA = kTileM * kTileK * 2;  // 16 KiB
constexpr int kStageB = kTileN * kTileK * 2;  // 16 KiB
constexpr long long kSpinG = 1LL << 22;

__device__ __forceinline__ uint32_t su32(const void *p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

// ---- mbarrier ----
__device__ __forceinline__ void mb_init(uint64_t *b, uint32_t n) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(n) : "memory");
}
__device__ __forceinline__ bool mb_try(uint64_t *b, uint32_t parity) {
  uint32_t ok;
  asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
               : "=r"(ok)
               : "r"(su32(b)), "r"(parity)
               : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mb_wait(uint64_t *b, uint32_t parity) {
  for (long long i = 0; i < kSpinG; ++i) {
    if (mb_try(b, parity)) return true;
    if (i > 32) __nanosleep(20);
  }
  return false;
}

// ---- tcgen05 ----
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row atoms of
// 1024 bytes (stride byte offset 1024), descriptor version 1.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFF) >> 4);       // start address
  d |= static_cast<uint64_t>(1) << 16;                      // leading byte offset (unused for SW128 K-major)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;              // stride byte offset
  d |= static_cast<uint64_t>(1) << 46;                      // version
  d |= static_cast<uint64_t>(2) << 61;                      // SWIZZLE_128B
  return d;
}

// Instruction descriptor, kind::f16: bf16 A and B, fp32 accumulator, both K-major.
__device__ __forceinline__ uint32_t idesc_bf16(int M, int N) {
  return (1u << 4)                                   // D format: f32
         | (1u << 7)                                 // A format: bf16
         | (1u << 10)                                // B format: bf16
         | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);    // M / 16
}

__device__ __forceinline__ void tc_mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(bar))
               : "memory");
}
// 32 lanes x 32 bit, 16 consecutive columns per thread.
__device__ __forceinline__ void tc_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Byte offset of 16-byte chunk c (0..7) of row r in a 128B-swizzled K-major tile.
__device__ __forceinline__ uint32_t sw128_off(int r, int c) {
  return static_cast<uint32_t>((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

// e2m1 pair byte -> two bf16 (packed) times 2^(s-127), exact.
__device__ __forceinline__ uint32_t e2m1x2_to_bf16x2_scaled(uint32_t f16x2, float scale) {
  const __half2 h = *reinterpret_cast<const __half2 *>(&f16x2);
  const float2 f = __half22float2(h);
  const __nv_bfloat162 b = __floats2bfloat162_rn(f.x * scale, f.y * scale);
  return *reinterpret_cast<const uint32_t *>(&b);
}

struct GemmTile {
  int kind;  // 0 gate/up, 1 down
  int u, e, p0, n, m0;  // active slot, expert, first bucket position, tokens, first weight row of the tile
};

// Tile t -> (u, token tile, row tile) by binary search over the per-slot inclusive prefix.
__device__ __forceinline__ bool decode_tile(const int32_t *pref, const int32_t *active, const int32_t *slot_p0,
                                            const int32_t *slot_cnt, int na, int mtiles, int tile, GemmTile &g) {
  if (na <= 0 || tile >= pref[na - 1]) return false;
  int lo = 0, hi = na - 1;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (pref[mid] > tile) hi = mid; else lo = mid + 1;
  }
  const int local = tile - (lo ? pref[lo - 1] : 0);
  const int nt = local / mtiles, mt = local % mtiles;
  g.u = lo;
  g.e = active[lo];
  g.p0 = slot_p0[lo] + nt * kTileN;
  g.n = min(kTileN, slot_cnt[lo] - nt * kTileN);
  g.m0 = mt * kTileM;
  return true;
}

struct GemmWs {
  size_t active, meta, sp0, scnt, pref_gu, pref_dn, hrow, total;
};
__host__ __device__ inline size_t g256(size_t v) { return (v + 255) & ~size_t(255); }
__host__ __device__ inline GemmWs gemm_ws(int T, int H, int I, int E, int k) {
  GemmWs w;
  const size_t A = static_cast<size_t>(T) * k;
  size_t o = 0;
  w.active = o;  o = g256(o + sizeof(int32_t) * E);
  w.meta = o;    o = g256(o + sizeof(int32_t) * 4);
  w.sp0 = o;     o = g256(o + sizeof(int32_t) * E);
  w.scnt = o;    o = g256(o + sizeof(int32_t) * E);
  w.pref_gu = o; o = g256(o + sizeof(int32_t) * E);
  w.pref_dn = o; o = g256(o + sizeof(int32_t) * E);
  w.hrow = o;    o = g256(o + sizeof(uint16_t) * A * I);
  w.total = o;
  return w;
}

}  // namespace

// ----------------------------------------------------------------------------
// prep: active experts, their token counts and the tile prefix of both GEMMs.
__global__ void __launch_bounds__(32)
    gemm_prep_kernel(const int32_t *__restrict__ offsets, int E, int A, int mt_gu, int mt_dn,
                     int32_t *__restrict__ active, int32_t *__restrict__ meta, int32_t *__restrict__ slot_p0,
                     int32_t *__restrict__ slot_cnt, int32_t *__restrict__ pref_gu, int32_t *__restrict__ pref_dn,
                     int32_t *status) {
  pdl_wait();
  const int lane = threadIdx.x;
  bool bad = offsets[0] != 0 || offsets[E] > A;
  int run = 0, sg = 0, sd = 0;
  for (int base = 0; base < E; base += 32) {
    const int e = base + lane;
    int cnt = 0;
    if (e < E) {
      cnt = offsets[e + 1] - offsets[e];
      if (cnt < 0) bad = true;
    }
    bad = __any_sync(0xFFFFFFFFu, bad);
    const bool f = cnt > 0 && !bad;
    const unsigned m = __ballot_sync(0xFFFFFFFFu, f);
    const int ntl = f ? (cnt + kTileN - 1) / kTileN : 0;
    int g = ntl * mt_gu, d = ntl * mt_dn;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int og = __shfl_up_sync(0xFFFFFFFFu, g, off), od = __shfl_up_sync(0xFFFFFFFFu, d, off);
      if (lane >= off) { g += og; d += od; }
    }
    if (f) {
      const int slot = run + __popc(m & ((1u << lane) - 1u));
      active[slot] = e;
      slot_p0[slot] = offsets[e];
      slot_cnt[slot] = cnt;
      pref_gu[slot] = sg + g;
      pref_dn[slot] = sd + d;
    }
    run += __popc(m);
    sg += __shfl_sync(0xFFFFFFFFu, g, 31);
    sd += __shfl_sync(0xFFFFFFFFu, d, 31);
  }
  if (lane == 0) {
    meta[0] = bad ? 0 : run;
    meta[1] = bad ? 0 : sg;
    meta[2] = bad ? 0 : sd;
    if (bad) set_status(status, K3MOE_DEV_BOUNDS);
  }
}

// ----------------------------------------------------------------------------
struct GemmParams {
  k3moe_weights w;
  int T, H, I, E, k, A;
  const int32_t *perm;
  const uint16_t *x;          // [T][H] bf16
  const int32_t *active, *meta, *slot_p0, *slot_cnt, *pref;
  uint16_t *hrow;             // [A][I] bf16 (gate/up output, down input)
  float *Y;                   // [A][H]
  int kind;                   // 0 gate/up, 1 down
  int32_t *status;
};

// dynamic shared memory: 1024 bytes of alignment slack, then max(stages, epilogue transpose buffer)
constexpr int kEpiBytes = kTileN * (kTileM + 1) * 4;
constexpr int kGemmSmem = 1024 + (kStagesG * (kStageA + kStageB) > kEpiBytes ? kStagesG * (kStageA + kStageB)
                                                                                 : kEpiBytes);

__global__ void __launch_bounds__(kThreadsG, 1) ffn_gemm_kernel(GemmParams P) {
  extern __shared__ __align__(1024) uint8_t gsm_raw[];
  // the 128B-swizzle atoms need 1024-byte aligned shared addresses: align explicitly
  uint8_t *gsm = gsm_raw + ((1024u - (su32(gsm_raw) & 1023u)) & 1023u);
  // stage s: A tile at gsm + s * (kStageA + kStageB), B tile right after (both 1024-aligned)
  __shared__ uint64_t mma_done[kStagesG];
  __shared__ uint32_t tmem_holder;
  __shared__ int tok_of_row[kTileN];
  const int tid = threadIdx.x, warp = tid >> 5;
  pdl_wait();
  pdl_trigger();

  const int kind = P.kind;
  const int K = kind == 0 ? P.H : P.I;          // reduction length
  const int mtiles = kind == 0 ? (2 * P.I) / kTileM : P.H / kTileM;
  GemmTile g;
  const int na = P.meta[0];
  if (!decode_tile(P.pref, P.active, P.slot_p0, P.slot_cnt, na, mtiles, blockIdx.x, g)) return;
  const int Npad = (g.n + 15) & ~15;  // MMA N: multiple of 16

  const uint8_t *codes, *scales;
  const uintptr_t al = reinterpret_cast<uintptr_t>(P.w.w13_codes[g.e]) | reinterpret_cast<uintptr_t>(P.w.w2_codes[g.e]);
  const bool present = P.w.w13_codes[g.e] && P.w.w13_scales[g.e] && P.w.w2_codes[g.e] && P.w.w2_scales[g.e] &&
                       (al & 15u) == 0;  // 16-byte code loads
  codes = kind == 0 ? P.w.w13_codes[g.e] : P.w.w2_codes[g.e];
  scales = kind == 0 ? P.w.w13_scales[g.e] : P.w.w2_scales[g.e];

  // token rows of this tile (gate/up gathers x rows by token id; down reads h rows in bucket order)
  for (int i = tid; i < kTileN; i += kThreadsG) {
    int t = -1;
    if (i < g.n) {
      const int p = g.p0 + i;
      if (kind == 0) {
        const int a = P.perm[p];
        t = (a >= 0 && a < P.A) ? a / P.k : -1;
        if (t < 0) set_status(P.status, K3MOE_DEV_BOUNDS);
      } else {
        t = p;
      }
    }
    tok_of_row[i] = t;
  }
  if (tid == 0) {
    for (int s = 0; s < kStagesG; ++s) mb_init(&mma_done[s], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {  // tensor memory: 128 lanes x 128 fp32 columns
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(&tmem_holder)),
                 "r"(kTileN)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_holder;
  const uint32_t idesc = idesc_bf16(kTileM, Npad);
  const int ksteps = K / kTileK;
  const int kbytes = K / 2, sbytes = K / 32;
  bool timeout = false;

  // Weight row held by tile row r: gate/up interleaves gate row i (even r) and
  // up row i (odd r) so the epilogue pairs g and u in neighbouring lanes.
  const int tile_row = tid;  // each thread fills one A row per stage
  int wrow;
  if (kind == 0) {
    const int i = (g.m0 >> 1) + (tile_row >> 1);
    wrow = (tile_row & 1) ? P.I + i : i;
  } else {
    wrow = g.m0 + tile_row;
  }

  for (int ks = 0; ks < ksteps; ++ks) {
    const int s = ks % kStagesG;
    uint8_t *sa = gsm + s * (kStageA + kStageB);
    uint8_t *sb = sa + kStageA;
    if (ks >= kStagesG) {  // the MMAs that last read this stage are done
      if (!mb_wait(&mma_done[s], static_cast<uint32_t>((ks / kStagesG) - 1) & 1u)) timeout = true;
      tc_fence_after();
    }
    // A: weight row `wrow`, columns ks*64 .. +63 -> bf16, exact
    {
      uint4 c0 = make_uint4(0, 0, 0, 0), c1 = make_uint4(0, 0, 0, 0);
      float s0 = 0.f, s1 = 0.f;
      if (present) {
        const uint8_t *rp = codes + static_cast<size_t>(wrow) * kbytes + ks * 32;
        c0 = *reinterpret_cast<const uint4 *>(rp);
        c1 = *reinterpret_cast<const uint4 *>(rp + 16);
        const uint8_t *sp = scales + static_cast<size_t>(wrow) * sbytes + ks * 2;
        s0 = e8m0_to_f32(sp[0]);
        s1 = e8m0_to_f32(sp[1]);
      }
      const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
      for (int c = 0; c < 8; ++c) {  // 16-byte chunk c = columns 8c .. 8c+7 of the 64
        uint32_t h[4];
        e2m1x8_to_f16x2(words[c], h);
        const float sc = c < 4 ? s0 : s1;
        uint4 o;
        o.x = e2m1x2_to_bf16x2_scaled(h[0], sc);
        o.y = e2m1x2_to_bf16x2_scaled(h[1], sc);
        o.z = e2m1x2_to_bf16x2_scaled(h[2], sc);
        o.w = e2m1x2_to_bf16x2_scaled(h[3], sc);
        *reinterpret_cast<uint4 *>(sa + sw128_off(tile_row, c)) = o;
      }
    }
    // B: token rows, columns ks*64 .. +63 (bf16), zero for padding rows
    for (int i = tid; i < kTileN * 8; i += kThreadsG) {
      const int r = i >> 3, c = i & 7;
      uint4 v = make_uint4(0, 0, 0, 0);
      const int t = tok_of_row[r];
      if (t >= 0) {
        const uint16_t *src = kind == 0 ? P.x + static_cast<size_t>(t) * P.H : P.hrow + static_cast<size_t>(t) * P.I;
        v = *reinterpret_cast<const uint4 *>(src + ks * kTileK + c * 8);
      }
      *reinterpret_cast<uint4 *>(sb + sw128_off(r, c)) = v;
    }
    // make the generic-proxy stores visible to the tensor core, then issue
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
      const uint32_t a0 = su32(sa), b0 = su32(sb);
#pragma unroll
      for (int kk = 0; kk < kTileK / 16; ++kk)  // K = 16 per MMA: +32 bytes inside the swizzle atom
        tc_mma_bf16(tmem, smem_desc_sw128(a0 + kk * 32), smem_desc_sw128(b0 + kk * 32), idesc,
                    (ks > 0 || kk > 0) ? 1u : 0u);
      tc_commit(&mma_done[s]);
    }
  }
  // wait for the last MMAs
  {
    const int last = ksteps - 1;
    if (!mb_wait(&mma_done[last % kStagesG], static_cast<uint32_t>(last / kStagesG) & 1u)) timeout = true;
    tc_fence_after();
  }
  if (timeout) set_status(P.status, K3MOE_DEV_TIMEOUT);

  // ---- epilogue: thread tid holds tile row tid (TMEM lane tid), columns 0..Npad-1
  float *stage = reinterpret_cast<float *>(gsm);  // [kTileN][kTileM + 1] fp32 transpose buffer (fits in stage 0+1)
  const uint32_t lane_addr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
  for (int c0 = 0; c0 < Npad; c0 += 16) {
    float v[16];
    tc_ld16(lane_addr + c0, v);
#pragma unroll
    for (int j = 0; j < 16; ++j) stage[(c0 + j) * (kTileM + 1) + tid] = present ? v[j] : 0.f;
  }
  __syncthreads();
  if (kind == 0) {
    // h[p0 + n][m0/2 + i] = bf16(silu(g) * u), g = row 2i, u = row 2i+1
    const int ncols = kTileM / 2;
    for (int idx = tid; idx < g.n * ncols; idx += kThreadsG) {
      const int n = idx / ncols, i = idx % ncols;
      const float gg = stage[n * (kTileM + 1) + 2 * i];
      const float uu = stage[n * (kTileM + 1) + 2 * i + 1];
      const float hv = (gg / (1.0f + expf(-gg))) * uu;
      P.hrow[static_cast<size_t>(g.p0 + n) * P.I + (g.m0 >> 1) + i] = f32_to_bf16_rne(hv);
    }
  } else {
    for (int idx = tid; idx < g.n * kTileM; idx += kThreadsG) {
      const int n = idx / kTileM, r = idx % kTileM;
      P.Y[static_cast<size_t>(g.p0 + n) * P.H + g.m0 + r] = stage[n * (kTileM + 1) + r];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTileN) : "memory");
  }
}

// ----------------------------------------------------------------------------
size_t ffn_gemm_workspace(const k3moe_shape &s) { return gemm_ws(s.T, s.H, s.I, s.E, s.k).total; }

bool ffn_gemm_supported(const k3moe_shape &s) {
  return (2 * s.I) % kTileM == 0 && s.H % kTileM == 0 && s.H % kTileK == 0 && s.I % kTileK == 0;
}

int launch_ffn_gemm(const k3moe_shape &s, const uint16_t *x, const k3moe_weights &w, const int32_t *offsets,
                    const int32_t *perm, float *Y, void *ws, int32_t *status, cudaStream_t st) {
  if (s.T == 0) return 0;
  const GemmWs L = gemm_ws(s.T, s.H, s.I, s.E, s.k);
  char *base = static_cast<char *>(ws);
  const int A = s.T * s.k;
  const int mt_gu = (2 * s.I) / kTileM, mt_dn = s.H / kTileM;
  int32_t *active = reinterpret_cast<int32_t *>(base + L.active);
  int32_t *meta = reinterpret_cast<int32_t *>(base + L.meta);
  int32_t *sp0 = reinterpret_cast<int32_t *>(base + L.sp0);
  int32_t *scnt = reinterpret_cast<int32_t *>(base + L.scnt);
  int32_t *pgu = reinterpret_cast<int32_t *>(base + L.pref_gu);
  int32_t *pdn = reinterpret_cast<int32_t *>(base + L.pref_dn);
  if (launch_pdl(gemm_prep_kernel, dim3(1), dim3(32), 0, st, offsets, s.E, A, mt_gu, mt_dn, active, meta, sp0,
                 scnt, pgu, pdn, status) != cudaSuccess)
    return -1;
  // upper bound of the token tiles: sum_e ceil(n_e / 128) <= A / 128 + min(A, E)
  const long long ntile_max = A / kTileN + (A < s.E ? A : s.E);
  const size_t smem = kGemmSmem;
  if (cudaFuncSetAttribute(ffn_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
      cudaSuccess)
    return -1;
  GemmParams P;
  P.w = w;
  P.T = s.T; P.H = s.H; P.I = s.I; P.E = s.E; P.k = s.k; P.A = A;
  P.perm = perm;
  P.x = x;
  P.active = active;
  P.meta = meta;
  P.slot_p0 = sp0;
  P.slot_cnt = scnt;
  P.hrow = reinterpret_cast<uint16_t *>(base + L.hrow);
  P.Y = Y;
  P.status = status;
  P.kind = 0;
  P.pref = pgu;
  if (launch_pdl(ffn_gemm_kernel, dim3(static_cast<unsigned>(ntile_max * mt_gu)), dim3(kThreadsG), smem, st, P) !=
      cudaSuccess)
    return -1;
  P.kind = 1;
  P.pref = pdn;
  if (launch_pdl(ffn_gemm_kernel, dim3(static_cast<unsigned>(ntile_max * mt_dn)), dim3(kThreadsG), smem, st, P) !=
      cudaSuccess)
    return -1;
  return 0;
}

}  // namespace k3moe
