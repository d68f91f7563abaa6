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
// Operands are f16 (kind::f16, fp32 accumulation):
//  * weights: e2m1 (exact in f16) times 2^(s - s_ref), where s_ref is the
//    largest block-scale byte of the weight row; exact for every block within
//    2^23 of the row's largest (smaller blocks round to f16 subnormals, below
//    2^-24 of the row's scale); the factor 2^(s_ref - 127) is applied in the
//    epilogue, exactly;
//  * activations: x (gate/up) and h (down) as f16 after an exact power-of-two
//    prescale per row (max|v| * 2^-p in [2^14, 2^15)), laid out in bucket order
//    by two small pre-pass kernels so that a 2-D TMA tile load fetches them.
//
// One CTA per tile (active expert, 128 weight rows, <= 128 tokens), 11 warps,
// two CTAs per SM:
//  * warp 8 (TMA, activations): per K step of 128 two boxes of 64 values of the
//    activation tile, as soon as the MMA has released the stage; a box is only
//    as high as the tile's tokens rounded up to 16 (one tensor map per height),
//    not 128 rows, which cuts the L2-to-shared-memory traffic of a prefill tile
//    (about 73 tokens per expert) by about a third;
//  * warp 9 (TMA, weights): per weight stage (256 K values) two 2-D boxes of
//    weight codes, 64 rows x 128 bytes each, 128B-swizzled, through the expert's
//    tensor map (built on the device by gemm_sched_kernel), as soon as the
//    dequantising warps have released the stage.  The two rings have their own
//    producers so that an activation load never waits for a weight stage to
//    drain (with one producer thread every activation tile, and its L2 latency,
//    joined the chain from one K step to the next);
//  * warps 0-7 (dequantisation): thread = one weight row (tensor-memory lane)
//    and one K half; reads 2 x 16 code bytes from shared memory, converts e2m1
//    pairs to f16, multiplies by 2^(s - s_ref) and stores the 128 x 128 A stage
//    to tensor memory with tcgen05.st; one mbarrier arrival per warp and stage;
//  * warp 10 (MMA): owns tensor memory, issues tcgen05.mma kind::f16 with A from
//    tensor memory and B (activations) from shared memory, M=128, K=16 each
//    (8 per stage, four per asm block: the issuing thread shares its scheduler
//    with dequantising warps, so each instruction it spends per MMA shows), and
//    commits every stage back to the producers.
// A K step of 128 rather than 64 halves the waits, arrivals and commits per MMA:
// on the issuing thread one satisfied wait plus one commit cost about as much as
// two MMAs.  Two A/activation stages and two weight stages.  The epilogue (warps 0-7)
// reads the accumulator with tcgen05.ld and writes h (bf16, the fixed rounding
// point) or Y (fp32) rows through shared memory.
#include <cuda.h>

#include <algorithm>
#include <cuda_fp16.h>
#include <cuda_bf16.h>

#include "k3moe_dev.cuh"
#include "k3moe_launch.h"
#include "mx_quant.cuh"
#include "tc_sm103.cuh"

namespace k3moe {

namespace {

constexpr int kDqWarps = 8;                     // dequantisation + epilogue warps
constexpr int kTmaWarp = kDqWarps;              // activation-tile TMA producer
constexpr int kWTmaWarp = kDqWarps + 1;         // weight-code TMA producer
constexpr int kMmaWarp = kDqWarps + 2;          // tensor-memory owner, MMA issuer
constexpr int kThreadsG = (kDqWarps + 3) * 32;  // 352
constexpr int kTileM = 128;     // weight rows per tile
constexpr int kTileN = 128;     // tokens per tile (max)
constexpr int kTileK = 128;     // K per stage: two 128-byte swizzle atoms of 16-bit values
constexpr int kBoxK = 64;       // K of one activation box (one 128-byte swizzle atom)
constexpr int kStagesG = 2;
constexpr int kStageB = kTileN * kTileK * 2;  // 32 KiB of shared memory per stage (activation tile)
constexpr int kBoxB = kTileN * kBoxK * 2;     // 16 KiB: one box of the stage
constexpr int kAcols = kTileK / 2;             // tensor-memory columns of one A stage (f16 pairs)
constexpr int kTmemCols = 256;                 // accumulator (kTileN columns) + kStagesG A stages
// weight codes reach shared memory by 2-D TMA boxes of 128 code bytes (256 K
// values) x 64 rows, 128-byte swizzled: 16-byte chunk c of tile row r sits at
// r * 128 + 16 * (c ^ (r % 8)), so the reads of 8 consecutive rows hit distinct banks
constexpr int kWK = 256;
constexpr int kWSteps = kWK / kTileK;           // MMA K steps per weight stage
constexpr int kWStages = 2;
constexpr int kWBoxRows = 64;
constexpr int kWStageB = kTileM * (kWK / 2);    // 16 KiB
constexpr int kMapBytes = 128;                  // one CUtensorMap
constexpr long long kSpinG = kSpinTc;

// 2-D TMA prefetch of one box into L2 (no shared memory, no completion).
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap *map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void prefetch_l2(const void *p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<uint64_t>(p)));
}
// ---- tcgen05 ----
// Instruction descriptor, kind::f16: f16 A and B, fp32 accumulator, both K-major.
__device__ __forceinline__ uint32_t idesc_f16(int M, int N) {
  return (1u << 4)                                   // D format: f32
         | (0u << 7)                                 // A format: f16
         | (0u << 10)                                // B format: f16
         | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);    // M / 16
}

// A operand from tensor memory (M lanes x K/2 columns of f16 pairs), B from shared memory:
// four MMAs over one 64-value box of the B stage (K = 16 each): A columns a,
// a + 8, a + 16, a + 24 and B descriptors b, b + 2, b + 4, b + 6 (32 bytes
// further each, in the descriptor's address field).  The first accumulates
// when `acc` is nonzero, the other three always.  One asm block keeps the
// issuing thread to about three instructions per MMA: it shares its scheduler
// with busy dequantisation warps, so every instruction it issues costs cycles.
__device__ __forceinline__ void tc_mma4_f16_ta(uint32_t tmem_d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t.reg .b32 a1, a2, a3;\n\t.reg .b64 b1, b2, b3;\n\t"
      "setp.ne.b32 p, %4, 0;\n\tsetp.eq.b32 q, %3, %3;\n\t"
      "add.u32 a1, %1, 8;\n\tadd.u32 a2, %1, 16;\n\tadd.u32 a3, %1, 24;\n\t"
      "add.u64 b1, %2, 2;\n\tadd.u64 b2, %2, 4;\n\tadd.u64 b3, %2, 6;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, q;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a2], b2, %3, q;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a3], b3, %3, q;\n\t}" ::"r"(tmem_d),
      "r"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
// 32 lanes x 32 bit, 16 consecutive columns per thread, registers -> tensor memory;
// completion is awaited by a later tc_st16 (tcgen05.wait::st covers every earlier store).
__device__ __forceinline__ void tc_st16_issue(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
// 32 lanes x 32 bit, 16 consecutive columns per thread, registers -> tensor memory.
__device__ __forceinline__ void tc_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}


// multiply by 2^p for |p| <= 252 (two exact steps)
__device__ __forceinline__ float mul_pow2(float v, int p) {
  const int p1 = p / 2, p2 = p - p1;
  return v * exp2i(p1) * exp2i(p2);
}

// Power-of-two exponent p such that max_abs * 2^-p lies in [2^14, 2^15); 0 for 0.
__device__ __forceinline__ int prescale_exp16(float max_abs) {
  if (!(max_abs > 0.f) || max_abs == INFINITY) return 0;
  int e;
  frexpf(max_abs, &e);
  return max(-100, min(100, (e - 1) - 14));
}

// f16 bit pattern of 2^d for d <= 0 (subnormal down to 2^-24, zero below).
__device__ __forceinline__ uint32_t f16_pow2_bits(int d) {
  if (d >= -14) return static_cast<uint32_t>(d + 15) << 10;
  if (d >= -24) return 1u << (d + 24);
  return 0u;
}

struct GemmTile {
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
  size_t active, meta, sp0, scnt, pref_gu, pref_dn, maps, tab_gu, tab_dn, xg, xexp, hrow, h16, hexp, xsc, hsc, total;
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
  w.maps = o;    o = g256(o + static_cast<size_t>(kMapBytes) * 2 * E);  // weight-code tensor maps per active slot
  // tile tables: an upper bound of the token tiles, sum_e ceil(n_e / 128) <= A / 128 + min(A, E), times the row tiles
  const size_t ntl = A / kTileN + (A < static_cast<size_t>(E) ? A : static_cast<size_t>(E));
  w.tab_gu = o;  o = g256(o + sizeof(int4) * ntl * ((2 * static_cast<size_t>(I)) / kTileM));
  w.tab_dn = o;  o = g256(o + sizeof(int4) * ntl * (static_cast<size_t>(H) / kTileM));
  w.xg = o;      o = g256(o + sizeof(uint16_t) * A * H);  // x rows in bucket order, prescaled f16
  w.xexp = o;    o = g256(o + sizeof(int32_t) * (A ? A : 1));
  w.hrow = o;    o = g256(o + sizeof(uint16_t) * A * I);  // h, bf16 (the rounding point)
  w.h16 = o;     o = g256(o + sizeof(uint16_t) * A * I);  // h prescaled to f16
  w.hexp = o;    o = g256(o + sizeof(int32_t) * (A ? A : 1));
  w.xsc = o;     o = g256(o + A * (static_cast<size_t>(H) / 32));  // MXFP4 block scales of x (W4A4)
  w.hsc = o;     o = g256(o + A * (static_cast<size_t>(I) / 32));  // MXFP4 block scales of h (W4A4)
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

// Tensor maps of the active experts' weight codes: maps[u] (w13) and
// maps[E + u] (w2) for active slot u, each the host-encoded template with its
// global address replaced by the expert's code pointer.  Experts whose code
// pointers are NULL or not 16-byte aligned keep the template's address; the
// GEMMs treat them as absent and never load through their map.  An expert whose
// four pointers are all given but whose codes are misaligned is reported
// (K3MOE_DEV_BOUNDS), once per map.
//
// The same launch writes the tile tables of both GEMMs: entry t of a table is
// {active slot, expert, first bucket position, (tokens << 16) | row tile} of
// tile t, so that a GEMM CTA finds its tile with one load.
__device__ __forceinline__ void write_tile(const int32_t *pref, const int32_t *active, const int32_t *slot_p0,
                                           const int32_t *slot_cnt, int na, int mtiles, int t, int4 *tab) {
  GemmTile g;
  if (decode_tile(pref, active, slot_p0, slot_cnt, na, mtiles, t, g))
    tab[t] = make_int4(g.u, g.e, g.p0, (g.n << 16) | (g.m0 / kTileM));
}

__global__ void __launch_bounds__(128)
    gemm_sched_kernel(const __grid_constant__ CUtensorMap t13, const __grid_constant__ CUtensorMap t2,
                      k3moe_weights w, const int32_t *__restrict__ active, const int32_t *__restrict__ meta, int E,
                      const int32_t *__restrict__ slot_p0, const int32_t *__restrict__ slot_cnt,
                      const int32_t *__restrict__ pref_gu, const int32_t *__restrict__ pref_dn, int mt_gu, int mt_dn,
                      int4 *__restrict__ tab_gu, int4 *__restrict__ tab_dn, uint8_t *__restrict__ maps,
                      int32_t *status) {
  pdl_wait();
  pdl_trigger();
  const int na = meta[0];
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t < meta[1]) write_tile(pref_gu, active, slot_p0, slot_cnt, na, mt_gu, t, tab_gu);
  if (t < meta[2]) write_tile(pref_dn, active, slot_p0, slot_cnt, na, mt_dn, t, tab_dn);
  if (t >= 2 * na) return;
  const int which = t >= na, u = which ? t - na : t;
  const int e = active[u];
  const uint4 *tmpl = reinterpret_cast<const uint4 *>(which ? &t2 : &t13);
  uint8_t *dst = maps + static_cast<size_t>(which * E + u) * kMapBytes;
  uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
  for (int i = 0; i < kMapBytes / 16; ++i) d4[i] = tmpl[i];
  const uint8_t *codes = which ? w.w2_codes[e] : w.w13_codes[e];
  if (w.w13_codes[e] && w.w13_scales[e] && w.w2_codes[e] && w.w2_scales[e] &&
      ((reinterpret_cast<uintptr_t>(w.w13_codes[e]) | reinterpret_cast<uintptr_t>(w.w2_codes[e])) & 15u) != 0)
    set_status(status, K3MOE_DEV_BOUNDS);
  if (codes && (reinterpret_cast<uintptr_t>(codes) & 15u) == 0)
    asm volatile("tensormap.replace.tile.global_address.global.b1024.b64 [%0], %1;" ::"l"(dst), "l"(codes)
                 : "memory");
  asm volatile("fence.proxy.tensormap::generic.release.gpu;" ::: "memory");
}

// The 8 values of row `s` at columns c .. c+7 (c a multiple of 8; ok = c < K) as
// fp32.  With A4 they are first quantised to MXFP4 and dequantised (exactly):
// the 4 lanes sharing a 32-block (lanes 4j..4j+3 hold its 4 pieces of 8) take
// its largest magnitude with shuffles.  Every lane of the warp must call it.
template <bool A4>
__device__ __forceinline__ void load8_act(const uint16_t *s, int c, bool ok, float (&v)[8]) {
  uint4 u = make_uint4(0, 0, 0, 0);
  if (ok) u = *reinterpret_cast<const uint4 *>(s + c);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    v[2 * m] = __uint_as_float(w[m] << 16);
    v[2 * m + 1] = __uint_as_float(w[m] & 0xFFFF0000u);
  }
  if (A4) {
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
    const int e = mx_shared_exp(amax);
    const float x = mx_pow2(e), inv_x = mx_pow2(-e);
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = mx_value(mx_code(v[i], inv_x), x);
  }
}

// Row p of `dst` (f16) = row of `src` (bf16, K values) times 2^-e, e chosen per
// row so the largest magnitude lands in [2^14, 2^15): exact for bf16 inputs.
// Gate/up: src row = x[perm[p] / k]; down: src row = h[p].  With A4 (the W4A4
// mode) the row is first quantised to MXFP4 and dequantised, per 32-block.
template <bool A4>
__global__ void __launch_bounds__(256)
    gemm_rows_to_f16_kernel(const uint16_t *__restrict__ src, const int32_t *__restrict__ perm, int k, int A,
                            int K, uint16_t *__restrict__ dst, int32_t *__restrict__ exps, int32_t *status) {
  pdl_wait();
  pdl_trigger();
  const int p = blockIdx.x;
  int row = p;
  if (perm) {
    const int a = perm[p];
    row = (a >= 0 && a < A) ? a / k : -1;
    if (row < 0) set_status(status, K3MOE_DEV_BOUNDS);
  }
  uint16_t *d = dst + static_cast<size_t>(p) * K;
  if (row < 0) {
    for (int c = threadIdx.x * 8; c < K; c += 256 * 8) *reinterpret_cast<uint4 *>(d + c) = make_uint4(0, 0, 0, 0);
    if (threadIdx.x == 0) exps[p] = 0;
    return;
  }
  const uint16_t *s = src + static_cast<size_t>(row) * K;
  __shared__ float red[8];
  float mx = 0.f;
  for (int c0 = 0; c0 < K; c0 += 256 * 8) {  // trip count uniform across the block
    const int c = c0 + threadIdx.x * 8;
    float v[8];
    load8_act<A4>(s, c, c < K, v);
#pragma unroll
    for (int i = 0; i < 8; ++i) mx = fmaxf(mx, fabsf(v[i]));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
  __syncthreads();
  mx = red[0];
  for (int i = 1; i < 8; ++i) mx = fmaxf(mx, red[i]);
  const int e = prescale_exp16(mx);
  if (threadIdx.x == 0) exps[p] = e;
  const float sc = mul_pow2(1.0f, -e);
  for (int c0 = 0; c0 < K; c0 += 256 * 8) {
    const int c = c0 + threadIdx.x * 8;
    float v[8];
    load8_act<A4>(s, c, c < K, v);
    uint32_t o[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const __half2 h = __floats2half2_rn(v[2 * m] * sc, v[2 * m + 1] * sc);
      o[m] = *reinterpret_cast<const uint32_t *>(&h);
    }
    if (c < K) *reinterpret_cast<uint4 *>(d + c) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// ----------------------------------------------------------------------------
struct GemmParams {
  k3moe_weights w;
  int H, I, A;
  const int32_t *meta;
  const int4 *tab;            // tile table of this GEMM
  const uint8_t *maps;        // weight-code tensor maps per active slot (w13 at u, w2 at E + u)
  int E;
  const int32_t *bexp;        // per bucket position: prescale exponent of the activation row
  uint16_t *hrow;             // [A][I] bf16 (gate/up output)
  float *Y;                   // [A][H]
  int kind;                   // 0 gate/up, 1 down
  int32_t *status;
};

// Activation-tile maps whose boxes are 16, 32, ..., 128 rows high: a tile loads
// only its expert's tokens (rounded up to 16), not 128 rows.
struct RowMaps {
  CUtensorMap m[kTileN / 16];
};

// dynamic shared memory: 1024 bytes of alignment slack, the activation stages,
// then the weight stages (the epilogue transpose buffer [kTileN][kTileM + 1]
// fp32 reuses them once every stage has been consumed)
constexpr int kEpiBytes = kTileN * (kTileM + 1) * 4;
constexpr int kStageBytes = kStagesG * kStageB + kWStages * kWStageB;
static_assert(kTileN + kStagesG * kAcols <= kTmemCols, "tensor-memory budget");
static_assert(kWStages >= 2 && kTileM == 2 * kWBoxRows, "weight ring");
constexpr int kGemmSmem = 1024 + (kStageBytes > kEpiBytes ? kStageBytes : kEpiBytes);

// weight row of tile row r: a gate/up tile holds gate rows m0/2 + [0, 64) in
// tile rows [0, 64) and the matching up rows I + m0/2 + [0, 64) in [64, 128)
__device__ __forceinline__ int tile_wrow(int kind, int m0, int r, int I) {
  if (kind == 0) return (r < kWBoxRows ? 0 : I - kWBoxRows) + (m0 >> 1) + r;
  return m0 + r;
}

__global__ void __launch_bounds__(kThreadsG, 1)
    ffn_gemm_kernel(const __grid_constant__ RowMaps bmaps, GemmParams P) {
  extern __shared__ __align__(1024) uint8_t gsm_raw[];
  // the 128B-swizzle atoms need 1024-byte aligned shared addresses: align explicitly
  uint8_t *gsm = gsm_raw + ((1024u - (su32(gsm_raw) & 1023u)) & 1023u);
  __shared__ uint64_t full_bar[kStagesG], empty_bar[kStagesG], acc_bar;
  __shared__ uint64_t wfull_bar[kWStages], wempty_bar[kWStages];
  __shared__ uint32_t tmem_holder;
  __shared__ int sref_s[kTileM];  // largest scale byte of each tile row
  __shared__ int smax_s[kTileM];  // partial maxima (second K half)
  __shared__ int bexp_s[kTileN];  // activation prescale exponent of each token column
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_wait();
  pdl_trigger();

  const int kind = P.kind;
  const int K = kind == 0 ? P.H : P.I;  // reduction length
  if (static_cast<int>(blockIdx.x) >= P.meta[1 + kind]) return;
  GemmTile g;
  {
    const int4 te = P.tab[blockIdx.x];
    g.u = te.x;
    g.e = te.y;
    g.p0 = te.z;
    g.n = te.w >> 16;
    g.m0 = (te.w & 0xFFFF) * kTileM;
  }
  const int Npad = (g.n + 15) & ~15;  // MMA N: multiple of 16
  const int ksteps = K / kTileK;

  const uint8_t *c13 = P.w.w13_codes[g.e], *s13 = P.w.w13_scales[g.e];
  const uint8_t *c2 = P.w.w2_codes[g.e], *s2 = P.w.w2_scales[g.e];
  const uintptr_t al = reinterpret_cast<uintptr_t>(c13) | reinterpret_cast<uintptr_t>(c2);
  const bool present = c13 && s13 && c2 && s2 && (al & 15u) == 0;  // TMA needs 16-byte aligned code rows
  const uint8_t *scales = kind == 0 ? s13 : s2;

  if (tid < kTileN) bexp_s[tid] = tid < g.n ? P.bexp[g.p0 + tid] : 0;
  if (tid == 0) {
    for (int s = 0; s < kStagesG; ++s) {
      mb_init(&full_bar[s], kDqWarps + 1);  // one arrival per dequantising warp + the TMA producer
      mb_init(&empty_bar[s], 1);                 // tcgen05.commit
    }
    mb_init(&acc_bar, 1);
    for (int s = 0; s < kWStages; ++s) {
      mb_init(&wfull_bar[s], 1);          // producer arrive + bulk-copy bytes
      mb_init(&wempty_bar[s], kDqWarps);  // one arrival per dequantising warp
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kMmaWarp) {  // tensor memory: accumulator columns [0, 128), A stages after
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(&tmem_holder)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_holder;
  bool timeout = false;

  if (warp < kDqWarps) {
    // ---------------------------------------------------- dequantisation
    // warp w fills tensor-memory lane quadrant w % 4 (tile rows 32(w%4) + lane)
    // for K half w / 4 of each stage; gate/up interleaves gate row i (even tile
    // row) and up row i (odd) so the epilogue pairs g and u.
    const int r = 32 * (warp & 3) + lane, hf = warp >> 2;
    const int wrow = tile_wrow(kind, g.m0, r, P.I);
    const int sbytes = K / 32;
    const uint8_t *srow = present ? scales + static_cast<size_t>(wrow) * sbytes : nullptr;
    // the row's scale bytes come 16 at a time (8 K steps) when the row is 16-byte aligned
    const bool svec = present && (sbytes & 15) == 0 && (reinterpret_cast<uintptr_t>(srow) & 15u) == 0;
    // largest block-scale byte of the row (the two K halves scan alternate
    // 16-byte chunks of the row's scale bytes)
    int smax = 0;
    if (svec) {
      // the thread's 16-byte chunks of scale bytes are loaded 8 at a time, all in
      // flight together (one memory latency per 8 chunks rather than one per chunk),
      // and reduced bytewise
      constexpr int kScanChunks = 8;
      uint32_t m4 = 0;
      for (int b0 = 16 * hf; b0 < sbytes; b0 += 32 * kScanChunks) {
        uint4 v[kScanChunks];
#pragma unroll
        for (int c = 0; c < kScanChunks; ++c)
          v[c] = b0 + 32 * c < sbytes ? *reinterpret_cast<const uint4 *>(srow + b0 + 32 * c) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int c = 0; c < kScanChunks; ++c)
          m4 = __vmaxu4(__vmaxu4(m4, __vmaxu4(v[c].x, v[c].y)), __vmaxu4(v[c].z, v[c].w));
      }
      smax = static_cast<int>(max(max(m4 & 0xFFu, (m4 >> 8) & 0xFFu), max((m4 >> 16) & 0xFFu, m4 >> 24)));
    } else if (present) {
      for (int b = hf; b < sbytes; b += 2) smax = max(smax, static_cast<int>(srow[b]));
    }
    if (hf == 1) smax_s[r] = smax;  // combine the two K halves of the row
    asm volatile("bar.sync 2, %0;" ::"r"(kDqWarps * 32) : "memory");
    if (hf == 0) {
      smax = max(smax, smax_s[r]);
      sref_s[r] = smax;
    }
    asm volatile("bar.sync 2, %0;" ::"r"(kDqWarps * 32) : "memory");
    smax = sref_s[r];
    const uint32_t a_lane = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
    const uint8_t *wsm = gsm + kStagesG * kStageB + r * (kWK / 2);
    // K steps in groups of 4 (a 16-byte window of the row's scale bytes: 4 blocks
    // of 32 values per step, two weight stages); the next window's scales are
    // loaded one group ahead
    uint4 scv = make_uint4(0, 0, 0, 0);
    if (svec) scv = *reinterpret_cast<const uint4 *>(srow);
    for (int kb = 0; kb < ksteps; kb += 4) {
      uint4 scn = make_uint4(0, 0, 0, 0);
      if (svec && kb + 4 < ksteps) scn = *reinterpret_cast<const uint4 *>(srow + 4 * (kb + 4));
      const uint32_t sw[4] = {scv.x, scv.y, scv.z, scv.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int ks = kb + j;
        if (ks >= ksteps) break;
        const int wst = ks / kWSteps, ws = wst % kWStages;
        if ((ks % kWSteps) == 0 && !mb_wait(&wfull_bar[ws], static_cast<uint32_t>(wst / kWStages) & 1u)) timeout = true;
        const int s = ks % kStagesG;
        const uint32_t lap = static_cast<uint32_t>(ks / kStagesG);
        if (!mb_wait(&empty_bar[s], (lap & 1u) ^ 1u)) timeout = true;
        // this thread's two blocks of the step: 4 ks + 2 hf + cc
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          int sbyte = 0;
          if (svec) sbyte = static_cast<int>((sw[j] >> (8 * (2 * hf + cc))) & 0xFFu);
          else if (present) sbyte = srow[4 * ks + 2 * hf + cc];
          uint4 cw = make_uint4(0, 0, 0, 0);
          if (present)
            cw = *reinterpret_cast<const uint4 *>(wsm + ws * kWStageB +
                                                  (((((ks % kWSteps) * 4) + 2 * hf + cc) ^ (r & 7)) << 4));
          const uint32_t mulbits = f16_pow2_bits(sbyte - smax);
          const uint32_t mul2 = mulbits | (mulbits << 16);
          const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
          uint32_t o[16];  // 32 f16 = columns 32 hf + 16 cc .. + 15 of the stage (two K values per column)
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t h[4];
            e2m1x8_to_f16x2(words[c], h);
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              const __half2 a = *reinterpret_cast<const __half2 *>(&h[m]);
              const __half2 b = *reinterpret_cast<const __half2 *>(&mul2);
              const __half2 prod = __hmul2(a, b);
              o[4 * c + m] = *reinterpret_cast<const uint32_t *>(&prod);
            }
          }
          if (cc == 0) tc_st16_issue(a_lane + kTileN + s * kAcols + 32 * hf, o);
          else tc_st16(a_lane + kTileN + s * kAcols + 32 * hf + 16, o);  // waits for both stores
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mb_arrive(&full_bar[s]);
          // the weight stage is free once this warp has read its last K step
          if ((ks % kWSteps) == kWSteps - 1 || ks == ksteps - 1) mb_arrive(&wempty_bar[ws]);
        }
      }
      scv = scn;
    }
  } else if (warp == kTmaWarp) {
    // ---------------------------------------------------- TMA: activation tiles
    if (lane == 0) {
      for (int ks = 0; ks < ksteps; ++ks) {
        const int s = ks % kStagesG;
        const uint32_t lap = static_cast<uint32_t>(ks / kStagesG);
        if (!mb_wait(&empty_bar[s], (lap & 1u) ^ 1u)) timeout = true;
        uint8_t *sbuf = gsm + s * kStageB;
        const CUtensorMap *bm = &bmaps.m[Npad / 16 - 1];
        mb_arrive_tx(&full_bar[s], static_cast<uint32_t>(2 * Npad * kBoxK * 2));
        tma_load_2d(sbuf, bm, ks * kTileK, g.p0, &full_bar[s]);
        tma_load_2d(sbuf + kBoxB, bm, ks * kTileK + kBoxK, g.p0, &full_bar[s]);
      }
    }
    __syncwarp();
  } else if (warp == kWTmaWarp) {
    // ---------------------------------------------------- TMA: weight codes
    if (lane == 0) {
      const int nws = (ksteps + kWSteps - 1) / kWSteps;
      uint8_t *wbase = gsm + kStagesG * kStageB;
      const CUtensorMap *wmap =
          reinterpret_cast<const CUtensorMap *>(P.maps + static_cast<size_t>(kind * P.E + g.u) * kMapBytes);
      // the map was written by the previous kernel: order its reads after those writes
      if (present) asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(wmap) : "memory");
      const int y0 = tile_wrow(kind, g.m0, 0, P.I), y1 = tile_wrow(kind, g.m0, kWBoxRows, P.I);
      for (int wst = 0; wst < nws; ++wst) {
        const int ws = wst % kWStages;
        if (!mb_wait(&wempty_bar[ws], (static_cast<uint32_t>(wst / kWStages) & 1u) ^ 1u)) timeout = true;
        mb_arrive_tx(&wfull_bar[ws], present ? static_cast<uint32_t>(kWStageB) : 0u);
        if (present) {
          uint8_t *dst = wbase + ws * kWStageB;
          tma_load_2d(dst, wmap, wst * (kWK / 2), y0, &wfull_bar[ws]);
          tma_load_2d(dst + kWStageB / 2, wmap, wst * (kWK / 2), y1, &wfull_bar[ws]);
        }
      }
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------- MMA issue
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(kTileM, Npad);
      for (int ks = 0; ks < ksteps; ++ks) {
        const int s = ks % kStagesG;
        const uint32_t lap = static_cast<uint32_t>(ks / kStagesG);
        if (!mb_wait(&full_bar[s], lap & 1u)) timeout = true;
        tc_fence_after();
        const uint64_t bd = smem_desc_sw128(su32(gsm + s * kStageB));
        const uint32_t a0 = tmem + kTileN + s * kAcols;
#pragma unroll
        for (int bx = 0; bx < kTileK / kBoxK; ++bx)  // per box 4 MMAs of K = 16: A +8 columns, B +32 bytes
          tc_mma4_f16_ta(tmem, a0 + bx * 32, bd + bx * (kBoxB >> 4), idesc, (ks > 0 || bx > 0) ? 1u : 0u);
        tc_commit(&empty_bar[s]);
      }
      tc_commit(&acc_bar);
    }
  }

  // ---- epilogue (dequantisation warps): TMEM lane quadrant = warp % 4,
  //      warps 0-3 take columns [0, 64), warps 4-7 columns [64, 128)
  if (warp < kDqWarps) {
    if (!mb_wait(&acc_bar, 0)) timeout = true;
    tc_fence_after();
    float *stage = reinterpret_cast<float *>(gsm);  // [kTileN][kTileM + 1]
    const int q = warp & 3, row = 32 * q + lane;
    const int cbeg = (warp >> 2) * 64;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * q) << 16);
    for (int c0 = cbeg; c0 < cbeg + 64 && c0 < Npad; c0 += 16) {
      float v[16];
      tc_ld16(lane_addr + c0, v);
#pragma unroll
      for (int j = 0; j < 16; ++j) stage[(c0 + j) * (kTileM + 1) + row] = v[j];
    }
    tc_fence_before();
    asm volatile("bar.sync 1, %0;" ::"r"(kDqWarps * 32) : "memory");
    if (kind == 0) {
      // h[p0 + n][m0/2 + i] = bf16(silu(g) * u), g = tile row i, u = tile row 64 + i
      const int ncols = kTileM / 2;
      for (int idx = tid; idx < g.n * ncols; idx += kDqWarps * 32) {
        const int n = idx / ncols, i = idx % ncols;
        float hv = 0.f;
        if (present) {
          const float gg = mul_pow2(stage[n * (kTileM + 1) + i], sref_s[i] - 127 + bexp_s[n]);
          const float uu = mul_pow2(stage[n * (kTileM + 1) + ncols + i], sref_s[ncols + i] - 127 + bexp_s[n]);
          hv = (gg / (1.0f + expf(-gg))) * uu;
        }
        P.hrow[static_cast<size_t>(g.p0 + n) * P.I + (g.m0 >> 1) + i] = f32_to_bf16_rne(hv);
      }
    } else {
      for (int idx = tid; idx < g.n * kTileM; idx += kDqWarps * 32) {
        const int n = idx / kTileM, r = idx % kTileM;
        P.Y[static_cast<size_t>(g.p0 + n) * P.H + g.m0 + r] =
            present ? mul_pow2(stage[n * (kTileM + 1) + r], sref_s[r] - 127 + bexp_s[n]) : 0.f;
      }
    }
  }
  if (timeout) set_status(P.status, K3MOE_DEV_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}


// ============================================================================
// W4A4 grouped GEMM on the block-scaled tensor core: tcgen05.mma kind::mxf4
// (scale_vec::2X, K = 64 per MMA) with the E8M0 block scales of both operands in
// tensor memory.  The weight codes go from TMA to the tensor core as they are
// stored (e2m1, two per byte, low nibble = even column) and the activations are
// the MXFP4 codes and scales of the quantiser rule (a pre-pass), so every product
// is exact and only the fp32 accumulation rounds.
// Tensor-memory layout of the scale factors (M = 128): the scale bytes of tile
// row r (or token column n) sit in lane r % 32 of every lane quadrant, column
// base + r / 32; a 32-bit cell holds the scales of 4 consecutive K blocks and the
// instruction descriptor's scale-factor id picks the byte pair of a K-64 step.
// Warps: 0-3 write the scale factors (tcgen05.st) and run the epilogue; 4 issues
// the TMA loads (weight codes through the expert's tensor map, activation codes);
// 5 owns tensor memory and issues the MMAs.  One ring of stages of 256 K values.
namespace {

constexpr int kMxSfWarps = 4;
constexpr int kMxTmaWarp = 4;
constexpr int kMxMmaWarp = 5;
constexpr int kMxThreads = 6 * 32;
constexpr int kMxAtomB = kTileN * 128;  // one 128-row x 128-byte swizzled tile (16 KiB)
constexpr int kMxColSf = kTileN;        // tensor-memory columns: accumulator [0, 128), then the scale slots
constexpr int kMxAhead = 8;             // weight-code stages prefetched into L2 ahead of the ring
constexpr int kMxKS = 256;              // K values per stage: one 128-byte row of codes per operand
constexpr int kMxSteps = kMxKS / 64;    // MMAs per stage
constexpr int kMxStages = 3;
constexpr int kMxStageB = 2 * kMxAtomB;  // weight tile + activation tile
constexpr int kMxSmem = kMxStages * kMxStageB;
constexpr int kMxDynSmem = 1024 + (kMxSmem > kEpiBytes ? kMxSmem : kEpiBytes);
// Scale factors travel in chunks of 16 bytes per row (512 K values, 2 stages).  A
// chunk takes 16 tensor-memory columns per operand: 4 words of 4 block scales x
// 4 row groups of 32.  Two chunk slots follow the accumulator.
constexpr int kMxCh = 512 / kMxKS;
constexpr int kMxSfChunkCols = 32;
static_assert(kMxColSf + 2 * kMxSfChunkCols <= kTmemCols, "tensor-memory budget");

// Instruction descriptor of kind::mxf4: B scale-factor id [4,6), A and B formats
// [7,10) and [10,13) (E2M1 = 1), N/8 [17,23), E8M0 scales (bit 23), M/16 [24,29),
// A scale-factor id [29,31).
__device__ __forceinline__ uint32_t idesc_mxf4(int M, int N, int sf_id) {
  return (static_cast<uint32_t>(sf_id) << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (1u << 23) | (static_cast<uint32_t>(M >> 4) << 24) | (static_cast<uint32_t>(sf_id) << 29);
}

// The four MMAs of one stage (K = 64 each, 256 K values): operand descriptors a
// and b advance 32 bytes (2 in the address field) per MMA; MMAs 0 and 2 take the
// scale-factor id 0 (idesc0), 1 and 3 id 2 (idesc2); MMAs 0 and 1 read the scale
// words at sfa / sfb, 2 and 3 the next word (+4 columns).  The first accumulates
// when `acc` is nonzero.  One asm block keeps the issuing thread to a few
// instructions per MMA.
__device__ __forceinline__ void tc_mma4_mxf4(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc0,
                                             uint32_t idesc2, uint32_t sfa, uint32_t sfb, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t.reg .b64 a1, a2, a3, b1, b2, b3;\n\t.reg .b32 sa1, sb1;\n\t"
      "setp.ne.b32 p, %7, 0;\n\tsetp.eq.b32 q, %3, %3;\n\t"
      "add.u64 a1, %1, 2;\n\tadd.u64 a2, %1, 4;\n\tadd.u64 a3, %1, 6;\n\t"
      "add.u64 b1, %2, 2;\n\tadd.u64 b2, %2, 4;\n\tadd.u64 b3, %2, 6;\n\t"
      "add.u32 sa1, %5, 4;\n\tadd.u32 sb1, %6, 4;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%5], [%6], p;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], a1, b1, %4, [%5], [%6], q;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], a2, b2, %3, [sa1], [sb1], q;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], a3, b3, %4, [sa1], [sb1], q;\n\t}" ::"r"(
          tmem_d),
      "l"(a), "l"(b), "r"(idesc0), "r"(idesc2), "r"(sfa), "r"(sfb), "r"(acc)
      : "memory");
}

// 32 lanes x 32 bit, 16 consecutive columns per thread, registers -> tensor
// memory (no wait: the caller waits once for several stores).
__device__ __forceinline__ void tc_st16_nw(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// `valid` (16 or 8) bytes of a byte array as four little-endian words, zero
// beyond `valid`; any alignment (the out-of-line path takes what is not one
// aligned 16-byte load).
__device__ __noinline__ uint4 ld_sf16_slow(const uint8_t *p, int valid) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  if ((a & 7u) == 0) {
    const uint2 lo = *reinterpret_cast<const uint2 *>(p);
    const uint2 hi = valid == 16 ? *reinterpret_cast<const uint2 *>(p + 8) : make_uint2(0u, 0u);
    return make_uint4(lo.x, lo.y, hi.x, hi.y);
  }
  uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int i = 0; i < 16; ++i)
    if (i < valid) w[i >> 2] |= static_cast<uint32_t>(p[i]) << (8 * (i & 3));
  return make_uint4(w[0], w[1], w[2], w[3]);
}
__device__ __forceinline__ uint4 ld_sf16(const uint8_t *p, int valid) {
  if (valid == 16 && (reinterpret_cast<uintptr_t>(p) & 15u) == 0) return *reinterpret_cast<const uint4 *>(p);
  return ld_sf16_slow(p, valid);
}

// One chunk of scale words for the 128 rows / token columns a lane covers
// (lane + 32 c): weights, then activations.
struct SfChunk {
  uint4 w[4];
  uint4 b[4];
};

// Bounded wait that also gives up as soon as another role has given up (`abort`
// in shared memory); a timeout raises the flag.  Returns true when the phase completed.
__device__ __forceinline__ bool mb_wait_or_abort(uint64_t *b, uint32_t parity, volatile int *abort) {
  if (mb_test(b, parity)) return true;
  for (long long i = 0; i < kSpinG; ++i) {
    if (mb_try(b, parity)) return true;
    if (*abort) return false;
    if (i > 32) __nanosleep(20);
  }
  *abort = 1;
  return false;
}


}  // namespace

struct Mx4Params {
  k3moe_weights w;
  int H, I, A, E;
  const int32_t *meta;
  const int4 *tab;         // tile table of this GEMM
  const uint8_t *maps;     // weight-code tensor maps per active slot (w13 at u, w2 at E + u)
  const uint8_t *ascale;   // activation block scales [A][K/32]
  uint16_t *hrow;          // [A][I] bf16 (gate/up output)
  float *Y;                // [A][H]
  int kind;                // 0 gate/up, 1 down
  int32_t *status;
};

__global__ void __launch_bounds__(kMxThreads, 2)
    ffn_gemm_mxf4_kernel(const __grid_constant__ RowMaps amaps, Mx4Params P) {
  extern __shared__ __align__(1024) uint8_t msm_raw[];
  uint8_t *msm = msm_raw + ((1024u - (su32(msm_raw) & 1023u)) & 1023u);
  __shared__ uint64_t full[kMxStages], empty[kMxStages], sf_full[2], sf_empty[2], acc_bar;
  __shared__ uint32_t tmem_holder;
  __shared__ int s_abort;
  volatile int *abort = &s_abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_wait();
  pdl_trigger();
  const int kind = P.kind;
  if (static_cast<int>(blockIdx.x) >= P.meta[1 + kind]) return;
  GemmTile g;
  {
    const int4 te = P.tab[blockIdx.x];
    g.u = te.x;
    g.e = te.y;
    g.p0 = te.z;
    g.n = te.w >> 16;
    g.m0 = (te.w & 0xFFFF) * kTileM;
  }
  const int K = kind == 0 ? P.H : P.I;
  const int nst = K / kMxKS;  // stages (K is a multiple of 256)
  const int Npad = (g.n + 15) & ~15;
  const uint8_t *c13 = P.w.w13_codes[g.e], *s13 = P.w.w13_scales[g.e];
  const uint8_t *c2 = P.w.w2_codes[g.e], *s2 = P.w.w2_scales[g.e];
  const uintptr_t al = reinterpret_cast<uintptr_t>(c13) | reinterpret_cast<uintptr_t>(c2);
  const bool present = c13 && s13 && c2 && s2 && (al & 15u) == 0;
  const uint8_t *wscales = kind == 0 ? s13 : s2;
  if (tid == 0) {
    for (int s = 0; s < kMxStages; ++s) {
      mb_init(&full[s], 1);  // TMA bytes
      mb_init(&empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mb_init(&sf_full[s], kMxSfWarps);  // one arrival per scale-factor warp
      mb_init(&sf_empty[s], 1);
    }
    mb_init(&acc_bar, 1);
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kMxMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(&tmem_holder)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_holder;
  bool timeout = false;

  if (warp < kMxSfWarps) {
    // ---------------------------------------------------- scale factors
    // Lane l of every warp writes rows / token columns l, l+32, l+64, l+96 into
    // its own lane quadrant (the same data in all four).  Chunk ch (stages
    // [2 ch, 2 ch + 2)) goes to slot ch & 1: weights at columns +0..15,
    // activations at +16..31; column 4 w + c holds scale word w of row group c.
    // Loads run two chunks ahead of the stores in two register sets.
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * warp) << 16);
    const int sbytes = K / 32;
    const int nch = (nst + kMxCh - 1) / kMxCh;
    const uint8_t *srow[4];
    const uint8_t *arow[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int r = lane + 32 * c;
      srow[c] = present ? wscales + static_cast<size_t>(tile_wrow(kind, g.m0, r, P.I)) * sbytes : nullptr;
      arow[c] = r < g.n ? P.ascale + static_cast<size_t>(g.p0 + r) * sbytes : nullptr;
      if (srow[c]) {  // the tile's weight-scale rows are read once, 16 bytes per chunk: pull them into L2 now
        for (int off = 0; off < sbytes; off += 128) prefetch_l2(srow[c] + off);
        prefetch_l2(srow[c] + sbytes - 1);
      }
    }
    auto load_chunk = [&](int ch, SfChunk &R) {
      const int off = 16 * ch;
      const int valid = sbytes - off < 16 ? sbytes - off : 16;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        R.w[c] = srow[c] ? ld_sf16(srow[c] + off, valid) : make_uint4(0u, 0u, 0u, 0u);
        R.b[c] = arow[c] ? ld_sf16(arow[c] + off, valid) : make_uint4(0u, 0u, 0u, 0u);
      }
    };
    auto words = [](const uint4 (&v)[4], uint32_t (&o)[16]) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        o[c] = v[c].x;
        o[4 + c] = v[c].y;
        o[8 + c] = v[c].z;
        o[12 + c] = v[c].w;
      }
    };
    auto store_chunk = [&](int ch, const SfChunk &R) -> bool {
      const int slot = ch & 1;
      if (!__all_sync(0xFFFFFFFFu,
                      mb_wait_or_abort(&sf_empty[slot], (static_cast<uint32_t>(ch >> 1) & 1u) ^ 1u, abort)))
        return false;
      const uint32_t base = lane_addr + kMxColSf + slot * kMxSfChunkCols;
      uint32_t o[16];
      words(R.w, o);
      tc_st16_nw(base, o);
      words(R.b, o);
      tc_st16_nw(base + 16, o);
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mb_arrive(&sf_full[slot]);
      return true;
    };
    SfChunk R0, R1;
    load_chunk(0, R0);
    if (nch > 1) load_chunk(1, R1);
    bool ok = true;
    for (int ch = 0; ch < nch && ok; ch += 2) {
      ok = store_chunk(ch, R0);
      if (ok && ch + 2 < nch) load_chunk(ch + 2, R0);
      if (ok && ch + 1 < nch) {
        ok = store_chunk(ch + 1, R1);
        if (ok && ch + 3 < nch) load_chunk(ch + 3, R1);
      }
    }
    if (!ok) timeout = true;
  } else if (warp == kMxTmaWarp) {
    // ---------------------------------------------------- TMA
    if (lane == 0) {
      const CUtensorMap *wmap =
          reinterpret_cast<const CUtensorMap *>(P.maps + static_cast<size_t>(kind * P.E + g.u) * kMapBytes);
      if (present) asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(wmap) : "memory");
      const int y0 = tile_wrow(kind, g.m0, 0, P.I), y1 = tile_wrow(kind, g.m0, kWBoxRows, P.I);
      if (present)
        for (int a = 0; a < kMxAhead && a < nst; ++a) {
          tma_prefetch_2d(wmap, a * 128, y0);
          tma_prefetch_2d(wmap, a * 128, y1);
        }
      for (int a = 0; a < nst; ++a) {
        const int s = a % kMxStages;
        if (!mb_wait_or_abort(&empty[s], (static_cast<uint32_t>(a / kMxStages) & 1u) ^ 1u, abort)) {
          timeout = true;
          break;
        }
        uint8_t *st = msm + s * kMxStageB;
        mb_arrive_tx(&full[s], static_cast<uint32_t>((present ? kMxAtomB : 0) + Npad * 128));
        if (present) {  // weight codes: K offset in bytes (128 per stage), two boxes of 64 rows
          tma_load_2d(st, wmap, a * 128, y0, &full[s]);
          tma_load_2d(st + kMxAtomB / 2, wmap, a * 128, y1, &full[s]);
          if (a + kMxAhead < nst) {
            tma_prefetch_2d(wmap, (a + kMxAhead) * 128, y0);
            tma_prefetch_2d(wmap, (a + kMxAhead) * 128, y1);
          }
        }
        tma_load_2d(st + kMxAtomB, &amaps.m[Npad / 16 - 1], a * 128, g.p0, &full[s]);
      }
    }
  } else {
    // ---------------------------------------------------- MMA issue
    if (lane == 0) {
      for (int a = 0; a < nst; ++a) {
        const int s = a % kMxStages;
        const int ch = a / kMxCh, t = a % kMxCh, slot = ch & 1;
        if (t == 0 && !mb_wait_or_abort(&sf_full[slot], static_cast<uint32_t>(ch >> 1) & 1u, abort)) {
          timeout = true;
          break;
        }
        if (!mb_wait_or_abort(&full[s], static_cast<uint32_t>(a / kMxStages) & 1u, abort)) {
          timeout = true;
          break;
        }
        tc_fence_after();
        const uint32_t wa = su32(msm + s * kMxStageB);
        const uint32_t sf = tmem + kMxColSf + slot * kMxSfChunkCols;
        // both operands advance 32 bytes (64 values) per MMA; MMA j's two 32-value
        // blocks are blocks 8 t + 2 j, 8 t + 2 j + 1 of the chunk: scale word
        // 2 t + j / 2, byte pair 2 (j % 2)
        static_assert(kMxSteps == 4, "one stage = four MMAs of K = 64");
        tc_mma4_mxf4(tmem, smem_desc_sw128(wa), smem_desc_sw128(wa + kMxAtomB), idesc_mxf4(kTileM, Npad, 0),
                     idesc_mxf4(kTileM, Npad, 2), sf + 8 * t, sf + 16 + 8 * t, a > 0 ? 1u : 0u);
        tc_commit(&empty[s]);
        if (t == kMxCh - 1 || a == nst - 1) tc_commit(&sf_empty[slot]);
      }
      tc_commit(&acc_bar);  // also after an abort: completes when every MMA issued so far has finished
    }
  }

  // ---- epilogue (scale-factor warps): lane quadrant = warp, all Npad columns
  if (warp < kMxSfWarps) {
    if (!mb_wait(&acc_bar, 0)) {
      timeout = true;
      *abort = 1;
    }
    tc_fence_after();
    float *stage = reinterpret_cast<float *>(msm);  // [kTileN][kTileM + 1]
    const int row = 32 * warp + lane;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * warp) << 16);
    for (int c0 = 0; c0 < Npad; c0 += 16) {
      float v[16];
      tc_ld16(lane_addr + c0, v);
#pragma unroll
      for (int j = 0; j < 16; ++j) stage[(c0 + j) * (kTileM + 1) + row] = v[j];
    }
    tc_fence_before();
    asm volatile("bar.sync 1, %0;" ::"r"(kMxSfWarps * 32) : "memory");
    if (kind == 0) {
      // h[p0 + n][m0/2 + i] = bf16(silu(g) * u), g = tile row i, u = tile row 64 + i
      const int ncols = kTileM / 2;
      for (int idx = tid; idx < g.n * ncols; idx += kMxSfWarps * 32) {
        const int n = idx / ncols, i = idx % ncols;
        float hv = 0.f;
        if (present) {
          const float gg = stage[n * (kTileM + 1) + i];
          const float uu = stage[n * (kTileM + 1) + ncols + i];
          hv = (gg / (1.0f + expf(-gg))) * uu;
        }
        P.hrow[static_cast<size_t>(g.p0 + n) * P.I + (g.m0 >> 1) + i] = f32_to_bf16_rne(hv);
      }
    } else {
      for (int idx = tid; idx < g.n * kTileM; idx += kMxSfWarps * 32) {
        const int n = idx / kTileM, r = idx % kTileM;
        P.Y[static_cast<size_t>(g.p0 + n) * P.H + g.m0 + r] = present ? stage[n * (kTileM + 1) + r] : 0.f;
      }
    }
  }
  if (timeout) set_status(P.status, K3MOE_DEV_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  if (*abort) {
    // a role gave up: copies it issued may still be landing in shared memory (and
    // their barrier may never complete), so wait a bounded 2 ms before leaving
    for (int i = 0; i < 2000; ++i) __nanosleep(1000);
    __syncthreads();
  }
  if (warp == kMxMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

// MXFP4 activations for the W4A4 GEMM, one block of 256 threads per bucket row p
// (source row x[perm[p] / k] for gate/up, h[p] for down; 4 lanes per 32-block, 8
// values each): codes [A][K/2] (two per byte, low nibble = even column) and
// scales [A][K/32] by the quantiser rule.
__global__ void __launch_bounds__(256)
    gemm_rows_to_mxfp4_kernel(const uint16_t *__restrict__ src, const int32_t *__restrict__ perm, int k, int A,
                              int K, uint8_t *__restrict__ codes, uint8_t *__restrict__ scales, int32_t *status) {
  pdl_wait();
  pdl_trigger();
  const int p = blockIdx.x;
  int row = p;
  if (perm) {
    const int a = perm[p];
    row = (a >= 0 && a < A) ? a / k : -1;
    if (row < 0) set_status(status, K3MOE_DEV_BOUNDS);
  }
  const uint16_t *s = row >= 0 ? src + static_cast<size_t>(row) * K : nullptr;
  const int sbytes = K / 32;
  for (int c0 = 0; c0 < K; c0 += 256 * 8) {  // trip count uniform across the block
    const int c = c0 + threadIdx.x * 8;
    const bool ok = c < K;
    float v[8];
    uint4 u = make_uint4(0, 0, 0, 0);
    if (ok && s) u = *reinterpret_cast<const uint4 *>(s + c);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      v[2 * m] = __uint_as_float(w[m] << 16);
      v[2 * m + 1] = __uint_as_float(w[m] & 0xFFFF0000u);
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
    const int e = mx_shared_exp(amax);
    const float inv_x = mx_pow2(-e);
    uint32_t code = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) code |= mx_code(v[i], inv_x) << (4 * i);
    if (ok) {
      *reinterpret_cast<uint32_t *>(codes + static_cast<size_t>(p) * (K / 2) + c / 2) = code;
      if ((threadIdx.x & 3) == 0) scales[static_cast<size_t>(p) * sbytes + c / 32] = static_cast<uint8_t>(e + 127);
    }
  }
}

// ----------------------------------------------------------------------------
namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 2-D map over the weight codes of one expert (rows x K/2 bytes): box = 128
// bytes x 64 rows, 128B swizzle.  `base` is a placeholder address that the
// device replaces per expert.
bool make_code_map(CUtensorMap *m, void *base, int rows, int kbytes) {
  EncodeTiledFn fn = encode_tiled();
  if (!fn) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kbytes), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kbytes)};
  const cuuint32_t box[2] = {kWK / 2, kWBoxRows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D map over activation bytes (rows x row_bytes): box = 128 bytes x 128 rows,
// 128B swizzle; rows past the end read as zero.
bool make_byte_map(CUtensorMap *m, void *base, int rows, int row_bytes, int box_rows = kTileN) {
  EncodeTiledFn fn = encode_tiled();
  if (!fn) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
  const cuuint32_t box[2] = {128, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D map over rows x K of 16-bit values: box = 64 (K) x box_rows, 128B swizzle,
// rows past the end read as zero.
bool make_row_map_box(CUtensorMap *m, void *base, int rows, int K, int box_rows) {
  EncodeTiledFn fn = encode_tiled();
  if (!fn) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
  const cuuint32_t box[2] = {kBoxK, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The maps of every box height over one buffer: 16-bit rows of K values (roles 0
// and 1: x and h for the W4A16 GEMM) or rows of K bytes of MXFP4 codes (roles 2
// and 3: x and h for the W4A4 GEMM).  The last encoding per role is kept per
// thread, since the workspace is normally reused.
bool make_row_maps(RowMaps *out, int role, void *base, int rows, int K) {
  struct Entry {
    void *base = nullptr;
    int rows = -1, K = -1;
    RowMaps maps;
  };
  thread_local Entry cache[4];
  Entry &c = cache[role];
  if (c.base != base || c.rows != rows || c.K != K) {
    c.base = nullptr;
    for (int i = 0; i < kTileN / 16; ++i)
      if (!(role < 2 ? make_row_map_box(&c.maps.m[i], base, rows, K, 16 * (i + 1))
                     : make_byte_map(&c.maps.m[i], base, rows, K, 16 * (i + 1))))
        return false;
    c.base = base;
    c.rows = rows;
    c.K = K;
  }
  *out = c.maps;
  return true;
}

// The W4A4 GEMM (both projections): MXFP4 activations of x -> gate/up -> MXFP4
// activations of h -> down.
int launch_gemm_mxf4(const k3moe_shape &s, const uint16_t *x, const int32_t *perm, int A, long long ntile_max,
                     int mt_gu, int mt_dn, Mx4Params P, const int4 *tab_dn, uint8_t *xq, uint8_t *xsc, uint8_t *hq,
                     uint8_t *hsc, int32_t *status, cudaStream_t st) {
  RowMaps xmaps, hmaps;
  if (!make_row_maps(&xmaps, 2, xq, A, s.H / 2) || !make_row_maps(&hmaps, 3, hq, A, s.I / 2)) return -1;
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(ffn_gemm_mxf4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMxDynSmem) !=
        cudaSuccess)
      return -1;
    attr = true;
  }
  if (launch_pdl(gemm_rows_to_mxfp4_kernel, dim3(A), dim3(256), 0, st, x, perm, s.k, A, s.H, xq, xsc, status) !=
      cudaSuccess)
    return -1;
  P.kind = 0;
  P.ascale = xsc;
  if (launch_pdl(ffn_gemm_mxf4_kernel, dim3(static_cast<unsigned>(ntile_max * mt_gu)), dim3(kMxThreads), kMxDynSmem,
                 st, xmaps, P) != cudaSuccess)
    return -1;
  if (launch_pdl(gemm_rows_to_mxfp4_kernel, dim3(A), dim3(256), 0, st, static_cast<const uint16_t *>(P.hrow),
                 static_cast<const int32_t *>(nullptr), 1, A, s.I, hq, hsc, status) != cudaSuccess)
    return -1;
  P.kind = 1;
  P.tab = tab_dn;
  P.ascale = hsc;
  if (launch_pdl(ffn_gemm_mxf4_kernel, dim3(static_cast<unsigned>(ntile_max * mt_dn)), dim3(kMxThreads), kMxDynSmem,
                 st, hmaps, P) != cudaSuccess)
    return -1;
  return 0;
}

}  // namespace


// 2-D map over rows x K of 16-bit values: box = 64 (K) x 128 rows, 128B swizzle,
// rows past the end read as zero.
bool make_row_map(CUtensorMap *m, void *base, int rows, int K) { return make_row_map_box(m, base, rows, K, kTileN); }

size_t ffn_gemm_workspace(const k3moe_shape &s) { return gemm_ws(s.T, s.H, s.I, s.E, s.k).total; }
size_t ffn_gemm_h_offset(const k3moe_shape &s) { return gemm_ws(s.T, s.H, s.I, s.E, s.k).hrow; }

bool ffn_gemm_supported(const k3moe_shape &s) {
  return (2 * s.I) % kTileM == 0 && s.H % kTileM == 0 && s.H % kTileK == 0 && s.I % kTileK == 0 &&
         encode_tiled() != nullptr;
}

int launch_ffn_gemm(const k3moe_shape &s, const uint16_t *x, const k3moe_weights &w, const int32_t *offsets,
                    const int32_t *perm, float *Y, void *ws, int32_t *status, cudaStream_t st, bool a4) {
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
  int4 *tab_gu = reinterpret_cast<int4 *>(base + L.tab_gu);
  int4 *tab_dn = reinterpret_cast<int4 *>(base + L.tab_dn);
  uint16_t *xg = reinterpret_cast<uint16_t *>(base + L.xg);
  int32_t *xexp = reinterpret_cast<int32_t *>(base + L.xexp);
  uint16_t *hrow = reinterpret_cast<uint16_t *>(base + L.hrow);
  uint16_t *h16 = reinterpret_cast<uint16_t *>(base + L.h16);
  int32_t *hexp = reinterpret_cast<int32_t *>(base + L.hexp);
  uint8_t *maps = reinterpret_cast<uint8_t *>(base + L.maps);
  CUtensorMap t13, t2;
  if (!make_code_map(&t13, maps, 2 * s.I, s.H / 2) || !make_code_map(&t2, maps, s.H, s.I / 2)) return -1;
  if (launch_pdl(gemm_prep_kernel, dim3(1), dim3(32), 0, st, offsets, s.E, A, mt_gu, mt_dn, active, meta, sp0,
                 scnt, pgu, pdn, status) != cudaSuccess)
    return -1;
  // upper bound of the token tiles: sum_e ceil(n_e / 128) <= A / 128 + min(A, E)
  const long long ntile_max = A / kTileN + (A < s.E ? A : s.E);
  const long long sched_threads = std::max<long long>(2LL * s.E, ntile_max * std::max(mt_gu, mt_dn));
  if (launch_pdl(gemm_sched_kernel, dim3(static_cast<unsigned>((sched_threads + 127) / 128)), dim3(128), 0, st, t13,
                 t2, w, static_cast<const int32_t *>(active), static_cast<const int32_t *>(meta), s.E,
                 static_cast<const int32_t *>(sp0), static_cast<const int32_t *>(scnt),
                 static_cast<const int32_t *>(pgu), static_cast<const int32_t *>(pdn), mt_gu, mt_dn, tab_gu, tab_dn,
                 maps, status) != cudaSuccess)
    return -1;
  if (a4 && s.H % kMxKS == 0 && s.I % kMxKS == 0) {  // W4A4 on the block-scaled tensor core
    Mx4Params B;
    B.w = w;
    B.H = s.H; B.I = s.I; B.A = A; B.E = s.E;
    B.meta = meta;
    B.tab = tab_gu;
    B.maps = maps;
    B.hrow = hrow;
    B.Y = Y;
    B.status = status;
    uint8_t *xq = reinterpret_cast<uint8_t *>(xg), *hq = reinterpret_cast<uint8_t *>(h16);
    uint8_t *xsc = reinterpret_cast<uint8_t *>(base + L.xsc), *hsc = reinterpret_cast<uint8_t *>(base + L.hsc);
    return launch_gemm_mxf4(s, x, perm, A, ntile_max, mt_gu, mt_dn, B, tab_dn, xq, xsc, hq, hsc, status, st);
  }
  auto rows_to_f16 = a4 ? gemm_rows_to_f16_kernel<true> : gemm_rows_to_f16_kernel<false>;
  if (launch_pdl(rows_to_f16, dim3(A), dim3(256), 0, st, x, perm, s.k, A, s.H, xg, xexp, status) !=
      cudaSuccess)
    return -1;
  RowMaps xmaps, hmaps;
  if (!make_row_maps(&xmaps, 0, xg, A, s.H) || !make_row_maps(&hmaps, 1, h16, A, s.I)) return -1;
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(ffn_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem) !=
        cudaSuccess)
      return -1;
    attr = true;
  }
  GemmParams P;
  P.w = w;
  P.H = s.H; P.I = s.I; P.A = A;
  P.meta = meta;
  P.maps = maps;
  P.E = s.E;
  P.hrow = hrow;
  P.Y = Y;
  P.status = status;
  P.kind = 0;
  P.tab = tab_gu;
  P.bexp = xexp;
  if (launch_pdl(ffn_gemm_kernel, dim3(static_cast<unsigned>(ntile_max * mt_gu)), dim3(kThreadsG), kGemmSmem, st,
                 xmaps, P) != cudaSuccess)
    return -1;
  if (launch_pdl(rows_to_f16, dim3(A), dim3(256), 0, st, static_cast<const uint16_t *>(hrow),
                 static_cast<const int32_t *>(nullptr), 1, A, s.I, h16, hexp, status) != cudaSuccess)
    return -1;
  P.kind = 1;
  P.tab = tab_dn;
  P.bexp = hexp;
  if (launch_pdl(ffn_gemm_kernel, dim3(static_cast<unsigned>(ntile_max * mt_dn)), dim3(kThreadsG), kGemmSmem, st,
                 hmaps, P) != cudaSuccess)
    return -1;
  return 0;
}

}  // namespace k3moe
