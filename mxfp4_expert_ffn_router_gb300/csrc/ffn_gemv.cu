// ffn_gemv.cu -- MXFP4 SwiGLU expert FFN for few tokens per expert (decode) as
// streaming matrix-vector products on the CUDA cores.
//
// The kimi-k3-in-c CHANGELOG walkthrough ("[0.1.0] Added") describes a matmul that
// reads the packed MXFP4 nibbles directly and never materialises a dequantised
// expert, and a gated-linear-unit expert.  Here every weight byte is read once
// per (expert, token group) with 16-byte coalesced loads, decoded in registers
// (cvt e2m1x2 -> f16x2, exact), multiplied by f16 activations with exact
// products accumulated in fp32, scaled per 32-block by the e8m0 scale, and
// reduced across the warp with shuffles.  The order of every sum is fixed.
//
// Activations are f16 after an exact power-of-two prescale per row (x' = x * 2^-p
// with max|x'| in [2^14, 2^15)), so bf16 values convert to f16 without rounding
// except for elements below 2^-28 * max|x| (error < 2^-25 of max).
//
// Kernels of one call:
//   gemv_prep    active-expert slots (block-parallel scan of the offsets),
//                x -> prescaled f16 (piece-major)
//   gemv_rows<0> item = (active slot u, row pair i): for each token p of u,
//                h[p][i] = bf16(silu(Wg_i x_p) * (Wu_i x_p)), plain stores
//   gemv_h16     h rows -> prescaled f16 (exponent from the row's max |h|)
//   gemv_rows<1> item = (active slot u, 4, 7 or 8 rows of W2): Y[p][rows] = W2 rows . h[p]
//
// Work is spread over warps, not blocks: warp w of the grid takes items w, w + W,
// w + 2W, ... (W = warps in the grid).  An item is streamed in steps of B chunks
// (32 K values = 16 code bytes) per lane and row; the next step's code and scale
// loads are issued before the current step is computed, so each warp keeps about
// one step of weight bytes in flight at all times, with no block-wide barrier.
// Activations (x16, h16), the slot table and the token ids are small and come
// through L1; weight codes bypass it.
#include <cuda_fp16.h>

#include "k3moe_dev.cuh"
#include "k3moe_launch.h"

namespace k3moe {

namespace {

constexpr int kGvWarps = 8;   // warps per block
constexpr int kDnRows = 4;    // W2 rows per down item (guarded kernel)

// Workspace layout (byte offsets, 256-aligned pieces).
struct GemvWs {
  size_t slots, meta, xexp, x16, hrow, h16, hexp, total;
};

__host__ __device__ inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

__host__ __device__ inline GemvWs gemv_ws(int T, int H, int I, int E, int k) {
  GemvWs w;
  const size_t A = static_cast<size_t>(T) * k;
  const size_t a1 = A ? A : 1;
  size_t o = 0;
  w.slots = o; o = align256(o + sizeof(int4) * E);                  // {e, p0, count, present} per active slot
  w.meta = o;  o = align256(o + sizeof(int32_t) * 4);              // active-slot count
  w.xexp = o;  o = align256(o + sizeof(int32_t) * (T > 0 ? T : 1));
  w.x16 = o;   o = align256(o + sizeof(uint16_t) * static_cast<size_t>(T) * H);
  w.hrow = o;  o = align256(o + sizeof(uint16_t) * A * I);          // h, bf16 (the rounding point)
  w.h16 = o;   o = align256(o + sizeof(uint16_t) * A * I);          // h, prescaled f16, piece-major
  w.hexp = o;  o = align256(o + sizeof(int32_t) * a1);
  w.total = o;
  return w;
}

// Power-of-two exponent p such that max_abs * 2^-p lies in [2^14, 2^15); 0 for 0.
__device__ __forceinline__ int prescale_exp(float max_abs) {
  if (!(max_abs > 0.f) || max_abs != max_abs) return 0;
  if (max_abs == INFINITY) return 0;
  int e;
  frexpf(max_abs, &e);  // max_abs = f * 2^e, f in [0.5, 1)
  int p = (e - 1) - 14;
  return max(-100, min(100, p));
}

// exact x * 2^-p to f16 bits
__device__ __forceinline__ uint32_t pack_f16x2_scaled(float a, float b, float s) {
  const __half2 h = __floats2half2_rn(a * s, b * s);
  return *reinterpret_cast<const uint32_t *>(&h);
}

// multiply by 2^p for |p| <= 200 (two exact steps)
__device__ __forceinline__ float scale_pow2(float v, int p) {
  const int p1 = p / 2, p2 = p - p1;
  return v * exp2i(p1) * exp2i(p2);
}

// bf16 row (K values) -> prescaled f16, piece-major: uint4 index q * (K/32) + c
// holds columns 32c + 8q .. 32c + 8q + 7, so a warp's lanes read consecutive 16 B.
__device__ __forceinline__ void row_to_f16_piece_major(const uint16_t *__restrict__ src, int K, float s,
                                                       uint4 *__restrict__ dst) {
  const int nch = K / 32;
  for (int piece = threadIdx.x; piece < K / 8; piece += blockDim.x) {  // piece = c * 4 + q (source order)
    const int c = piece >> 2, q = piece & 3;
    const uint4 v = *reinterpret_cast<const uint4 *>(src + 8 * piece);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int m = 0; m < 4; ++m)
      o[m] = pack_f16x2_scaled(__uint_as_float(w[m] << 16), __uint_as_float(w[m] & 0xFFFF0000u), s);
    dst[q * nch + c] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

__device__ __forceinline__ float block_max_256(float mx, float *red) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
  __syncthreads();
  mx = red[0];
  for (int i = 1; i < 8; ++i) mx = fmaxf(mx, red[i]);
  return mx;
}

}  // namespace

// An expert takes part when its four pointers are non-NULL and its code arrays
// are 16-byte aligned (the 128-bit loads need it); otherwise its rows are zero.
__device__ __forceinline__ bool expert_present(const k3moe_weights &w, int e) {
  const uint8_t *a = w.w13_codes[e], *b = w.w13_scales[e], *c = w.w2_codes[e], *d = w.w2_scales[e];
  return a && b && c && d && ((reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(c)) & 15u) == 0;
}
// Of an expert's four pointers (w13 codes and scales, w2 codes and scales):
// 1 present (as expert_present); 2 all given but the codes misaligned (absent,
// and reported); 0 absent.
__device__ __forceinline__ int expert_flags(const uint8_t *a, const uint8_t *b, const uint8_t *c, const uint8_t *d) {
  if (!(a && b && c && d)) return 0;
  return ((reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(c)) & 15u) == 0 ? 1 : 2;
}

// ----------------------------------------------------------------------------
// prep.  Block 0: slots of the active experts in expert order, from a
// block-parallel scan of the bucket offsets (thread i reads experts
// [i*m, (i+1)*m), m = ceil(E/256) <= 16).
// Block 1 + t: x[t] -> prescaled f16.
__global__ void __launch_bounds__(256)
    gemv_prep_kernel(k3moe_weights w, const uint16_t *__restrict__ x, int T, int H, int E, int A,
                     const int32_t *__restrict__ offsets, int4 *__restrict__ slots, int32_t *__restrict__ meta,
                     int32_t *__restrict__ xexp, uint4 *__restrict__ x16, int32_t *status) {
  pdl_wait();
  pdl_trigger();
  if (blockIdx.x == 0) {
    __shared__ int wsum[8];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int m = (E + 255) / 256;
    const int e0 = tid * m;
    int cnt[16], beg[16];
    int nf = 0;
    bool bad = false;
    int prev = e0 <= E ? offsets[e0 < E ? e0 : E] : 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      cnt[i] = 0;
      beg[i] = prev;
      const int e = e0 + i;
      if (i < m && e < E) {
        const int nx = offsets[e + 1];
        cnt[i] = nx - prev;
        if (cnt[i] < 0) bad = true;
        nf += cnt[i] > 0;
        prev = nx;
      }
    }
    if (tid == 0 && (offsets[0] != 0 || offsets[E] > A)) bad = true;
    bad = __syncthreads_or(bad) != 0;
    int inc = nf;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, inc, off);
      if (lane >= off) inc += v;
    }
    if (lane == 31) wsum[warp] = inc;
    __syncthreads();
    int base = 0, total = 0;
    for (int i = 0; i < 8; ++i) {
      base += i < warp ? wsum[i] : 0;
      total += wsum[i];
    }
    int slot = base + inc - nf;
    if (!bad) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int e = e0 + i;
        if (i < m && e < E && cnt[i] > 0) {
          const bool pr = expert_present(w, e);
          if (!pr && w.w13_codes[e] && w.w13_scales[e] && w.w2_codes[e] && w.w2_scales[e])
            set_status(status, K3MOE_DEV_BOUNDS);  // non-NULL but misaligned: treated as absent
          slots[slot++] = make_int4(e, beg[i], cnt[i], pr ? 1 : 0);
        }
      }
    }
    if (tid == 0) {
      meta[0] = bad ? 0 : total;
      if (bad) set_status(status, K3MOE_DEV_BOUNDS);
    }
    return;
  }
  const int t = blockIdx.x - 1;
  if (t >= T) return;
  const uint16_t *xr = x + static_cast<size_t>(t) * H;
  __shared__ float red[8];
  float mx = 0.f;
  for (int c = threadIdx.x; c < H; c += 256) mx = fmaxf(mx, fabsf(bf16_bits_to_f32(xr[c])));
  const int p = prescale_exp(block_max_256(mx, red));
  if (threadIdx.x == 0) xexp[t] = p;
  row_to_f16_piece_major(xr, H, scale_pow2(1.0f, -p), x16 + static_cast<size_t>(t) * (H / 8));
}

// h row p -> prescaled f16 (piece-major), exponent from the row's max |h| (a row
// holding a NaN takes exponent 0, as prescale_exp gives for a NaN maximum).  The
// block finds the maximum itself: the gate/up kernels write h with plain stores
// and no per-row atomics.
__global__ void __launch_bounds__(256)
    gemv_h16_kernel(const uint16_t *__restrict__ hrow, int I, uint4 *__restrict__ h16, int32_t *__restrict__ hexp) {
  // dependents first: the down projection may then start on the SMs the gate/up
  // kernel frees and prefetch its first weight rows while this kernel waits
  pdl_trigger();
  pdl_wait();
  const int p = blockIdx.x;
  const uint16_t *row = hrow + static_cast<size_t>(p) * I;
  __shared__ float red[8];
  float mx = 0.f;
  bool nan_here = false;
  for (int c = threadIdx.x * 8; c < I; c += 256 * 8) {
    const uint4 v = *reinterpret_cast<const uint4 *>(row + c);
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const float a = fabsf(__uint_as_float(u[m] << 16)), b = fabsf(__uint_as_float(u[m] & 0xFFFF0000u));
      nan_here |= (a != a) || (b != b);
      mx = fmaxf(mx, fmaxf(a, b));
    }
  }
  const bool any_nan = __syncthreads_or(nan_here) != 0;
  const int e = any_nan ? 0 : prescale_exp(block_max_256(mx, red));
  if (threadIdx.x == 0) hexp[p] = e;
  row_to_f16_piece_major(row, I, scale_pow2(1.0f, -e), h16 + static_cast<size_t>(p) * (I / 8));
}

// ----------------------------------------------------------------------------
struct RowsParams {
  k3moe_weights w;
  int H, I, k, A, E;
  const int32_t *perm;
  const int4 *slots;
  const int32_t *meta;
  const int32_t *aexp;   // activation prescale exponent: per token (gate/up) or per bucket position (down)
  const uint4 *act;      // activations, f16 piece-major: x16 [T][H] (gate/up) or h16 [A][I] (down)
  uint16_t *hrow;        // gate/up output, bf16 [A][I]
  float *Y;              // down output, [A][H]
  int32_t *status;
  // gate/up of the decode layer only (NULL otherwise): the routing weights of the
  // rw_T tokens, computed by the grid's last rw_T warps once their items are done
  const float *rw_logits;  // [rw_T][E]
  const int32_t *rw_idx;   // [rw_T][k], the picks of the layer's front
  float *rw_w;             // [rw_T][k]
  int rw_T;
};

// Routing weights of token t = (warps in the grid - 1 - this warp), the same
// arithmetic as route_kernel (exp in double of each pick's logit minus the
// largest, xor-butterfly sum, one division, then float; a largest logit of +inf
// splits the weight among the +inf picks, one of -inf gives 1/k), or 1/k for a
// row holding a NaN, whose picks are experts 0..k-1.  Only the combine reads
// them, so they need not hold up the front of the layer.  The warp is converged.
__device__ __forceinline__ void route_weights_tail(const RowsParams &P) {
  const long long gw = static_cast<long long>(blockIdx.x) * kGvWarps + (threadIdx.x >> 5);
  const long long t = static_cast<long long>(gridDim.x) * kGvWarps - 1 - gw;
  if (t >= P.rw_T) return;
  const int lane = threadIdx.x & 31, k = P.k, E = P.E;
  const float *row = P.rw_logits + t * E;
  bool nan_here = false;
  for (int e = lane; e < E; e += 32) {
    const float v = __ldg(row + e);
    nan_here |= v != v;
  }
  const bool active = lane < k;
  float wj;
  if (__any_sync(0xFFFFFFFFu, nan_here)) {
    wj = 1.0f / static_cast<float>(k);
  } else {
    const int pick = active ? min(max(P.rw_idx[t * k + lane], 0), E - 1) : 0;
    wj = warp_route_weight(active ? __ldg(row + pick) : 0.f, k);  // the first pick holds the largest logit
  }
  if (active) P.rw_w[t * k + lane] = wj;
}

__device__ __forceinline__ const uint8_t *ldg_ptr(const uint8_t *const *arr, int e) {
  return reinterpret_cast<const uint8_t *>(__ldg(reinterpret_cast<const unsigned long long *>(arr) + e));
}

// KIND 0 (gate/up): an item is one row pair (gate row i, up row I + i), K = H.
// KIND 1 (down):    an item is R = 4 consecutive rows of W2, K = I.
// A warp issues every 16-byte code load of its item's K segment (NJ chunks per
// lane and row, one segment when K <= 32 * 32 * NJ) before it computes, and many
// warps per SM keep loads in flight while others compute.  EXACT instances serve
// K = 1024 * NJ exactly (every lane has NJ chunks, no guards in the loop).
template <int KIND, int R, int NT, int NJ, bool EXACT>
__global__ void __launch_bounds__(kGvWarps * 32, 2) gemv_rows_kernel(RowsParams P) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int K = EXACT ? 1024 * NJ : (KIND == 0 ? P.H : P.I);
  const int nch = K / 32;                                  // 32-value chunks per row (a constant when EXACT)
  const int nseg = EXACT ? 1 : (nch + 32 * NJ - 1) / (32 * NJ);  // K segments
  const int per_slot = KIND == 0 ? P.I : (P.H + R - 1) / R;
  const long long nitems = static_cast<long long>(P.meta[0]) * per_slot;
  const long long stride = static_cast<long long>(gridDim.x) * kGvWarps;
  const size_t cbytes = static_cast<size_t>(K) / 2, sbytes = static_cast<size_t>(nch);
  for (long long item = static_cast<long long>(blockIdx.x) * kGvWarps + (threadIdx.x >> 5); item < nitems;
       item += stride) {
    const int4 sl = __ldg(P.slots + static_cast<int>(item / per_slot));  // {expert, first position, tokens, present}
    const int rb = static_cast<int>(item % per_slot);
    const bool present = sl.w != 0;
    // row pointers, advanced to the lane's first chunk
    const uint8_t *cr[R], *sr[R];
    if (present) {
      const uint8_t *cb = ldg_ptr(KIND == 0 ? P.w.w13_codes : P.w.w2_codes, sl.x);
      const uint8_t *sb = ldg_ptr(KIND == 0 ? P.w.w13_scales : P.w.w2_scales, sl.x);
#pragma unroll
      for (int r = 0; r < R; ++r) {
        int row;
        if (KIND == 0) row = r == 0 ? rb : P.I + rb;
        else row = min(rb * R + r, P.H - 1);  // rows past H are computed (duplicates), not stored
        cr[r] = cb + row * cbytes + 16 * lane;
        sr[r] = sb + row * sbytes + lane;
      }
    }
    uint4 cw[R][NJ];
    uint32_t sc[R][NJ];
    for (int g = 0; g * NT < sl.z; ++g) {
      const int p0 = sl.y + g * NT;
      const int nt = min(NT, sl.z - g * NT);
      const uint4 *arow[NT];
      int aexp[NT];
      float acc[R][NT];
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        int row = 0, ex = 0;
        if (t < nt) {
          if (KIND == 0) {
            const int a = __ldg(P.perm + p0 + t);
            const bool ok = a >= 0 && a < P.A;
            if (!ok) set_status(P.status, K3MOE_DEV_BOUNDS);
            row = ok ? a / P.k : 0;
          } else {
            row = p0 + t;
          }
          ex = __ldg(P.aexp + row);
        }
        arow[t] = P.act + static_cast<size_t>(row) * (K / 8) + lane;
        aexp[t] = ex;
#pragma unroll
        for (int r = 0; r < R; ++r) acc[r][t] = 0.f;
      }
      for (int seg = 0; present && seg < nseg; ++seg) {
        const int c0 = seg * 32 * NJ;  // first chunk of the segment (lane 0)
        if (seg > 0 || g == 0 || nseg > 1) {
          // every code and scale load of the segment, then the arithmetic
#pragma unroll
          for (int j = 0; j < NJ; ++j) {
            const bool ok = EXACT || c0 + 32 * j + lane < nch;
#pragma unroll
            for (int r = 0; r < R; ++r) {
              cw[r][j] = ok ? ldg_nc_v4(cr[r] + 16 * (c0 + 32 * j)) : make_uint4(0, 0, 0, 0);
              sc[r][j] = ok ? __ldg(sr[r] + c0 + 32 * j) : 127u;
            }
          }
        }
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
          const int cj = c0 + 32 * j;  // chunk of lane 0; the lane's chunk is cj + lane
          if (EXACT || cj + lane < nch) {
            constexpr int kP = NT == 1 ? 2 : 1;  // partial sums per (row, token)
            float d[kP][R][NT];
#pragma unroll
            for (int i = 0; i < kP; ++i)
#pragma unroll
              for (int r = 0; r < R; ++r)
#pragma unroll
                for (int t = 0; t < NT; ++t) d[i][r][t] = 0.f;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint32_t wh[R][4];
#pragma unroll
              for (int r = 0; r < R; ++r) {
                const uint32_t word = q == 0 ? cw[r][j].x : q == 1 ? cw[r][j].y : q == 2 ? cw[r][j].z : cw[r][j].w;
                e2m1x8_to_f16x2(word, wh[r]);
              }
#pragma unroll
              for (int t = 0; t < NT; ++t) {
                if (t == 0 || t < nt) {  // a group has at least one token
                  const uint4 xv = __ldg(arow[t] + q * nch + cj);
#pragma unroll
                  for (int r = 0; r < R; ++r) {
                    d[0][r][t] = fma2_f16_f32(wh[r][0], xv.x, d[0][r][t]);
                    d[kP - 1][r][t] = fma2_f16_f32(wh[r][1], xv.y, d[kP - 1][r][t]);
                    d[0][r][t] = fma2_f16_f32(wh[r][2], xv.z, d[0][r][t]);
                    d[kP - 1][r][t] = fma2_f16_f32(wh[r][3], xv.w, d[kP - 1][r][t]);
                  }
                }
              }
            }
#pragma unroll
            for (int r = 0; r < R; ++r) {
              const float sf = e8m0_to_f32(sc[r][j]);
#pragma unroll
              for (int t = 0; t < NT; ++t)
                acc[r][t] = fmaf(kP == 2 ? d[0][r][t] + d[kP - 1][r][t] : d[0][r][t], sf, acc[r][t]);
            }
          }
        }
      }
      // reduce across the warp and write
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) acc[r][t] += __shfl_xor_sync(0xFFFFFFFFu, acc[r][t], off);
      if (KIND == 0) {
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          if (lane == t && t < nt) {
            float hv = 0.f;
            if (present) {
              const float gg = scale_pow2(acc[0][t], aexp[t]);
              const float uu = scale_pow2(acc[R - 1][t], aexp[t]);
              hv = (gg / (1.0f + expf(-gg))) * uu;
            }
            const uint16_t hb = f32_to_bf16_rne(hv);
            P.hrow[static_cast<size_t>(p0 + t) * P.I + rb] = hb;
          }
        }
      } else {
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
          for (int t = 0; t < NT; ++t)
            if (lane == r * NT + t && t < nt && rb * R + r < P.H)
              P.Y[static_cast<size_t>(p0 + t) * P.H + rb * R + r] = present ? scale_pow2(acc[r][t], aexp[t]) : 0.f;
      }
    }
  }
  if (KIND == 0 && P.rw_logits) route_weights_tail(P);
}

// ----------------------------------------------------------------------------
// Exact shapes (K = 1024 * NJ), software-pipelined chunk by chunk: a lane holds
// its NJ chunks per row of one item in registers; as soon as chunk j of item i has
// been computed, chunk j of the warp's next item is loaded into its registers, so
// while the warp computes it keeps the rest of item i and the start of item i + 1
// in flight, with the registers of one item.  Tokens are taken one at a time; with
// several tokens on an item the next item's chunks load during its last token.
// Gate/up (KIND 0) keeps a pointer per row (rows i and I + i).  The down rows of
// an item are consecutive (the pipelined down kernel runs only when H is a
// multiple of R, so every row of an item lies below H): one pointer per item, and
// row r at a fixed stride from it, an immediate offset in the loads.
template <int KIND, int R>
struct ItemRows {
  static constexpr int NP = KIND == 1 ? 1 : R;
  int4 sl;                      // slot record {expert, first position, tokens, present}
  int rb;                       // row block of the item
  const uint8_t *cr[NP], *sr[NP];  // the lane's first code chunk and scale byte of each row (or of row 0)
};

template <int KIND, int R, int NJ>
__device__ __forceinline__ const uint8_t *row_codes(const ItemRows<KIND, R> &it, int r) {
  if constexpr (KIND == 1) return it.cr[0] + r * (512 * NJ);
  else return it.cr[r];
}
template <int KIND, int R, int NJ>
__device__ __forceinline__ const uint8_t *row_scales(const ItemRows<KIND, R> &it, int r) {
  if constexpr (KIND == 1) return it.sr[0] + r * (32 * NJ);
  else return it.sr[r];
}

template <int KIND, int R, int NJ>
__device__ __forceinline__ void item_rows_at(const RowsParams &P, long long item, int per_slot,
                                             ItemRows<KIND, R> &it) {
  const int lane = threadIdx.x & 31;
  constexpr size_t cbytes = 512 * NJ, sbytes = 32 * NJ;  // K/2 and K/32 for K = 1024 * NJ
  it.sl = __ldg(P.slots + static_cast<int>(item / per_slot));
  it.rb = static_cast<int>(item % per_slot);
  const uint8_t *cb = nullptr, *sb = nullptr;
  if (it.sl.w) {
    cb = ldg_ptr(KIND == 0 ? P.w.w13_codes : P.w.w2_codes, it.sl.x);
    sb = ldg_ptr(KIND == 0 ? P.w.w13_scales : P.w.w2_scales, it.sl.x);
  }
  if constexpr (KIND == 1) {
    const int row = it.rb * R;
    it.cr[0] = cb + row * cbytes + 16 * lane;
    it.sr[0] = sb + row * sbytes + lane;
  } else {
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int row = r == 0 ? it.rb : P.I + it.rb;
      it.cr[r] = cb + row * cbytes + 16 * lane;
      it.sr[r] = sb + row * sbytes + lane;
    }
  }
}

// 16-byte code load / scale byte load kept in program order (issued ahead of use).
__device__ __forceinline__ uint4 ldg_code_pf(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ldg_u8_pf(const void *p) {
  uint32_t v;
  asm volatile("ld.global.nc.u8 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// Chunks J0 .. J0 + NH - 1 of an item's rows into registers (the lane's 16-byte
// code chunk and scale byte of each row and chunk), in program order.
template <int KIND, int R, int NJ, int J0, int NH>
__device__ __forceinline__ void load_span(const ItemRows<KIND, R> &it, uint4 (&cw)[R][NJ], uint32_t (&sc)[R][NJ]) {
#pragma unroll
  for (int j = 0; j < NH; ++j)
#pragma unroll
    for (int r = 0; r < R; ++r) {
      cw[r][J0 + j] = ldg_code_pf(row_codes<KIND, R, NJ>(it, r) + 16 * 32 * (J0 + j));
      sc[r][J0 + j] = ldg_u8_pf(row_scales<KIND, R, NJ>(it, r) + 32 * (J0 + j));
    }
}

// acc[r] += lane's share of row r . activation over chunks J0 .. J0 + NH - 1.
// Rows are taken in groups of at most four (the activation words are loaded
// again for each group), so that only a group's partial sums are live; each
// row's sums are formed in the same order whatever the grouping.
template <int R, int NJ, int J0, int NH, int NCH>
__device__ __forceinline__ void compute_span(const uint4 (&cw)[R][NJ], const uint32_t (&sc)[R][NJ],
                                             const uint4 *arow, float (&acc)[R]) {
  constexpr int RG = R < 4 ? R : 4;
#pragma unroll
  for (int j = J0; j < J0 + NH; ++j) {
#pragma unroll
    for (int g = 0; g < R; g += RG) {
      float d0[RG], d1[RG];
#pragma unroll
      for (int r = 0; r < RG; ++r) d0[r] = d1[r] = 0.f;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 xv = __ldg(arow + q * NCH + 32 * j);
#pragma unroll
        for (int r = 0; r < RG; ++r) {
          if (g + r >= R) break;  // the last group may be short
          uint32_t wh[4];
          const uint4 &c = cw[g + r][j];
          const uint32_t word = q == 0 ? c.x : q == 1 ? c.y : q == 2 ? c.z : c.w;
          e2m1x8_to_f16x2(word, wh);
          d0[r] = fma2_f16_f32(wh[0], xv.x, d0[r]);
          d1[r] = fma2_f16_f32(wh[1], xv.y, d1[r]);
          d0[r] = fma2_f16_f32(wh[2], xv.z, d0[r]);
          d1[r] = fma2_f16_f32(wh[3], xv.w, d1[r]);
        }
      }
#pragma unroll
      for (int r = 0; r < RG; ++r)
        if (g + r < R) acc[g + r] = fmaf(d0[r] + d1[r], e8m0_to_f32(sc[g + r][j]), acc[g + r]);
    }
  }
}

// Spans of PS chunks from chunk J on: each is computed from the registers, then,
// when the warp moves on to the next item after this token, the same chunks of the
// next item are loaded into those registers.  While a span is computed, the rest
// of the item and the next item's earlier spans are in flight: with PS = 1 about
// NJ - 1 of the NJ chunks of a row, and each load has most of an item's compute
// time to arrive.  The chunks are summed in the same order whatever PS is.
template <int KIND, int R, int NJ, int NCH, int PS, int J>
__device__ __forceinline__ void spans_from(const ItemRows<KIND, R> &nxt, bool present, bool reload,
                                          uint4 (&cw)[R][NJ], uint32_t (&sc)[R][NJ], const uint4 *arow,
                                          float (&acc)[R]) {
  if constexpr (J < NJ) {
    constexpr int NH = NJ - J < PS ? NJ - J : PS;
    if (present) compute_span<R, NJ, J, NH, NCH>(cw, sc, arow, acc);
    if (reload) load_span<KIND, R, NJ, J, NH>(nxt, cw, sc);
    spans_from<KIND, R, NJ, NCH, PS, J + NH>(nxt, present, reload, cw, sc, arow, acc);
  }
}

__device__ __forceinline__ void prefetch_line_l2(const void *p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<uint64_t>(p)));
}

// Down projection only: the weight rows of the warp's first two items into L2
// before the kernel waits for its predecessor.  The slot table comes from a kernel
// that completed before this one was launched and is read through L2 (bounds
// checked all the same); the weights are not written by the predecessor.  It is a
// hint: the rows are loaded again after the wait.
template <int R, int NJ>
__device__ __forceinline__ void prefetch_first_items(const RowsParams &P, int per_slot, long long item,
                                                     long long stride) {
  const int lane = threadIdx.x & 31;
  const int nsl = min(__ldcg(P.meta), min(P.A, P.E));
  const long long nit = static_cast<long long>(max(nsl, 0)) * per_slot;
  for (int q = 0; q < 2; ++q, item += stride) {
    if (item >= nit) return;
    const int4 sl = __ldcg(P.slots + static_cast<int>(item / per_slot));
    if (!sl.w || sl.x < 0 || sl.x >= P.E) continue;
    const uint8_t *cb = ldg_ptr(P.w.w2_codes, sl.x), *sb = ldg_ptr(P.w.w2_scales, sl.x);
    if (!cb || !sb) continue;
    const int rb = static_cast<int>(item % per_slot);
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int row = min(rb * R + r, P.H - 1);
#pragma unroll
      for (int j = 0; j < NJ; ++j) prefetch_line_l2(cb + static_cast<size_t>(row) * (512 * NJ) + 16 * lane + 512 * j);
      if (lane == 0) prefetch_line_l2(sb + static_cast<size_t>(row) * (32 * NJ));
    }
  }
}

// Chunks per span of the software pipeline (spans_from).
constexpr int kSpanChunks = 1;

// The warp's items item, item + stride, ... below nitems.
template <int KIND, int R, int NJ>
__device__ __forceinline__ void rows_pipe_items(const RowsParams &P, long long item, long long stride, int per_slot,
                                                long long nitems) {
  constexpr int NCH = 32 * NJ;  // chunks per row
  const int lane = threadIdx.x & 31;
  if (item >= nitems) return;
  ItemRows<KIND, R> cur;
  item_rows_at<KIND, R, NJ>(P, item, per_slot, cur);
  uint4 cw[R][NJ];
  uint32_t sc[R][NJ];
  if (cur.sl.w) load_span<KIND, R, NJ, 0, NJ>(cur, cw, sc);
  for (;;) {
    const long long nitem = item + stride;
    const bool has_next = nitem < nitems;
    ItemRows<KIND, R> nxt;
    if (has_next) item_rows_at<KIND, R, NJ>(P, nitem, per_slot, nxt);
    const bool pf = has_next && nxt.sl.w;
    for (int t = 0; t < cur.sl.z; ++t) {
      const int p = cur.sl.y + t;
      const bool last = t == cur.sl.z - 1;
      int row, ex;
      if (KIND == 0) {
        const int a = __ldg(P.perm + p);
        const bool ok = a >= 0 && a < P.A;
        if (!ok) set_status(P.status, K3MOE_DEV_BOUNDS);
        row = ok ? a / P.k : 0;
      } else {
        row = p;
      }
      ex = __ldg(P.aexp + row);
      const uint4 *arow = P.act + static_cast<size_t>(row) * (NCH * 4) + lane;
      float acc[R];
#pragma unroll
      for (int r = 0; r < R; ++r) acc[r] = 0.f;
      spans_from<KIND, R, NJ, NCH, kSpanChunks, 0>(nxt, cur.sl.w != 0, last && pf, cw, sc, arow, acc);
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc[r] += __shfl_xor_sync(0xFFFFFFFFu, acc[r], off);
      if (KIND == 0) {
        if (lane == 0) {
          float hv = 0.f;
          if (cur.sl.w) {
            const float gg = scale_pow2(acc[0], ex);
            const float uu = scale_pow2(acc[R - 1], ex);
            hv = (gg / (1.0f + expf(-gg))) * uu;
          }
          const uint16_t hb = f32_to_bf16_rne(hv);
          P.hrow[static_cast<size_t>(p) * P.I + cur.rb] = hb;
        }
      } else {
#pragma unroll
        for (int r = 0; r < R; ++r)
          if (lane == r && cur.rb * R + r < P.H)
            P.Y[static_cast<size_t>(p) * P.H + cur.rb * R + r] = cur.sl.w ? scale_pow2(acc[r], ex) : 0.f;
      }
    }
    if (!has_next) break;
    item = nitem;
    cur = nxt;
  }
}

template <int KIND, int R, int NJ>
__global__ void __launch_bounds__(kGvWarps * 32, 2) gemv_rows_pipe_kernel(RowsParams P) {
  const int per_slot = KIND == 0 ? P.I : (P.H + R - 1) / R;
  const long long stride = static_cast<long long>(gridDim.x) * kGvWarps;
  const long long item = static_cast<long long>(blockIdx.x) * kGvWarps + (threadIdx.x >> 5);
  if (KIND == 1) prefetch_first_items<R, NJ>(P, per_slot, item, stride);
  pdl_wait();
  pdl_trigger();
  rows_pipe_items<KIND, R, NJ>(P, item, stride, per_slot, static_cast<long long>(P.meta[0]) * per_slot);
  if (KIND == 0 && P.rw_logits) route_weights_tail(P);
}

// ----------------------------------------------------------------------------
size_t ffn_gemv_workspace(const k3moe_shape &s) { return gemv_ws(s.T, s.H, s.I, s.E, s.k).total; }
size_t ffn_gemv_h_offset(const k3moe_shape &s) { return gemv_ws(s.T, s.H, s.I, s.E, s.k).hrow; }

namespace {

// Blocks of a persistent grid: resident blocks per SM (occupancy, cached per kernel) x SMs.
template <int KIND, int R, int NT, int NJ, bool EXACT>
int persistent_grid(int nsm) {
  static int nb = 0;
  if (nb == 0) {
    int v = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, gemv_rows_kernel<KIND, R, NT, NJ, EXACT>, kGvWarps * 32,
                                                      0) !=
            cudaSuccess ||
        v < 1)
      v = 1;
    nb = v;
  }
  return nsm * nb;
}

template <int KIND, int R, int NT, int NJ, bool EXACT>
cudaError_t launch_rows_kernel(const RowsParams &P, int nsm, cudaStream_t st) {
  return launch_pdl(gemv_rows_kernel<KIND, R, NT, NJ, EXACT>, dim3(persistent_grid<KIND, R, NT, NJ, EXACT>(nsm)),
                    dim3(kGvWarps * 32), 0, st, P);
}

// One token.  Gate/up (2 rows): exact instances for K/32 = 32 * NJ with NJ in
// {2, 4, 7}.  Down (7 or 8 consecutive rows): 2 chunks per lane and row (exact
// for K = 2048).
template <int KIND, int R, int NJ>
cudaError_t launch_rows_pipe(const RowsParams &P, int nsm, cudaStream_t st) {
  static int nb = 0;
  if (nb == 0) {
    int v = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, gemv_rows_pipe_kernel<KIND, R, NJ>, kGvWarps * 32, 0) !=
            cudaSuccess ||
        v < 1)
      v = 1;
    nb = v;
  }
  return launch_pdl(gemv_rows_pipe_kernel<KIND, R, NJ>, dim3(nsm * nb), dim3(kGvWarps * 32), 0, st, P);
}

// Gate/up (2 rows): pipelined exact instances for K/32 = 32 * NJ with NJ in
// {2, 4, 7}, else the guarded kernel holding 8 chunks per lane and row (several
// segments past K = 8192).  Down: the pipelined exact instance for K = 2048 (7 or
// 8 rows per item), else the guarded kernel with 4 rows and 2 chunks per lane and
// row.
template <int KIND, int R>
cudaError_t launch_rows_nt1(const RowsParams &P, int K, int nsm, cudaStream_t st) {
  const int nch = K / 32;
  if constexpr (KIND == 1) {
    // the pipelined kernel takes 7 rows per item when 7 divides H (H = 7 x 1024 in
    // the decode shape; 7 rows of codes fit the 128 registers, 8 spill ten words),
    // else 8 (H is a multiple of 32): every row of an item lies below H
    if (nch == 64 && P.H % 7 == 0) return launch_rows_pipe<KIND, 7, 2>(P, nsm, st);
    if (nch == 64 && P.H % 8 == 0) return launch_rows_pipe<KIND, 8, 2>(P, nsm, st);
    return launch_rows_kernel<KIND, R, 1, 2, false>(P, nsm, st);
  } else {
    if (nch == 64) return launch_rows_pipe<KIND, R, 2>(P, nsm, st);
    if (nch == 128) return launch_rows_pipe<KIND, R, 4>(P, nsm, st);
    if (nch == 224) return launch_rows_pipe<KIND, R, 7>(P, nsm, st);
    return launch_rows_kernel<KIND, R, 1, 8, false>(P, nsm, st);
  }
}

// gate/up -> h to f16 -> down.  P holds the gate/up activations (x16, xexp);
// h16/hexp are the down activations.  Tokens are taken one at a time: an item's
// weight codes stay in registers while the warp loops over the expert's tokens.
int launch_rows(RowsParams P, int nsm, cudaStream_t st, int A, uint4 *h16, int32_t *hexp) {
  if (launch_rows_nt1<0, 2>(P, P.H, nsm, st) != cudaSuccess) return -1;
  if (launch_pdl(gemv_h16_kernel, dim3(A), dim3(256), 0, st, static_cast<const uint16_t *>(P.hrow), P.I, h16,
                 hexp) != cudaSuccess)
    return -1;
  P.aexp = hexp;
  P.act = h16;
  return launch_rows_nt1<1, kDnRows>(P, P.I, nsm, st) == cudaSuccess ? 0 : -1;
}

}  // namespace

GemvBufs gemv_bufs(const k3moe_shape &s, void *ws) {
  const GemvWs L = gemv_ws(s.T, s.H, s.I, s.E, s.k);
  char *base = static_cast<char *>(ws);
  GemvBufs b;
  b.slots = reinterpret_cast<int4 *>(base + L.slots);
  b.meta = reinterpret_cast<int32_t *>(base + L.meta);
  b.xexp = reinterpret_cast<int32_t *>(base + L.xexp);
  b.x16 = reinterpret_cast<uint4 *>(base + L.x16);
  b.hrow = reinterpret_cast<uint16_t *>(base + L.hrow);
  b.h16 = reinterpret_cast<uint4 *>(base + L.h16);
  b.hexp = reinterpret_cast<int32_t *>(base + L.hexp);
  return b;
}

int launch_gemv_prep(const k3moe_shape &s, const uint16_t *x, const k3moe_weights &w, const int32_t *offsets,
                     const GemvBufs &b, int32_t *status, cudaStream_t st) {
  return launch_pdl(gemv_prep_kernel, dim3(1 + s.T), dim3(256), 0, st, w, x, s.T, s.H, s.E, s.T * s.k, offsets,
                    b.slots, b.meta, b.xexp, b.x16, status) == cudaSuccess
             ? 0
             : -1;
}

int launch_gemv_h16(const k3moe_shape &s, const GemvBufs &b, cudaStream_t st) {
  return launch_pdl(gemv_h16_kernel, dim3(s.T * s.k), dim3(256), 0, st, static_cast<const uint16_t *>(b.hrow), s.I,
                    b.h16, b.hexp) == cudaSuccess
             ? 0
             : -1;
}

int sm_count() {
  static int nsm = 0;
  if (nsm == 0) {
    int dev = 0, v = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    nsm = v < 1 ? 1 : v;
  }
  return nsm;
}

// ----------------------------------------------------------------------------
// Decode front in one block: route, bucket and the GEMV prep of a small batch
// (T <= 4 tokens, E <= 1024 experts, A = T k <= 128), writing what the route,
// bucket and prep kernels write (same selection order, same stable bucket order,
// same slots and prescaled activations) but the routing weights, which the
// gate/up kernel's last warps compute once their items are done
// (route_weights_tail): only the combine reads them.
//  * before the block waits for its predecessor it hints its inputs into L2:
//    the logits and x rows and the four per-expert pointer arrays, which are cold
//    after a step's weight stream (a prefetch returns nothing to the block, so it
//    cannot let the block see a value that the predecessor has yet to write);
//  * route: warp t takes token t with warp-level operations only: lane l holds
//    the order-preserving keys of experts l, l + 32, ...; k rounds of a warp
//    arg-max (two warp reductions each: the largest key, then the smallest
//    index holding it) give the picks in (key desc, index asc) order, the
//    winning lane finding its next best by a pairwise tree over its keys;
//    meanwhile warps 4..31 take the presence flags of every expert (from its
//    four weight pointers) and the max |x| of row slices;
//  * bucket, by counting over the A <= 128 assignments: assignment a's place is
//    #{a' : (idx[a'], a') < (idx[a], a)}, which sorts the experts; meanwhile
//    warps 4..31 write the x rows as prescaled f16; offsets and counts come
//    from binary searches in the sorted experts;
//  * prep: the first position of each expert writes its active slot (the number
//    of distinct experts before it).
// Two block barriers in all.
namespace {

constexpr int kFrontMaxT = 4, kFrontMaxE = 1024, kFrontMaxA = 128;
constexpr int kFrontKeys = kFrontMaxE / 32;            // keys per lane
constexpr int kFrontAux = 1024 - 32 * kFrontMaxT;      // threads of warps 4..31

}  // namespace

__global__ void __launch_bounds__(1024)
    layer_front_kernel(const float *__restrict__ logits, const uint16_t *__restrict__ x, k3moe_weights w, int T,
                       int H, int E, int k, int32_t *__restrict__ idx, int32_t *__restrict__ counts,
                       int32_t *__restrict__ offsets, int32_t *__restrict__ perm, int32_t *__restrict__ inv,
                       int4 *__restrict__ slots, int32_t *__restrict__ meta, int32_t *__restrict__ xexp,
                       uint4 *__restrict__ x16, int32_t *status) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  {  // L2 hints, one 128-byte line per thread and pass
    const long long bl = 4LL * T * E, bx = 2LL * T * H, bp = 8LL * E;
    const long long nl = (bl + 127) / 128, nx = (bx + 127) / 128, np = (bp + 127) / 128;
    for (long long i = tid; i < nl + nx + 4 * np; i += 1024) {
      const char *p;
      if (i < nl) {
        p = reinterpret_cast<const char *>(logits) + min(128 * i, bl - 1);
      } else if (i < nl + nx) {
        p = reinterpret_cast<const char *>(x) + min(128 * (i - nl), bx - 1);
      } else {
        const long long j = i - nl - nx, a = j / np, o = j - a * np;
        const void *arr = a == 0 ? static_cast<const void *>(w.w13_codes)
                          : a == 1 ? static_cast<const void *>(w.w13_scales)
                          : a == 2 ? static_cast<const void *>(w.w2_codes)
                                   : static_cast<const void *>(w.w2_scales);
        p = reinterpret_cast<const char *>(arr) + min(128 * o, bp - 1);
      }
      prefetch_line_l2(p);
    }
  }
  pdl_wait();
  pdl_trigger();
  __shared__ int s_idx[kFrontMaxA];
  __shared__ int s_sorted[kFrontMaxA];
  __shared__ int s_pres_sorted[kFrontMaxA];  // expert_flags per bucket position
  __shared__ unsigned char s_flag[kFrontMaxE];  // expert_flags per expert
  __shared__ float s_xpart[32];
  const int A = T * k;
  // ---- phase A: warp t < T routes token t; warps 4..31 take the experts' flags
  //      and the max |x| of row slices
  if (warp < T) {
    const int t = warp;
    const float *row = logits + static_cast<size_t>(t) * E;
    uint32_t key[kFrontKeys];
    bool nan_here = false;
#pragma unroll
    for (int i = 0; i < kFrontKeys; ++i) {
      const int e = lane + 32 * i;
      float v = 0.f;
      if (e < E) v = __ldg(row + e);
      nan_here |= e < E && v != v;
      key[i] = e < E ? order_key(v) : 0u;  // 0: no expert (every real key is larger)
    }
    if (__any_sync(0xFFFFFFFFu, nan_here)) {  // a NaN row: experts 0..k-1 (weights 1/k)
      if (lane < k) {
        idx[t * k + lane] = lane;
        s_idx[t * k + lane] = lane;
      }
      if (lane == 0) set_status(status, K3MOE_DEV_NONFINITE);
    } else {
      // the k picks in (key desc, index asc) order (warp_top_k: one warp arg-max
      // per pick); every expert e < E has a key above 0 and k <= E
      const int pick = warp_top_k<kFrontKeys>(key, k);
      if (lane < k) {
        idx[t * k + lane] = pick;
        s_idx[t * k + lane] = pick;
      }
    }
  } else if (warp >= kFrontMaxT) {
    for (int e = tid - 32 * kFrontMaxT; e < E; e += kFrontAux)
      s_flag[e] = static_cast<unsigned char>(expert_flags(ldg_ptr(w.w13_codes, e), ldg_ptr(w.w13_scales, e),
                                                          ldg_ptr(w.w2_codes, e), ldg_ptr(w.w2_scales, e)));
    // partial max |x| of a slice of one token's row (16-byte loads)
    const int nw = 32 - kFrontMaxT, wpt = nw / T, wr = warp - kFrontMaxT;
    if (wr < wpt * T) {
      const int t = wr / wpt, part = wr % wpt;
      const int n16 = H / 8, per = (n16 + wpt - 1) / wpt;
      const uint4 *xr = reinterpret_cast<const uint4 *>(x + static_cast<size_t>(t) * H);
      float mx = 0.f;
#pragma unroll 4
      for (int c = part * per + lane; c < min(n16, (part + 1) * per); c += 32) {
        const uint4 v = __ldg(xr + c);
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int m = 0; m < 4; ++m)
          mx = fmaxf(mx, fmaxf(fabsf(__uint_as_float(u[m] << 16)), fabsf(__uint_as_float(u[m] & 0xFFFF0000u))));
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
      if (lane == 0) s_xpart[wr] = mx;
    }
  }
  __syncthreads();
  // ---- phase B: each assignment's place in (expert, assignment) order (warps
  //      0..3, as A <= 128); warps 4..31 write x as prescaled f16 (piece-major)
  if (tid < A) {
    const int e = s_idx[tid];
    int p = 0;
    for (int a = 0; a < A; ++a) p += s_idx[a] < e || (s_idx[a] == e && a < tid);
    perm[p] = tid;
    inv[tid] = p;
    s_sorted[p] = e;
    s_pres_sorted[p] = s_flag[e];
  }
  if (warp >= kFrontMaxT) {
    const int wpt = (32 - kFrontMaxT) / T, n8 = H / 8, nch = H / 32;
    for (int i = tid - 32 * kFrontMaxT; i < T * n8; i += kFrontAux) {
      const int t = i / n8, piece = i - t * n8;  // piece = c * 4 + q (source order)
      float mx = 0.f;
      for (int j = 0; j < wpt; ++j) mx = fmaxf(mx, s_xpart[t * wpt + j]);
      const int pe = prescale_exp(mx);
      if (piece == 0) xexp[t] = pe;
      const float sc = scale_pow2(1.0f, -pe);
      const uint4 v = __ldg(reinterpret_cast<const uint4 *>(x + static_cast<size_t>(t) * H) + piece);
      const uint32_t u[4] = {v.x, v.y, v.z, v.w};
      uint32_t o[4];
#pragma unroll
      for (int m = 0; m < 4; ++m)
        o[m] = pack_f16x2_scaled(__uint_as_float(u[m] << 16), __uint_as_float(u[m] & 0xFFFF0000u), sc);
      x16[static_cast<size_t>(t) * n8 + (piece & 3) * nch + (piece >> 2)] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
  __syncthreads();
  // ---- phase C: offsets and counts by binary search in the sorted experts,
  //      active slots (first position of each expert)
  for (int e = tid; e <= E; e += 1024) {
    int lo = 0, hi = A;  // first position with expert >= e
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (s_sorted[mid] < e) lo = mid + 1; else hi = mid;
    }
    offsets[e] = lo;
    if (e < E) {
      int lo2 = lo, hi2 = A;  // first position with expert > e
      while (lo2 < hi2) {
        const int mid = (lo2 + hi2) >> 1;
        if (s_sorted[mid] <= e) lo2 = mid + 1; else hi2 = mid;
      }
      counts[e] = lo2 - lo;
    }
  }
  if (tid < A && (tid == 0 || s_sorted[tid] != s_sorted[tid - 1])) {
    const int e = s_sorted[tid];
    int slot = 0, end = tid + 1;
    for (int p = 1; p <= tid; ++p) slot += s_sorted[p] != s_sorted[p - 1];
    while (end < A && s_sorted[end] == e) ++end;
    const int fl = s_pres_sorted[tid];
    const bool pr = (fl & 1) != 0;
    if (fl == 2) set_status(status, K3MOE_DEV_BOUNDS);  // non-NULL but misaligned: treated as absent
    slots[slot] = make_int4(e, tid, end - tid, pr ? 1 : 0);
  }
  if (tid == 0) {
    int n = A > 0 ? 1 : 0;
    for (int p = 1; p < A; ++p) n += s_sorted[p] != s_sorted[p - 1];
    meta[0] = n;
  }
}

bool layer_front_fits(const k3moe_shape &s) {
  return s.T <= kFrontMaxT && s.E <= kFrontMaxE && s.T * s.k <= kFrontMaxA;
}

// route + bucket + GEMV prep in one block, then the GEMV kernels (the gate/up
// kernel also writes the routing weights) and the combine.
int launch_layer_gemv_fast(const k3moe_shape &s, const float *logits, const uint16_t *x, const k3moe_weights &w,
                           int32_t *idx, float *wts, int32_t *counts, int32_t *offsets, int32_t *perm, int32_t *inv,
                           float *Y, uint16_t *out, float *out_f32, void *ws, int32_t *status, cudaStream_t st) {
  if (s.T == 0) return 0;
  const GemvBufs b = gemv_bufs(s, ws);
  if (launch_pdl(layer_front_kernel, dim3(1), dim3(1024), 0, st, logits, x, w, s.T, s.H, s.E, s.k, idx, counts,
                 offsets, perm, inv, b.slots, b.meta, b.xexp, b.x16, status) != cudaSuccess)
    return -1;
  RowsParams P;
  P.w = w;
  P.H = s.H;
  P.I = s.I;
  P.k = s.k;
  P.A = s.T * s.k;
  P.E = s.E;
  P.perm = perm;
  P.slots = b.slots;
  P.meta = b.meta;
  P.aexp = b.xexp;
  P.act = b.x16;
  P.hrow = b.hrow;
  P.Y = Y;
  P.status = status;
  P.rw_logits = logits;
  P.rw_idx = idx;
  P.rw_w = wts;
  P.rw_T = s.T;
  if (launch_rows(P, sm_count(), st, P.A, b.h16, b.hexp)) return -1;
  return launch_combine(s, Y, wts, inv, nullptr, out, out_f32, st);
}

int launch_ffn_gemv(const k3moe_shape &s, const uint16_t *x, const k3moe_weights &w,
                    const int32_t *offsets, const int32_t *perm, float *Y, void *ws,
                    int32_t *status, cudaStream_t st) {
  if (s.T == 0) return 0;
  const GemvBufs b = gemv_bufs(s, ws);
  if (launch_gemv_prep(s, x, w, offsets, b, status, st)) return -1;
  RowsParams P;
  P.w = w;
  P.H = s.H;
  P.I = s.I;
  P.k = s.k;
  P.A = s.T * s.k;
  P.E = s.E;
  P.perm = perm;
  P.slots = b.slots;
  P.meta = b.meta;
  P.aexp = b.xexp;
  P.act = b.x16;
  P.hrow = b.hrow;
  P.Y = Y;
  P.status = status;
  P.rw_logits = nullptr;
  P.rw_idx = nullptr;
  P.rw_w = nullptr;
  P.rw_T = 0;
  return launch_rows(P, sm_count(), st, P.A, b.h16, b.hexp);
}

}  // namespace k3moe
