// ffn_gemv.cu -- MXFP4 SwiGLU expert FFN as streaming GEMVs on the CUDA cores.
//
// The kimi-k3-in-c CHANGELOG walkthrough ("[0.1.0] Added") describes a matmul that
// reads the packed MXFP4 nibbles directly and never materialises a dequantised
// expert, and a gated-linear-unit expert.  Here every weight byte is read once
// per (expert, token chunk) with 128-bit coalesced loads, decoded in registers
// (cvt e2m1x2 -> f16x2, exact), multiplied by f16 activations with exact
// products accumulated in fp32, scaled per 32-block by the e8m0 scale, and
// reduced across the warp with shuffles.  The order of every sum is fixed.
//
// Activations are staged as f16 after an exact power-of-two prescale per row
// (x' = x * 2^-p with max|x'| in [2^14, 2^15)), so bf16 values convert to f16
// without rounding except for elements below 2^-28 * max|x| (error < 2^-25 of max).
//
// Kernels (one expert FFN call):
//   ffn_prep     active-expert list, offsets check, x -> prescaled f16 (piece-major)
//   ffn_gateup   h[p] = bf16(silu(Wg x) * (Wu x)) for every bucket position p
//   ffn_down     Y[p] = Wd h[p]
#include <cuda_fp16.h>

#include "k3moe_dev.cuh"
#include "k3moe_launch.h"

namespace k3moe {

namespace {

constexpr int kWarps = 8;  // warps per block
constexpr int kNT = 4;     // tokens per pass over a weight tile

// Workspace layout (byte offsets, 256-aligned pieces).
struct GemvWs {
  size_t active, nactive, xexp, x16, hrow, total;
};

__host__ __device__ inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

__host__ __device__ inline GemvWs gemv_ws(int T, int H, int I, int E, int k) {
  GemvWs w;
  size_t o = 0;
  w.active = o;
  o = align256(o + sizeof(int32_t) * E);
  w.nactive = o;
  o = align256(o + sizeof(int32_t));
  w.xexp = o;
  o = align256(o + sizeof(int32_t) * (T > 0 ? T : 1));
  w.x16 = o;
  o = align256(o + sizeof(uint16_t) * static_cast<size_t>(T) * H);
  w.hrow = o;
  o = align256(o + sizeof(uint16_t) * static_cast<size_t>(T) * k * I);
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

}  // namespace

// An expert takes part when its four pointers are non-NULL and its code arrays
// are 16-byte aligned (the 128-bit loads need it); otherwise its rows are zero.
__device__ __forceinline__ bool expert_present(const k3moe_weights &w, int e) {
  const uint8_t *a = w.w13_codes[e], *b = w.w13_scales[e], *c = w.w2_codes[e], *d = w.w2_scales[e];
  return a && b && c && d && ((reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(c)) & 15u) == 0;
}

// ----------------------------------------------------------------------------
// prep: block 0 builds the active-expert list; block 1 + t converts x[t].
// x16 layout per token: piece-major, uint4 index q * (H/32) + c holds the f16 of
// columns 32c + 8q .. 32c + 8q + 7 (so a warp's lanes read consecutive 16 B).
__global__ void __launch_bounds__(256)
    ffn_prep_kernel(k3moe_weights w, const uint16_t *__restrict__ x, int T, int H, int E, int A,
                    const int32_t *__restrict__ offsets, int32_t *__restrict__ active,
                    int32_t *__restrict__ nactive, int32_t *__restrict__ xexp,
                    uint4 *__restrict__ x16, int32_t *status) {
  pdl_wait();
  pdl_trigger();
  if (blockIdx.x == 0) {
    if (threadIdx.x >= 32) return;
    const int lane = threadIdx.x;
    int run = 0;
    bool bad = offsets[0] != 0 || offsets[E] > A;
    for (int base = 0; base < E; base += 32) {
      const int e = base + lane;
      int cnt = 0;
      if (e < E) {
        cnt = offsets[e + 1] - offsets[e];
        if (cnt < 0) bad = true;
      }
      const bool f = cnt > 0 && !bad;
      if (f && !expert_present(w, e) && w.w13_codes[e] && w.w13_scales[e] && w.w2_codes[e] &&
          w.w2_scales[e])
        set_status(status, K3MOE_DEV_BOUNDS);  // non-NULL but misaligned: treated as absent
      const unsigned m = __ballot_sync(0xFFFFFFFFu, f);
      if (f) active[run + __popc(m & ((1u << lane) - 1u))] = e;
      run += __popc(m);
    }
    bad = __any_sync(0xFFFFFFFFu, bad);
    if (lane == 0) {
      *nactive = bad ? 0 : run;
      if (bad) set_status(status, K3MOE_DEV_BOUNDS);
    }
    return;
  }
  const int t = blockIdx.x - 1;
  if (t >= T) return;
  const uint16_t *xr = x + static_cast<size_t>(t) * H;
  __shared__ float red[kWarps];
  float mx = 0.f;
  for (int c = threadIdx.x; c < H; c += 256) mx = fmaxf(mx, fabsf(bf16_bits_to_f32(xr[c])));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
  __syncthreads();
  mx = red[0];
  for (int i = 1; i < kWarps; ++i) mx = fmaxf(mx, red[i]);
  const int p = prescale_exp(mx);
  if (threadIdx.x == 0) xexp[t] = p;
  const float s = scale_pow2(1.0f, -p);
  const int nch = H / 32;
  uint4 *dst = x16 + static_cast<size_t>(t) * (H / 8);
  for (int piece = threadIdx.x; piece < H / 8; piece += 256) {  // piece = c*4 + q (source order)
    const int c = piece >> 2, q = piece & 3;
    const uint4 src = *reinterpret_cast<const uint4 *>(xr + 8 * piece);
    const uint32_t w[4] = {src.x, src.y, src.z, src.w};
    uint32_t o[4];
#pragma unroll
    for (int m = 0; m < 4; ++m)
      o[m] = pack_f16x2_scaled(__uint_as_float(w[m] << 16), __uint_as_float(w[m] & 0xFFFF0000u), s);
    dst[q * nch + c] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// ----------------------------------------------------------------------------
// R rows of one expert matrix against NT staged activation rows.
// codes[r], scales[r]: row pointers; nch = K/32 chunks; xs: smem piece-major f16,
// NT rows of K/8 uint4 each.  acc[r][t] accumulates the lane's partial sums.
template <int R, int NT, int B>
__device__ __forceinline__ void mx_rows_dot(const uint8_t *const (&codes)[R],
                                            const uint8_t *const (&scales)[R], int nch,
                                            const uint4 *__restrict__ xs, float (&acc)[R][NT]) {
  const int lane = threadIdx.x & 31;
  for (int c0 = lane; c0 < nch; c0 += 32 * B) {
    uint4 cw[B][R];
    uint32_t sb[B][R];
#pragma unroll
    for (int b = 0; b < B; ++b) {
      const int c = c0 + 32 * b;
#pragma unroll
      for (int r = 0; r < R; ++r) {
        if (c < nch) {
          cw[b][r] = ldg_nc_v4(codes[r] + 16 * static_cast<size_t>(c));
          sb[b][r] = __ldg(scales[r] + c);
        } else {
          cw[b][r] = make_uint4(0, 0, 0, 0);
          sb[b][r] = 0;
        }
      }
    }
#pragma unroll
    for (int b = 0; b < B; ++b) {
      const int c = c0 + 32 * b;
      if (c >= nch) break;
      float d[R][NT];
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int t = 0; t < NT; ++t) d[r][t] = 0.f;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t wh[R][4];  // decoded once, used for all NT tokens
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const uint32_t word = q == 0 ? cw[b][r].x : q == 1 ? cw[b][r].y : q == 2 ? cw[b][r].z : cw[b][r].w;
          e2m1x8_to_f16x2(word, wh[r]);
        }
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const uint4 xv = xs[static_cast<size_t>(t) * (nch * 4) + q * nch + c];
          const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
          for (int r = 0; r < R; ++r)
#pragma unroll
            for (int m = 0; m < 4; ++m) d[r][t] = fma2_f16_f32(wh[r][m], xw[m], d[r][t]);
        }
      }
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const float sf = e8m0_to_f32(sb[b][r]);
#pragma unroll
        for (int t = 0; t < NT; ++t) acc[r][t] = fmaf(d[r][t], sf, acc[r][t]);
      }
    }
  }
}

template <int R, int NT>
__device__ __forceinline__ void warp_allreduce(float (&acc)[R][NT]) {
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc[r][t] += __shfl_xor_sync(0xFFFFFFFFu, acc[r][t], off);
}

// ----------------------------------------------------------------------------
// gate/up: item = (active slot u, block of kWarps * RPW row pairs).
template <int NT>
__device__ void gateup_item_tokens(const uint8_t *__restrict__ w13c, const uint8_t *__restrict__ w13s,
                                   int H, int I, int r0, int rows, const uint4 *xs, const int *ptok_p,
                                   const int *ptok_exp, uint16_t *__restrict__ hrow) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nch = H / 32;
  for (int rr = warp; rr < rows; rr += kWarps) {
    const int r = r0 + rr;
    const uint8_t *codes[2] = {w13c + static_cast<size_t>(r) * (H / 2),
                               w13c + static_cast<size_t>(I + r) * (H / 2)};
    const uint8_t *scales[2] = {w13s + static_cast<size_t>(r) * nch,
                                w13s + static_cast<size_t>(I + r) * nch};
    float acc[2][NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[0][t] = acc[1][t] = 0.f;
    mx_rows_dot<2, NT, 4>(codes, scales, nch, xs, acc);
    warp_allreduce<2, NT>(acc);
    if (lane < NT) {
#pragma unroll
      for (int t = 0; t < NT; ++t)
        if (t == lane) {
          const float g = scale_pow2(acc[0][t], ptok_exp[t]);
          const float u = scale_pow2(acc[1][t], ptok_exp[t]);
          const float hv = (g / (1.0f + expf(-g))) * u;
          hrow[static_cast<size_t>(ptok_p[t]) * I + r] = f32_to_bf16_rne(hv);
        }
    }
  }
}

__global__ void __launch_bounds__(kWarps * 32)
    ffn_gateup_kernel(k3moe_weights w, int T, int H, int I, int k, int E, int A,
                      const int32_t *__restrict__ offsets, const int32_t *__restrict__ perm,
                      const int32_t *__restrict__ active, const int32_t *__restrict__ nactive,
                      const int32_t *__restrict__ xexp, const uint4 *__restrict__ x16,
                      uint16_t *__restrict__ hrow, int rows_per_item, int ntmax, int32_t *status) {
  extern __shared__ uint4 xs[];  // ntmax tokens x H/8 uint4
  __shared__ int tok_p[kNT], tok_t[kNT], tok_exp[kNT];
  pdl_wait();
  pdl_trigger();
  const int n_act = *nactive;
  const int items_per_e = (I + rows_per_item - 1) / rows_per_item;
  const long long n_items = static_cast<long long>(n_act) * items_per_e;
  for (long long item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int u = static_cast<int>(item / items_per_e);
    const int r0 = static_cast<int>(item % items_per_e) * rows_per_item;
    const int rows = min(rows_per_item, I - r0);
    const int e = active[u];
    const int p0 = offsets[e], p1 = offsets[e + 1];
    const bool present = expert_present(w, e);
    for (int pc = p0; pc < p1; pc += ntmax) {
      const int nt = min(ntmax, p1 - pc);
      __syncthreads();  // previous users of xs / tok_* are done
      if (threadIdx.x < nt) {
        const int p = pc + threadIdx.x;
        const int a = perm[p];
        int t = a / k;
        if (a < 0 || a >= A) {
          set_status(status, K3MOE_DEV_BOUNDS);
          t = -1;
        }
        tok_p[threadIdx.x] = p;
        tok_t[threadIdx.x] = t;
        tok_exp[threadIdx.x] = t >= 0 ? xexp[t] : 0;
      }
      __syncthreads();
      if (!present) {
        for (int i = threadIdx.x; i < nt * rows; i += blockDim.x)
          hrow[static_cast<size_t>(tok_p[i / rows]) * I + r0 + i % rows] = 0;
        continue;
      }
      const int row_u4 = H / 8;
      for (int i = threadIdx.x; i < nt * row_u4; i += blockDim.x) {
        const int tt = i / row_u4, j = i % row_u4;
        const int t = tok_t[tt];
        xs[i] = t >= 0 ? x16[static_cast<size_t>(t) * row_u4 + j] : make_uint4(0, 0, 0, 0);
      }
      __syncthreads();
      const uint8_t *w13c = w.w13_codes[e], *w13s = w.w13_scales[e];
      switch (nt) {
        case 1: gateup_item_tokens<1>(w13c, w13s, H, I, r0, rows, xs, tok_p, tok_exp, hrow); break;
        case 2: gateup_item_tokens<2>(w13c, w13s, H, I, r0, rows, xs, tok_p, tok_exp, hrow); break;
        case 3: gateup_item_tokens<3>(w13c, w13s, H, I, r0, rows, xs, tok_p, tok_exp, hrow); break;
        default: gateup_item_tokens<4>(w13c, w13s, H, I, r0, rows, xs, tok_p, tok_exp, hrow); break;
      }
    }
  }
}

// ----------------------------------------------------------------------------
// down: item = (active slot u, block of rows of W2).  Each warp takes 4 rows at a time.
template <int NT>
__device__ void down_item_tokens(const uint8_t *__restrict__ w2c, const uint8_t *__restrict__ w2s,
                                 int H, int I, int r0, int rows, const uint4 *xs, const int *ptok_p,
                                 const int *ptok_exp, float *__restrict__ Y) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nch = I / 32;
  for (int rr = warp * 4; rr < rows; rr += kWarps * 4) {
    const uint8_t *codes[4], *scales[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = r0 + min(rr + i, rows - 1);  // clamp: duplicate rows are computed, not stored
      codes[i] = w2c + static_cast<size_t>(r) * (I / 2);
      scales[i] = w2s + static_cast<size_t>(r) * nch;
    }
    float acc[4][NT];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int t = 0; t < NT; ++t) acc[i][t] = 0.f;
    mx_rows_dot<4, NT, 2>(codes, scales, nch, xs, acc);
    warp_allreduce<4, NT>(acc);
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int t = 0; t < NT; ++t)
        if (lane == i * NT + t && rr + i < rows)
          Y[static_cast<size_t>(ptok_p[t]) * H + r0 + rr + i] = scale_pow2(acc[i][t], ptok_exp[t]);
  }
}

__global__ void __launch_bounds__(kWarps * 32)
    ffn_down_kernel(k3moe_weights w, int H, int I, int E, const int32_t *__restrict__ offsets,
                    const int32_t *__restrict__ active, const int32_t *__restrict__ nactive,
                    const uint16_t *__restrict__ hrow, float *__restrict__ Y, int rows_per_item,
                    int ntmax) {
  extern __shared__ uint4 xs[];  // ntmax rows x I/8 uint4
  __shared__ int tok_p[kNT], tok_exp[kNT];
  __shared__ float red[kNT][kWarps];
  pdl_wait();
  pdl_trigger();
  const int n_act = *nactive;
  const int items_per_e = (H + rows_per_item - 1) / rows_per_item;
  const long long n_items = static_cast<long long>(n_act) * items_per_e;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (long long item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int u = static_cast<int>(item / items_per_e);
    const int r0 = static_cast<int>(item % items_per_e) * rows_per_item;
    const int rows = min(rows_per_item, H - r0);
    const int e = active[u];
    const int p0 = offsets[e], p1 = offsets[e + 1];
    const bool present = expert_present(w, e);
    for (int pc = p0; pc < p1; pc += ntmax) {
      const int nt = min(ntmax, p1 - pc);
      __syncthreads();
      if (!present) {
        for (int i = threadIdx.x; i < nt * rows; i += blockDim.x)
          Y[static_cast<size_t>(pc + i / rows) * H + r0 + i % rows] = 0.f;
        continue;
      }
      // per-row max |h| (exact prescale), warp tt handles token tt's max
      for (int tt = 0; tt < nt; ++tt) {
        const uint16_t *hr = hrow + static_cast<size_t>(pc + tt) * I;
        float mx = 0.f;
        for (int c = threadIdx.x; c < I; c += blockDim.x) mx = fmaxf(mx, fabsf(bf16_bits_to_f32(hr[c])));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
        if (lane == 0) red[tt][warp] = mx;
      }
      __syncthreads();
      if (threadIdx.x < nt) {
        float mx = red[threadIdx.x][0];
        for (int i = 1; i < kWarps; ++i) mx = fmaxf(mx, red[threadIdx.x][i]);
        tok_exp[threadIdx.x] = prescale_exp(mx);
        tok_p[threadIdx.x] = pc + threadIdx.x;
      }
      __syncthreads();
      const int nch = I / 32, row_u4 = I / 8;
      for (int i = threadIdx.x; i < nt * row_u4; i += blockDim.x) {
        const int tt = i / row_u4, piece = i % row_u4, c = piece >> 2, q = piece & 3;
        const float s = scale_pow2(1.0f, -tok_exp[tt]);
        const uint4 src = *reinterpret_cast<const uint4 *>(hrow + static_cast<size_t>(pc + tt) * I + 8 * piece);
        const uint32_t wv[4] = {src.x, src.y, src.z, src.w};
        uint32_t o[4];
#pragma unroll
        for (int m = 0; m < 4; ++m)
          o[m] = pack_f16x2_scaled(__uint_as_float(wv[m] << 16), __uint_as_float(wv[m] & 0xFFFF0000u), s);
        xs[static_cast<size_t>(tt) * row_u4 + q * nch + c] = make_uint4(o[0], o[1], o[2], o[3]);
      }
      __syncthreads();
      const uint8_t *w2c = w.w2_codes[e], *w2s = w.w2_scales[e];
      switch (nt) {
        case 1: down_item_tokens<1>(w2c, w2s, H, I, r0, rows, xs, tok_p, tok_exp, Y); break;
        case 2: down_item_tokens<2>(w2c, w2s, H, I, r0, rows, xs, tok_p, tok_exp, Y); break;
        case 3: down_item_tokens<3>(w2c, w2s, H, I, r0, rows, xs, tok_p, tok_exp, Y); break;
        default: down_item_tokens<4>(w2c, w2s, H, I, r0, rows, xs, tok_p, tok_exp, Y); break;
      }
    }
  }
}

// ----------------------------------------------------------------------------
size_t ffn_gemv_workspace(const k3moe_shape &s) { return gemv_ws(s.T, s.H, s.I, s.E, s.k).total; }

int launch_ffn_gemv(const k3moe_shape &s, const uint16_t *x, const k3moe_weights &w,
                    const int32_t *offsets, const int32_t *perm, float *Y, void *ws,
                    int32_t *status, cudaStream_t st) {
  if (s.T == 0) return 0;
  const GemvWs L = gemv_ws(s.T, s.H, s.I, s.E, s.k);
  char *base = static_cast<char *>(ws);
  int32_t *active = reinterpret_cast<int32_t *>(base + L.active);
  int32_t *nactive = reinterpret_cast<int32_t *>(base + L.nactive);
  int32_t *xexp = reinterpret_cast<int32_t *>(base + L.xexp);
  uint4 *x16 = reinterpret_cast<uint4 *>(base + L.x16);
  uint16_t *hrow = reinterpret_cast<uint16_t *>(base + L.hrow);
  const int A = s.T * s.k;
  int dev = 0, nsm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  if (launch_pdl(ffn_prep_kernel, dim3(1 + s.T), dim3(256), 0, st, w, x, s.T, s.H, s.E, A, offsets,
                 active, nactive, xexp, x16, status) != cudaSuccess)
    return -1;
  const int max_act = A < s.E ? A : s.E;
  const int ntmax = s.T < kNT ? s.T : kNT;
  // gate/up: kWarps row pairs per item
  {
    const int rows_per_item = kWarps;
    const size_t smem = static_cast<size_t>(ntmax) * s.H * 2;
    static bool attr_set = false;
    if (!attr_set) {
      cudaFuncSetAttribute(ffn_gateup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 4 * 16384 * 2);
      attr_set = true;
    }
    const long long items = static_cast<long long>(max_act) * ((s.I + rows_per_item - 1) / rows_per_item);
    int nb = 1;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, ffn_gateup_kernel, kWarps * 32, smem);
    const long long cap = static_cast<long long>(nsm) * (nb > 0 ? nb : 1);
    const int grid = static_cast<int>(items < cap ? items : cap);
    if (launch_pdl(ffn_gateup_kernel, dim3(grid), dim3(kWarps * 32), smem, st, w, s.T, s.H, s.I, s.k,
                   s.E, A, offsets, perm, static_cast<const int32_t *>(active),
                   static_cast<const int32_t *>(nactive), static_cast<const int32_t *>(xexp),
                   static_cast<const uint4 *>(x16), hrow, rows_per_item, ntmax, status) != cudaSuccess)
      return -1;
  }
  {
    const int rows_per_item = kWarps * 4;
    const size_t smem = static_cast<size_t>(ntmax) * s.I * 2;
    static bool attr_set = false;
    if (!attr_set) {
      cudaFuncSetAttribute(ffn_down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 4 * 16384 * 2);
      attr_set = true;
    }
    const long long items = static_cast<long long>(max_act) * ((s.H + rows_per_item - 1) / rows_per_item);
    int nb = 1;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, ffn_down_kernel, kWarps * 32, smem);
    const long long cap = static_cast<long long>(nsm) * (nb > 0 ? nb : 1);
    const int grid = static_cast<int>(items < cap ? items : cap);
    if (launch_pdl(ffn_down_kernel, dim3(grid), dim3(kWarps * 32), smem, st, w, s.H, s.I, s.E, offsets,
                   static_cast<const int32_t *>(active), static_cast<const int32_t *>(nactive),
                   static_cast<const uint16_t *>(hrow), Y, rows_per_item, ntmax) != cudaSuccess)
      return -1;
  }
  return 0;
}

}  // namespace k3moe
