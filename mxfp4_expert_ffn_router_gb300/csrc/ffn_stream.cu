// ffn_stream.cu -- the MXFP4 expert FFN as one persistent streaming kernel.
//
// Same arithmetic as the CUDA-core GEMV path (ffn_gemv.cu): packed e2m1 codes
// are decoded in registers (cvt e2m1x2 -> f16x2, exact) and multiplied by f16
// activations (exact power-of-two prescale) with fp32 accumulation, scaled per
// 32-block by the e8m0 scale, reduced across the warp; h = bf16(silu(g) * u).
// The kimi-k3-in-c CHANGELOG walkthrough, "[0.1.0] Added": the matmul consumes
// the packed nibbles directly and never materialises a dequantised expert;
// "[1.0.0] Added": each unique routed expert is fetched once per token chunk.
//
// Structure (one CTA per SM, 1 producer warp + 11 consumer warps):
//  * Work is a queue of tasks taken with an atomic counter: first every gate/up
//    task (active expert u, token chunk, block of 22 row pairs), then every down
//    task (u, chunk, block of 88 rows).  A task is 22 stages of the ring.
//  * The producer thread streams each stage's weight rows (codes + scales) into a
//    ring of shared-memory stages with cp.async.bulk (TMA, 1-D), completing on a
//    per-stage mbarrier, and writes the stage's descriptor (expert, rows, tokens).
//  * Consumer warp w takes ring stages w, w+11, w+22, ... and works alone: no
//    block-wide barriers, so the ring stays full.  Activations come from global
//    memory (L1/L2 resident): x as prescaled f16 for gate/up, h as bf16 for down.
//  * A down stage of expert u waits (bounded) until every h row of u is written:
//    gate/up warps publish each row pair through a per-expert counter (fence +
//    atomic), and the per-(token, expert) max |h| through an integer atomicMax
//    (order-free), from which the down stage takes its exact f16 prescale.
//  Every wait is bounded; on timeout the kernel sets K3MOE_DEV_TIMEOUT and goes
//  on (results are then invalid but the kernel returns).
#include <cuda_fp16.h>

#include "k3moe_dev.cuh"
#include "k3moe_launch.h"

namespace k3moe {

namespace {

// The kernel is instantiated for W consumer warps (plus one producer warp) and at
// most NTMAX tokens per chunk (1 for single-token decode, else 4).  A task is 2W
// stages; consumer warp w takes stages w and w + W of every task.  The ring has
// a multiple of W stages (each slot owned by one consumer warp; two or more
// slots per warp let a warp compute one stage while its next one is in flight).
constexpr int kDownRowsPerStage = 4;
constexpr int kNT = 4;              // tokens per chunk (the task descriptor stores 4)
constexpr int kTableCap = 1024;     // active experts whose task table lives in shared memory
constexpr int kHSlots = 3;         // h buffers for down tasks (reused round-robin)
constexpr long long kSpinLimit = 1LL << 22;  // ~0.1-0.3 s per wait

// Per-stage descriptor (one 16-byte store by the producer).
struct StageDesc {
  int seq;    // ring sequence number of this stage
  int tslot;  // task-ring slot of the stage's task (-1 = end of work)
  int row0;   // first row of this stage (gate/up: gate row r; down: W2 row)
  int nrows;  // valid rows in this stage (0 = padding stage)
};

// Per-task descriptor, in a ring of kTaskRing entries (a slot is rewritten only
// after every stage of its previous task has been consumed: the stage ring is
// shorter than kTaskRing - 1 tasks).
constexpr int kTaskRing = 8;
struct TaskDesc {
  int kind;   // 0 gate/up, 1 down
  int u;      // active slot
  int p0, nt; // first bucket position of the token chunk, tokens in it
  int present;
  int hslot, hphase;  // down: h buffer of the task and the phase of its fill
  int tok[kNT];       // token ids of the chunk (-1 = invalid)
};

struct StreamWs {
  size_t active, nactive, xexp, x16, hrow, hmax, tokid, pref, sp0, scnt, counter, done, total;
};

__host__ __device__ inline size_t a256(size_t v) { return (v + 255) & ~size_t(255); }

__host__ __device__ inline StreamWs stream_ws(int T, int H, int I, int E, int k) {
  StreamWs w;
  const size_t A = static_cast<size_t>(T) * k;
  size_t o = 0;
  w.active = o;   o = a256(o + sizeof(int32_t) * E);
  w.nactive = o;  o = a256(o + sizeof(int32_t) * 4);
  w.xexp = o;     o = a256(o + sizeof(int32_t) * (T > 0 ? T : 1));
  w.x16 = o;      o = a256(o + sizeof(uint16_t) * static_cast<size_t>(T) * H);
  w.hrow = o;     o = a256(o + sizeof(uint16_t) * A * I);
  w.hmax = o;     o = a256(o + 4 * sizeof(int32_t) * (A ? A : 1));  // 16 B per position (bulk-copyable)
  w.tokid = o;    o = a256(o + sizeof(int32_t) * (A ? A : 1));
  w.pref = o;     o = a256(o + sizeof(int32_t) * 2 * (E + 1));
  w.sp0 = o;      o = a256(o + sizeof(int32_t) * E);
  w.scnt = o;     o = a256(o + sizeof(int32_t) * E);
  w.counter = o;  o = a256(o + sizeof(int32_t) * 4);
  w.done = o;     o = a256(o + sizeof(int32_t) * E);
  w.total = o;
  return w;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait on an mbarrier phase.  After any wait of the CTA has timed out
// (*abort set), every later wait returns at once, so a stuck kernel ends after
// one time limit instead of one per wait.  Returns false on timeout or abort.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort) {
  for (long long i = 0; i < kSpinLimit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255) == 255 && *abort) return false;
    if (i > 64) __nanosleep(32);
  }
  *abort = 1;
  return false;
}
// 1-D bulk copy global -> this CTA's shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ int ld_acquire(const int32_t *p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ int prescale_exp(float max_abs) {
  if (!(max_abs > 0.f) || max_abs == INFINITY) return 0;
  int e;
  frexpf(max_abs, &e);
  return max(-100, min(100, (e - 1) - 14));
}
__device__ __forceinline__ float scale_pow2(float v, int p) {
  const int p1 = p / 2, p2 = p - p1;
  return v * exp2i(p1) * exp2i(p2);
}
__device__ __forceinline__ uint32_t pack_f16x2(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t *>(&h);
}


// Partial dot products of R smem rows (codes at `codes + r*rstride`, scales at
// `scl + r*sstride`) with NT activation rows (piece-major f16 in xs), then a warp
// all-reduce.  Two chunks per iteration and two partial sums per chunk keep the
// dependent FMA chains short.

// acc[r][t] += the lane's share of sum_c row_r(c) * act_t(c) over the stage's chunks.
// codes/scales of R rows in shared memory (row strides rstride / sstride bytes);
// activation chunk c of token t comes from `act(t, c, q)` as four f16x2 words.
template <int R, int NT, typename Act>
__device__ __forceinline__ void chunk_dot(const uint8_t *codes, int rstride, const uint8_t *scl, int sstride,
                                          int c, const Act &act, float (&acc)[R][NT]) {
  float d0[R][NT], d1[R][NT];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int t = 0; t < NT; ++t) d0[r][t] = d1[r][t] = 0.f;
  uint4 cw[R];
#pragma unroll
  for (int r = 0; r < R; ++r) cw[r] = *reinterpret_cast<const uint4 *>(codes + r * rstride + 16 * c);
  uint4 xv[NT][4];
#pragma unroll
  for (int t = 0; t < NT; ++t)
#pragma unroll
    for (int q = 0; q < 4; ++q) xv[t][q] = act(t, c, q);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t wh[R][4];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const uint32_t word = q == 0 ? cw[r].x : q == 1 ? cw[r].y : q == 2 ? cw[r].z : cw[r].w;
      e2m1x8_to_f16x2(word, wh[r]);
    }
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int r = 0; r < R; ++r) {
        d0[r][t] = fma2_f16_f32(wh[r][0], xv[t][q].x, d0[r][t]);
        d1[r][t] = fma2_f16_f32(wh[r][1], xv[t][q].y, d1[r][t]);
        d0[r][t] = fma2_f16_f32(wh[r][2], xv[t][q].z, d0[r][t]);
        d1[r][t] = fma2_f16_f32(wh[r][3], xv[t][q].w, d1[r][t]);
      }
  }
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const float sf = e8m0_to_f32(scl[r * sstride + c]);
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[r][t] = fmaf(d0[r][t] + d1[r][t], sf, acc[r][t]);
  }
}

// All chunks of R stage rows against NT activation rows, then a warp all-reduce.
template <int R, int NT, typename Act>
__device__ __forceinline__ void stage_dot(const uint8_t *codes, int rstride, const uint8_t *scl, int sstride,
                                          int nch, const Act &act, float (&acc)[R][NT]) {
  const int lane = threadIdx.x & 31;
  float acc2[R][NT];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[r][t] = acc2[r][t] = 0.f;
  int c = lane;
  for (; c + 32 < nch; c += 64) {
    chunk_dot<R, NT>(codes, rstride, scl, sstride, c, act, acc);
    chunk_dot<R, NT>(codes, rstride, scl, sstride, c + 32, act, acc2);
  }
  if (c < nch) chunk_dot<R, NT>(codes, rstride, scl, sstride, c, act, acc);
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      acc[r][t] += acc2[r][t];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc[r][t] += __shfl_xor_sync(0xFFFFFFFFu, acc[r][t], off);
    }
}

struct Params {
  k3moe_weights w;
  int T, H, I, E, k, A;
  const int32_t *active, *nactive, *xexp, *pref, *slot_p0, *slot_cnt, *tokid;
  const uint4 *x16;
  uint16_t *hrow;
  int32_t *hmax;
  float *Y;
  int32_t *counter, *done, *status;
  int stages;       // ring depth
  int stage_bytes;  // bytes per stage buffer (multiple of 128)
  int x_in_smem;    // 1: every token's x (prescaled f16) is staged once in shared memory
  int ntcap;        // token rows a down stage carries (min(T, kNT))
};

// Task id -> (kind, active slot u, token chunk, row block) by binary search over
// the inclusive task prefix of the active slots.
__device__ __forceinline__ void decode_task(const int *pf_gu, const int *pf_dn, int na, int task, int n_gu,
                                            int rb_gu, int rb_dn, int &kind, int &u, int &chunk, int &rb) {
  kind = task < n_gu ? 0 : 1;
  const int local = kind ? task - n_gu : task;
  const int *pf = kind ? pf_dn : pf_gu;
  int lo = 0, hi = na - 1;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (pf[mid] > local) hi = mid; else lo = mid + 1;
  }
  u = lo;
  const int before = u ? pf[u - 1] : 0;
  const int per = kind ? rb_dn : rb_gu;
  chunk = (local - before) / per;
  rb = (local - before) % per;
}

}  // namespace

// ----------------------------------------------------------------------------
// prep: active list, task prefix tables, token ids, zeroed counters and maxima,
// x -> prescaled f16 (piece-major: uint4 index q * (H/32) + c holds columns
// 32c + 8q .. 32c + 8q + 7).
__global__ void __launch_bounds__(256)
    stream_prep_kernel(const uint16_t *__restrict__ x, int T, int H, int E, int k, int A,
                       const int32_t *__restrict__ offsets, const int32_t *__restrict__ perm,
                       int32_t *__restrict__ active, int32_t *__restrict__ nactive, int32_t *__restrict__ xexp,
                       uint4 *__restrict__ x16, int32_t *__restrict__ pref, int32_t *__restrict__ slot_p0,
                       int32_t *__restrict__ slot_cnt, int32_t *__restrict__ tokid, int32_t *__restrict__ hmax,
                       int32_t *__restrict__ counter, int32_t *__restrict__ done, int rb_gu, int rb_dn,
                       int32_t *status) {
  pdl_wait();
  if (blockIdx.x == 0) {
    for (int e = threadIdx.x; e < E; e += 256) done[e] = 0;
    if (threadIdx.x == 0) counter[0] = 0;
    if (threadIdx.x >= 32) return;
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
      const int nch = f ? (cnt + kNT - 1) / kNT : 0;
      int g = nch * rb_gu, d = nch * rb_dn;  // inclusive prefix of task counts
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
        pref[slot] = sg + g;
        pref[E + 1 + slot] = sd + d;
      }
      run += __popc(m);
      sg += __shfl_sync(0xFFFFFFFFu, g, 31);
      sd += __shfl_sync(0xFFFFFFFFu, d, 31);
    }
    if (lane == 0) {
      nactive[0] = bad ? 0 : run;
      nactive[1] = bad ? 0 : sg;  // gate/up tasks
      nactive[2] = bad ? 0 : sd;  // down tasks
      if (bad) set_status(status, K3MOE_DEV_BOUNDS);
    }
    return;
  }
  if (blockIdx.x == 1) {  // token id of every bucket position, zeroed maxima
    bool bad = false;
    for (int p = threadIdx.x; p < A; p += 256) {
      const int a = perm[p];
      int t = -1;
      if (a >= 0 && a < A) t = a / k; else bad = true;
      tokid[p] = t;
      hmax[4 * p] = 0;
    }
    if (bad) set_status(status, K3MOE_DEV_BOUNDS);
    return;
  }
  const int t = blockIdx.x - 2;
  if (t >= T) return;
  const uint16_t *xr = x + static_cast<size_t>(t) * H;
  __shared__ float red[8];
  float mx = 0.f;
  for (int c = threadIdx.x; c < H; c += 256) mx = fmaxf(mx, fabsf(bf16_bits_to_f32(xr[c])));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
  __syncthreads();
  mx = red[0];
  for (int i = 1; i < 8; ++i) mx = fmaxf(mx, red[i]);
  const int p = prescale_exp(mx);
  if (threadIdx.x == 0) xexp[t] = p;
  const float s = scale_pow2(1.0f, -p);
  const int nch = H / 32;
  uint4 *dst = x16 + static_cast<size_t>(t) * (H / 8);
  for (int piece = threadIdx.x; piece < H / 8; piece += 256) {
    const int c = piece >> 2, q = piece & 3;
    const uint4 src = *reinterpret_cast<const uint4 *>(xr + 8 * piece);
    const uint32_t w[4] = {src.x, src.y, src.z, src.w};
    uint32_t o[4];
#pragma unroll
    for (int m = 0; m < 4; ++m)
      o[m] = pack_f16x2(__uint_as_float(w[m] << 16) * s, __uint_as_float(w[m] & 0xFFFF0000u) * s);
    dst[q * nch + c] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// ----------------------------------------------------------------------------
// x chunk of a token, prescaled f16, piece-major rows (shared or global memory).
struct XAct {
  const uint4 *rows[kNT];
  int nch;
  __device__ __forceinline__ uint4 operator()(int t, int c, int q) const { return rows[t][q * nch + c]; }
};

// h chunk of a (token, expert) row: raw bf16 in the stage buffer, converted to
// f16 after the exact power-of-two prescale s_t.
struct HAct {
  const uint4 *rows[kNT];  // bf16 rows, 4 uint4 (32 values) per chunk
  float s[kNT];
  __device__ __forceinline__ uint4 operator()(int t, int c, int q) const {
    const uint4 v = rows[t][4 * c + q];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int m = 0; m < 4; ++m)
      o[m] = pack_f16x2(__uint_as_float(w[m] << 16) * s[t], __uint_as_float(w[m] & 0xFFFF0000u) * s[t]);
    return make_uint4(o[0], o[1], o[2], o[3]);
  }
};

template <int NT>
__device__ void gateup_stage(const Params &P, const TaskDesc &d, int row0, const uint8_t *buf, const uint4 *xs) {
  const int lane = threadIdx.x & 31;
  const int nch = P.H / 32, cbytes = P.H / 2;
  float acc[2][NT];
  XAct act;
  act.nch = nch;
  const uint4 *xbase = P.x_in_smem ? xs : P.x16;
#pragma unroll
  for (int t = 0; t < NT; ++t) act.rows[t] = xbase + static_cast<size_t>(d.tok[t] < 0 ? 0 : d.tok[t]) * (P.H / 8);
  if (d.present) {
    stage_dot<2, NT>(buf, cbytes, buf + 2 * cbytes, nch, nch, act, acc);
  } else {
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[0][t] = acc[1][t] = 0.f;
  }
#pragma unroll
  for (int t = 0; t < NT; ++t)
    if (lane == t) {
      float hv = 0.f;
      if (d.present && d.tok[t] >= 0) {
        const int ex = P.xexp[d.tok[t]];
        const float g = scale_pow2(acc[0][t], ex);
        const float u = scale_pow2(acc[1][t], ex);
        hv = (g / (1.0f + expf(-g))) * u;
      }
      const uint16_t hb = f32_to_bf16_rne(hv);
      P.hrow[static_cast<size_t>(d.p0 + t) * P.I + row0] = hb;
      atomicMax(P.hmax + 4 * (d.p0 + t), static_cast<int>(__float_as_uint(fabsf(bf16_bits_to_f32(hb)))));
    }
}

template <int NT>
__device__ void down_stage(const Params &P, const TaskDesc &d, int row0, int nrows, const uint8_t *buf,
                           const uint8_t *hbuf) {
  const int lane = threadIdx.x & 31;
  const int nch = P.I / 32, cbytes = P.I / 2;
  float acc[kDownRowsPerStage][NT];
  HAct act;
  // h slot: ntcap rows of bf16 h, then ntcap 16-byte records whose first word is max|h|
  const int *hmx = reinterpret_cast<const int *>(hbuf + static_cast<size_t>(P.ntcap) * P.I * 2);
  int hexp[NT];
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    hexp[t] = prescale_exp(__int_as_float(hmx[4 * t]));
    act.s[t] = scale_pow2(1.0f, -hexp[t]);
    act.rows[t] = reinterpret_cast<const uint4 *>(hbuf + static_cast<size_t>(t) * P.I * 2);
  }
  if (d.present) {
    stage_dot<kDownRowsPerStage, NT>(buf, cbytes, buf + kDownRowsPerStage * cbytes, nch, nch, act, acc);
  } else {
#pragma unroll
    for (int r = 0; r < kDownRowsPerStage; ++r)
#pragma unroll
      for (int t = 0; t < NT; ++t) acc[r][t] = 0.f;
  }
#pragma unroll
  for (int r = 0; r < kDownRowsPerStage; ++r)
#pragma unroll
    for (int t = 0; t < NT; ++t)
      if (lane == r * NT + t && r < nrows)
        P.Y[static_cast<size_t>(d.p0 + t) * P.H + row0 + r] = scale_pow2(acc[r][t], hexp[t]);
}

__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// What the producer needs to issue a task, fetched one task ahead so the global
// loads (expert pointers, token ids) are in flight while the previous task issues.
struct TaskFetch {
  int task, kind, u, rb, e, cnt, p0, nt;
  const uint8_t *c13, *s13, *c2, *s2;
  int tok[kNT];
};

__device__ __forceinline__ void fetch_task(const Params &P, int task, int n_tasks, int n_gu, int na, int rb_gu,
                                           int rb_dn, const int *t_e, const int *t_p0, const int *t_cnt,
                                           const int *t_gu, const int *t_dn, TaskFetch &f) {
  f.task = task;
  f.kind = 0; f.u = 0; f.rb = 0; f.e = 0; f.cnt = 0; f.p0 = 0; f.nt = 0;
  f.c13 = f.s13 = f.c2 = f.s2 = nullptr;
  if (task >= n_tasks) return;
  int chunk;
  decode_task(t_gu, t_dn, na, task, n_gu, rb_gu, rb_dn, f.kind, f.u, chunk, f.rb);
  f.e = t_e[f.u];
  f.cnt = t_cnt[f.u];
  f.p0 = t_p0[f.u] + chunk * kNT;
  f.nt = min(kNT, f.cnt - chunk * kNT);
  f.c13 = P.w.w13_codes[f.e];
  f.s13 = P.w.w13_scales[f.e];
  f.c2 = P.w.w2_codes[f.e];
  f.s2 = P.w.w2_scales[f.e];
#pragma unroll
  for (int t = 0; t < kNT; ++t) f.tok[t] = t < f.nt ? P.tokid[f.p0 + t] : -1;
}

template <int W, int NTMAX>
__global__ void __launch_bounds__((W + 1) * 32, 1) ffn_stream_kernel(Params P) {
  constexpr int kThreads = (W + 1) * 32;
  constexpr int kStagesPerTask = 2 * W;
  extern __shared__ __align__(128) uint8_t smem[];
  // layout: ring [stages * stage_bytes] | h slots [kHSlots * ntcap * I bf16] | xs [T * H f16
  //         when staged] | task table [5 * min(E, kTableCap) int, 16-B padded] |
  //         barriers [2 * stages + 2 * kHSlots] | stage descs [stages] | task descs [kTaskRing]
  uint8_t *ring = smem;
  const int tcap = P.E < kTableCap ? P.E : kTableCap;
  uint8_t *hslots = ring + static_cast<size_t>(P.stages) * P.stage_bytes;
  const size_t hslot_bytes = static_cast<size_t>(P.ntcap) * (P.I * 2 + 16);
  uint4 *xs = reinterpret_cast<uint4 *>(hslots + kHSlots * hslot_bytes);
  const size_t xs_bytes = P.x_in_smem ? static_cast<size_t>(P.T) * P.H * 2 : 0;
  int *tab = reinterpret_cast<int *>(reinterpret_cast<uint8_t *>(xs) + xs_bytes);
  uint64_t *full = reinterpret_cast<uint64_t *>(reinterpret_cast<uint8_t *>(tab) + ((20 * tcap + 15) & ~15));
  uint64_t *empty = full + P.stages;
  uint64_t *hfull = empty + P.stages;
  uint64_t *hempty = hfull + kHSlots;
  StageDesc *desc = reinterpret_cast<StageDesc *>(hempty + kHSlots);
  TaskDesc *tdesc = reinterpret_cast<TaskDesc *>(desc + P.stages);
  __shared__ int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < P.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      desc[s].seq = -1;
    }
    for (int k = 0; k < kHSlots; ++k) {
      mbar_init(&hfull[k], 1);
      mbar_init(&hempty[k], kStagesPerTask);  // every stage of a down task releases its h slot
    }
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  pdl_wait();  // prep's tables, counters and x16 are ready
  pdl_trigger();
  const int na = P.nactive[0];
  const int n_gu = P.nactive[1], n_dn = P.nactive[2];
  const int n_tasks = n_gu + n_dn;
  const bool in_smem = na <= tcap;
  if (in_smem) {
    for (int i = threadIdx.x; i < na; i += kThreads) {
      tab[i] = P.active[i];
      tab[tcap + i] = P.slot_p0[i];
      tab[2 * tcap + i] = P.slot_cnt[i];
      tab[3 * tcap + i] = P.pref[i];
      tab[4 * tcap + i] = P.pref[P.E + 1 + i];
    }
  }
  if (P.x_in_smem) {
    const int n = P.T * P.H / 8;
    for (int i = threadIdx.x; i < n; i += kThreads) xs[i] = P.x16[i];
  }
  __syncthreads();
  volatile int *abort = &s_abort;

  const int rb_gu = (P.I + kStagesPerTask - 1) / kStagesPerTask;
  const int rows_dn = kStagesPerTask * kDownRowsPerStage;
  const int rb_dn = (P.H + rows_dn - 1) / rows_dn;

  if (warp == W) {
    // ------------------------------------------------------------ producer
    // The whole warp produces: task set-up is computed by every lane (same
    // values), and the stages of a task are issued in groups of G <= stages, lane
    // i issuing stage base + i (distinct ring slots within a group).
    const int *t_e = in_smem ? tab : P.active;
    const int *t_p0 = in_smem ? tab + tcap : P.slot_p0;
    const int *t_cnt = in_smem ? tab + 2 * tcap : P.slot_cnt;
    const int *t_gu = in_smem ? tab + 3 * tcap : P.pref;
    const int *t_dn = in_smem ? tab + 4 * tcap : P.pref + P.E + 1;
    const int G = P.stages < 32 ? P.stages : 32;
    int seq = 0;        // stages issued so far
    int slot = 0;       // seq % stages
    uint32_t lap = 0;   // seq / stages
    int ntask = 0, ndown = 0;  // tasks / down tasks issued by this CTA
    const int cb13 = P.H / 2, sb13 = P.H / 32, cb2 = P.I / 2, sb2 = P.I / 32;
    const uint32_t hbytes = static_cast<uint32_t>(P.I) * 2;
    int ready_u = -1;
    TaskFetch cur, nxt;
    int first = 0;
    if (lane == 0) first = atomicAdd(P.counter, 1);
    first = __shfl_sync(0xFFFFFFFFu, first, 0);
    fetch_task(P, first, n_tasks, n_gu, na, rb_gu, rb_dn, t_e, t_p0, t_cnt, t_gu, t_dn, cur);
    int next_id = n_tasks;
    if (cur.task < n_tasks && lane == 0) next_id = atomicAdd(P.counter, 1);
    next_id = __shfl_sync(0xFFFFFFFFu, next_id, 0);
    for (;;) {
      const bool end = cur.task >= n_tasks;
      if (!end) {
        // the task after this one: its loads fly while this task's stages issue
        fetch_task(P, next_id, n_tasks, n_gu, na, rb_gu, rb_dn, t_e, t_p0, t_cnt, t_gu, t_dn, nxt);
        int nid = n_tasks;
        if (next_id < n_tasks && lane == 0) nid = atomicAdd(P.counter, 1);
        next_id = __shfl_sync(0xFFFFFFFFu, nid, 0);
      }
      const int ts = ntask % kTaskRing;
      int present = 0;
      if (!end) {
        const uintptr_t al = reinterpret_cast<uintptr_t>(cur.c13) | reinterpret_cast<uintptr_t>(cur.s13) |
                             reinterpret_cast<uintptr_t>(cur.c2) | reinterpret_cast<uintptr_t>(cur.s2);
        const bool nonnull = cur.c13 && cur.s13 && cur.c2 && cur.s2;
        present = nonnull && (al & 15u) == 0;
        if (lane == 0 && nonnull && !present) set_status(P.status, K3MOE_DEV_BOUNDS);  // misaligned: absent
        int hslot = 0, hphase = 0;
        if (cur.kind == 1) {
          if (ready_u != cur.u) {
            // down: wait (bounded) until every h row of expert u is published
            if (lane == 0) {
              const int want = P.I * ((cur.cnt + kNT - 1) / kNT);
              long long it = 0;
              while (ld_acquire(P.done + cur.u) < want) {
                if (++it > kSpinLimit || *abort) {
                  *abort = 1;
                  set_status(P.status, K3MOE_DEV_TIMEOUT);
                  break;
                }
                __nanosleep(64);
              }
            }
            __syncwarp();
            (void)ld_acquire(P.done + cur.u);
            fence_proxy_async_global();  // h is read below by bulk copies (async proxy)
            ready_u = cur.u;
          }
          // this task's h rows (raw bf16) and their max|h| records into an h slot,
          // released by the task's stages
          const int k = ndown % kHSlots;
          const uint32_t ph = static_cast<uint32_t>(ndown / kHSlots) & 1u;
          hslot = k;
          hphase = static_cast<int>(ph);
          if (lane == 0) {
            if (!mbar_wait(&hempty[k], ph ^ 1u, abort)) set_status(P.status, K3MOE_DEV_TIMEOUT);
            if (present) {
              uint8_t *hs = hslots + k * hslot_bytes;
              mbar_arrive_expect_tx(&hfull[k], cur.nt * (hbytes + 16));
              for (int t = 0; t < cur.nt; ++t) {
                bulk_g2s(hs + static_cast<size_t>(t) * hbytes, P.hrow + static_cast<size_t>(cur.p0 + t) * P.I,
                         hbytes, &hfull[k]);
                bulk_g2s(hs + static_cast<size_t>(P.ntcap) * hbytes + 16 * t, P.hmax + 4 * (cur.p0 + t), 16,
                         &hfull[k]);
              }
            } else {
              mbar_arrive(&hfull[k]);
            }
          }
          ++ndown;
        }
        // task descriptor: lane i < 15 writes word i
        int word = 0;
        switch (lane) {
          case 0: word = cur.kind; break;
          case 1: word = cur.u; break;
          case 2: word = cur.p0; break;
          case 3: word = cur.nt; break;
          case 4: word = present; break;
          case 5: word = hslot; break;
          case 6: word = hphase; break;
          default: break;
        }
        if (lane == 7) word = cur.tok[0];
        if (lane == 8) word = cur.tok[1];
        if (lane == 9) word = cur.tok[2];
        if (lane == 10) word = cur.tok[3];
        if (lane < 7 + kNT) reinterpret_cast<int *>(&tdesc[ts])[lane] = word;
        __syncwarp();  // descriptor stores before any stage of the task is released
      }
      const int nst = end ? W : kStagesPerTask;
      const uint8_t *wc = cur.kind == 0 ? cur.c13 : cur.c2;
      const uint8_t *wsc = cur.kind == 0 ? cur.s13 : cur.s2;
      for (int j0 = 0; j0 < nst; j0 += G) {
        const int cnt = min(G, nst - j0);
        if (lane < cnt) {
          const int j = j0 + lane;
          int s = slot + lane;
          uint32_t n = lap;
          while (s >= P.stages) {
            s -= P.stages;
            ++n;
          }
          if (!mbar_wait(&empty[s], (n & 1u) ^ 1u, abort)) set_status(P.status, K3MOE_DEV_TIMEOUT);
          uint8_t *buf = ring + static_cast<size_t>(s) * P.stage_bytes;
          int row0 = 0, nrows = 0;
          uint32_t bytes = 0;
          if (!end && cur.kind == 0) {
            row0 = cur.rb * kStagesPerTask + j;
            nrows = row0 < P.I ? 1 : 0;
            if (nrows && present) bytes = 2u * (cb13 + sb13);
          } else if (!end) {
            row0 = cur.rb * rows_dn + j * kDownRowsPerStage;
            nrows = max(0, min(kDownRowsPerStage, P.H - row0));
            if (nrows && present) bytes = static_cast<uint32_t>(nrows) * (cb2 + sb2);
          }
          *reinterpret_cast<int4 *>(&desc[s]) = make_int4(seq + lane, end ? -1 : ts, row0, nrows);
          if (!bytes) {
            mbar_arrive(&full[s]);
          } else if (cur.kind == 0) {
            mbar_arrive_expect_tx(&full[s], bytes);
            bulk_g2s(buf, wc + static_cast<size_t>(row0) * cb13, cb13, &full[s]);
            bulk_g2s(buf + cb13, wc + static_cast<size_t>(P.I + row0) * cb13, cb13, &full[s]);
            bulk_g2s(buf + 2 * cb13, wsc + static_cast<size_t>(row0) * sb13, sb13, &full[s]);
            bulk_g2s(buf + 2 * cb13 + sb13, wsc + static_cast<size_t>(P.I + row0) * sb13, sb13, &full[s]);
          } else {
            mbar_arrive_expect_tx(&full[s], bytes);
            bulk_g2s(buf, wc + static_cast<size_t>(row0) * cb2, nrows * cb2, &full[s]);
            bulk_g2s(buf + kDownRowsPerStage * cb2, wsc + static_cast<size_t>(row0) * sb2, nrows * sb2, &full[s]);
          }
        }
        seq += cnt;
        slot += cnt;
        while (slot >= P.stages) {
          slot -= P.stages;
          ++lap;
        }
        __syncwarp();
      }
      if (end) break;
      ++ntask;
      cur = nxt;
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  int pending = 0;  // gate/up rows of the current task not yet published
  int s = warp;     // ring slot of stage q (q % stages)
  uint32_t n = 0;   // lap of stage q (q / stages)
  for (int q = warp;; q += W, s += W) {
    if (s >= P.stages) {
      s -= P.stages;
      ++n;
    }
    // Every ring slot belongs to one consumer warp (stages is a multiple of
    // W), so the slot's previous fill was consumed by this warp and
    // the parity wait is unambiguous; the sequence check below is a second guard.
    if (!mbar_wait(&full[s], n & 1u, abort)) set_status(P.status, K3MOE_DEV_TIMEOUT);
    const int4 dv = *reinterpret_cast<const int4 *>(&desc[s]);
    if (dv.x != q) {
      *abort = 1;
      set_status(P.status, K3MOE_DEV_TIMEOUT);
    }
    if (dv.y < 0 || *abort) break;
    const TaskDesc &d = tdesc[dv.y];
    const int row0 = dv.z, nrows = dv.w;
    const uint8_t *buf = ring + static_cast<size_t>(s) * P.stage_bytes;
    if (d.kind == 0) {
      if (nrows > 0) {
        if (NTMAX == 1) {
          gateup_stage<1>(P, d, row0, buf, xs);
        } else {
          switch (d.nt) {
            case 1: gateup_stage<1>(P, d, row0, buf, xs); break;
            case 2: gateup_stage<2>(P, d, row0, buf, xs); break;
            case 3: gateup_stage<3>(P, d, row0, buf, xs); break;
            default: gateup_stage<4>(P, d, row0, buf, xs); break;
          }
        }
      }
      const int u = d.u;
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      pending += nrows;
      if (q % kStagesPerTask >= W) {  // constant divisor
        // this warp's second (last) stage of the task: publish its h rows and
        // their maxima with one fence and one count
        __threadfence();
        __syncwarp();
        if (lane == 0 && pending) atomicAdd(P.done + u, pending);
        pending = 0;
      }
    } else {
      const int hs = d.hslot;
      if (!mbar_wait(&hfull[hs], static_cast<uint32_t>(d.hphase), abort)) set_status(P.status, K3MOE_DEV_TIMEOUT);
      if (nrows > 0) {
        const uint8_t *hb = hslots + hs * hslot_bytes;
        if (NTMAX == 1) {
          down_stage<1>(P, d, row0, nrows, buf, hb);
        } else {
          switch (d.nt) {
            case 1: down_stage<1>(P, d, row0, nrows, buf, hb); break;
            case 2: down_stage<2>(P, d, row0, nrows, buf, hb); break;
            case 3: down_stage<3>(P, d, row0, nrows, buf, hb); break;
            default: down_stage<4>(P, d, row0, nrows, buf, hb); break;
          }
        }
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&empty[s]);
        mbar_arrive(&hempty[hs]);
      }
    }
  }
}

// ----------------------------------------------------------------------------
size_t ffn_stream_workspace(const k3moe_shape &s) { return stream_ws(s.T, s.H, s.I, s.E, s.k).total; }
size_t ffn_stream_h_offset(const k3moe_shape &s) { return stream_ws(s.T, s.H, s.I, s.E, s.k).hrow; }

static int stream_ntcap(const k3moe_shape &s) { return s.T < kNT ? s.T : kNT; }

static int stream_stage_bytes(const k3moe_shape &s) {
  const int gu = 2 * (s.H / 2 + s.H / 32);
  const int dn = kDownRowsPerStage * (s.I / 2 + s.I / 32);
  const int b = gu > dn ? gu : dn;
  return (b + 127) & ~127;
}

// x of every token is staged in shared memory when it takes at most this much
static constexpr size_t kXsMax = 64 * 1024;

static bool stream_x_in_smem(const k3moe_shape &s) {
  return static_cast<size_t>(s.T) * s.H * 2 <= kXsMax;
}

// must match the device-side layout in ffn_stream_kernel
static size_t stream_fixed_smem(const k3moe_shape &s, int stages) {
  const int tcap = s.E < kTableCap ? s.E : kTableCap;
  const size_t xs = stream_x_in_smem(s) ? static_cast<size_t>(s.T) * s.H * 2 : 0;
  const size_t hs = static_cast<size_t>(kHSlots) * stream_ntcap(s) * (s.I * 2 + 16);
  return hs + xs + ((20 * static_cast<size_t>(tcap) + 15) & ~size_t(15)) + 16 * stages + 16 * kHSlots +
         sizeof(StageDesc) * stages + sizeof(TaskDesc) * kTaskRing;
}

// consumer warps of the instance a shape uses
static int stream_warps(const k3moe_shape &) { return 11; }

bool ffn_stream_supported(const k3moe_shape &s) {
  // bulk copies need 16-byte multiples for every row of codes and scales
  if ((s.H / 32) % 16 || (s.I / 32) % 16) return false;
  if (s.H > 8192 || s.I > 8192) return false;
  const int W = stream_warps(s);
  const size_t need = stream_fixed_smem(s, W) + W * static_cast<size_t>(stream_stage_bytes(s));
  return need <= 224 * 1024;
}

int launch_ffn_stream(const k3moe_shape &s, const uint16_t *x, const k3moe_weights &w,
                      const int32_t *offsets, const int32_t *perm, float *Y, void *ws,
                      int32_t *status, cudaStream_t st) {
  if (s.T == 0) return 0;
  const StreamWs L = stream_ws(s.T, s.H, s.I, s.E, s.k);
  char *base = static_cast<char *>(ws);
  Params P;
  P.w = w;
  P.T = s.T; P.H = s.H; P.I = s.I; P.E = s.E; P.k = s.k; P.A = s.T * s.k;
  P.active = reinterpret_cast<const int32_t *>(base + L.active);
  P.nactive = reinterpret_cast<const int32_t *>(base + L.nactive);
  P.xexp = reinterpret_cast<const int32_t *>(base + L.xexp);
  P.pref = reinterpret_cast<const int32_t *>(base + L.pref);
  P.slot_p0 = reinterpret_cast<const int32_t *>(base + L.sp0);
  P.slot_cnt = reinterpret_cast<const int32_t *>(base + L.scnt);
  P.tokid = reinterpret_cast<const int32_t *>(base + L.tokid);
  P.x16 = reinterpret_cast<const uint4 *>(base + L.x16);
  P.hrow = reinterpret_cast<uint16_t *>(base + L.hrow);
  P.hmax = reinterpret_cast<int32_t *>(base + L.hmax);
  P.Y = Y;
  P.counter = reinterpret_cast<int32_t *>(base + L.counter);
  P.done = reinterpret_cast<int32_t *>(base + L.done);
  P.status = status;
  P.stage_bytes = stream_stage_bytes(s);
  P.x_in_smem = stream_x_in_smem(s) ? 1 : 0;
  P.ntcap = stream_ntcap(s);
  const size_t budget = 224 * 1024;
  const size_t fixed = stream_fixed_smem(s, 0);
  int stages = static_cast<int>((budget - fixed) / (P.stage_bytes + sizeof(StageDesc) + 16));
  if (stages > 66) stages = 66;
  // a multiple of the consumer-warp count: every ring slot is then owned by one
  // consumer warp, which consumes the slot's fills in order
  const int W = stream_warps(s);
  stages -= stages % W;
  if (stages < W) return -1;
  P.stages = stages;
  const size_t smem = static_cast<size_t>(stages) * P.stage_bytes + stream_fixed_smem(s, stages);
  const int spt = 2 * W;  // stages per task
  const int rb_gu = (s.I + spt - 1) / spt;
  const int rb_dn = (s.H + spt * kDownRowsPerStage - 1) / (spt * kDownRowsPerStage);
  if (launch_pdl(stream_prep_kernel, dim3(2 + s.T), dim3(256), 0, st, x, s.T, s.H, s.E, s.k, P.A, offsets, perm,
                 reinterpret_cast<int32_t *>(base + L.active), reinterpret_cast<int32_t *>(base + L.nactive),
                 reinterpret_cast<int32_t *>(base + L.xexp), reinterpret_cast<uint4 *>(base + L.x16),
                 reinterpret_cast<int32_t *>(base + L.pref), reinterpret_cast<int32_t *>(base + L.sp0),
                 reinterpret_cast<int32_t *>(base + L.scnt), reinterpret_cast<int32_t *>(base + L.tokid),
                 reinterpret_cast<int32_t *>(base + L.hmax), P.counter, P.done, rb_gu, rb_dn,
                 status) != cudaSuccess)
    return -1;
  void (*kern)(Params) = P.ntcap == 1 ? ffn_stream_kernel<11, 1> : ffn_stream_kernel<11, kNT>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess)
    return -1;
  int dev = 0, nsm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  if (launch_pdl(kern, dim3(nsm), dim3((W + 1) * 32), smem, st, P) != cudaSuccess) return -1;
  return 0;
}

}  // namespace k3moe
